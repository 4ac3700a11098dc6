"""Context split of one sequence's cache over G shards, one per rank (or G logical shards on one GPU).

Shard g holds the cache entries [lo_g, hi_g) of every sequence of the batch (`shard_bounds`).  A
decode step of a Full layer and the Reuse layers after it then runs as:

  local_pairs     (every shard)  score its own entries, keep its local Top-k as (score, position)
  exchange 1                     all shards' pairs, stacked in shard order      [G, rows, k]
  merge           (every shard)  the exact global Top-k of the G x k pairs        [rows, k]
  local_attention (every shard)  attend the selected rows it holds (the shard holding the newest
                                 entries also the window rows): bf16 out and lse per layer
  exchange 2                     all shards' out and lse, stacked in shard order
  combine         (every shard)  attention over the union of the rows

Every phase is a call of the C library (`csa2_index_score`, `csa2_shard_topk_pairs`,
`csa2_merge_topk_pairs`, `csa2_shard_indices`, `csa2_sparse_attn_decode`, `csa2_attn_merge_shards`);
this module only orders them and moves their buffers.  The exchanges are `gather` callables that
return a tensor's copies from all shards stacked along a new leading axis in shard order:
`dist_gather` does that with torch.distributed.all_gather (NCCL between GPUs, gloo on CPU); a
single-process run of logical shards stacks the shards' tensors itself.

The result is the unsplit step's: the same indices, and attention within the extra rounding of each
shard's bf16 output.
"""
from __future__ import annotations

from . import (csa2_attn_merge_shards, csa2_index_score, csa2_merge_topk_pairs, csa2_shard_indices,
               csa2_shard_topk_pairs, csa2_sparse_attn_decode)


def shard_bounds(cap, G):
    """[lo_g, hi_g) of G shards splitting `cap` cache entries into contiguous, nearly equal ranges."""
    return [(g * cap // G, (g + 1) * cap // G) for g in range(G)]


def dist_gather(group=None):
    """An exchange over torch.distributed: every rank passes its tensor and gets all ranks' tensors
    stacked along a new leading axis in rank order (ranks hold the shards in order)."""
    import torch
    import torch.distributed as dist

    def gather(t):
        parts = [torch.empty_like(t) for _ in range(dist.get_world_size(group))]
        dist.all_gather(parts, t.contiguous(), group=group)
        return torch.stack(parts)
    return gather


class Shard:
    """One shard's slice of the cache: entries [lo, hi) of every sequence.  codes [B, hi-lo, 256],
    scales [B, hi-lo, 32], KI [B, hi-lo, 128] on this shard's device; lens int32 [B]: the entries
    present in the whole sequence (global)."""

    def __init__(self, lo, hi, codes, scales, KI, lens, owns_window):
        import torch
        self.lo, self.hi = int(lo), int(hi)
        self.codes, self.scales, self.KI = codes, scales, KI
        self.owns_window = bool(owns_window)
        self.lens = lens
        self.lens_local = torch.clamp(lens - self.lo, 0, self.hi - self.lo).to(torch.int32).contiguous()

    @property
    def n(self):
        return self.hi - self.lo


def local_pairs(shard, qI, w, k, q_pos, ratio=1):
    """Score the shard's entries with the queries' indexer Q (qI [B, Nq, 4, 128] bf16, w [B, Nq, 4]
    fp32; query positions q_pos int32 [B*Nq], global) and keep the local Top-k as pairs.
    Returns (pair_score fp32 [rows, k], pair_pos int32 [rows, k], pair_n int32 [rows])."""
    import torch
    B, Nq = qI.shape[0], qI.shape[1]
    rows, dev = B * Nq, qI.device
    n = max(shard.n, 1)
    scores = torch.empty((rows, n), dtype=torch.float32, device=dev)
    n_valid = torch.empty(rows, dtype=torch.int32, device=dev)
    # the shard's entry j is global entry lo + j: visible to position p iff ratio*(lo+j) + ratio-1 <= p
    q_local = (q_pos - ratio * shard.lo).to(torch.int32).contiguous()
    csa2_index_score(qI, w, shard.KI, shard.lens_local, scores, ratio=ratio, q_pos=q_local, n_valid=n_valid)
    pair_score = torch.empty((rows, k), dtype=torch.float32, device=dev)
    pair_pos = torch.empty((rows, k), dtype=torch.int32, device=dev)
    pair_n = torch.empty(rows, dtype=torch.int32, device=dev)
    csa2_shard_topk_pairs(scores, k, pair_score, pair_pos, n_valid=n_valid, n=shard.n, pos_offset=shard.lo,
                          pair_n=pair_n)
    return pair_score, pair_pos, pair_n


def merge(pair_score, pair_pos, pair_n):
    """The exact global Top-k from all shards' pairs ([G, rows, k], [G, rows, k], [G, rows])."""
    import torch
    G, rows, k = pair_score.shape
    idx = torch.empty((rows, k), dtype=torch.int32, device=pair_score.device)
    csa2_merge_topk_pairs(pair_score, pair_pos, idx, pair_n=pair_n)
    return idx


def local_attention(shard, idx, q, swa, swa_len, W, softmax_scale=None):
    """Attention of the queries (q [B, Nq, 16, 512] bf16) over the selected rows this shard holds and,
    if it holds the newest entries, the window rows (swa [B, W-1+Nq, 512], swa_len int32 [B]).
    Returns (out bf16 [B, Nq, 16, 512], lse fp32 [B, Nq, 16])."""
    import torch
    idx_local = torch.empty_like(idx)
    csa2_shard_indices(idx, shard.lo, shard.hi, idx_local)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    own = shard.owns_window and swa is not None
    csa2_sparse_attn_decode(q, shard.codes, shard.scales, idx_local, out, swa=swa if own else None,
                            swa_len=swa_len if own else None, W=W if own else 0, softmax_scale=softmax_scale, lse=lse)
    return out, lse


def combine(out_g, lse_g):
    """All shards' (out, lse) stacked [G, ...] -> attention over the union of their rows."""
    import torch
    out = torch.empty(out_g.shape[1:], dtype=torch.bfloat16, device=out_g.device)
    lse = torch.empty(lse_g.shape[1:], dtype=torch.float32, device=lse_g.device)
    csa2_attn_merge_shards(out_g, lse_g, out, lse)
    return out, lse


def split_group_step(shard, gather, *, q, qI, w, swa, swa_len, k=512, W=128, q_pos=None, ratio=1,
                     softmax_scale=None):
    """One decode step of a Full layer followed by Reuse layers on this rank's shard: q and swa are
    per-layer lists, qI / w the Full layer's indexer Q.  `gather` is the exchange (dist_gather() under
    torch.distributed).  Returns (idx int32 [rows, k] global, [out per layer], [lse per layer]), the
    same on every rank."""
    import torch
    B, Nq = qI.shape[0], qI.shape[1]
    if q_pos is None:   # query i of sequence b at ratio * T_b - Nq + i
        q_pos = (ratio * shard.lens.view(B, 1) - Nq + torch.arange(Nq, device=qI.device).view(1, Nq)).reshape(-1)
    ps, pp, pn = local_pairs(shard, qI, w, k, q_pos.to(torch.int32), ratio)
    idx = merge(gather(ps), gather(pp), gather(pn))
    outs, lses = [], []
    for l in range(len(q)):
        o, s = local_attention(shard, idx, q[l], swa[l] if swa is not None else None, swa_len, W, softmax_scale)
        o, s = combine(gather(o), gather(s))
        outs.append(o)
        lses.append(s)
    return idx, outs, lses

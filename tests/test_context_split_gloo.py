"""The context split's exchange on CPU: two and three gloo ranks (127.0.0.1), each holding one
contiguous shard of a sequence's cache, exchange their local Top-k pairs and their attention partials
with context_split.dist_gather, in rank order.  The oracle stands in for the library on each rank (no
GPU here): the union of the local Top-k pairs, selected by the oracle's Top-k with the positions as
its map, must equal the unsplit Top-k, and the log-sum-exp combination of the shards' attention must
equal the unsplit attention over the union of the rows."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

T, K, W, SEED = 3000, 128, 32, 81


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    import csa2_synth as syn
    import oracle
    kv = syn.normal_bf16(SEED, syn.T_KV, 0, (T, 512))
    codes, scales = oracle.fp4_quantize(kv)
    KI = syn.normal_bf16(SEED, syn.T_KI, 0, (T, 128))
    qI = syn.normal_bf16(SEED, syn.T_QI, 0, (4, 128))
    w = syn.normal_f32(SEED, syn.T_W, 0, (4,))
    q = syn.normal_bf16(SEED, syn.T_Q, 0, (16, 512))
    swa = syn.normal_bf16(SEED, syn.T_SWA, 0, (W, 512))
    return codes, scales, KI, qI, w, q, swa


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from compressed_sparse_attention_step_gb300 import context_split as cs
    oracle.build()
    codes, scales, KI, qI, w, q, swa = _inputs()
    lo, hi = cs.shard_bounds(T, world)[rank]
    gather = cs.dist_gather()
    # exchange 1: the shard's local Top-k as (score, global position) pairs, padded to k
    s_loc = oracle.index_score(qI, w, KI[lo:hi])
    sel, n = oracle.topk(s_loc, K)
    ps = np.full(K, -np.inf, np.float32)
    pp = np.full(K, -1, np.int32)
    ps[:n], pp[:n] = s_loc[sel[:n]], sel[:n] + lo
    ps_all = gather(torch.from_numpy(ps)).numpy()
    pp_all = gather(torch.from_numpy(pp)).numpy()
    pn_all = gather(torch.tensor([n], dtype=torch.int32)).numpy()[:, 0]
    keep = [np.arange(pn_all[g]) for g in range(world)]
    union_s = np.concatenate([ps_all[g][keep[g]] for g in range(world)])
    union_p = np.concatenate([pp_all[g][keep[g]] for g in range(world)])
    idx, _ = oracle.topk(union_s, K, union_p)
    # exchange 2: attention over the selected rows this shard holds (+ the window on the last shard)
    mine = idx[(idx >= lo) & (idx < hi)]
    rows = swa if rank == world - 1 else np.zeros((0, 512), np.uint16)
    o, l = oracle.sparse_attn(q, codes, scales, mine, rows, float(np.float32(512 ** -0.5)))
    o_all = gather(torch.from_numpy(o)).numpy()
    l_all = gather(torch.from_numpy(l)).numpy()
    out[rank] = (idx, o_all, l_all, lo, hi)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_context_split_exchange_matches_unsplit(world):
    import oracle
    oracle.build()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert sorted(res) == list(range(world))
    codes, scales, KI, qI, w, q, swa = _inputs()
    ref_idx, _ = oracle.topk(oracle.index_score(qI, w, KI), K)
    ref_o, ref_l = oracle.sparse_attn(q, codes, scales, ref_idx, swa, float(np.float32(512 ** -0.5)))
    bounds = [res[r][3:] for r in range(world)]
    assert bounds[0][0] == 0 and bounds[-1][1] == T and all(bounds[g][1] == bounds[g + 1][0] for g in range(world - 1))
    for r in range(world):
        idx, o_all, l_all = res[r][:3]
        assert np.array_equal(idx, ref_idx), f"rank {r}: merged indices differ from the unsplit Top-k"
        assert np.array_equal(o_all, res[0][1]) and np.array_equal(l_all, res[0][2])   # same exchange everywhere
        # log-sum-exp combination of the shards' attention = attention over the union
        L = np.logaddexp.reduce(l_all, axis=0)
        comb = sum(np.exp(l_all[g] - L)[:, None] * np.where(np.isfinite(l_all[g])[:, None], o_all[g], 0.0)
                   for g in range(world))
        assert np.allclose(L, ref_l, rtol=0, atol=1e-9)
        assert np.allclose(comb, ref_o, rtol=0, atol=1e-9)
    # the selection spans more than one shard, so the exchange matters
    assert len({int(np.searchsorted([b[1] for b in bounds], p, side="right")) for p in ref_idx}) > 1

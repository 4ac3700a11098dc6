"""GPU parity of the context split (one sequence's cache over G shards), run as G logical shards on
one GPU: every shard scores its slice and keeps its local Top-k pairs (csa2_shard_topk_pairs), the
stacked pairs are merged (csa2_merge_topk_pairs), each shard attends the rows it holds
(csa2_shard_indices + csa2_sparse_attn_decode, the window on the newest shard) and the partials are
combined (csa2_attn_merge_shards).  The indices must equal the oracle's unsplit step bit for bit and
the outputs lie within the attention tolerance, for ragged batches, shards with no visible entries,
contexts shorter than k, ties across a shard boundary, and one 2^20-entry sequence over four shards."""
import numpy as np
import pytest

import csa2_synth as syn
from tests._cases import HOST_THREADS, SCALE, assert_attn_close, bf16_dev, bf16_host, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)
import compressed_sparse_attention_step_gb300 as c  # noqa: E402
from compressed_sparse_attention_step_gb300 import context_split as cs  # noqa: E402

W = 128


def _case(seed, T, L, cap, zero_keys=()):
    B = len(T)
    kv = [syn.normal_bf16(seed, syn.T_KV, b, (cap, 512)) for b in range(B)]
    KI = np.stack([syn.normal_bf16(seed, syn.T_KI, b, (cap, 128)) for b in range(B)])
    for b in zero_keys:
        KI[b] = 0
    q = np.stack([np.stack([syn.normal_bf16(seed, syn.T_Q + l, b, (1, 16, 512)) for b in range(B)]) for l in range(L)])
    qI = np.stack([syn.normal_bf16(seed, syn.T_QI, b, (1, 4, 128)) for b in range(B)])
    w = np.stack([syn.normal_f32(seed, syn.T_W, b, (1, 4)) for b in range(B)])
    swa = np.stack([np.stack([syn.normal_bf16(seed, syn.T_SWA + l, b, (W, 512)) for b in range(B)]) for l in range(L)])
    swa_len = np.minimum(np.array(T), W).astype(np.int32)
    return kv, KI, q, qI, w, swa, swa_len


def _run_split(G, T, cap, kv, KI, q, qI, w, swa, swa_len, K):
    B, L = len(T), q.shape[0]
    codes = torch.empty((B, cap, 256), dtype=torch.uint8, device="cuda")
    scales = torch.empty((B, cap, 32), dtype=torch.uint8, device="cuda")
    for b in range(B):
        c.csa2_fp4_quantize_append(bf16_dev(kv[b])[None], codes[b:b + 1], scales[b:b + 1])
    KI_d = bf16_dev(KI)
    lens = to_dev(np.array(T, np.int32))
    shards = [cs.Shard(lo, hi, codes[:, lo:hi].contiguous(), scales[:, lo:hi].contiguous(),
                       KI_d[:, lo:hi].contiguous(), lens, owns_window=(g == G - 1))
              for g, (lo, hi) in enumerate(cs.shard_bounds(cap, G))]
    qI_d, w_d = bf16_dev(qI), to_dev(w)
    q_pos = (lens - 1).to(torch.int32)
    pairs = [cs.local_pairs(sh, qI_d, w_d, K, q_pos) for sh in shards]
    idx = cs.merge(*(torch.stack([p[i] for p in pairs]) for i in range(3)))
    swa_len_d = to_dev(swa_len)
    outs, lses = [], []
    for l in range(L):
        q_l, swa_l = bf16_dev(q[l]), bf16_dev(swa[l])
        parts = [cs.local_attention(sh, idx, q_l, swa_l, swa_len_d, W, SCALE) for sh in shards]
        o, s = cs.combine(torch.stack([p[0] for p in parts]), torch.stack([p[1] for p in parts]))
        outs.append(o)
        lses.append(s)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), [bf16_host(o) for o in outs], [s.cpu().numpy() for s in lses]


def _check(orc, G, T, cap, K, seed, L=3, zero_keys=()):
    kv, KI, q, qI, w, swa, swa_len = _case(seed, T, L, cap, zero_keys)
    idx, outs, lses = _run_split(G, T, cap, kv, KI, q, qI, w, swa, swa_len, K)
    B = len(T)
    codes = np.zeros((B, cap, 256), np.uint8)
    scales = np.zeros((B, cap, 32), np.uint8)
    for b in range(B):
        codes[b], scales[b] = orc.fp4_quantize(kv[b], threads=HOST_THREADS)
    # the Reuse layers' indexer inputs are unused; the oracle takes one per layer
    ref = orc.group_step([0] + [2] * (L - 1), T, codes, scales, KI, q, np.repeat(qI[None], L, 0),
                         np.repeat(w[None], L, 0), swa, swa_len, K=K, W=W, softmax_scale=SCALE, threads=HOST_THREADS)
    assert np.array_equal(idx.reshape(B, 1, K), ref["idx"][0]), "merged indices differ from the unsplit Top-k"
    for l in range(L):
        assert_attn_close(outs[l], ref["out"][l], f"layer {l}")
        fin = np.isfinite(ref["lse"][l])
        assert np.array_equal(np.isfinite(lses[l]), fin)
        assert np.all(np.abs(lses[l][fin] - ref["lse"][l][fin]) <= 1e-2)
    return idx


@pytest.mark.parametrize("G", [1, 2, 3, 5])
def test_context_split_ragged_batch(orc, G):
    """Three sequences of 20000, 7000 and 300 entries in a 20000-entry cache: the later shards hold no
    visible entries of the short sequences, and the shortest has fewer than k entries in all."""
    _check(orc, G, [20000, 7000, 300], 20000, 512, 91)


def test_context_split_ties_across_shards(orc):
    """All-zero keys: every score ties and the Top-512 is positions 0..511, which span two of the five
    shards of a 2000-entry cache (ties go to the lower position across the shard boundary)."""
    idx = _check(orc, 5, [2000, 1500], 2000, 512, 92, L=2, zero_keys=(0,))
    assert np.array_equal(idx[0], np.arange(512))


def test_context_split_one_sequence_1m_over_4_shards(orc):
    """One sequence of 2^20 entries over four shards of 2^18, Full + 3 Reuse, Top-512."""
    _check(orc, 4, [1 << 20], 1 << 20, 512, 93, L=4)

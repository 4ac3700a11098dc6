"""Pins for the oracle's sparse attention, hierarchical pool and layer-group modes.

Attention: with every position selected and no window it must equal dense softmax
attention (scipy's softmax/logsumexp over independently dequantised rows); one row
returns that row; equal logits return the mean; order of the selected rows does not
matter; a token present both as a selected row and a window row counts twice.
Pool: block keys are exact means on integer data; when all blocks fit, the pool is
every complete block and hierarchical selection equals flat selection over them.
Groups: Reuse layers use bit-identical indices; a Reindex layer fed the Full layer's
indexer Q reproduces its indices."""
import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import csa2_synth as syn

SCALE = float(np.float32(1.0 / np.sqrt(512)))


def _deq(codes, scales):
    """Independent dequantisation: E2M1 magnitudes and torch's E4M3 decoder."""
    tab = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])
    nib = np.stack([codes & 15, codes >> 4], -1).reshape(codes.shape[:-1] + (512,))
    sv = torch.tensor(scales.reshape(-1)).view(torch.float8_e4m3fn).float().numpy()
    return tab[nib] * np.repeat(sv.reshape(scales.shape).astype(np.float64), 16, -1)


def _cache(orc, seed, T):
    kv = syn.normal_bf16(seed, syn.T_KV, 0, (T, 512))
    codes, scales = orc.fp4_quantize(kv)
    return codes, scales


def _dense(q, rows):
    qf = syn.bf16_bits_to_f32(q).astype(np.float64)
    logits = SCALE * (qf @ rows.T)
    return softmax(logits, axis=1) @ rows, logsumexp(logits, axis=1)


def test_attention_equals_dense_when_k_covers_context(orc):
    codes, scales = _cache(orc, 1, 300)
    q = syn.normal_bf16(1, syn.T_Q, 0, (16, 512))
    idx = np.arange(512, dtype=np.int32)
    idx[300:] = -1
    out, lse = orc.sparse_attn(q, codes, scales, idx, np.zeros((0, 512), np.uint16), SCALE)
    ref, rlse = _dense(q, _deq(codes, scales))
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, rlse, rtol=1e-12, atol=1e-12)


def test_attention_with_window_equals_dense_over_union(orc):
    codes, scales = _cache(orc, 2, 200)
    q = syn.normal_bf16(2, syn.T_Q, 0, (16, 512))
    swa = syn.normal_bf16(2, syn.T_SWA, 0, (37, 512))
    idx = np.array([5, 17, 199, 0, 64], np.int32)
    out, lse = orc.sparse_attn(q, codes, scales, idx, swa, SCALE)
    rows = np.concatenate([_deq(codes, scales)[idx], syn.bf16_bits_to_f32(swa).astype(np.float64)])
    ref, rlse = _dense(q, rows)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, rlse, rtol=1e-12, atol=1e-12)


def test_attention_closed_forms(orc):
    codes, scales = _cache(orc, 3, 64)
    deq = _deq(codes, scales)
    q = syn.normal_bf16(3, syn.T_Q, 0, (16, 512))
    none = np.zeros((0, 512), np.uint16)
    # a single row: the output is that row for every head
    out, _ = orc.sparse_attn(q, codes, scales, np.array([9], np.int32), none, SCALE)
    assert np.allclose(out, np.broadcast_to(deq[9], (16, 512)), rtol=0, atol=1e-12)
    # q = 0: equal logits, the output is the mean of the rows
    z = np.zeros((16, 512), np.uint16)
    sel = np.array([1, 2, 3, 40, 63], np.int32)
    out, lse = orc.sparse_attn(z, codes, scales, sel, none, SCALE)
    assert np.allclose(out, np.broadcast_to(deq[sel].mean(0), (16, 512)), atol=1e-12)
    assert np.allclose(lse, np.log(5.0))
    # selected-row order does not matter
    perm = sel[::-1].copy()
    a, _ = orc.sparse_attn(q, codes, scales, sel, none, SCALE)
    b, _ = orc.sparse_attn(q, codes, scales, perm, none, SCALE)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-13)
    # no rows at all: zero output, lse = -inf
    out, lse = orc.sparse_attn(q, codes, scales, np.full(4, -1, np.int32), none, SCALE)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_attention_counts_duplicate_rows_twice(orc):
    """A token both selected and present in the window is attended twice (no
    de-duplication): with rows u (selected) and u, v (window) the weights are 2e^a : e^b."""
    codes, scales = _cache(orc, 4, 16)
    deq = _deq(codes, scales)
    u = deq[3]
    swa = np.stack([syn.f32_to_bf16_bits(u.astype(np.float32)),
                    syn.normal_bf16(4, syn.T_SWA, 0, (512,))])
    assert np.array_equal(syn.bf16_bits_to_f32(swa[0]).astype(np.float64), u)   # exact in bf16
    v = syn.bf16_bits_to_f32(swa[1]).astype(np.float64)
    q = syn.normal_bf16(4, syn.T_Q, 0, (16, 512))
    out, _ = orc.sparse_attn(q, codes, scales, np.array([3], np.int32), swa, SCALE)
    qf = syn.bf16_bits_to_f32(q).astype(np.float64)
    a, b = SCALE * (qf @ u), SCALE * (qf @ v)
    m = np.maximum(a, b)
    wu, wv = 2 * np.exp(a - m), np.exp(b - m)
    ref = (wu[:, None] * u + wv[:, None] * v) / (wu + wv)[:, None]
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# Hierarchical pool
# ---------------------------------------------------------------------------
def test_block_keys_exact_on_integer_data(orc):
    KI = syn.integer_bf16(5, syn.T_KI, 0, (8 * 50 + 3, 128), -8, 8)   # partial trailing block
    bk = orc.block_keys(KI)
    assert bk.shape == (50, 128)
    k = syn.bf16_bits_to_f32(KI).astype(np.float64)[:400].reshape(50, 8, 128)
    assert np.array_equal(syn.bf16_bits_to_f32(bk).astype(np.float64), k.mean(1))


def test_block_keys_within_one_bf16_ulp_of_mean(orc):
    KI = syn.normal_bf16(6, syn.T_KI, 0, (8 * 300, 128))
    bk = syn.bf16_bits_to_f32(orc.block_keys(KI)).astype(np.float64)
    mean = syn.bf16_bits_to_f32(KI).astype(np.float64).reshape(300, 8, 128).mean(1)
    ulp = np.ldexp(1.0, np.frexp(np.abs(mean) + 1e-300)[1] - 8)
    assert np.all(np.abs(bk - mean) <= ulp)


def test_constant_block_keys_keep_lowest_blocks(orc):
    bk = np.tile(syn.normal_bf16(7, syn.T_KI, 0, (1, 128)), (5000, 1))
    qI = syn.normal_bf16(7, syn.T_QI, 0, (4, 128))
    w = syn.normal_f32(7, syn.T_W, 0, (4,))
    pool, n = orc.block_pool(qI, w, bk, 5000, 2048)
    assert n == 16384 and np.array_equal(pool, np.arange(16384))


def test_pool_covers_all_complete_blocks_when_they_fit(orc):
    T = 8 * 1500 + 5
    KI = syn.normal_bf16(8, syn.T_KI, 0, (T, 128))
    qI = syn.normal_bf16(8, syn.T_QI, 0, (4, 128))
    w = syn.normal_f32(8, syn.T_W, 0, (4,))
    pool, n = orc.block_pool(qI, w, orc.block_keys(KI), T // 8, 2048)
    assert n == 12000 and np.array_equal(pool[:n], np.arange(12000)) and np.all(pool[n:] == -1)


def test_pool_blocks_are_the_top_blocks(orc):
    nb = 3000
    bk = syn.normal_bf16(9, syn.T_KI, 0, (nb, 128))
    qI = syn.normal_bf16(9, syn.T_QI, 0, (4, 128))
    w = syn.normal_f32(9, syn.T_W, 0, (4,))
    pool, n = orc.block_pool(qI, w, bk, nb, 2048)
    assert n == 2048 * 8
    blocks = pool.reshape(2048, 8)
    assert np.all(blocks == blocks[:, :1] + np.arange(8)) and np.all(blocks[:, 0] % 8 == 0)
    bsel = blocks[:, 0] // 8
    s = orc.index_score(qI, w, bk)
    mask = np.zeros(nb, bool)
    mask[bsel] = True
    assert s[mask].min() >= s[~mask].max()


# ---------------------------------------------------------------------------
# Layer groups
# ---------------------------------------------------------------------------
def _group_inputs(orc, seed, B, T, L, Nq=1, W=128):
    cap = max(T)
    kv = np.stack([syn.normal_bf16(seed, syn.T_KV, b, (cap, 512)) for b in range(B)])
    codes, scales = orc.fp4_quantize(kv)
    KI = np.stack([syn.normal_bf16(seed, syn.T_KI, b, (cap, 128)) for b in range(B)])
    q = np.stack([np.stack([syn.normal_bf16(seed, syn.T_Q + l, b, (Nq, 16, 512)) for b in range(B)])
                  for l in range(L)])
    qI = np.stack([np.stack([syn.normal_bf16(seed, syn.T_QI + l, b, (Nq, 4, 128)) for b in range(B)])
                   for l in range(L)])
    w = np.stack([np.stack([syn.normal_f32(seed, syn.T_W + l, b, (Nq, 4)) for b in range(B)])
                  for l in range(L)])
    swa = np.stack([np.stack([syn.normal_bf16(seed, syn.T_SWA + l, b, (W - 1 + Nq, 512))
                              for b in range(B)]) for l in range(L)])
    swa_len = np.minimum(np.array(T), W - 1 + Nq).astype(np.int32)
    return codes, scales, KI, q, qI, w, swa, swa_len


def test_reuse_layers_share_bit_identical_indices(orc):
    T = [3000, 700]
    codes, scales, KI, q, qI, w, swa, swa_len = _group_inputs(orc, 10, 2, T, 4)
    r = orc.group_step([0, 2, 2, 2], T, codes, scales, KI, q, qI, w, swa, swa_len)
    for l in (1, 2, 3):
        assert np.array_equal(r["idx"][l], r["idx"][0])
    # the Full layer's indices are the flat Top-512 of its own scores
    for b in range(2):
        s = orc.index_score(qI[0, b, 0], w[0, b, 0], KI[b], n=T[b])
        idx, _ = orc.topk(s, 512)
        assert np.array_equal(r["idx"][0, b, 0], idx)
    # each Reuse layer's output is the attention of its own q / window over those rows
    for l in (1, 3):
        for b in range(2):
            rows = swa[l, b][128 - swa_len[b]:]
            out, _ = orc.sparse_attn(q[l, b, 0], codes[b], scales[b], r["idx"][0, b, 0], rows, SCALE)
            assert np.array_equal(out, r["out"][l, b, 0])


def test_reindex_with_full_queries_reproduces_full_indices(orc):
    T = [2500]
    codes, scales, KI, q, qI, w, swa, swa_len = _group_inputs(orc, 11, 1, T, 3)
    qI[1] = qI[0]
    w[1] = w[0]
    r = orc.group_step([0, 1, 1], T, codes, scales, KI, q, qI, w, swa, swa_len)
    assert np.array_equal(r["idx"][1], r["idx"][0])
    assert not np.array_equal(r["idx"][2], r["idx"][0])     # own indexer Q: fresh selection


def test_hierarchical_equals_flat_when_every_block_fits(orc):
    T = [8 * 1200 + 3]          # 1200 complete blocks <= 2048 kept
    codes, scales, KI, q, qI, w, swa, swa_len = _group_inputs(orc, 12, 1, T, 3)
    r = orc.group_step([0, 1, 2], T, codes, scales, KI, q, qI, w, swa, swa_len,
                       hierarchical=True)
    assert r["pool_len"][0, 0] == 9600
    for l in (0, 1):
        s = orc.index_score(qI[l, 0, 0], w[l, 0, 0], KI[0], n=9600)   # complete blocks only
        idx, _ = orc.topk(s, 512)
        assert np.array_equal(r["idx"][l, 0, 0], idx)
    assert np.array_equal(r["idx"][2], r["idx"][1])


def test_hierarchical_reindex_stays_inside_pool(orc):
    T = [8 * 4000]
    codes, scales, KI, q, qI, w, swa, swa_len = _group_inputs(orc, 13, 1, T, 2)
    r = orc.group_step([0, 1], T, codes, scales, KI, q, qI, w, swa, swa_len, hierarchical=True)
    pool = r["pool"][0, 0]
    assert r["pool_len"][0, 0] == 16384
    assert np.all(np.isin(r["idx"][1, 0, 0], pool))
    s = orc.index_score(qI[1, 0, 0], w[1, 0, 0], KI[0], pos=pool)
    idx, _ = orc.topk(s, 512, pool)
    assert np.array_equal(r["idx"][1, 0, 0], idx)


def test_causal_prefill_indices_and_windows(orc):
    """Ratio-2 prefill chunk: entry j is visible to token position p iff 2j+1 <= p; the
    window of query i is its own W rows."""
    Nq, W, T = 6, 8, [40]
    codes, scales, KI, q, qI, w, swa, swa_len = _group_inputs(orc, 14, 1, T, 2, Nq=Nq, W=W)
    q_pos = np.array([[70, 71, 72, 73, 74, 79]], np.int32)
    r = orc.group_step([0, 2], T, codes, scales, KI, q, qI, w, swa, swa_len, Nq=Nq, K=16,
                       W=W, ratio=2, q_pos=q_pos)
    for i in range(Nq):
        nvis = min(40, (q_pos[0, i] + 1) // 2)
        sel = r["idx"][0, 0, i]
        assert np.all(sel[sel >= 0] < nvis)
        s = orc.index_score(qI[0, 0, i], w[0, 0, i], KI[0], n=nvis)
        idx, _ = orc.topk(s, 16)
        assert np.array_equal(sel, idx)
        rows = swa[1, 0][i:i + W]
        out, _ = orc.sparse_attn(q[1, 0, i], codes[0], scales[0], sel, rows, SCALE)
        assert np.array_equal(out, r["out"][1, 0, i])


@pytest.mark.parametrize("hier", [False, True])
def test_group_step_rows_are_independent_of_thread_count(orc, hier):
    """The group step runs its query rows on host threads; a chunk of queries over ragged
    sequences gives identical indices, pools, outputs and lse on 1 and on 5 threads."""
    Nq, W = 6, 16
    T = [8 * 700 + 5, 8 * 300] if hier else [700, 333]
    codes, scales, KI, q, qI, w, swa, swa_len = _group_inputs(orc, 15, 2, T, 3, Nq=Nq, W=W)
    kw = dict(Nq=Nq, K=64, W=W, ratio=1 if hier else 2, hierarchical=hier, keep=256)
    r1 = orc.group_step([0, 1, 2], T, codes, scales, KI, q, qI, w, swa, swa_len, threads=1, **kw)
    r5 = orc.group_step([0, 1, 2], T, codes, scales, KI, q, qI, w, swa, swa_len, threads=5, **kw)
    for key in ("idx", "out", "lse") + (("pool", "pool_len") if hier else ()):
        assert np.array_equal(r1[key], r5[key]), key

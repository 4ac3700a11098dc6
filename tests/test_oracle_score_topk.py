"""Pins for the oracle's indexer score and exact Top-K.

Score: exact integer arithmetic (small-integer data makes every partial sum exact in
fp32, so any correct summation order gives the same bits), one-hot queries, and an
fp64 error bound on N(0, 1) data.  Top-K: the defining properties of the selected
set (size, order, and "every selected key beats every unselected key" under
(score desc, position asc)), checked exhaustively on small rows with heavy ties."""
import numpy as np
import pytest

import csa2_synth as syn


def _int_case(seed, T):
    qI = syn.integer_bf16(seed, 1, 0, (4, 128), -8, 8)
    KI = syn.integer_bf16(seed, 2, 0, (T, 128), -8, 8)
    w = np.array([3.0, -2.0, 0.5, 5.0], np.float32)          # distinct per head, one negative
    return qI, w, KI


def test_score_exact_on_integer_data(orc):
    qI, w, KI = _int_case(3, 777)
    got = orc.index_score(qI, w, KI)
    q = syn.bf16_bits_to_f32(qI).astype(np.int64)
    k = syn.bf16_bits_to_f32(KI).astype(np.int64)
    dots = k @ q.T                                           # [T, 4], exact
    exp = (np.maximum(dots, 0).astype(np.float64) * w.astype(np.float64)[None]).sum(1)
    assert np.array_equal(got.astype(np.float64), exp)


def test_score_one_hot_queries(orc):
    KI = syn.normal_bf16(9, 2, 0, (300, 128))
    kf = syn.bf16_bits_to_f32(KI)
    for h in range(4):
        for c in [0, 15, 16, 77, 127]:
            q = np.zeros((4, 128), np.float32)
            q[h, c] = 1.0
            w = np.zeros(4, np.float32)
            w[h] = 1.0
            got = orc.index_score(syn.f32_to_bf16_bits(q), w, KI)
            assert np.array_equal(got, np.maximum(kf[:, c], 0)), (h, c)


def test_score_positions_and_error_bound(orc):
    qI = syn.normal_bf16(4, 1, 0, (4, 128))
    KI = syn.normal_bf16(4, 2, 0, (2000, 128))
    w = syn.normal_f32(4, 3, 0, (4,))
    pos = np.random.default_rng(0).permutation(2000)[:700].astype(np.int32)
    got = orc.index_score(qI, w, KI, pos=pos)
    q = syn.bf16_bits_to_f32(qI).astype(np.float64)
    k = syn.bf16_bits_to_f32(KI).astype(np.float64)[pos]
    dots = k @ q.T
    exp = (np.maximum(dots, 0) * w.astype(np.float64)[None]).sum(1)
    # 16-term fma chains + a depth-3 tree per head, then 4 products and a depth-2 tree
    mag = (np.abs(k) @ np.abs(q).T * np.abs(w.astype(np.float64))[None]).sum(1)
    assert np.all(np.abs(got - exp) <= 32 * 2.0 ** -24 * mag + 1e-30)


# ---------------------------------------------------------------------------
# Rounding order of the score.  bf16 x bf16 products are exact in fp32 (8-bit significands give a
# 16-bit product), so each fused multiply-add of a chain is exactly one fp32 addition of an exact
# product.  With products of 2^24 and 1 an addition of 1 to 2^24 is a tie that rounds to even
# (back to 2^24), while 2^24 + 2 and 2^24 + 4 are exact: the cases below give different bits for
# every plausible reordering, and their canonical values follow by hand.
# ---------------------------------------------------------------------------
BIG = 2.0 ** 12          # BIG * BIG = 2^24


def _crafted(products, w):
    """qI / KI rows whose per-(head, channel) products are the given values: products[h] maps a
    channel to (q, k) with q * k the product."""
    q = np.zeros((4, 128), np.float32)
    k = np.zeros(128, np.float32)
    for h, chans in products.items():
        for ch, (qv, kv) in chans.items():
            q[h, ch] = qv
            k[ch] = kv
    return syn.f32_to_bf16_bits(q), np.asarray(w, np.float32), syn.f32_to_bf16_bits(k[None])


def test_score_chain_runs_in_increasing_channel_order(orc):
    # head 0, chain 0: 2^24 at channel 0, then 1 at channels 1..15.  In increasing order every +1 is a
    # tie that rounds back to 2^24; summed the other way round the ones reach 15 first and
    # 2^24 + 15 rounds (tie, to even) to 2^24 + 16.
    prods = {0: {0: (BIG, BIG), **{c: (1.0, 1.0) for c in range(1, 16)}}}
    qI, w, k = _crafted(prods, [1.0, 0.0, 0.0, 0.0])
    assert orc.index_score(qI, w, k)[0] == np.float32(2.0 ** 24)


def test_score_chain_partials_combine_as_a_fixed_tree(orc):
    # p0 = 2^24, p1 = p2 = p3 = 1: ((p0 + p1) + (p2 + p3)) = 2^24 + 2, whereas one running sum
    # gives 2^24 and the reversed running sum 2^24 + 4.
    prods = {0: {0: (BIG, BIG), 16: (1.0, 1.0), 32: (1.0, 1.0), 48: (1.0, 1.0)}}
    qI, w, k = _crafted(prods, [1.0, 0.0, 0.0, 0.0])
    assert orc.index_score(qI, w, k)[0] == np.float32(2.0 ** 24 + 2)
    # p0 = 2^24 and p4 = p5 = p6 = 1: (2^24) + ((1 + 1) + (1 + 0)) = 2^24 + 3, a tie that rounds
    # to 2^24 + 4; a running sum keeps 2^24.
    prods = {0: {0: (BIG, BIG), 64: (1.0, 1.0), 80: (1.0, 1.0), 96: (1.0, 1.0)}}
    qI, w, k = _crafted(prods, [1.0, 0.0, 0.0, 0.0])
    assert orc.index_score(qI, w, k)[0] == np.float32(2.0 ** 24 + 4)


def test_score_heads_combine_in_pairs(orc):
    # r0 = 2^24, r1 = r2 = r3 = 1 with unit weights: (w0 r0 + w1 r1) + (w2 r2 + w3 r3) = 2^24 + 2;
    # a running sum over the heads gives 2^24.
    prods = {0: {0: (BIG, BIG)}, 1: {1: (1.0, 1.0)}, 2: {2: (1.0, 1.0)}, 3: {3: (1.0, 1.0)}}
    qI, w, k = _crafted(prods, [1.0, 1.0, 1.0, 1.0])
    assert orc.index_score(qI, w, k)[0] == np.float32(2.0 ** 24 + 2)
    # each weighted product is rounded on its own before the sums: with r0 = r1 = 3, w0 = -1 and
    # w1 = 1 + 2^-23, w1 r1 = 3 + 1.5 * 2^-22 is a tie between 3 + 2^-22 and 3 + 2^-21 (spacing 2^-22
    # above 2) and rounds to the even 3 + 2^-21, so the score is -3 + (3 + 2^-21) = 2^-21 exactly.
    # Fusing w1 r1 into the sum with w0 r0 would give 1.5 * 2^-22 instead.
    prods = {0: {0: (3.0, 1.0)}, 1: {1: (3.0, 1.0)}}
    w1 = np.float32(1.0 + 2.0 ** -23)
    qI, w, k = _crafted(prods, [-1.0, w1, 0.0, 0.0])
    assert orc.index_score(qI, w, k)[0] == np.float32(2.0 ** -21)


def test_score_relu_and_signed_zero(orc):
    # a negative head dot contributes w * (+0); all heads negative with negative weights give -0,
    # which is an exact zero (Top-K treats -0 and +0 alike)
    prods = {h: {h: (-1.0, 2.0)} for h in range(4)}
    qI, w, k = _crafted(prods, [-1.0, -2.0, -3.0, -4.0])
    s = orc.index_score(qI, w, k)[0]
    assert s == 0.0
    # one positive head: only it counts
    prods = {0: {0: (3.0, 2.0)}, 1: {1: (-1.0, 2.0)}, 2: {2: (-5.0, 1.0)}, 3: {3: (-1.0, 1.0)}}
    qI, w, k = _crafted(prods, [0.5, 100.0, 100.0, 100.0])
    assert orc.index_score(qI, w, k)[0] == np.float32(3.0)


def _numpy_score(qI, w, KI):
    """The canonical score restated with numpy fp32 array arithmetic: every product of two bf16
    values is exact in fp32, so adding it to the chain's running sum is the fused multiply-add."""
    q = syn.bf16_bits_to_f32(qI)
    k = syn.bf16_bits_to_f32(KI)
    w = np.asarray(w, np.float32)
    r = []
    for h in range(4):
        p = []
        for j in range(8):
            acc = np.zeros(k.shape[0], np.float32)
            for ch in range(16 * j, 16 * j + 16):
                acc = acc + q[h, ch] * k[:, ch]
            p.append(acc)
        dot = ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]))
        r.append(np.where(dot > 0, dot, np.float32(0.0)))
    m = [w[h] * r[h] for h in range(4)]
    return (m[0] + m[1]) + (m[2] + m[3])


def test_score_matches_numpy_restatement_bitwise(orc):
    for seed in (11, 12):
        qI = syn.normal_bf16(seed, 1, 0, (4, 128))
        KI = syn.normal_bf16(seed, 2, 0, (3000, 128))
        w = syn.normal_f32(seed, 3, 0, (4,))
        exp = _numpy_score(qI, w, KI)
        assert exp.dtype == np.float32
        got = orc.index_score(qI, w, KI)
        assert np.array_equal(got.view(np.uint32), exp.view(np.uint32)), seed


def test_index_select_is_rowwise_score_then_topk(orc):
    """The batched flat selection equals index_score + topk per row (ragged, causal ratio 2, explicit
    positions, fewer visible entries than k) and does not depend on the thread count."""
    B, Nq, cap, k = 3, 5, 900, 64
    T = np.array([900, 401, 30], np.int64)
    KI = np.stack([syn.normal_bf16(21, syn.T_KI, b, (cap, 128)) for b in range(B)])
    qI = np.stack([syn.normal_bf16(21, syn.T_QI, b, (Nq, 4, 128)) for b in range(B)])
    w = np.stack([syn.normal_f32(21, syn.T_W, b, (Nq, 4)) for b in range(B)])
    q_pos = np.array([[0, 1, 500, 1700, 1799], [3, 100, 700, 801, 900], [1, 9, 59, 61, 3000]], np.int32)
    for qp in (None, q_pos):
        idx1, n1 = orc.index_select(KI, qI, w, T, k, ratio=2, q_pos=qp, threads=1)
        idx4, n4 = orc.index_select(KI, qI, w, T, k, ratio=2, q_pos=qp, threads=4)
        assert np.array_equal(idx1, idx4) and np.array_equal(n1, n4)
        for b in range(B):
            for i in range(Nq):
                p = int(qp[b, i]) if qp is not None else 2 * int(T[b]) - Nq + i
                nv = max(0, min(int(T[b]), (p + 1) // 2))
                s = orc.index_score(qI[b, i], w[b, i], KI[b], n=nv) if nv else np.zeros(0, np.float32)
                e, cnt = orc.topk(s, k) if nv else (np.full(k, -1, np.int32), 0)
                assert np.array_equal(idx1[b, i], e) and n1[b, i] == cnt


# ---------------------------------------------------------------------------
# Top-K
# ---------------------------------------------------------------------------
def _check_topk(scores, k, idx, cnt, n_valid=None):
    n = scores.size if n_valid is None else n_valid
    s = scores[:n].astype(np.float64)
    m = min(k, n)
    assert cnt == m
    assert np.all(idx[m:] == -1)
    sel = idx[:m]
    assert np.all(np.diff(sel) > 0), "ascending, unique"
    assert np.all((sel >= 0) & (sel < n))
    mask = np.zeros(n, bool)
    mask[sel] = True
    if m == n or m == 0:
        return
    # every selected (score, -pos) beats every unselected one
    smin = s[mask].min()
    smax_un = s[~mask].max()
    assert smin >= smax_un
    if smin == smax_un:
        tied_sel = np.nonzero(mask & (s == smin))[0]
        tied_un = np.nonzero(~mask & (s == smin))[0]
        assert tied_sel.max() < tied_un.min()


@pytest.mark.parametrize("n,k", [(1, 512), (5, 3), (511, 512), (512, 512), (513, 512),
                                 (1000, 7), (4096, 512), (4096, 2048), (3000, 1)])
def test_topk_properties_random_with_ties(orc, n, k):
    g = np.random.default_rng(n * 7 + k)
    for trial in range(3):
        if trial == 0:
            s = g.standard_normal(n).astype(np.float32)
        elif trial == 1:
            s = np.round(g.standard_normal(n) * 2).astype(np.float32)      # many ties
        else:
            s = g.choice(np.array([0.0, -0.0, 1.0, -1.0], np.float32), n)  # +-0 mixed
        idx, cnt = orc.topk(s, k)
        _check_topk(s, k, idx, cnt)


def test_topk_all_equal_takes_lowest_positions(orc):
    s = np.full(4096, 0.25, np.float32)
    idx, cnt = orc.topk(s, 512)
    assert cnt == 512 and np.array_equal(idx, np.arange(512))
    s = np.where(np.arange(4096) % 2 == 0, 0.0, -0.0).astype(np.float32)
    idx, _ = orc.topk(s, 512)
    assert np.array_equal(idx, np.arange(512))


def test_topk_extremes_and_map(orc):
    s = np.array([-np.inf, 3.0, np.inf, -1e38, 1e38, 0.0], np.float32)
    idx, cnt = orc.topk(s, 3)
    assert cnt == 3 and list(idx) == [1, 2, 4]
    # a map turns column indices into positions (ascending maps keep the order)
    g = np.random.default_rng(1)
    s = g.standard_normal(900).astype(np.float32)
    mp = np.sort(g.choice(100000, 900, replace=False)).astype(np.int32)
    idx, _ = orc.topk(s, 100, mp)
    base, _ = orc.topk(s, 100)
    assert np.array_equal(idx, mp[base])


def test_topk_brute_force_tiny_exhaustive(orc):
    """All score rows over a 3-value alphabet of length 6, every k: the result equals the
    first k of a full lexicographic sort (numpy lexsort on (-score, position))."""
    vals = np.array([-1.0, 0.0, 2.0], np.float32)
    for code in range(3 ** 6):
        digits = [(code // 3 ** i) % 3 for i in range(6)]
        s = vals[digits]
        order = np.lexsort((np.arange(6), -s.astype(np.float64)))
        for k in range(1, 8):
            idx, cnt = orc.topk(s, k)
            exp = np.sort(order[:min(k, 6)])
            assert np.array_equal(idx[:cnt], exp)

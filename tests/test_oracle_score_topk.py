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

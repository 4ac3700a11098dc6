"""Host model of the prefill selection's split rows (no GPU).  The rows with the most marked keys are
rescored by several CTAs: CTA s takes the marked keys of ranks [s total / S, (s + 1) total / S) in
column order, streams them through a list of at most 4096 candidates that is cut back to its k
best (score key descending, column ascending; kept in column order) whenever more keys remain, and
keeps its k best at the end; the last CTA concatenates the S lists in slice order, cutting the
list back whenever the next slice would overflow it, and selects the k best.  The model checks,
against the oracle's exact Top-k of the whole row, that this returns the same columns for rows with
heavy ties, signed zeros, one repeated value and integer scores, marked sets from just above k to
several list lengths, and k from 64 to 2048 (where eight slices' lists overflow the merge list)."""
import numpy as np
import pytest

CAP = 4096


def keys_of(s):
    u = s.astype(np.float32).view(np.uint32).copy()
    u[u == 0x80000000] = 0
    return np.where(u & 0x80000000, ~u, u | 0x80000000).astype(np.uint32)


def keep_top(key, col, k):
    """The k best of a column-ordered list by (key desc, column asc), still in column order."""
    order = np.lexsort((col, -key.astype(np.int64)))[:k]
    keep = np.sort(order)
    return key[keep], col[keep]


def slice_list(key, col, k):
    """One CTA's pass over its column-ordered marked keys: chunks into a list of at most CAP,
    cut back to the k best while keys remain, and to the k best at the end."""
    lk, lc = key[:0], col[:0]
    lo = 0
    while lo < key.size:
        hi = min(key.size, lo + CAP - lk.size)
        lk, lc = np.concatenate([lk, key[lo:hi]]), np.concatenate([lc, col[lo:hi]])
        lo = hi
        if lo < key.size:
            lk, lc = keep_top(lk, lc, k)
    if lk.size > k:
        lk, lc = keep_top(lk, lc, k)
    return lk, lc


def split_select(s, marked, k, n_slices):
    key, col = keys_of(s)[marked], marked.astype(np.int64)
    total = key.size
    lists = []
    for sl in range(n_slices):
        a, b = total * sl // n_slices, total * (sl + 1) // n_slices
        lists.append(slice_list(key[a:b], col[a:b], k))
    lk, lc = key[:0], col[:0]
    for sk, sc in lists:
        if lk.size + sk.size > CAP:
            assert lk.size >= k
            lk, lc = keep_top(lk, lc, k)
        lk, lc = np.concatenate([lk, sk]), np.concatenate([lc, sc])
    if lk.size > k:
        lk, lc = keep_top(lk, lc, k)
    return lc


def rows(n, g):
    return {
        "normal": g.standard_normal(n).astype(np.float32),
        "ties": np.round(g.standard_normal(n) * 3).astype(np.float32),
        "one_key": np.full(n, 0.5, np.float32),
        "signed_zero": g.choice(np.array([0.0, -0.0, 2.0, -2.0], np.float32), n),
        "relu_zeros": np.minimum(g.standard_normal(n), 0).astype(np.float32),
        "integers": g.integers(-20, 20, n).astype(np.float32),
    }


@pytest.mark.parametrize("k", [64, 512, 2048])
@pytest.mark.parametrize("n_slices", [1, 3, 8])
def test_split_rows_select_the_exact_topk(orc, k, n_slices):
    g = np.random.default_rng(k + 7 * n_slices)
    n = 24000
    for name, s in rows(n, g).items():
        exp, cnt = orc.topk(s, k)
        assert cnt == k
        kth = np.sort(keys_of(s))[::-1][k - 1]
        keys = keys_of(s)
        # marked sets: every key at or above the k-th key (ties included), a few thousand more, and
        # every key; each contains the exact Top-k
        for extra in (0, 3000, n):
            if extra == n:
                marked = np.arange(n)
            else:
                above = np.nonzero(keys >= kth)[0]
                rest = np.setdiff1d(np.arange(n), above)
                marked = np.sort(np.concatenate([above, g.choice(rest, min(extra, rest.size), replace=False)]))
            got = split_select(s, marked, k, n_slices)
            assert np.array_equal(got, np.sort(exp)), (name, extra)


def test_merge_cuts_when_the_slices_overflow_the_list(orc):
    """k = 2048 and eight full slices: the merge list overflows and is cut back twice or more."""
    g = np.random.default_rng(11)
    s = g.standard_normal(40000).astype(np.float32)
    marked = np.arange(s.size)
    got = split_select(s, marked, 2048, 8)
    exp, _ = orc.topk(s, 2048)
    assert np.array_equal(got, np.sort(exp))

"""Host model of the long-row Top-K's bound (no GPU): rows longer than 8192 columns are cut into
slices of whole 4096-key sweep steps; in each sweep step, thread t of a 256-thread CTA takes the 16
keys s[b0 + 4 (u 256 + t) + e] (u, e < 4) as one group.  The bin (top 12 key bits) of the k-th
largest group maximum gives the bound, and only groups whose maximum reaches it are read.  The
model checks, against the oracle's exact Top-k, that the keys so listed are exactly the keys at or
above the bound and include the Top-k, on rows with heavy ties, signed zeros, one repeated value,
negative scores and valid prefixes that end inside a group."""
import numpy as np
import pytest

NT, SWEEP, BINS = 256, 4096, 4096


def keys_of(s):
    u = s.astype(np.float32).view(np.uint32).copy()
    u[u == 0x80000000] = 0
    return np.where(u & 0x80000000, ~u, u | 0x80000000).astype(np.uint32)


def group_ids(nv):
    """Group index of every column below nv: (sweep, thread)."""
    col = np.arange(nv)
    sweep, r = np.divmod(col, SWEEP)
    t = (r // 4) % NT
    return sweep * NT + t


def listed_keys(s, nv, k):
    key = keys_of(s[:nv])
    gid = group_ids(nv)
    ng = gid.max() + 1
    gmax = np.zeros(ng, np.uint32)
    np.maximum.at(gmax, gid, key)
    present = np.zeros(ng, bool)
    present[gid] = True
    gmax = gmax[present]
    bound = 0
    if gmax.size >= k:
        hist = np.bincount(gmax >> 20, minlength=BINS)
        cum = np.cumsum(hist[::-1])
        b1 = BINS - 1 - int(np.searchsorted(cum, k))
        bound = b1 << 20
    full_max = np.zeros(ng, np.uint32)
    np.maximum.at(full_max, gid, key)
    reach = full_max >= bound                      # groups the filter reads
    listed = np.nonzero(reach[gid] & (key >= bound))[0]
    return listed, np.nonzero(key >= bound)[0], bound


def rows(n, g):
    return {
        "normal": g.standard_normal(n).astype(np.float32),
        "ties": np.round(g.standard_normal(n) * 3).astype(np.float32),
        "one_key": np.full(n, 0.5, np.float32),
        "signed_zero": g.choice(np.array([0.0, -0.0, 2.0, -2.0], np.float32), n),
        "relu_zeros": np.minimum(g.standard_normal(n), 0).astype(np.float32),
        "narrow": (g.standard_normal(n) * 1e-4 + 3.0).astype(np.float32),
    }


@pytest.mark.parametrize("n,k", [(8193, 512), (20000, 64), (40000, 2048), (131072, 512)])
def test_listed_keys_cover_the_topk(orc, n, k):
    g = np.random.default_rng(n + k)
    for name, s in rows(n, g).items():
        for nv in (n, n - 5, 16 * k + 3, 9000):
            if nv <= k or nv > n:
                continue
            listed, at_or_above, bound = listed_keys(s, nv, k)
            assert np.array_equal(listed, at_or_above), (name, nv)
            exp, cnt = orc.topk(s[:nv], k)
            assert cnt == k
            assert np.isin(exp, listed).all(), (name, nv)
            assert listed.size >= k


def test_bound_is_a_bin_floor_below_the_kth_key(orc):
    g = np.random.default_rng(7)
    s = g.standard_normal(65536).astype(np.float32)
    listed, _, bound = listed_keys(s, s.size, 512)
    kth = np.sort(keys_of(s))[::-1][511]
    assert bound & 0xFFFFF == 0 and bound <= kth

"""Host model of the prefill threshold's bound (no GPU).  Per query row the threshold kernel keeps
the row's group maxima as ordered 32-bit score keys and runs two radix rounds of 11 bits (key bits
31..21, then 20..10), each picking the bin that holds the k-th largest key among the keys that
match the bits fixed so far.  The bound L is the key so found with its low 10 bits zero.  The
model checks that L never exceeds the exact k-th largest key (so L - 2 delta stays a valid
threshold), that it agrees with it in the top 22 bits, and that the float it stands for is at most
the k-th largest maximum, on rows of normal, tied, negative, signed-zero and narrow values."""
import numpy as np
import pytest


def keys_of(s):
    u = s.astype(np.float32).view(np.uint32).copy()
    u[u == 0x80000000] = 0
    return np.where(u & 0x80000000, ~u, u | 0x80000000).astype(np.uint32)


def key_score(key):
    key = np.uint32(key)
    bits = (key & np.uint32(0x7FFFFFFF)) if key & np.uint32(0x80000000) else ~key
    return np.array([bits], np.uint32).view(np.float32)[0]


def two_round_bound(keys, k):
    prefix, mask, need = 0, 0, k
    for shift in (21, 10):
        sel = keys[(keys & np.uint32(mask)) == np.uint32(prefix)]
        b = (sel >> np.uint32(shift)) & np.uint32(0x7FF)
        hist = np.bincount(b, minlength=2048)
        cum = 0
        for bin_ in range(2047, -1, -1):  # from the top bin down, as the kernel's scan does
            if cum + hist[bin_] >= need:
                break
            cum += hist[bin_]
        prefix |= bin_ << shift
        mask |= 0x7FF << shift
        need -= cum
    return np.uint32(prefix)


def rows(n, g):
    return {
        "normal": g.standard_normal(n).astype(np.float32),
        "ties": np.round(g.standard_normal(n) * 3).astype(np.float32),
        "negative": -np.abs(g.standard_normal(n)).astype(np.float32),
        "signed_zero": g.choice(np.array([0.0, -0.0, 1.5, -1.5], np.float32), n),
        "narrow": (g.standard_normal(n) * 1e-4 + 3.0).astype(np.float32),
        "one_value": np.full(n, 0.25, np.float32),
    }


@pytest.mark.parametrize("k", [1, 64, 512, 2048])
def test_two_round_bound_is_below_the_kth_key(k):
    g = np.random.default_rng(k)
    for name, s in rows(4096, g).items():
        keys = keys_of(s)
        kth = np.sort(keys)[::-1][k - 1]
        bound = two_round_bound(keys, k)
        assert bound <= kth, name
        assert (bound >> 10) == (kth >> 10), name  # the top 22 bits are exact
        assert key_score(bound) <= key_score(kth), name


def test_the_bound_keeps_the_low_bits_zero():
    """A plausible mistake, keeping the k-th key's low bits from an earlier key instead of zeroing
    them, can exceed the k-th key; the zeroed prefix cannot."""
    keys = np.array([0x80000000 | (7 << 10) | 0x3FF] + [0x80000000 | (7 << 10)] * 3, np.uint32)
    kth = np.sort(keys)[::-1][1]
    bound = two_round_bound(keys, 2)
    assert bound <= kth
    assert (bound | np.uint32(0x3FF)) > kth  # filling the low bits would overshoot

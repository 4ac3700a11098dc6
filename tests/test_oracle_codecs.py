"""Pins for the oracle's FP4 (E2M1) / FP8 (E4M3) codecs and the NVFP4-style row
quantiser, against facts fixed outside the oracle: the format tables (golden
files), torch's float8_e4m3fn decoder/encoder, brute-force nearest-value search
and exact rational arithmetic."""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import csa2_synth as syn

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, b = line.split()
            rows.append((int(a, 0), float(b)))
    return rows


def _e2m1_table():
    return {k: v for k, v in _golden("e2m1_values.txt")}


def _torch_e4m3(b):
    """Decode E4M3 bytes with torch's float8_e4m3fn (a library decoder)."""
    t = torch.tensor(np.asarray(b, dtype=np.uint8).reshape(-1)).view(torch.float8_e4m3fn)
    return t.float().numpy().astype(np.float64)


def test_e2m1_decode_matches_format_table(orc):
    for code, val in _e2m1_table().items():
        got = orc.e2m1_value(code)
        assert got == val and np.signbit(got) == np.signbit(val), (code, got, val)


def test_e4m3_decode_landmarks_and_torch(orc):
    for b, v in _golden("e4m3_landmarks.txt"):
        got = orc.e4m3_value(b)
        if np.isnan(v):
            assert np.isnan(got)
        else:
            assert got == v and np.signbit(got) == np.signbit(v), (hex(b), got, v)
    ref = _torch_e4m3(np.arange(256))
    got = np.array([orc.e4m3_value(b) for b in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def _e2m1_brute(v):
    """Nearest E2M1 magnitude by exhaustive search; ties to the even code; saturate at 6."""
    tab = _e2m1_table()
    a = abs(v)
    if a > 6.0:                                   # satfinite
        return 7 | (8 if np.signbit(v) else 0)
    best, bestd = None, None
    for k in range(8):
        d = abs(a - tab[k])
        if best is None or d < bestd or (d == bestd and k % 2 == 0):
            best, bestd = k, d
    return best | (8 if np.signbit(v) else 0)


def test_e2m1_encode_brute_force(orc):
    grid = np.concatenate([
        np.arange(-8.0, 8.0 + 1e-9, 1.0 / 64),                 # includes every midpoint
        np.random.default_rng(5).normal(0, 3, 3000),
        [1e-30, -1e-30, 0.0, -0.0, 5.999999, 6.000001, 1e30, -1e30],
    ]).astype(np.float32)
    for v in grid:
        assert orc.e2m1_encode(float(v)) == _e2m1_brute(float(v)), float(v)


def test_e2m1_rounding_landmarks(orc):
    # round-to-nearest-even at every midpoint of the E2M1 grid, saturation above 6
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6, 7.0: 7, 100.0: 7}
    for v, c in cases.items():
        assert orc.e2m1_encode(v) == c and orc.e2m1_encode(-v) == c | 8


def test_e4m3_encode_matches_torch_in_range(orc):
    vals = np.array([orc.e4m3_value(b) for b in range(0x7F)])        # 0 .. 448
    mids = (vals[:-1] + vals[1:]) / 2                                   # exact ties
    rng = np.random.default_rng(7)
    x = np.concatenate([vals, mids, rng.uniform(0, 448, 20000),
                        np.exp(rng.uniform(np.log(1e-4), np.log(448), 20000))]).astype(np.float32)
    x = x[x <= 448]
    ref = torch.tensor(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_saturates(orc):
    for v in [448.0, 449.0, 463.9, 464.0, 465.0, 1e6, 3.0e38]:
        assert orc.e4m3_encode(v) == 0x7E
        assert orc.e4m3_encode(-v) == 0xFE


_E4M3_POS = None


def _e4m3_nearest_exact(fr):
    """E4M3 byte of the exact rational fr >= 0: nearest value, ties to the even code, satfinite."""
    global _E4M3_POS
    if _E4M3_POS is None:
        ref = _torch_e4m3(np.arange(0x7F))
        _E4M3_POS = [Fraction(float(v)) for v in ref]          # 0x00 .. 0x7E ascending
    vals = _E4M3_POS
    if fr >= vals[-1]:
        return 0x7E
    lo, hi = 0, len(vals) - 1
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if vals[mid] <= fr:
            lo = mid
        else:
            hi = mid
    dl, dh = fr - vals[lo], vals[hi] - fr
    if dl < dh:
        return lo
    if dh < dl:
        return hi
    return lo if lo % 2 == 0 else hi


def test_scale_rounding_is_exact_for_every_bf16_amax(orc):
    """amax / 6 rounded in fp32 and then to E4M3 equals E4M3 rounding of the exact quotient,
    for every positive finite bf16 amax (no double rounding).  Checked through the row
    quantiser itself: each 16-channel group carries one amax value."""
    bits = np.arange(1, 0x7F80, dtype=np.uint16)                  # positive finite bf16
    n = bits.size
    groups = np.zeros((n, 16), np.uint16)
    groups[:, 0] = bits
    pad = (-n) % 32
    groups = np.concatenate([groups, np.zeros((pad, 16), np.uint16)])
    rows = groups.reshape(-1, 512)
    _, scales = orc.fp4_quantize(rows)
    got = scales.reshape(-1)[:n]
    amax = syn.bf16_bits_to_f32(bits).astype(np.float64)
    exp = np.array([_e4m3_nearest_exact(Fraction(float(a)) / 6) for a in amax], dtype=np.uint8)
    assert np.array_equal(got, exp)


def _dequant_indep(codes, scales):
    """Dequantise with the golden E2M1 table and torch's E4M3 decoder (independent of the oracle)."""
    tab = np.array([v for _, v in sorted(_e2m1_table().items())])
    lo = codes & 15
    hi = codes >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(codes.shape[:-1] + (codes.shape[-1] * 2,))
    sv = _torch_e4m3(scales).reshape(scales.shape)
    return tab[nib] * np.repeat(sv, 16, axis=-1)


def _rows(seed, n):
    g = np.random.default_rng(seed)
    x = g.standard_normal((n, 512)).astype(np.float32)
    x[0] *= 1e-4            # tiny scales (subnormal E4M3 region)
    x[1] *= 1e3             # saturating scales
    x[2] = 0.0              # all-zero groups
    x[3, :16] = -0.0
    x[4] = np.where(g.random(512) < 0.05, x[4] * 20, x[4])
    x[5, ::16] = 6.0 * 2.0 ** -12   # amax/6 below half the smallest subnormal: zero scale
    return syn.f32_to_bf16_bits(x)


def test_quantize_brute_force_nearest(orc):
    """Every code is the E2M1 value whose product with the group's decoded scale is nearest
    to x (ties are covered by the codec tests), saturating at +-6 * scale."""
    xb = _rows(11, 64)
    codes, scales = orc.fp4_quantize(xb)
    x = syn.bf16_bits_to_f32(xb).astype(np.float64)
    xh = _dequant_indep(codes, scales)
    s = np.repeat(_torch_e4m3(scales).reshape(scales.shape), 16, axis=-1)
    tab = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])
    cand = tab[None, None, :] * s[..., None]
    best = np.min(np.abs(cand - x[..., None]), axis=-1)
    nz = s > 0
    assert np.all(np.abs(xh - x)[nz] == best[nz])
    assert np.all(xh[~nz] == 0)


def test_quantize_invariants(orc):
    xb = _rows(12, 128)
    codes, scales = orc.fp4_quantize(xb)
    x = syn.bf16_bits_to_f32(xb).astype(np.float64).reshape(128, 32, 16)
    nib = np.stack([codes & 15, codes >> 4], -1).reshape(128, 32, 16)
    sv = _torch_e4m3(scales).reshape(128, 32)
    amax = np.abs(x).max(-1)
    # the largest-magnitude element gets code +-6 whenever the scale is normal and unsaturated
    normal = (sv >= 2.0 ** -6) & (amax / 6 <= 448)
    am = np.abs(x).argmax(-1)
    top = np.take_along_axis(nib, am[..., None], -1)[..., 0]
    assert np.all((top[normal] & 7) == 7)
    # zero scale <=> all-zero codes
    assert np.all(nib[sv == 0] == 0)
    # sign bit follows the sign of x wherever the scale is nonzero
    sgn = np.signbit(x)
    assert np.all(((nib & 8) > 0)[sv > 0] == sgn[sv > 0])
    # dequantisation is exact in bf16 and matches the independent decode
    deq = orc.fp4_dequantize(codes, scales)
    ind = _dequant_indep(codes, scales)
    assert np.array_equal(syn.bf16_bits_to_f32(deq).astype(np.float64), ind.reshape(128, 512))
    # idempotence: Q(DQ(Q(x))) == Q(x)
    c2, s2 = orc.fp4_quantize(deq)
    assert np.array_equal(c2, codes) and np.array_equal(s2, scales)


def test_nibble_order_and_layout(orc):
    # channel 0 = 6, channel 1 = 0, channel 17 = -3 (group 1): scale_0 = scale_1 = 1.0
    x = np.zeros(512, np.float32)
    x[0] = 6.0
    x[17] = -3.0
    x[16] = 6.0
    codes, scales = orc.fp4_quantize(syn.f32_to_bf16_bits(x)[None])
    assert codes[0, 0] == 0x07                     # even channel in the low nibble
    assert codes[0, 8] == (0x07 | (0x0D << 4))     # channels 16 (6.0) and 17 (-3.0)
    assert scales[0, 0] == 0x38 and scales[0, 1] == 0x38
    assert np.all(scales[0, 2:] == 0) and np.all(codes[0, 9:] == 0)


def test_fp8_window_rows_every_bf16_value(orc):
    """8-bit window rows: every finite bf16 value quantises to the nearest E4M3 value of its
    magnitude (exact rationals; ties to the even code; saturating at 448) with its sign, a zero
    result keeping the sign; dequantisation returns the E4M3 value exactly (in bf16)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = syn.bf16_bits_to_f32(bits)
    bits = bits[np.isfinite(f)]
    f = f[np.isfinite(f)]
    got = orc.fp8_quantize(bits)
    sign = ((bits >> 15).astype(np.uint8) << 7)
    exp = np.array([_e4m3_nearest_exact(Fraction(abs(float(v)))) for v in f], np.uint8) | sign
    assert np.array_equal(got, exp)
    back = syn.bf16_bits_to_f32(orc.fp8_dequantize(got)).astype(np.float64)
    ref = _torch_e4m3(got)
    assert np.array_equal(back, ref)

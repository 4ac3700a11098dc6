"""GPU parity of the FP4 quantise-append and dequantise kernels against the oracle: bit-exact
codes and scales, on ragged appends, an exhaustive value-by-scale sweep and the full-size
64 x 8192 x 512 round-trip workload (sampled sequences against the oracle, every row against
the idempotence property)."""
import numpy as np
import pytest

import csa2_synth as syn
from tests._cases import bf16_dev, bf16_host, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)
import compressed_sparse_attention_step_gb300 as c  # noqa: E402


def test_quantize_append_ragged_offsets(orc):
    B, n_new, cap = 3, 37, 100
    x = syn.normal_bf16(21, syn.T_X, 0, (B, n_new, 512))
    x[1, 3] = syn.f32_to_bf16_bits(np.zeros(512, np.float32))
    x[2, 5, :64] = 0x8000                                   # -0.0
    codes = torch.full((B, cap, 256), 0xAB, dtype=torch.uint8, device="cuda")
    scales = torch.full((B, cap, 32), 0xCD, dtype=torch.uint8, device="cuda")
    offs = torch.tensor([0, 10, 63], dtype=torch.int32, device="cuda")
    c.csa2_fp4_quantize_append(bf16_dev(x), codes, scales, offs)
    torch.cuda.synchronize()
    gc, gs = codes.cpu().numpy(), scales.cpu().numpy()
    oc, os_ = orc.fp4_quantize(x)
    for b, o in enumerate([0, 10, 63]):
        assert np.array_equal(gc[b, o:o + n_new], oc[b]) and np.array_equal(gs[b, o:o + n_new], os_[b])
        keep = np.ones(cap, bool)
        keep[o:o + n_new] = False
        assert np.all(gc[b, keep] == 0xAB) and np.all(gs[b, keep] == 0xCD)
    assert c.csa2_device_flags() == 0


def test_quantize_out_of_range_rows_are_flagged_and_skipped():
    x = bf16_dev(syn.normal_bf16(22, syn.T_X, 0, (2, 8, 512)))
    codes = torch.zeros((2, 10, 256), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((2, 10, 32), dtype=torch.uint8, device="cuda")
    c.csa2_device_flags(clear=True)
    c.csa2_fp4_quantize_append(x, codes, scales, torch.tensor([0, 5], dtype=torch.int32, device="cuda"))
    assert c.csa2_device_flags(clear=True) == c.FLAG_APPEND_OOB
    assert torch.all(codes[0, :8].sum(-1) > 0) and torch.all(codes[1, 5:].sum(-1) > 0)


def _sweep_rows():
    """Every finite bf16 value as x, each against 16 group maxima; and every positive finite bf16
    value as the group maximum."""
    bits = np.arange(65536, dtype=np.uint32)
    exp = (bits >> 7) & 0xFF
    finite = bits[exp != 0xFF].astype(np.uint16)
    xs = syn.bf16_bits_to_f32(finite)
    g = np.random.default_rng(3)
    amaxes = np.float32(2.0) ** g.uniform(-140, 127, 16).astype(np.float32)
    groups = []
    for a in amaxes:
        v = xs[np.abs(xs) <= a]
        v = np.concatenate([v, np.zeros((-v.size) % 15, np.float32)]).reshape(-1, 15)
        head = np.full((v.shape[0], 1), a, np.float32)
        groups.append(np.concatenate([head, v], 1))
    amax_all = xs[(xs > 0)]
    fill = amax_all[:, None] * g.uniform(-1, 1, (amax_all.size, 15)).astype(np.float32)
    groups.append(np.concatenate([amax_all[:, None], fill], 1))
    gr = np.concatenate(groups)
    perm = g.permutation(16)          # the maximum anywhere in the group
    gr = gr[:, perm]
    gr = np.concatenate([gr, np.zeros(((-gr.shape[0]) % 32, 16), np.float32)])
    return syn.f32_to_bf16_bits(gr).reshape(-1, 512)


def test_quantize_exhaustive_values_and_scales(orc):
    x = _sweep_rows()
    n = x.shape[0]
    codes = torch.empty((1, n, 256), dtype=torch.uint8, device="cuda")
    scales = torch.empty((1, n, 32), dtype=torch.uint8, device="cuda")
    c.csa2_fp4_quantize_append(bf16_dev(x[None]), codes, scales)
    oc, os_ = orc.fp4_quantize(x)
    assert np.array_equal(scales.cpu().numpy()[0], os_)
    assert np.array_equal(codes.cpu().numpy()[0], oc)
    out = torch.empty((n, 512), dtype=torch.bfloat16, device="cuda")
    c.csa2_fp4_dequantize(codes, scales, out)
    assert np.array_equal(bf16_host(out), orc.fp4_dequantize(oc, os_))


def test_dequantize_every_code_byte_and_scale_byte(orc):
    """Every packed code byte (both nibbles) under every finite non-negative E4M3 scale byte
    (0x00 .. 0x7E): one row per scale byte, whose 256 code bytes are 0 .. 255."""
    scale_bytes = np.arange(0x7F, dtype=np.uint8)
    codes = np.tile(np.arange(256, dtype=np.uint8), (scale_bytes.size, 1))
    scales = np.repeat(scale_bytes[:, None], 32, 1)
    out = torch.empty((scale_bytes.size, 512), dtype=torch.bfloat16, device="cuda")
    c.csa2_fp4_dequantize(to_dev(codes), to_dev(scales), out)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_host(out), orc.fp4_dequantize(codes, scales))


def test_fp4_roundtrip_full_size_64x8192x512(orc):
    """The FP4 round-trip workload: 64 sequences x 8192 tokens x 512 channels, N(0,1) with 1% of
    entries x20, quantised then dequantised in one launch each."""
    B, T = 64, 8192
    seed = syn.SEEDS["fp4_roundtrip_64x8192x512"]
    x = syn.device_outlier_bf16((B, T, 512), seed, syn.T_X)
    sampled = [0, 29, 63]
    host = {b: syn.outlier_bf16(seed, syn.T_X, b, (T, 512)) for b in sampled}
    for b in sampled:
        x[b].copy_(bf16_dev(host[b]))
    codes = torch.empty((B, T, 256), dtype=torch.uint8, device="cuda")
    scales = torch.empty((B, T, 32), dtype=torch.uint8, device="cuda")
    c.csa2_fp4_quantize_append(x, codes, scales)
    deq = torch.empty((B, T, 512), dtype=torch.bfloat16, device="cuda")
    c.csa2_fp4_dequantize(codes, scales, deq)
    torch.cuda.synchronize()
    for b in sampled:
        oc, os_ = orc.fp4_quantize(host[b])
        assert np.array_equal(codes[b].cpu().numpy(), oc)
        assert np.array_equal(scales[b].cpu().numpy(), os_)
        assert np.array_equal(bf16_host(deq[b]), orc.fp4_dequantize(oc, os_))
    # every row: quantising the dequantised tensor reproduces the codes (idempotence)
    c2 = torch.empty_like(codes)
    s2 = torch.empty_like(scales)
    c.csa2_fp4_quantize_append(deq, c2, s2)
    torch.cuda.synchronize()
    assert torch.equal(c2, codes) and torch.equal(s2, scales)

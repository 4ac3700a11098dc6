"""The allocation-free attention entry point.

csa2_sparse_attn_decode_static serves callers that cannot allocate device memory when they call
(for instance code running inside a memory allocator's callbacks, or a plugin that is handed only
its input and output buffers): it keeps its split-KV scratch in a fixed array inside the library.
These tests call it through the C ABI and check that it reproduces csa2_sparse_attn_decode (which
takes a caller workspace) bit for bit, on calls in a row of different sizes (the array keeps the
previous call's contents), and that an oversized problem is refused.  The file is collected last so
that a run stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import csa2_synth as syn
from tests._cases import SCALE, assert_attn_close, bf16_dev, bf16_host, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)
import compressed_sparse_attention_step_gb300 as c  # noqa: E402


def _inputs(seed, B, cap, k, W):
    kv = np.stack([syn.normal_bf16(seed, syn.T_KV, b, (cap, 512)) for b in range(B)])
    q = np.stack([syn.normal_bf16(seed, syn.T_Q, b, (1, 16, 512)) for b in range(B)])
    swa = np.stack([syn.normal_bf16(seed, syn.T_SWA, b, (W, 512)) for b in range(B)])
    g = np.random.default_rng(seed)
    idx = np.stack([np.sort(g.choice(cap, k, replace=False)) for _ in range(B)]).astype(np.int32)
    codes = torch.empty((B, cap, 256), dtype=torch.uint8, device="cuda")
    scales = torch.empty((B, cap, 32), dtype=torch.uint8, device="cuda")
    c.csa2_fp4_quantize_append(bf16_dev(kv), codes, scales)
    swa_len = np.minimum(np.full(B, W), np.arange(B) * 37 + 5).astype(np.int32)
    return bf16_dev(q), codes, scales, to_dev(idx), bf16_dev(swa), to_dev(swa_len)


def _call_static(q, codes, scales, idx, swa, swa_len, out, lse, n_split=0):
    B, cap, k = q.shape[0], codes.shape[1], idx.shape[1]
    st = c.lib().csa2_sparse_attn_decode_static(
        q.data_ptr(), B, 1, codes.data_ptr(), scales.data_ptr(), cap, idx.data_ptr(), None, k,
        swa.data_ptr(), swa_len.data_ptr(), 128, SCALE, out.data_ptr(), lse.data_ptr(), n_split,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_static_scratch_matches_workspace_entry_point():
    """Calls alternate between a batch of 7 queries (automatic split 10) and one of 64 (split 4), so
    each call starts from the previous call's partials and tickets, over a different ticket range.
    Both entry points run the same kernel at the same split, so outputs and lse must be identical
    bit for bit; the first case is also checked against the attention tolerance of the oracle tests'
    reference, the workspace entry point."""
    cases = []
    for seed, B in ((71, 7), (72, 64)):
        q, codes, scales, idx, swa, swa_len = _inputs(seed, B, 2000, 512, 128)
        ref = torch.empty((B, 1, 16, 512), dtype=torch.bfloat16, device="cuda")
        ref_lse = torch.empty((B, 1, 16), dtype=torch.float32, device="cuda")
        c.csa2_sparse_attn_decode(q, codes, scales, idx, ref, swa=swa, swa_len=swa_len, W=128,
                                  softmax_scale=SCALE, lse=ref_lse)
        cases.append(((q, codes, scales, idx, swa, swa_len), ref, ref_lse))
    torch.cuda.synchronize()
    assert c.lib().csa2_attn_auto_split(7, 512, 128) > 1 and c.lib().csa2_attn_auto_split(64, 512, 128) > 1
    for call in (0, 1, 0, 1, 1, 0):
        args, ref, ref_lse = cases[call]
        B = ref.shape[0]
        out = torch.full((B, 1, 16, 512), 9.0, dtype=torch.bfloat16, device="cuda")
        lse = torch.zeros((B, 1, 16), dtype=torch.float32, device="cuda")
        assert _call_static(*args, out, lse) == 0
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call of batch {B}: outputs differ from the workspace entry point"
        assert torch.equal(lse, ref_lse), f"call of batch {B}: lse differs from the workspace entry point"
        assert_attn_close(bf16_host(out), syn.bf16_bits_to_f32(bf16_host(ref)).astype(np.float64),
                          "static-scratch attention")


def test_static_scratch_refuses_oversized_split():
    cap_bytes = int(c.lib().csa2_sparse_attn_static_scratch_bytes())
    B = 128
    q, codes, scales, idx, swa, swa_len = _inputs(73, B, 600, 512, 128)
    out = torch.zeros((B, 1, 16, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, 1, 16), dtype=torch.float32, device="cuda")
    n_split = 5                               # 128 queries x 5 splits of 32 KiB exceed 16 MiB
    assert B * n_split * (16 * 512 + 32) * 4 > cap_bytes
    assert _call_static(q, codes, scales, idx, swa, swa_len, out, lse, n_split=n_split) == 5
    assert c.lib().csa2_status_string(5) == b"problem exceeds the library's built-in scratch"

"""GPU parity of the 8-bit (E4M3) window: the quantiser is bit-exact with the oracle on every finite
bf16 value, and group steps whose windows hold E4M3 rows (decode with ragged contexts and partial
windows, prefill chunks on both selection paths, the full-size decode group) match the oracle
reading the same bytes."""
import numpy as np
import pytest

import csa2_synth as syn
from tests._cases import GroupCase

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)
import compressed_sparse_attention_step_gb300 as c  # noqa: E402

F, RX, R = c.MODE_FULL, c.MODE_REINDEX, c.MODE_REUSE


def test_fp8_quantize_every_bf16_value(orc):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    bits = bits[np.isfinite(syn.bf16_bits_to_f32(bits))]
    for n in (bits.size, bits.size - 5):   # a tail shorter than a thread's 8 values
        x = torch.from_numpy(bits[:n].view(np.int16).copy()).cuda().view(torch.bfloat16)
        out = torch.full((n,), 0xAA, dtype=torch.uint8, device="cuda")
        c.csa2_fp8_quantize(x, out)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), orc.fp8_quantize(bits[:n]))


def test_decode_group_fp8_window_ragged(orc):
    """Contexts shorter than the window (partial windows) and than K; Reuse and Reindex layers."""
    gc = GroupCase(81, [3000, 700, 130, 9], [F, R, RX, R], swa_fp8=True)
    gc.run()
    gc.check(orc)


def test_prefill_chunk_fp8_window_cuda_core_path(orc):
    Nq, T = 24, 300
    q_pos = np.arange(2 * T - Nq, 2 * T, dtype=np.int32)[None]
    gc = GroupCase(82, [T], [F, R, R], Nq=Nq, ratio=2, K=128, W=32, append=False, q_pos=q_pos, swa_fp8=True)
    gc.run()
    gc.check(orc)


def test_prefill_chunk_fp8_window_tensor_core_path(orc):
    Nq, T = 64, 6000
    q_pos = np.arange(2 * T - Nq, 2 * T, dtype=np.int32)[None]
    gc = GroupCase(83, [T], [F, R, R], Nq=Nq, ratio=2, K=256, W=64, append=False, q_pos=q_pos, swa_fp8=True)
    gc.run()
    gc.check(orc)


def test_prefill_chunk_fp8_window_many_queries(orc):
    """256 queries x 3 layers sharing their selection: one attention launch of 768 queries, which
    runs the kernel with two CTAs per SM."""
    Nq, T = 256, 6000
    q_pos = np.arange(2 * T - Nq, 2 * T, dtype=np.int32)[None]
    gc = GroupCase(84, [T], [F, R, R], Nq=Nq, ratio=2, K=256, W=64, append=False, q_pos=q_pos, swa_fp8=True)
    gc.run()
    gc.check(orc)


def test_decode_group_fp8_window_full_size_b64_t131072(orc):
    """The decode workload with 8-bit windows: batch 64, 128K context, 1 Full + 3 Reuse, sampled
    sequences."""
    gc = GroupCase(syn.SEEDS["decode_group_1f3r_b64_t131072"], [131072] * 64, [F, R, R, R],
                   host_seqs=[0, 63], swa_fp8=True)
    gc.run()
    gc.check(orc, seqs=[0, 63], threads=2)

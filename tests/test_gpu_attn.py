"""GPU parity of split-KV sparse attention against the oracle (fp64): outputs within
max-abs 2e-2 and relative (Frobenius) 1e-2, lse within 1e-2, over ragged selections, empty
slots, partial windows, several queries per sequence, every split count, and the empty case."""
import numpy as np
import pytest

import csa2_synth as syn
from tests._cases import SCALE, assert_attn_close, bf16_dev, bf16_host, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)
import compressed_sparse_attention_step_gb300 as c  # noqa: E402


def _case(seed, B, Nq, cap, k, W):
    kv = np.stack([syn.normal_bf16(seed, syn.T_KV, b, (cap, 512)) for b in range(B)])
    q = np.stack([syn.normal_bf16(seed, syn.T_Q, b, (Nq, 16, 512)) for b in range(B)])
    swa = np.stack([syn.normal_bf16(seed, syn.T_SWA, b, (max(W - 1 + Nq, 1), 512)) for b in range(B)])
    g = np.random.default_rng(seed)
    idx = np.stack([np.sort(g.choice(cap, k, replace=False)) for _ in range(B * Nq)]).astype(np.int32)
    return kv, q, swa, idx


def _run(kv, q, swa, idx, nvalid, swa_len, W, n_split, use_swa=True):
    B, cap = kv.shape[0], kv.shape[1]
    Nq = q.shape[1]
    codes = torch.empty((B, cap, 256), dtype=torch.uint8, device="cuda")
    scales = torch.empty((B, cap, 32), dtype=torch.uint8, device="cuda")
    c.csa2_fp4_quantize_append(bf16_dev(kv), codes, scales)
    out = torch.zeros((B, Nq, 16, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, Nq, 16), dtype=torch.float32, device="cuda")
    c.csa2_sparse_attn_decode(bf16_dev(q), codes, scales, to_dev(idx), out,
                              n_valid=None if nvalid is None else to_dev(nvalid),
                              swa=bf16_dev(swa) if use_swa else None,
                              swa_len=to_dev(swa_len) if use_swa else None, W=W,
                              softmax_scale=SCALE, lse=lse, n_split=n_split)
    torch.cuda.synchronize()
    return bf16_host(out), lse.cpu().numpy()


def _oracle(orc, kv, q, swa, idx, nvalid, swa_len, W, use_swa=True):
    B, Nq = q.shape[0], q.shape[1]
    k = idx.shape[1]
    outs, lses = [], []
    for b in range(B):
        codes, scales = orc.fp4_quantize(kv[b])
        SW = W - 1 + Nq
        for i in range(Nq):
            r = b * Nq + i
            sel = idx[r].copy()
            if nvalid is not None:
                sel[nvalid[r]:] = -1
            if use_swa:
                lo = SW - swa_len[b]
                rows = [swa[b, j] for j in range(i, i + W) if j >= lo]
                rows = np.stack(rows) if rows else np.zeros((0, 512), np.uint16)
            else:
                rows = np.zeros((0, 512), np.uint16)
            o, l = orc.sparse_attn(q[b, i], codes, scales, sel, rows, SCALE)
            outs.append(o)
            lses.append(l)
    return np.stack(outs).reshape(B, Nq, 16, 512), np.stack(lses).reshape(B, Nq, 16)


def _cmp(got, glse, ref, rlse):
    assert_attn_close(got, ref, "attention")
    fin = np.isfinite(rlse)
    assert np.array_equal(np.isfinite(glse), fin)
    assert np.all(np.abs(glse[fin] - rlse[fin]) <= 1e-2)


@pytest.mark.parametrize("n_split", [0, 1, 3, 20])
def test_decode_attention_ragged(orc, n_split):
    B, Nq, cap, k, W = 3, 1, 900, 512, 128
    kv, q, swa, idx = _case(41, B, Nq, cap, k, W)
    idx[0, 7] = -1
    idx[1, 100:130] = -1
    nvalid = np.array([512, 300, 17], np.int32)
    swa_len = np.array([128, 50, 0], np.int32)
    got, glse = _run(kv, q, swa, idx, nvalid, swa_len, W, n_split)
    ref, rlse = _oracle(orc, kv, q, swa, idx, nvalid, swa_len, W)
    _cmp(got, glse, ref, rlse)


def test_multi_query_windows_and_no_window(orc):
    B, Nq, cap, k, W = 2, 5, 600, 512 - 64, 16
    kv, q, swa, idx = _case(42, B, Nq, cap, k, W)
    swa_len = np.array([W - 1 + Nq, 9], np.int32)
    got, glse = _run(kv, q, swa, idx, None, swa_len, W, 0)
    ref, rlse = _oracle(orc, kv, q, swa, idx, None, swa_len, W)
    _cmp(got, glse, ref, rlse)
    got, glse = _run(kv, q, swa, idx, None, swa_len, W, 2, use_swa=False)
    ref, rlse = _oracle(orc, kv, q, swa, idx, None, swa_len, W, use_swa=False)
    _cmp(got, glse, ref, rlse)


def test_empty_rows_give_zero_and_neg_inf(orc):
    B, Nq, cap, k, W = 1, 1, 64, 512, 128
    kv, q, swa, idx = _case(43, B, Nq, cap, 64, W)
    idx = np.full((1, k), -1, np.int32)
    got, glse = _run(kv, q, swa, idx, None, np.array([0], np.int32), W, 4)
    assert np.all(syn.bf16_bits_to_f32(got) == 0) and np.all(np.isneginf(glse))


def test_index_out_of_range_is_flagged_not_read(orc):
    B, Nq, cap, k, W = 1, 1, 64, 64, 128
    kv, q, swa, idx = _case(44, B, Nq, cap, k, W)
    bad = idx.copy()
    bad[0, 3] = 10_000_000
    c.csa2_device_flags(clear=True)
    got, glse = _run(kv, q, swa, bad, None, np.array([128], np.int32), W, 0)
    assert c.csa2_device_flags(clear=True) & c.FLAG_INDEX_OOB
    sel = bad.copy()
    sel[0, 3] = -1
    ref, rlse = _oracle(orc, kv, q, swa, sel, None, np.array([128], np.int32), W)
    _cmp(got, glse, ref, rlse)


@pytest.mark.parametrize("n_split", [2, 4, 10])
def test_split_partials_of_empty_splits_are_never_read(orc, n_split):
    """Splits whose tiles hold no rows write no partial output; the workspace is filled with NaN
    first, so reading such a slot (even with a zero weight) would corrupt the merged result."""
    B, Nq, cap, k, W = 3, 1, 900, 512, 128
    kv, q, swa, idx = _case(43, B, Nq, cap, k, W)
    nvalid = np.array([512, 300, 17], np.int32)
    swa_len = np.array([128, 50, 0], np.int32)
    codes = torch.empty((B, cap, 256), dtype=torch.uint8, device="cuda")
    scales = torch.empty((B, cap, 32), dtype=torch.uint8, device="cuda")
    c.csa2_fp4_quantize_append(bf16_dev(kv), codes, scales)
    nb = c.workspace_size(c.OP_SPARSE_ATTN, B=B, Nq=Nq, k=k, W=W, n_split=n_split)
    ws = torch.full((max(nb, 256) // 4,), float("nan"), dtype=torch.float32, device="cuda")
    out = torch.zeros((B, Nq, 16, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, Nq, 16), dtype=torch.float32, device="cuda")
    c.csa2_sparse_attn_decode(bf16_dev(q), codes, scales, to_dev(idx), out, n_valid=to_dev(nvalid),
                              swa=bf16_dev(swa), swa_len=to_dev(swa_len), W=W, softmax_scale=SCALE, lse=lse,
                              n_split=n_split, ws=ws)
    torch.cuda.synchronize()
    ref, rlse = _oracle(orc, kv, q, swa, idx, nvalid, swa_len, W)
    _cmp(bf16_host(out), lse.cpu().numpy(), ref, rlse)


@pytest.mark.parametrize("n_split", [0, 2])
def test_many_queries_ragged(orc, n_split):
    """640 queries (more than one CTA per SM): the launch runs the kernel with two CTAs per SM
    instead of the warp-specialised one.  Ragged selections, empty slots and partial windows; with
    a forced split of 2 its partials are merged too."""
    B, Nq, cap, k, W = 4, 160, 2000, 512, 128
    kv, q, swa, idx = _case(45, B, Nq, cap, k, W)
    g = np.random.default_rng(45)
    nvalid = g.integers(0, k + 1, size=B * Nq).astype(np.int32)
    nvalid[:3] = [k, 0, 1]
    idx[g.random(idx.shape) < 0.02] = -1
    swa_len = np.array([W - 1 + Nq, 100, 0, 60], np.int32)
    got, glse = _run(kv, q, swa, idx, nvalid, swa_len, W, n_split)
    ref, rlse = _oracle(orc, kv, q, swa, idx, nvalid, swa_len, W)
    _cmp(got, glse, ref, rlse)

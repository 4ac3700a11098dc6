"""Python binding of the CSA2 step library (`_lib/libcsa2.so`, C ABI in `include/csa2.h`).

Argument marshalling only: every function below checks dtypes, shapes and devices of torch
tensors, passes their device pointers and the current CUDA stream to the C entry point of the
same name, and raises `Csa2Error` on a non-OK status.  All computation runs in the library's
CUDA kernels; there is no CPU or PyTorch fallback, and importing a function whose library is
not built raises immediately.

bf16 tensors may be torch.bfloat16 or torch.int16/uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

D, H, HI, DI, GROUP, BLOCK = 512, 16, 4, 128, 16, 8
CODE_BYTES, SCALE_BYTES = 256, 32
MAX_LAYERS = 16
MODE_FULL, MODE_REINDEX, MODE_REUSE = 0, 1, 2
OP_TOPK, OP_BLOCK_POOL, OP_SPARSE_ATTN, OP_GROUP_STEP, OP_INDEX_SELECT_PREFILL, OP_MERGE_PAIRS = 1, 2, 3, 4, 5, 6
FLAG_APPEND_OOB, FLAG_INDEX_OOB, FLAG_TIMEOUT = 1, 2, 4
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE, ERR_TOO_LARGE = 0, 1, 2, 3, 4, 5
SWA_BF16, SWA_E4M3 = 0, 1

LIB_PATH = _build.LIB


class Csa2Error(RuntimeError):
    def __init__(self, fn, status, text):
        super().__init__(f"{fn}: {text} (status {status})")
        self.status = status


P = ctypes.c_void_p
I32 = ctypes.c_int
I64 = ctypes.c_int64
SZ = ctypes.c_size_t
F32 = ctypes.c_float


class GroupDesc(ctypes.Structure):
    """Mirror of `csa2_group_desc` (checked against csa2_group_desc_size at load)."""
    _fields_ = [
        ("n_layers", I32), ("modes", I32 * MAX_LAYERS),
        ("B", I32), ("Nq", I32), ("K", I32), ("W", I32), ("ratio", I32),
        ("hierarchical", I32), ("n_blocks_keep", I32), ("n_split", I32), ("n_new", I32), ("seq_chunks", I32),
        ("swa_format", I32), ("cap", I64), ("lens", P), ("q_pos", P),
        ("codes", P), ("scales", P), ("KI", P), ("block_keys", P),
        ("kv_new", P), ("ki_new", P),
        ("q", P * MAX_LAYERS), ("qI", P * MAX_LAYERS), ("w", P * MAX_LAYERS),
        ("swa", P * MAX_LAYERS), ("swa_len", P),
        ("out", P * MAX_LAYERS), ("lse", P * MAX_LAYERS), ("idx", P * MAX_LAYERS),
        ("pool", P), ("pool_len", P),
        ("softmax_scale", F32),
        ("ev_score_begin", P), ("ev_score_end", P),
        ("ev_attn_begin", P), ("ev_attn_end", P),
    ]


class Dims(ctypes.Structure):
    _fields_ = [("B", I32), ("Nq", I32), ("cap", I64), ("n", I64), ("k", I32), ("W", I32),
                ("n_split", I32), ("hierarchical", I32), ("n_blocks_keep", I32)]


_lib = None


def lib():
    """Load the built library (never builds implicitly; raises if it is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CSA2 library not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "csa2_fp4_quantize_append": [P, I32, I32, I32, P, P, I64, P, P],
            "csa2_fp4_dequantize": [P, P, I64, I32, P, P],
            "csa2_index_score": [P, P, I32, I32, P, I64, P, P, P, I64, I32, P, P, P, P],
            "csa2_topk": [P, I32, I64, I64, P, I32, P, I64, P, P, P, SZ, P],
            "csa2_block_keys_build": [P, I32, I64, P, P, P],
            "csa2_block_pool": [P, P, I32, I32, P, I64, P, I32, P, I32, P, P, P, SZ, P],
            "csa2_sparse_attn_decode": [P, I32, I32, P, P, I64, P, P, I32, P, P, I32, F32, P, P, I32, P,
                                        SZ, P],
            "csa2_group_step": [ctypes.POINTER(GroupDesc), P, SZ, P],
            "csa2_stack_step": [ctypes.POINTER(GroupDesc), I32, P, SZ, P],
            "csa2_fp8_quantize": [P, I64, P, P],
            "csa2_workspace_size": [I32, ctypes.POINTER(Dims)],
            "csa2_attn_auto_split": [I64, I32, I32],
            "csa2_status_string": [I32],
            "csa2_device_flags": [ctypes.POINTER(ctypes.c_uint32), I32, P],
            "csa2_group_desc_size": [],
            "csa2_sparse_attn_decode_static": [P, I32, I32, P, P, I64, P, P, I32, P, P, I32, F32, P, P, I32, P],
            "csa2_sparse_attn_static_scratch_bytes": [],
            "csa2_index_select_prefill": [P, P, I32, I32, P, I64, P, I32, P, I32, P, P, P, SZ, P],
            "csa2_shard_topk_pairs": [P, I32, I64, I64, P, I32, P, I64, I64, P, P, P, P, SZ, P],
            "csa2_merge_topk_pairs": [P, P, P, I32, I32, I32, P, P, P, SZ, P],
            "csa2_shard_indices": [P, I32, I32, I64, I64, P, P],
            "csa2_attn_merge_shards": [P, P, I32, I32, P, P, P],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = I32
        L.csa2_workspace_size.restype = SZ
        L.csa2_status_string.restype = ctypes.c_char_p
        L.csa2_group_desc_size.restype = SZ
        L.csa2_sparse_attn_static_scratch_bytes.restype = SZ
        if L.csa2_group_desc_size() != ctypes.sizeof(GroupDesc):
            raise RuntimeError("csa2_group_desc layout mismatch between binding and library")
        _lib = L
    return _lib


# ---------------------------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _ptr(t, name, dtypes=None, numel=None, cuda=True):
    if t is None:
        return None
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name}: expected at least {numel} elements, got {t.numel()}")
    return t.data_ptr()


def _bf16_types():
    torch = _torch()
    return (torch.bfloat16, torch.int16, torch.uint16)


def _stream(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(fn, st):
    if st != 0:
        raise Csa2Error(fn, st, lib().csa2_status_string(st).decode())


# ---------------------------------------------------------------------------------------------
# C-ABI entry points (same names)
# ---------------------------------------------------------------------------------------------
def csa2_fp4_quantize_append(x, codes, scales, offsets=None, stream=None):
    """x [B, n_new, 512] bf16 -> codes [B, cap, 256] u8 and scales [B, cap, 32] u8 at rows
    offsets[b] + r (offsets int32 [B] or None)."""
    torch = _torch()
    B, n_new, d = x.shape
    cap = codes.shape[1]
    _check("csa2_fp4_quantize_append", lib().csa2_fp4_quantize_append(
        _ptr(x, "x", _bf16_types()), B, n_new, d,
        _ptr(codes, "codes", (torch.uint8,), B * cap * CODE_BYTES),
        _ptr(scales, "scales", (torch.uint8,), B * cap * SCALE_BYTES), cap,
        _ptr(offsets, "offsets", (torch.int32,), B), _stream(stream)))


def csa2_fp4_dequantize(codes, scales, out, stream=None):
    torch = _torch()
    rows = codes.numel() // CODE_BYTES
    _check("csa2_fp4_dequantize", lib().csa2_fp4_dequantize(
        _ptr(codes, "codes", (torch.uint8,)), _ptr(scales, "scales", (torch.uint8,), rows * SCALE_BYTES),
        rows, D, _ptr(out, "out", _bf16_types(), rows * D), _stream(stream)))


def csa2_index_score(qI, w, KI, lens, scores, *, cand=None, cand_len=None, ratio=1, q_pos=None,
                     n_valid=None, stream=None):
    """qI [B, Nq, 4, 128], w [B, Nq, 4] fp32, KI [B, cap, 128], lens int32 [B];
    scores fp32 [B*Nq, cap] (or [B*Nq, n_cand] with cand int32 [B*Nq, n_cand])."""
    torch = _torch()
    B, Nq = qI.shape[0], qI.shape[1]
    cap = KI.shape[1]
    n_cand = cand.shape[-1] if cand is not None else 0
    _check("csa2_index_score", lib().csa2_index_score(
        _ptr(qI, "qI", _bf16_types(), B * Nq * HI * DI), _ptr(w, "w", (torch.float32,), B * Nq * HI), B, Nq,
        _ptr(KI, "KI", _bf16_types(), B * cap * DI), cap, _ptr(lens, "lens", (torch.int32,), B),
        _ptr(cand, "cand", (torch.int32,)), _ptr(cand_len, "cand_len", (torch.int32,)), n_cand, ratio,
        _ptr(q_pos, "q_pos", (torch.int32,), B * Nq),
        _ptr(scores, "scores", (torch.float32,), B * Nq * (n_cand if cand is not None else cap)),
        _ptr(n_valid, "n_valid", (torch.int32,)), _stream(stream)))


def csa2_topk(scores, k, idx, *, n_valid=None, n=None, map_=None, n_sel=None, ws=None, stream=None):
    """scores fp32 [rows, ld] -> idx int32 [rows, k] (ascending, -1 padded)."""
    torch = _torch()
    rows, ld = scores.shape
    n = ld if n is None else n
    map_ld = map_.shape[-1] if map_ is not None else 0
    need = workspace_size(OP_TOPK, B=rows, Nq=1, n=n, k=k)
    if ws is None and need:
        ws = _ws(need, scores.device)
    _check("csa2_topk", lib().csa2_topk(
        _ptr(scores, "scores", (torch.float32,)), rows, n, ld, _ptr(n_valid, "n_valid", (torch.int32,), rows),
        k, _ptr(map_, "map", (torch.int32,)), map_ld, _ptr(idx, "idx", (torch.int32,), rows * k),
        _ptr(n_sel, "n_sel", (torch.int32,), rows), _ptr(ws, "ws"), _nbytes(ws),
        _stream(stream)))


def csa2_block_keys_build(KI, lens, block_keys, stream=None):
    torch = _torch()
    B, cap = KI.shape[0], KI.shape[1]
    _check("csa2_block_keys_build", lib().csa2_block_keys_build(
        _ptr(KI, "KI", _bf16_types()), B, cap, _ptr(lens, "lens", (torch.int32,), B),
        _ptr(block_keys, "block_keys", _bf16_types(), B * (cap // BLOCK) * DI), _stream(stream)))


def workspace_size(op, *, B=0, Nq=1, cap=0, n=0, k=0, W=0, n_split=0, hierarchical=0, n_blocks_keep=0):
    d = Dims(B, Nq, cap, n, k, W, n_split, hierarchical, n_blocks_keep)
    return int(lib().csa2_workspace_size(op, ctypes.byref(d)))


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def _ws(nbytes, device):
    torch = _torch()
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def csa2_index_select_prefill(qI, w, KI, lens, idx, *, k=512, ratio=1, q_pos=None, n_sel=None, ws=None,
                              stream=None):
    """Exact Top-k per query of a prefill chunk via the tensor-core filter: qI [B, Nq, 4, 128] bf16,
    w [B, Nq, 4] fp32, KI [B, cap, 128] bf16, lens int32 [B] -> idx int32 [B*Nq, k]."""
    torch = _torch()
    B, Nq = qI.shape[0], qI.shape[1]
    cap = KI.shape[1]
    rows = B * Nq
    need = workspace_size(OP_INDEX_SELECT_PREFILL, B=B, Nq=Nq, cap=cap)
    if ws is None:
        ws = _ws(need, qI.device)
    _check("csa2_index_select_prefill", lib().csa2_index_select_prefill(
        _ptr(qI, "qI", _bf16_types(), rows * HI * DI), _ptr(w, "w", (torch.float32,), rows * HI), B, Nq,
        _ptr(KI, "KI", _bf16_types(), B * cap * DI), cap, _ptr(lens, "lens", (torch.int32,), B), ratio,
        _ptr(q_pos, "q_pos", (torch.int32,), rows), k, _ptr(idx, "idx", (torch.int32,), rows * k),
        _ptr(n_sel, "n_sel", (torch.int32,), rows), _ptr(ws, "ws"), _nbytes(ws), _stream(stream)))


def csa2_block_pool(qI, w, block_keys, cap, lens, keep, pool, pool_len, *, ratio=1, q_pos=None, ws=None,
                    stream=None):
    torch = _torch()
    B, Nq = qI.shape[0], qI.shape[1]
    need = workspace_size(OP_BLOCK_POOL, B=B, Nq=Nq, cap=cap)
    ws = ws if ws is not None else _ws(need, qI.device)
    _check("csa2_block_pool", lib().csa2_block_pool(
        _ptr(qI, "qI", _bf16_types()), _ptr(w, "w", (torch.float32,)), B, Nq,
        _ptr(block_keys, "block_keys", _bf16_types()), cap, _ptr(lens, "lens", (torch.int32,), B), ratio,
        _ptr(q_pos, "q_pos", (torch.int32,), B * Nq), keep,
        _ptr(pool, "pool", (torch.int32,), B * Nq * keep * BLOCK), _ptr(pool_len, "pool_len", (torch.int32,), B * Nq),
        _ptr(ws, "ws"), _nbytes(ws), _stream(stream)))


def csa2_sparse_attn_decode(q, codes, scales, idx, out, *, n_valid=None, swa=None, swa_len=None, W=0,
                            softmax_scale=None, lse=None, n_split=0, ws=None, stream=None):
    """q [B, Nq, 16, 512]; codes/scales [B, cap, *]; idx int32 [B*Nq, k]; swa [B, W-1+Nq, 512]."""
    torch = _torch()
    B, Nq = q.shape[0], q.shape[1]
    cap = codes.shape[1]
    k = idx.shape[-1]
    if softmax_scale is None:
        softmax_scale = D ** -0.5
    if swa is None:
        W = 0
    ns = n_split or int(lib().csa2_attn_auto_split(B * Nq, k, W))
    need = workspace_size(OP_SPARSE_ATTN, B=B, Nq=Nq, k=k, W=W, n_split=ns)
    if ws is None and need:
        ws = _ws(need, q.device)
    _check("csa2_sparse_attn_decode", lib().csa2_sparse_attn_decode(
        _ptr(q, "q", _bf16_types(), B * Nq * H * D), B, Nq, _ptr(codes, "codes", (torch.uint8,)),
        _ptr(scales, "scales", (torch.uint8,)), cap, _ptr(idx, "idx", (torch.int32,), B * Nq * k),
        _ptr(n_valid, "n_valid", (torch.int32,), B * Nq), k, _ptr(swa, "swa", _bf16_types()),
        _ptr(swa_len, "swa_len", (torch.int32,), B), W, float(softmax_scale),
        _ptr(out, "out", _bf16_types(), B * Nq * H * D), _ptr(lse, "lse", (torch.float32,), B * Nq * H), ns,
        _ptr(ws, "ws"), _nbytes(ws), _stream(stream)))


def group_workspace_size(B, Nq, cap, K=512, W=128, hierarchical=False, keep=2048, n_split=0):
    return workspace_size(OP_GROUP_STEP, B=B, Nq=Nq, cap=cap, k=K, W=W, n_split=n_split,
                          hierarchical=int(bool(hierarchical)), n_blocks_keep=keep)


def make_group_desc(modes, *, B, Nq, cap, lens, codes, scales, KI, q, qI, w, swa, swa_len, out, idx,
                    K=512, W=128, ratio=1, hierarchical=False, keep=2048, n_split=0, q_pos=None,
                    block_keys=None, pool=None, pool_len=None, kv_new=None, ki_new=None, lse=None,
                    softmax_scale=None, events=None, seq_chunks=0, swa_fp8=False, attn_events=None):
    """Build a csa2_group_desc from torch tensors (per-layer arguments are lists; entries of
    qI/w/idx may be None for Reuse layers; swa_fp8: the window buffers are uint8 E4M3 rows, as
    csa2_fp8_quantize writes them; events / attn_events: (begin, end) torch.cuda.Event pairs
    recorded around the step's first indexer scan / first attention launch)."""
    torch = _torch()
    L = len(modes)
    if not 1 <= L <= MAX_LAYERS:
        raise ValueError("1..16 layers per group")
    g = GroupDesc()
    g.n_layers = L
    for l, m in enumerate(modes):
        g.modes[l] = int(m)
    g.B, g.Nq, g.K, g.W, g.ratio = B, Nq, K, W, ratio
    g.hierarchical, g.n_blocks_keep, g.n_split = int(bool(hierarchical)), keep, n_split
    n_new = 0
    if kv_new is not None:
        n_new = kv_new.shape[1]
    elif ki_new is not None:
        n_new = ki_new.shape[1]
    g.n_new = n_new
    g.seq_chunks = int(seq_chunks)
    g.swa_format = SWA_E4M3 if swa_fp8 else SWA_BF16
    g.cap = cap
    bf = _bf16_types()
    g.lens = _ptr(lens, "lens", (torch.int32,), B)
    g.q_pos = _ptr(q_pos, "q_pos", (torch.int32,), B * Nq)
    g.codes = _ptr(codes, "codes", (torch.uint8,), B * cap * CODE_BYTES)
    g.scales = _ptr(scales, "scales", (torch.uint8,), B * cap * SCALE_BYTES)
    g.KI = _ptr(KI, "KI", bf, B * cap * DI)
    g.block_keys = _ptr(block_keys, "block_keys", bf)
    g.kv_new = _ptr(kv_new, "kv_new", bf)
    g.ki_new = _ptr(ki_new, "ki_new", bf)
    for l in range(L):
        g.q[l] = _ptr(q[l], f"q[{l}]", bf, B * Nq * H * D)
        g.qI[l] = _ptr(qI[l], f"qI[{l}]", bf) if qI[l] is not None else None
        g.w[l] = _ptr(w[l], f"w[{l}]", (torch.float32,)) if w[l] is not None else None
        g.swa[l] = (_ptr(swa[l], f"swa[{l}]", (torch.uint8,) if swa_fp8 else bf)
                    if (swa is not None and swa[l] is not None) else None)
        g.out[l] = _ptr(out[l], f"out[{l}]", bf, B * Nq * H * D)
        g.lse[l] = _ptr(lse[l], f"lse[{l}]", (torch.float32,)) if (lse is not None and lse[l] is not None) else None
        g.idx[l] = _ptr(idx[l], f"idx[{l}]", (torch.int32,), B * Nq * K) if idx[l] is not None else None
    g.swa_len = _ptr(swa_len, "swa_len", (torch.int32,), B)
    g.pool = _ptr(pool, "pool", (torch.int32,))
    g.pool_len = _ptr(pool_len, "pool_len", (torch.int32,))
    g.softmax_scale = float(D ** -0.5 if softmax_scale is None else softmax_scale)
    if events is not None:
        g.ev_score_begin = events[0].cuda_event
        g.ev_score_end = events[1].cuda_event
    if attn_events is not None:
        g.ev_attn_begin = attn_events[0].cuda_event
        g.ev_attn_end = attn_events[1].cuda_event
    return g


def csa2_group_step(desc, ws, stream=None):
    _check("csa2_group_step", lib().csa2_group_step(ctypes.byref(desc), _ptr(ws, "ws"), _nbytes(ws),
                                                    _stream(stream)))


def csa2_fp8_quantize(x, out, stream=None):
    """8-bit window rows: bf16 tensor x -> uint8 E4M3 tensor out of the same number of elements."""
    torch = _torch()
    n = x.numel()
    _check("csa2_fp8_quantize", lib().csa2_fp8_quantize(_ptr(x, "x", _bf16_types(), n), n,
                                                        _ptr(out, "out", (torch.uint8,), n), _stream(stream)))


def csa2_stack_step(descs, ws, stream=None):
    """The groups of a decoder stack in order (csa2_stack_step): descs is a list of group
    descriptors sharing one batch and cache; ws is sized for the largest group."""
    arr = (GroupDesc * len(descs))(*descs)
    _check("csa2_stack_step", lib().csa2_stack_step(arr, len(descs), _ptr(ws, "ws"), _nbytes(ws), _stream(stream)))


def csa2_device_flags(clear=True, stream=None):
    v = ctypes.c_uint32(0)
    _check("csa2_device_flags", lib().csa2_device_flags(ctypes.byref(v), int(clear), _stream(stream)))
    return int(v.value)


# ---------------------------------------------------------------------------------------------
# context split of one sequence over G shards
# ---------------------------------------------------------------------------------------------
def csa2_shard_topk_pairs(scores, k, pair_score, pair_pos, *, n_valid=None, n=None, pos_offset=0, map_=None,
                          pair_n=None, ws=None, stream=None):
    """A shard's local Top-k of scores fp32 [rows, ld] as (score, global position) pairs: pair_score
    fp32 [rows, k], pair_pos int32 [rows, k] (ascending, -1 padded), pair_n int32 [rows]."""
    torch = _torch()
    rows, ld = scores.shape
    n = ld if n is None else n
    map_ld = map_.shape[-1] if map_ is not None else 0
    need = workspace_size(OP_TOPK, B=rows, Nq=1, n=n, k=k)
    if ws is None and need:
        ws = _ws(need, scores.device)
    _check("csa2_shard_topk_pairs", lib().csa2_shard_topk_pairs(
        _ptr(scores, "scores", (torch.float32,)), rows, n, ld, _ptr(n_valid, "n_valid", (torch.int32,), rows), k,
        _ptr(map_, "map", (torch.int32,)), map_ld, int(pos_offset),
        _ptr(pair_score, "pair_score", (torch.float32,), rows * k), _ptr(pair_pos, "pair_pos", (torch.int32,), rows * k),
        _ptr(pair_n, "pair_n", (torch.int32,), rows), _ptr(ws, "ws"), _nbytes(ws), _stream(stream)))


def csa2_merge_topk_pairs(pair_score, pair_pos, idx, *, pair_n=None, n_sel=None, ws=None, stream=None):
    """The exact Top-k of G shards' pairs: pair_score fp32 [G, rows, k], pair_pos int32 [G, rows, k],
    pair_n int32 [G, rows] (shards in ascending order of their position ranges) -> idx int32 [rows, k]."""
    torch = _torch()
    G, rows, k = pair_score.shape
    need = workspace_size(OP_MERGE_PAIRS, B=rows, Nq=1, n=G, k=k)
    if ws is None:
        ws = _ws(need, pair_score.device)
    _check("csa2_merge_topk_pairs", lib().csa2_merge_topk_pairs(
        _ptr(pair_score, "pair_score", (torch.float32,), G * rows * k),
        _ptr(pair_pos, "pair_pos", (torch.int32,), G * rows * k), _ptr(pair_n, "pair_n", (torch.int32,), G * rows),
        G, rows, k, _ptr(idx, "idx", (torch.int32,), rows * k), _ptr(n_sel, "n_sel", (torch.int32,), rows),
        _ptr(ws, "ws"), _nbytes(ws), _stream(stream)))


def csa2_shard_indices(idx, lo, hi, idx_local, stream=None):
    """The selected positions a shard holding entries [lo, hi) attends, as its local rows (-1 elsewhere)."""
    torch = _torch()
    rows, k = idx.shape
    _check("csa2_shard_indices", lib().csa2_shard_indices(
        _ptr(idx, "idx", (torch.int32,)), rows, k, int(lo), int(hi),
        _ptr(idx_local, "idx_local", (torch.int32,), rows * k), _stream(stream)))


def csa2_attn_merge_shards(out_g, lse_g, out, lse=None, stream=None):
    """out_g [G, rows, 16, 512] bf16 and lse_g fp32 [G, rows, 16] -> out [rows, 16, 512], lse [rows, 16]."""
    torch = _torch()
    G = out_g.shape[0]
    rows = out_g[0].numel() // (H * D)
    _check("csa2_attn_merge_shards", lib().csa2_attn_merge_shards(
        _ptr(out_g, "out_g", _bf16_types(), G * rows * H * D), _ptr(lse_g, "lse_g", (torch.float32,), G * rows * H),
        G, rows, _ptr(out, "out", _bf16_types(), rows * H * D), _ptr(lse, "lse", (torch.float32,), rows * H),
        _stream(stream)))

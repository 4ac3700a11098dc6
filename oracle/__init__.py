"""CSA2 step oracle (test infrastructure).

A plain, slow CPU implementation of the CSA2 step, written in C++ in
`csa2_oracle.cpp` and loaded here through ctypes with numpy arrays.  It shares
no code with the CUDA path.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg use it; the product path never imports it.

Parity is pinned by the `-m "not gpu"` tests in `tests/test_oracle_*.py`:
every function below is checked there against facts fixed independently of
this code (format tables, brute force, closed forms, library routines).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa2_oracle.cpp")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle_csa2.so")

MODE_FULL, MODE_REINDEX, MODE_REUSE = 0, 1, 2
D, H, HI, DI, GROUP, BLOCK = 512, 16, 4, 128, 16, 8


def build(force: bool = False) -> str:
    """Compile the oracle with the host C++ compiler (no implicit FMA contraction)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-pthread", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
        _lib.oracle_e4m3_value.restype = ctypes.c_double
        _lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        _lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        _lib.oracle_e4m3_encode.argtypes = [f32]
        _lib.oracle_e2m1_value.restype = f32
        _lib.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
        _lib.oracle_e2m1_encode.restype = ctypes.c_uint8
        _lib.oracle_e2m1_encode.argtypes = [f32]
        _lib.oracle_fp4_quantize.argtypes = [P, i64, P, P, i32]
        _lib.oracle_fp4_dequantize.argtypes = [P, P, i64, P]
        _lib.oracle_index_score.argtypes = [P, P, P, P, i64, P]
        _lib.oracle_topk.restype = i32
        _lib.oracle_topk.argtypes = [P, i64, i32, P, P]
        _lib.oracle_block_keys.argtypes = [P, i64, P]
        _lib.oracle_block_pool.restype = i32
        _lib.oracle_block_pool.argtypes = [P, P, P, i64, i32, P]
        _lib.oracle_sparse_attn.argtypes = [P, P, P, P, i32, P, i32, f32, P, P]
        _lib.oracle_group_step.restype = i32
        _lib.oracle_group_step.argtypes = [i32, i32, P, i32, i32, i32, i32, i32, i32, P, i64,
                                           P, P, P, P, P, P, P, P, P, f32, P, P, P, P, P, i32, i32]
        _lib.oracle_fp8_quantize.argtypes = [P, i64, P]
        _lib.oracle_index_select.argtypes = [i32, i32, P, i64, P, P, P, i32, P, i32, P, P, i32]
        _lib.oracle_fp8_dequantize.argtypes = [P, i64, P]
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


# ---------------------------------------------------------------------------
# Scalar codecs
# ---------------------------------------------------------------------------
def e4m3_value(b: int) -> float:
    return lib().oracle_e4m3_value(int(b))


def e4m3_encode(v: float) -> int:
    return int(lib().oracle_e4m3_encode(float(v)))


def e2m1_value(n: int) -> float:
    return float(lib().oracle_e2m1_value(int(n)))


def e2m1_encode(v: float) -> int:
    return int(lib().oracle_e2m1_encode(float(v)))


# ---------------------------------------------------------------------------
# Array functions
# ---------------------------------------------------------------------------
def fp4_quantize(x_bf16: np.ndarray, threads: int = 1):
    """x: uint16 bf16 bits [..., 512] -> (codes uint8 [..., 256], scales uint8 [..., 32]).
    Rows are quantised independently, on up to `threads` host threads."""
    x = _c(x_bf16, np.uint16)
    rows = x.size // D
    codes = np.empty(x.shape[:-1] + (D // 2,), np.uint8)
    scales = np.empty(x.shape[:-1] + (D // GROUP,), np.uint8)
    lib().oracle_fp4_quantize(_p(x), rows, _p(codes), _p(scales), int(threads))
    return codes, scales


def fp8_quantize(x_bf16: np.ndarray) -> np.ndarray:
    """8-bit window rows: bf16 bits -> E4M3 bytes (RNE, saturating to +-448), same shape."""
    x = _c(x_bf16, np.uint16)
    out = np.empty(x.shape, np.uint8)
    lib().oracle_fp8_quantize(_p(x), x.size, _p(out))
    return out


def fp8_dequantize(b: np.ndarray) -> np.ndarray:
    """E4M3 bytes -> bf16 bits (exact), same shape."""
    b = _c(b, np.uint8)
    out = np.empty(b.shape, np.uint16)
    lib().oracle_fp8_dequantize(_p(b), b.size, _p(out))
    return out


def fp4_dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    rows = codes.size // (D // 2)
    out = np.empty(codes.shape[:-1] + (D,), np.uint16)
    lib().oracle_fp4_dequantize(_p(codes), _p(scales), rows, _p(out))
    return out


def index_score(qI: np.ndarray, w: np.ndarray, KI: np.ndarray, pos=None, n=None) -> np.ndarray:
    """One indexer query qI [4,128] bf16 bits, w [4] fp32, keys KI [T,128] bf16 bits.
    Scores keys pos[i] (or 0..n-1) -> fp32 [n]."""
    qI = _c(qI, np.uint16)
    w = _c(w, np.float32)
    KI = _c(KI, np.uint16)
    if pos is not None:
        pos = _c(pos, np.int32)
        n = pos.size
    elif n is None:
        n = KI.shape[0]
    out = np.empty(n, np.float32)
    lib().oracle_index_score(_p(qI), _p(w), _p(KI), _p(pos), int(n), _p(out))
    return out


def topk(scores: np.ndarray, k: int, map_=None):
    """Exact Top-k of a score row -> (idx int32 [k] ascending, -1 padded; count)."""
    s = _c(scores, np.float32)
    m = None if map_ is None else _c(map_, np.int32)
    out = np.empty(k, np.int32)
    cnt = lib().oracle_topk(_p(s), s.size, int(k), _p(m), _p(out))
    return out, cnt


def index_select(KI, qI, w, T, k: int, *, ratio=1, q_pos=None, threads=1):
    """Flat Top-k of every query row of a batch, as a flat Full layer selects: KI [B,cap,128] bf16
    bits, qI [B,Nq,4,128] bf16 bits, w [B,Nq,4] fp32, T [B] entries present; query i of sequence b
    at q_pos[b,i] (or ratio*T_b - Nq + i).  Returns (idx int32 [B,Nq,k] ascending, -1 padded;
    n_sel int32 [B,Nq])."""
    KI = _c(KI, np.uint16)
    qI = _c(qI, np.uint16)
    w = _c(w, np.float32)
    B, cap = KI.shape[0], KI.shape[1]
    Nq = qI.shape[1]
    T = _c(T, np.int64)
    qp = None if q_pos is None else _c(q_pos, np.int32)
    idx = np.empty((B, Nq, k), np.int32)
    n_sel = np.empty((B, Nq), np.int32)
    lib().oracle_index_select(B, Nq, _p(T), cap, _p(KI), _p(qI), _p(w), int(ratio), _p(qp), int(k), _p(idx),
                              _p(n_sel), int(threads))
    return idx, n_sel


def block_keys(KI: np.ndarray) -> np.ndarray:
    KI = _c(KI, np.uint16)
    T = KI.shape[0]
    out = np.zeros((max(T // BLOCK, 0), DI), np.uint16)
    lib().oracle_block_keys(_p(KI), T, _p(out))
    return out


def block_pool(qI, w, bkeys, n_blocks: int, keep: int):
    qI = _c(qI, np.uint16)
    w = _c(w, np.float32)
    bkeys = _c(bkeys, np.uint16)
    pool = np.full(keep * BLOCK, -1, np.int32)
    n = lib().oracle_block_pool(_p(qI), _p(w), _p(bkeys), int(n_blocks), int(keep), _p(pool))
    return pool, n


def sparse_attn(q, codes, scales, idx, swa_rows, softmax_scale: float):
    """One query: q [16,512] bf16 bits; codes/scales of one sequence's cache; idx [k];
    swa_rows [n,512] bf16 bits -> (out fp64 [16,512], lse fp64 [16])."""
    q = _c(q, np.uint16)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    idx = _c(idx, np.int32)
    swa_rows = _c(swa_rows, np.uint16).reshape(-1, D)
    out = np.empty((H, D), np.float64)
    lse = np.empty(H, np.float64)
    lib().oracle_sparse_attn(_p(q), _p(codes), _p(scales), _p(idx), idx.size, _p(swa_rows),
                             swa_rows.shape[0], float(softmax_scale), _p(out), _p(lse))
    return out, lse


def group_step(modes, T, codes, scales, KI, q, qI, w, swa, swa_len, *, Nq=1, K=512, W=128,
               ratio=1, hierarchical=False, keep=2048, q_pos=None, softmax_scale=None,
               threads=1, swa_fp8=False):
    """One layer group over a batch.  Shapes: codes [B,cap,256], scales [B,cap,32],
    KI [B,cap,128]; q [L,B,Nq,16,512]; qI [L,B,Nq,4,128]; w [L,B,Nq,4];
    swa [L,B,W-1+Nq,512] (bf16 bits, or E4M3 bytes when swa_fp8); T and swa_len [B].
    Returns dict of out (fp64), lse, idx, pool, pool_len."""
    modes = _c(modes, np.int32)
    L = modes.size
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    KI = _c(KI, np.uint16)
    B, cap = codes.shape[0], codes.shape[1]
    T = _c(T, np.int64)
    q = _c(q, np.uint16)
    qI = _c(qI, np.uint16)
    w = _c(w, np.float32)
    swa = _c(swa, np.uint8 if swa_fp8 else np.uint16)
    swa_len = _c(swa_len, np.int32)
    qp = None if q_pos is None else _c(q_pos, np.int32)
    if softmax_scale is None:
        softmax_scale = float(np.float32(1.0 / np.sqrt(D)))
    out = np.empty((L, B, Nq, H, D), np.float64)
    lse = np.empty((L, B, Nq, H), np.float64)
    idx = np.empty((L, B, Nq, K), np.int32)
    pool = np.full((B, Nq, keep * BLOCK), -1, np.int32) if hierarchical else None
    pool_len = np.zeros((B, Nq), np.int32) if hierarchical else None
    rc = lib().oracle_group_step(B, L, _p(modes), Nq, K, W, ratio, int(bool(hierarchical)), keep,
                                 _p(T), cap, _p(codes), _p(scales), _p(KI), _p(qp), _p(q), _p(qI),
                                 _p(w), _p(swa), _p(swa_len), float(softmax_scale), _p(out),
                                 _p(lse), _p(idx), _p(pool), _p(pool_len), int(threads), int(bool(swa_fp8)))
    if rc != 0:
        raise ValueError("oracle_group_step: bad arguments")
    return {"out": out, "lse": lse, "idx": idx, "pool": pool, "pool_len": pool_len}

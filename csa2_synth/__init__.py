"""Seeded synthetic inputs for the CSA2 step, shared by the oracle tests, the GPU
tests and the benchmark.

This module holds none of the method's arithmetic: it only draws numbers and
formats them as the storage types the step consumes (bf16 bit patterns, fp32).
Every tensor is drawn from its own stream, keyed by (seed, tensor id, index),
where index is normally the sequence number.  A single sequence of a large
workload can therefore be regenerated on the host without drawing the others,
which is how full-size parity tests obtain oracle inputs for sampled sequences.

Host draws use numpy's PCG64 generator seeded with the key triple and its
float32 standard normal sampler; values are then rounded to bf16 with
round-to-nearest-even.  Large device-resident fills (benchmark sizes) use
torch's CUDA Philox generator seeded from the same key; those values follow the
same N(0, 1) law but are different numbers, so a parity test that samples a
sequence overwrites that sequence with the host draw before running.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# Tensor ids (part of the stream key).  Per-layer tensors add the layer number.
# ---------------------------------------------------------------------------
T_KI = 1            # cached indexer keys  [T, 128] bf16
T_KV = 2            # main KV latent rows  [T, 512] bf16 (quantised to FP4 by the step)
T_QI = 100          # indexer queries      [Nq, 4, 128] bf16      (+ layer)
T_W = 200           # indexer head weights [Nq, 4] fp32           (+ layer)
T_Q = 300           # main queries         [Nq, 16, 512] bf16     (+ layer)
T_SWA = 400         # sliding-window rows  [W - 1 + Nq, 512] bf16 (+ layer)
T_X = 500           # rows to quantise (FP4 round-trip workload)
T_XMASK = 501       # outlier mask draw for T_X
T_KV_NEW = 600      # new main-KV rows appended by a decode step
T_KI_NEW = 601      # new indexer-key rows appended by a decode step

# Seeds per workload, by workload name.
SEEDS = {
    "full_layer_decode_b1_t4096": 0,
    "fp4_roundtrip_64x8192x512": 1,
    "decode_group_1f3r_b64_t131072": 0,
    "prefill_group_1f5r_ratio2_q2048": 3,
    "hier_decode_b8_t1m": 4,
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even) and return
    the 16-bit patterns as uint16.  Inputs are finite."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u >> 16) & np.uint32(1)
    r += np.uint32(0x7FFF)
    r += u                       # finite inputs: no carry out of 32 bits
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 values (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int, tensor_id: int, index: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(tensor_id), int(index)])


def normal_f32(seed: int, tensor_id: int, index: int, shape) -> np.ndarray:
    """N(0, 1) float32 draws for one (seed, tensor, index) stream."""
    return _rng(seed, tensor_id, index).standard_normal(shape, dtype=np.float32)


def normal_bf16(seed: int, tensor_id: int, index: int, shape, chunk_elems: int = 1 << 22) -> np.ndarray:
    """N(0, 1) draws rounded to bf16, as uint16 bit patterns.  The same numbers as rounding
    normal_f32(...) (successive draws continue one stream), drawn and rounded chunk by chunk so
    that a large tensor holds only its bf16 result and one small fp32 temporary."""
    g = _rng(seed, tensor_id, index)
    out = np.empty(shape, np.uint16)
    flat = out.reshape(-1)
    buf = np.empty(min(chunk_elems, max(flat.size, 1)), np.float32)
    for s in range(0, flat.size, buf.size):
        n = min(buf.size, flat.size - s)
        g.standard_normal(out=buf[:n], dtype=np.float32)
        flat[s:s + n] = f32_to_bf16_bits(buf[:n])
    return out


def outlier_bf16(seed: int, tensor_id: int, index: int, shape,
                 frac: float = 0.01, mult: float = 20.0) -> np.ndarray:
    """N(0, 1) draws in which each entry independently (Bernoulli(frac), drawn
    from the same stream after the normals) is multiplied by `mult`, then
    rounded to bf16."""
    g = _rng(seed, tensor_id, index)
    x = g.standard_normal(shape, dtype=np.float32)
    m = g.random(shape, dtype=np.float32) < frac
    x = np.where(m, x * np.float32(mult), x).astype(np.float32)
    return f32_to_bf16_bits(x)


def integer_bf16(seed: int, tensor_id: int, index: int, shape, lo: int, hi: int) -> np.ndarray:
    """Uniform integers in [lo, hi] stored as bf16 (exact for |v| <= 256).
    Used by tests whose dot products must be exact in any summation order."""
    v = _rng(seed, tensor_id, index).integers(lo, hi + 1, size=shape).astype(np.float32)
    return f32_to_bf16_bits(v)


# ---------------------------------------------------------------------------
# Device fills (benchmark-sized tensors); torch is imported lazily so that the
# host generators above work without it.
# ---------------------------------------------------------------------------
def device_normal_bf16(shape, seed: int, tensor_id: int, device="cuda", chunk_elems=1 << 28):
    """Fill a bf16 device tensor with N(0, 1) draws from torch's CUDA generator,
    seeded from (seed, tensor_id).  Generated in chunks to bound the fp32
    temporary."""
    import torch
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) << 20) ^ (int(tensor_id) * 0x9E3779B1 & 0xFFFFF))
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        flat[s:e].copy_(torch.randn(e - s, generator=g, device=device, dtype=torch.float32))
    return out


def device_outlier_bf16(shape, seed: int, tensor_id: int, frac=0.01, mult=20.0, device="cuda",
                        chunk_elems=1 << 28):
    """Device analogue of `outlier_bf16` (different numbers, same law)."""
    import torch
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) << 20) ^ (int(tensor_id) * 0x9E3779B1 & 0xFFFFF))
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        x = torch.randn(e - s, generator=g, device=device, dtype=torch.float32)
        m = torch.rand(e - s, generator=g, device=device, dtype=torch.float32) < frac
        flat[s:e].copy_(torch.where(m, x * mult, x))
    return out

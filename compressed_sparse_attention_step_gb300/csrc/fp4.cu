// FP4 main-KV codec: E2M1 codes with one E4M3 scale per 16 channels, NVFP4 without the global
// scale (ai-maestro.online "DeepSeek AI released DeepSeek-V4.1-Flash with 1M context, FP4",
// section "FP4 KV, Bounded Replay, and other extensions").  Also the plain row-append copy, the
// decode append in one launch (new KV rows quantised, new indexer-K rows copied, the step's
// counters cleared), the 8-bit window encoder and the block-key builder of the hierarchical
// indexer.
//
// All kernels here stream: one thread per 16-channel group (32 B of bf16 in, 8 B of codes and
// 1 B of scale out), so a warp covers one 512-channel row with fully coalesced accesses.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "attn_common.cuh"

namespace csa2 {
namespace {

// E4M3 (FN) byte -> fp32 value (exact).  Scale bytes are never NaN (encoded with satfinite).
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  const float v = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : float(m) * 0.001953125f;
  return (b & 0x80u) ? -v : v;
}

// Quantise one 16-channel group held as 8 packed bf16 pairs.
//
// The E2M1 code of q = fp32(x / s) under round-to-nearest-even is the number of midpoints
// {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5} that |q| passes, where a midpoint between codes c and
// c+1 counts on equality only when c+1 is even (ties to the even mantissa); magnitudes above 6
// saturate to code 7.  The comparison is done as |x| against midpoint * s instead of dividing:
// each product has at most 3 + 4 significant bits, so it is exact in fp32, and x (8 significant
// bits) either equals a product or differs from it by at least 2^-9 of its size, far more than
// the 2^-24 rounding of the quotient.  Hence |x| > m*s <=> fp32(|x|/s) > m and equality holds
// exactly when the quotient is the tie, which makes the codes bit-identical to dividing.  The
// midpoints increase, so the count is found by a three-level search: 4 [|x| >= 1.75 s], then
// 2 [|x| >= 3.5 s or 0.75 s], then [|x| > the lower midpoint of the remaining pair] (the midpoints
// taken with >= are exactly those whose upper code is even).
__device__ __forceinline__ void quantize_group(const uint32_t (&wv)[8], uint32_t& lo, uint32_t& hi,
                                               uint32_t& sb) {
  uint32_t amax = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = max(amax, max(wv[i] & 0x7FFFu, (wv[i] >> 16) & 0x7FFFu));
  const float s32 = __fdiv_rn(__uint_as_float(amax << 16), 6.0f);
  sb = __nv_cvt_float_to_fp8(s32, __NV_SATFINITE, __NV_E4M3);
  const float s = e4m3_value(sb);
  lo = 0u;
  hi = 0u;
  if (s > 0.0f) {
    // the midpoints m s as bf16 pairs: each has at most 3 + 4 significant bits, so it is exact in
    // bf16, and as |x| is a bf16 value the pairwise bf16 comparisons decide exactly as fp32 ones
    // (s >= 2^-9 keeps every midpoint normal, so a subnormal |x| compares the same either way)
    auto pair = [&](float m) {
      const uint32_t bits = __float_as_uint(m * s) >> 16;
      return bits | (bits << 16);
    };
    auto bf2 = [](uint32_t u) { return *reinterpret_cast<const __nv_bfloat162*>(&u); };
    const uint32_t T0 = pair(0.25f), T1 = pair(0.75f), T2 = pair(1.25f), T3 = pair(1.75f);
    const uint32_t T4 = pair(2.5f), T5 = pair(3.5f), T6 = pair(5.0f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // channels 2 i (low half) and 2 i + 1 (high half)
      const uint32_t m2 = wv[i] & 0x7FFF7FFFu;
      const uint32_t b2 = __hge2_mask(bf2(m2), bf2(T3));
      const uint32_t b1 = __hge2_mask(bf2(m2), bf2((T5 & b2) | (T1 & ~b2)));
      const uint32_t tl = (((T6 & b1) | (T4 & ~b1)) & b2) | (((T2 & b1) | (T0 & ~b1)) & ~b2);
      const uint32_t b0 = __hgt2_mask(bf2(m2), bf2(tl));
      const uint32_t c = (b2 & 0x00040004u) | (b1 & 0x00020002u) | (b0 & 0x00010001u) |
                         ((wv[i] >> 12) & 0x00080008u);  // signs of x
      const uint32_t byte = (c & 0xFu) | ((c >> 12) & 0xF0u);
      if (i < 4) lo |= byte << (8 * i);
      else hi |= byte << (8 * (i - 4));
    }
  }
}

// One 16-value group (gid = row * 32 + group) of the rows being appended: FP4 codes and its scale.
__device__ __forceinline__ void quantize_append_group(const uint16_t* __restrict__ x, int64_t gid, int n_new,
                                                      uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                                      int64_t cap, const int32_t* __restrict__ offsets,
                                                      int offset_bias, unsigned int* flags) {
  const int64_t row = gid >> 5;
  const int g = int(gid & 31);
  // rows fit in 32 bits (2^32 rows of 1 KiB would be 4 TiB of input): a 32-bit division
  const uint32_t b32 = uint32_t(row) / uint32_t(n_new);
  const int64_t b = b32, r = int64_t(uint32_t(row) - b32 * uint32_t(n_new));
  const int64_t pos = (offsets ? int64_t(offsets[b]) + offset_bias : 0) + r;
  if (pos < 0 || pos >= cap) {
    if (g == 0) atomicOr(flags, CSA2_FLAG_APPEND_OOB);
    return;
  }
  const uint16_t* src = x + row * CSA2_D + g * CSA2_GROUP;
  const uint4 v0 = ld_stream16(src), v1 = ld_stream16(src + 8);
  const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  uint32_t lo, hi, sb;
  quantize_group(wv, lo, hi, sb);
  const int64_t crow = b * cap + pos;
  *reinterpret_cast<uint2*>(codes + crow * CSA2_CODE_BYTES + g * 8) = make_uint2(lo, hi);
  scales[crow * CSA2_SCALE_BYTES + g] = uint8_t(sb);
}

// 16 bytes (vector v of row `row`) of the rows being appended: dst row (lens[b] - n_new + r) of
// sequence b <- src row r of sequence b.
__device__ __forceinline__ void copy_append_vec(const uint16_t* __restrict__ src, int64_t row, int v, int n_new,
                                                int row_vecs, uint16_t* __restrict__ dst, int64_t cap,
                                                const int32_t* __restrict__ lens, unsigned int* flags) {
  const int64_t b = row / n_new, r = row - b * n_new;
  const int64_t pos = int64_t(lens[b]) - n_new + r;
  if (pos < 0 || pos >= cap) {
    if (v == 0) atomicOr(flags, CSA2_FLAG_APPEND_OOB);
    return;
  }
  const uint4 val = reinterpret_cast<const uint4*>(src)[row * row_vecs + v];
  reinterpret_cast<uint4*>(dst)[(b * cap + pos) * row_vecs + v] = val;
}

__global__ void __launch_bounds__(256) fp4_quantize_kernel(
    const uint16_t* __restrict__ x, int64_t n_groups, int n_new, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales, int64_t cap, const int32_t* __restrict__ offsets, int offset_bias,
    unsigned int* flags) {
  pdl_wait();
  pdl_trigger();
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= n_groups) return;
  quantize_append_group(x, gid, n_new, codes, scales, cap, offsets, offset_bias, flags);
}

// The decode append in one launch: threads [0, n_groups) quantise the new main-KV rows, the next
// n_vecs copy the new indexer-K rows (16 bytes each), the next n_zero clear 16 bytes each of
// `zero` (a step's counters, which must start at zero), and the last n_bk refresh the keys of the
// blocks the append completes (as block_keys_kernel with only_new, bps blocks per sequence, 16
// threads of 8 channels per block): a block's rows from before this step are read from the cache,
// its new rows from ki_new itself, so nothing this launch writes is read, and the sum runs in the
// same row order.
__global__ void __launch_bounds__(256) append_kernel(const uint16_t* __restrict__ kv_new,
                                                     const uint16_t* __restrict__ ki_new, int64_t n_groups,
                                                     int64_t n_vecs, int n_new, int ki_vecs,
                                                     uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                                     uint16_t* __restrict__ KI, int64_t cap,
                                                     const int32_t* __restrict__ lens, uint4* __restrict__ zero,
                                                     int64_t n_zero, uint16_t* __restrict__ bkeys, int64_t bps,
                                                     int64_t n_bk, unsigned int* flags) {
  pdl_wait();
  pdl_trigger();
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid < n_groups) {
    quantize_append_group(kv_new, gid, n_new, codes, scales, cap, lens, -n_new, flags);
  } else if (gid - n_groups < n_vecs) {
    const int64_t q = gid - n_groups, row = q / ki_vecs;
    copy_append_vec(ki_new, row, int(q - row * ki_vecs), n_new, ki_vecs, KI, cap, lens, flags);
  } else if (gid - n_groups - n_vecs < n_zero) {
    zero[gid - n_groups - n_vecs] = make_uint4(0u, 0u, 0u, 0u);
  } else if (gid - n_groups - n_vecs - n_zero < n_bk) {
    const int64_t q = gid - n_groups - n_vecs - n_zero;
    const int sl = int(q & 15);
    const int64_t tb = q >> 4, b = tb / bps;
    const int64_t lb = lens[b], T = min(lb, cap), first_new = lb - n_new;
    const int64_t j = tb - b * bps + max(int64_t(0), (T - n_new) / CSA2_BLOCK);
    if (j >= T / CSA2_BLOCK) return;
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.0f;
#pragma unroll
    for (int i = 0; i < CSA2_BLOCK; ++i) {
      const int64_t p = j * CSA2_BLOCK + i;
      const uint16_t* src = p >= first_new ? ki_new + ((b * n_new + (p - first_new)) * CSA2_DI + sl * 8)
                                           : KI + ((b * cap + p) * CSA2_DI + sl * 8);
      const uint4 v = *reinterpret_cast<const uint4*>(src);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        acc[2 * c] = __fadd_rn(acc[2 * c], bf16lo(wv[c]));
        acc[2 * c + 1] = __fadd_rn(acc[2 * c + 1], bf16hi(wv[c]));
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
      o[c] = pack_bf16x2(__fmul_rn(acc[2 * c], 0.125f), __fmul_rn(acc[2 * c + 1], 0.125f));
    *reinterpret_cast<uint4*>(bkeys + ((b * (cap / CSA2_BLOCK) + j) * CSA2_DI + sl * 8)) =
        make_uint4(o[0], o[1], o[2], o[3]);
  }
}

__global__ void __launch_bounds__(256) zero_kernel(uint4* __restrict__ p, int64_t n16) {
  pdl_wait();
  pdl_trigger();
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n16) p[i] = make_uint4(0u, 0u, 0u, 0u);
}

// One 16-channel group per thread.  The codes go through the hardware E2M1 -> f16x2 conversion and
// one f16x2 multiply by the group's scale (E4M3 -> f16x2, also exact): the product of a code (at
// most 2 significant bits) and a scale (at most 4) has at most 6 significant bits and lies in f16's
// normal range (2^-10 .. 2688) or is a signed zero, so the f16 product is exact, and so are its
// widening to fp32 and its rounding to bf16.  A code of -0 gives -0 (bf16 0x8000).
__global__ void __launch_bounds__(256) fp4_dequantize_kernel(const uint8_t* __restrict__ codes,
                                                             const uint8_t* __restrict__ scales,
                                                             int64_t n_groups,
                                                             uint16_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= n_groups) return;
  const int64_t row = gid >> 5;
  const int g = int(gid & 31);
  const uint2 c = __ldcs(reinterpret_cast<const uint2*>(codes + row * CSA2_CODE_BYTES + g * 8));
  const uint32_t sb = scales[row * CSA2_SCALE_BYTES + g];
  const __half2 sc = attn::bits_h2(attn::e4m3x2_to_f16x2(uint16_t(sb | (sb << 8))));
  uint32_t o[8];
  const uint32_t words[2] = {c.x, c.y};
#pragma unroll
  for (int wi = 0; wi < 2; ++wi) {
    uint32_t f[4];
    attn::e2m1x8_to_f16x2x4(words[wi], f[0], f[1], f[2], f[3]);  // channels 8 wi + 2 j (low), + 1 (high)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 v = __hmul2(attn::bits_h2(f[j]), sc);
      const __nv_bfloat162 bv = __floats2bfloat162_rn(__low2float(v), __high2float(v));
      o[4 * wi + j] = *reinterpret_cast<const uint32_t*>(&bv);
    }
  }
  uint4* dst = reinterpret_cast<uint4*>(out + row * CSA2_D + g * CSA2_GROUP);
  __stcs(dst, make_uint4(o[0], o[1], o[2], o[3]));
  __stcs(dst + 1, make_uint4(o[4], o[5], o[6], o[7]));
}

// 8-bit window rows (kongchang.com "DeepSeek V4.1 Flash Deep Dive", section "Compressed Absorption
// Attention (2nd Gen)": the sliding window is kept in 8-bit precision): every bf16 value to E4M3FN
// with round-to-nearest-even, saturating to +-448, by the hardware conversion; 8 values per thread.
__global__ void __launch_bounds__(256) fp8_quantize_kernel(const uint16_t* __restrict__ x, int64_t n,
                                                           uint8_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t i = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) * 8;
  if (i >= n) return;
  auto cvt2 = [](float lo, float hi) -> uint32_t {  // two E4M3 bytes, lo's in the low byte
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
  };
  if (i + 8 <= n) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + i));
    const uint32_t o0 = cvt2(bf16lo(v.x), bf16hi(v.x)) | (cvt2(bf16lo(v.y), bf16hi(v.y)) << 16);
    const uint32_t o1 = cvt2(bf16lo(v.z), bf16hi(v.z)) | (cvt2(bf16lo(v.w), bf16hi(v.w)) << 16);
    *reinterpret_cast<uint2*>(out + i) = make_uint2(o0, o1);
  } else {
    for (int64_t j = i; j < n; ++j) out[j] = uint8_t(cvt2(bf16f(x[j]), 0.0f) & 0xFFu);
  }
}

// dst row (lens[b] - n_new + r) of sequence b <- src row r of sequence b; 16 B per thread.
__global__ void __launch_bounds__(256) copy_rows_append_kernel(const uint16_t* __restrict__ src,
                                                               int B, int n_new, int row_vecs,
                                                               uint16_t* __restrict__ dst,
                                                               int64_t cap,
                                                               const int32_t* __restrict__ lens,
                                                               unsigned int* flags) {
  pdl_wait();
  pdl_trigger();
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t total = int64_t(B) * n_new * row_vecs;
  if (gid >= total) return;
  const int64_t row = gid / row_vecs;
  copy_append_vec(src, row, int(gid - row * row_vecs), n_new, row_vecs, dst, cap, lens, flags);
}

// Block keys: key of block j = bf16_RNE(0.125 * sum_{i<8} KI[8j+i]) with the sum in token order
// in fp32 (ai-maestro "Compressed Sparse Attention 2": blocks of eight tokens).  One thread per
// (sequence, block, 8-channel slice).  With only_new, just the blocks completed by the last
// n_new appended rows: j in [floor((lens-n_new)/8), floor(lens/8)).
__global__ void __launch_bounds__(256) block_keys_kernel(const uint16_t* __restrict__ KI, int B,
                                                         int64_t cap, const int32_t* __restrict__ lens,
                                                         uint16_t* __restrict__ bkeys,
                                                         int64_t blocks_per_seq, int only_new,
                                                         int n_new) {
  pdl_wait();
  pdl_trigger();
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t total = int64_t(B) * blocks_per_seq * 16;
  if (gid >= total) return;
  const int sl = int(gid & 15);
  const int64_t t = gid >> 4;
  const int64_t b = t / blocks_per_seq;
  int64_t j = t - b * blocks_per_seq;
  const int64_t T = min(int64_t(lens[b]), cap);
  const int64_t nb = T / CSA2_BLOCK;
  if (only_new) j += max(int64_t(0), (T - n_new) / CSA2_BLOCK);
  if (j >= nb) return;
  float acc[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) acc[c] = 0.0f;
#pragma unroll
  for (int i = 0; i < CSA2_BLOCK; ++i) {
    const uint4 v = *reinterpret_cast<const uint4*>(KI + ((b * cap + j * CSA2_BLOCK + i) * CSA2_DI + sl * 8));
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      acc[2 * c] = __fadd_rn(acc[2 * c], bf16lo(wv[c]));
      acc[2 * c + 1] = __fadd_rn(acc[2 * c + 1], bf16hi(wv[c]));
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int c = 0; c < 4; ++c)
    o[c] = pack_bf16x2(__fmul_rn(acc[2 * c], 0.125f), __fmul_rn(acc[2 * c + 1], 0.125f));
  *reinterpret_cast<uint4*>(bkeys + ((b * (cap / CSA2_BLOCK) + j) * CSA2_DI + sl * 8)) =
      make_uint4(o[0], o[1], o[2], o[3]);
}

inline unsigned grid_for(int64_t threads, int block) { return unsigned((threads + block - 1) / block); }

}  // namespace

cudaError_t launch_fp4_quantize(const uint16_t* x, int B, int n_new, uint8_t* codes, uint8_t* scales,
                                int64_t cap, const int32_t* offsets, int offset_bias,
                                cudaStream_t st) {
  const int64_t n_groups = int64_t(B) * n_new * (CSA2_D / CSA2_GROUP);
  if (n_groups == 0) return cudaSuccess;
  unsigned int* flags = device_flags_ptr();
  if (!flags) return cudaErrorUnknown;
  return launch_pdl(fp4_quantize_kernel, grid_for(n_groups, 256), dim3(256), 0, st, x, n_groups, n_new, codes, scales,
                    cap, offsets, offset_bias, flags);
}

cudaError_t launch_fp8_quantize(const uint16_t* x, int64_t n, uint8_t* out, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  return launch_pdl(fp8_quantize_kernel, grid_for((n + 7) / 8, 256), dim3(256), 0, st, x, n, out);
}

cudaError_t launch_copy_rows_append(const uint16_t* src, int B, int n_new, int row_elems,
                                    uint16_t* dst, int64_t cap, const int32_t* lens, cudaStream_t st) {
  const int row_vecs = row_elems / 8;
  const int64_t total = int64_t(B) * n_new * row_vecs;
  if (total == 0) return cudaSuccess;
  unsigned int* flags = device_flags_ptr();
  if (!flags) return cudaErrorUnknown;
  return launch_pdl(copy_rows_append_kernel, grid_for(total, 256), dim3(256), 0, st, src, B, n_new, row_vecs, dst, cap,
                                                                lens, flags);
}

cudaError_t launch_append(const uint16_t* kv_new, const uint16_t* ki_new, int B, int n_new, uint8_t* codes,
                          uint8_t* scales, uint16_t* KI, int64_t cap, const int32_t* lens, void* zero,
                          size_t zero_bytes, uint16_t* block_keys, cudaStream_t st) {
  const int64_t n_groups = int64_t(B) * n_new * (CSA2_D / CSA2_GROUP);
  const int ki_vecs = CSA2_DI / 8;
  const int64_t n_vecs = int64_t(B) * n_new * ki_vecs;
  if ((reinterpret_cast<uintptr_t>(zero) | zero_bytes) & 15u) return cudaErrorInvalidValue;
  const int64_t n_zero = zero ? int64_t(zero_bytes / 16) : 0;
  const int64_t bps = int64_t(n_new / CSA2_BLOCK + 1);  // blocks the append may complete, per sequence
  const int64_t n_bk = block_keys ? int64_t(B) * bps * 16 : 0;
  if (n_groups + n_vecs + n_zero + n_bk == 0) return cudaSuccess;
  unsigned int* flags = device_flags_ptr();
  if (!flags) return cudaErrorUnknown;
  return launch_pdl(append_kernel, grid_for(n_groups + n_vecs + n_zero + n_bk, 256), dim3(256), 0, st, kv_new, ki_new,
                    n_groups, n_vecs, n_new, ki_vecs, codes, scales, KI, cap, lens, static_cast<uint4*>(zero), n_zero,
                    block_keys, bps, n_bk, flags);
}

cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t st) {
  if (bytes == 0) return cudaSuccess;
  if ((reinterpret_cast<uintptr_t>(p) | bytes) & 15u) return cudaMemsetAsync(p, 0, bytes, st);
  const int64_t n16 = int64_t(bytes / 16);
  return launch_pdl(zero_kernel, grid_for(n16, 256), dim3(256), 0, st, static_cast<uint4*>(p), n16);
}

cudaError_t launch_block_keys(const uint16_t* KI, int B, int64_t cap, const int32_t* lens,
                              uint16_t* block_keys, int only_new, int n_new, cudaStream_t st) {
  const int64_t bps = only_new ? int64_t(n_new / CSA2_BLOCK + 1) : cap / CSA2_BLOCK;
  const int64_t total = int64_t(B) * bps * 16;
  if (total == 0) return cudaSuccess;
  return launch_pdl(block_keys_kernel, grid_for(total, 256), dim3(256), 0, st, KI, B, cap, lens, block_keys, bps, only_new,
                                                          n_new);
}

}  // namespace csa2

// ------------------------------------------------------------------------------------------------
// C ABI
// ------------------------------------------------------------------------------------------------
namespace {
inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

extern "C" csa2_status csa2_fp4_quantize_append(const uint16_t* x, int B, int n_new, int d,
                                                uint8_t* codes, uint8_t* scales, int64_t cap,
                                                const int32_t* offsets, csa2_stream_t stream) {
  if (d != CSA2_D) return CSA2_ERR_UNSUPPORTED;
  if (B < 0 || n_new < 0 || cap < 0 || (!offsets && n_new > cap)) return CSA2_ERR_INVALID_ARG;
  if (int64_t(B) * n_new == 0) return CSA2_OK;
  if (!x || !codes || !scales || !al16(x) || !al16(codes) || !al16(scales)) return CSA2_ERR_INVALID_ARG;
  if (offsets && (reinterpret_cast<uintptr_t>(offsets) & 3u)) return CSA2_ERR_INVALID_ARG;
  return csa2::launch_fp4_quantize(x, B, n_new, codes, scales, cap, offsets, 0,
                                   reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? CSA2_OK
             : CSA2_ERR_CUDA;
}

extern "C" csa2_status csa2_fp8_quantize(const uint16_t* x, int64_t n, uint8_t* out, csa2_stream_t stream) {
  if (n < 0) return CSA2_ERR_INVALID_ARG;
  if (n == 0) return CSA2_OK;
  if (!x || !out || !al16(x) || !al16(out)) return CSA2_ERR_INVALID_ARG;
  return csa2::launch_fp8_quantize(x, n, out, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? CSA2_OK
                                                                                                   : CSA2_ERR_CUDA;
}

extern "C" csa2_status csa2_fp4_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t rows,
                                           int d, uint16_t* out, csa2_stream_t stream) {
  if (d != CSA2_D) return CSA2_ERR_UNSUPPORTED;
  if (rows < 0) return CSA2_ERR_INVALID_ARG;
  if (rows == 0) return CSA2_OK;
  if (!codes || !scales || !out || !al16(codes) || !al16(scales) || !al16(out)) return CSA2_ERR_INVALID_ARG;
  const int64_t n_groups = rows * (CSA2_D / CSA2_GROUP);
  const cudaError_t e = csa2::launch_pdl(csa2::fp4_dequantize_kernel, dim3(csa2::grid_for(n_groups, 256)), dim3(256), 0,
                                        reinterpret_cast<cudaStream_t>(stream), codes, scales, n_groups, out);
  if (e != cudaSuccess) return CSA2_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}

extern "C" csa2_status csa2_block_keys_build(const uint16_t* KI, int B, int64_t cap, const int32_t* lens,
                                             uint16_t* block_keys, csa2_stream_t stream) {
  if (B < 0 || cap < 0) return CSA2_ERR_INVALID_ARG;
  if (B == 0 || cap < CSA2_BLOCK) return CSA2_OK;
  if (!KI || !lens || !block_keys || !al16(KI) || !al16(block_keys)) return CSA2_ERR_INVALID_ARG;
  return csa2::launch_block_keys(KI, B, cap, lens, block_keys, 0, 0,
                                 reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? CSA2_OK
             : CSA2_ERR_CUDA;
}

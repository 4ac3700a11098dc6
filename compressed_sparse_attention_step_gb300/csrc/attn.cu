// Sparse attention of each query's 16 heads over its selected FP4 main-KV rows plus its
// sliding-window rows ("Every layer retains its own main Q and sliding-window key-value cache",
// ai-maestro.online "DeepSeek AI released DeepSeek-V4.1-Flash with 1M context, FP4", section
// "Compressed Sparse Attention 2"; the 128-token window: section "Causal Encoder-Decoder
// architecture"; E2M1 codes with an E4M3 scale per 16 channels: section "FP4 KV, Bounded Replay,
// and other extensions").  K = V = the dequantised row.
//
// Split-KV flash decoding.  A query's rows form a list of 32-row chunks (selected FP4 rows, then
// window rows); each CTA takes an equal share of consecutive chunks and keeps an online softmax
// (m, l, O) over them.  The selected positions of the share are staged in shared memory once and
// every row of the share is prefetched into L2 up front, so the double-buffered per-chunk copies
// wait on L2 rather than on HBM.  The last CTA of a query to finish (an atomic ticket) merges the
// splits in split order, so the result does not depend on which CTA finishes last.
//
// Inside a CTA, warp w (of 8) owns latent channels [64w, 64w+64) for everything: it gathers only
// its slice of each row (cp.async, 16-byte pieces, XOR-swizzled in shared memory), converts it to
// f16 in shared memory, keeps its Q slice in registers, and computes S_w = Q[:, slice] K[:, slice]^T
// and O[:, slice] += P V[:, slice]
// on tensor cores with the 16 heads as the M = 16 dimension of mma.m16n8k16 (f16 inputs, fp32
// accumulate).  The eight partial S are summed in a fixed order, so the only block-wide barriers
// are the two around each chunk's softmax.
//
// Tensor-core inputs are f16: an FP4 row is dequantised with the hardware E2M1 -> f16x2 and
// E4M3 -> f16x2 conversions and one f16 multiply by the scale, which is exact (at most 6 significant bits,
// magnitudes in [2^-10, 2688]); window rows and Q are converted from bf16, which is exact for
// magnitudes in [2^-14, 65504] (and rounds below); P is rounded to f16.
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"

namespace csa2 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kCH = 32;          // rows per chunk
constexpr int kPitchP = 40;      // f16 per row of the P tile (80 B: conflict-free ldmatrix)
constexpr int kPitchS = 36;      // floats per row of the partial-S tiles
constexpr int kMaxSplit = 32;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnSmem {
  uint16_t kv[2][kCH * CSA2_D];                    // f16, swizzled 16-byte chunks (kv[1] first stages Q)
  uint8_t raw_codes[2][kCH * CSA2_CODE_BYTES];     // swizzled 16-byte pieces
  uint8_t raw_scales[2][kCH * CSA2_SCALE_BYTES];
  uint16_t p[CSA2_H * kPitchP];
  float s[kWarps][CSA2_H * kPitchS];
  float corr[CSA2_H];
  float m_fin[CSA2_H];
  float l_fin[CSA2_H];
  int32_t pos[CSA2_MAX_ATTN_K];  // cache row of each selected slot of this split, -1 if empty
  int is_last;
};

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Four code bytes (eight E2M1 codes, the even channel in the low nibble of each byte) -> four f16x2
// (even channel in the low half), with the hardware conversion.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t& o0, uint32_t& o1, uint32_t& o2,
                                                  uint32_t& o3) {
  asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
      : "r"(w));
}
// Two E4M3 (FN) scale bytes (first in the low byte) -> f16x2 (first in the low half); exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}
// bf16x2 -> f16x2 (round to nearest)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t u) {
  return h2_bits(__floats2half2_rn(bf16lo(u), bf16hi(u)));
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) { return h2_bits(__floats2half2_rn(lo, hi)); }

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// byte offset of logical 16-byte chunk cc (0..63) of row r in a 1 KiB-per-row swizzled tile
__device__ __forceinline__ int swz(int r, int cc) { return r * (CSA2_D * 2) + ((cc ^ (r & 7)) << 4); }

__global__ void __launch_bounds__(kThreads, 2) sparse_attn_kernel(
    const uint16_t* __restrict__ q, int Nq, const uint8_t* __restrict__ codes,
    const uint8_t* __restrict__ scales, int64_t cap, const int32_t* __restrict__ idx,
    const int32_t* __restrict__ n_valid, int k, const uint16_t* __restrict__ swa,
    const int32_t* __restrict__ swa_len, int W, float scale_log2, uint16_t* __restrict__ out,
    float* __restrict__ lse, int n_split, float* __restrict__ ws, unsigned int* __restrict__ tickets,
    unsigned int* flags) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>(smem_raw);
  const int inst = blockIdx.y;
  const int split = blockIdx.x;
  const int b = inst / Nq, qi = inst - b * Nq;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int g = lane >> 2, tq = lane & 3;
  const int mat = lane >> 3, mrow = lane & 7;
  const uint32_t kv0 = smem_u32(sm.kv[0]);
  auto kv_addr = [&](int buf) -> uint32_t { return kv0 + uint32_t(buf) * uint32_t(kCH * CSA2_D * 2); };

  // ---- this split's chunks ------------------------------------------------------------------
  const int nfp4 = (k + kCH - 1) / kCH;
  const int nswa = swa ? (W + kCH - 1) / kCH : 0;
  const int nch = nfp4 + nswa;
  const int c_begin = split * nch / n_split, c_end = (split + 1) * nch / n_split;

  const int n_fp4_valid = min(k, n_valid ? max(n_valid[inst], 0) : k);
  const int32_t* irow = idx + int64_t(inst) * k;
  const int SW = W - 1 + Nq;
  const int swa_lo = swa ? SW - min(max(swa_len[b], 0), SW) : SW;
  const uint8_t* cbase = codes + int64_t(b) * cap * CSA2_CODE_BYTES;
  const uint8_t* sbase = scales + int64_t(b) * cap * CSA2_SCALE_BYTES;
  const uint16_t* swbase = swa ? swa + int64_t(b) * SW * CSA2_D : nullptr;

  // stage the cache rows of this split's selected slots and pull every row of the share into L2
  for (int slot = c_begin * kCH + t; slot < min(c_end, nfp4) * kCH; slot += kThreads) {
    int32_t p = slot < n_fp4_valid ? __ldg(irow + slot) : -1;
    if (int64_t(p) >= cap) {
      atomicOr(flags, CSA2_FLAG_INDEX_OOB);
      p = -1;
    }
    sm.pos[slot] = p < 0 ? -1 : p;
    if (p >= 0) {
      const uint8_t* cr = cbase + int64_t(p) * CSA2_CODE_BYTES;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(cr));
      asm volatile("prefetch.global.L2 [%0];" ::"l"(cr + 128));
      asm volatile("prefetch.global.L2 [%0];" ::"l"(sbase + int64_t(p) * CSA2_SCALE_BYTES));
    }
  }
  if (swa) {
    const int w0 = max(c_begin, nfp4) * kCH - nfp4 * kCH, w1 = min(c_end * kCH - nfp4 * kCH, W);
    for (int e = t; e < max(w1 - w0, 0) * 8; e += kThreads) {   // 8 lines of 128 B per row
      const int br = qi + w0 + (e >> 3);
      if (br >= swa_lo) asm volatile("prefetch.global.L2 [%0];" ::"l"(swbase + int64_t(br) * CSA2_D + (e & 7) * 64));
    }
  }
  __syncthreads();

  auto swa_row = [&](int wr) -> int {
    if (wr >= W) return -1;
    const int br = qi + wr;
    return br >= swa_lo ? br : -1;
  };
  auto row_valid = [&](int c, int r) -> bool {
    return (c < nfp4) ? sm.pos[c * kCH + r] >= 0 : swa_row((c - nfp4) * kCH + r) >= 0;
  };

  // gather of chunk c into buffer buf: this warp's channel slice only
  auto issue = [&](int c, int buf) {
    if (c < nfp4) {
#pragma unroll
      for (int it = 0; it < 2; ++it) {  // 32 rows x 2 pieces of 16 code bytes
        const int task = it * 32 + lane, r = task >> 1, piece = 2 * warp + (task & 1);
        const int32_t pos = sm.pos[c * kCH + r];
        if (pos >= 0)
          cp_async16(smem_u32(sm.raw_codes[buf] + r * CSA2_CODE_BYTES + ((piece ^ (r & 7)) << 4)),
                     cbase + int64_t(pos) * CSA2_CODE_BYTES + 16 * piece, 16);
      }
      const int32_t pos = sm.pos[c * kCH + lane];  // 4 scale bytes of row `lane`
      if (pos >= 0)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(
                         smem_u32(sm.raw_scales[buf] + lane * CSA2_SCALE_BYTES + 4 * warp)),
                     "l"(sbase + int64_t(pos) * CSA2_SCALE_BYTES + 4 * warp)
                     : "memory");
    } else {
      const int cw = c - nfp4;
#pragma unroll
      for (int it = 0; it < 8; ++it) {  // 32 rows x 8 pieces of 16 B (64 bf16)
        const int task = it * 32 + lane, r = task >> 3, cc = 8 * warp + (task & 7);
        const int br = swa_row(cw * kCH + r);
        const uint16_t* src = br >= 0 ? swbase + int64_t(br) * CSA2_D + 8 * cc : swa;
        cp_async16(kv_addr(buf) + swz(r, cc), src, br >= 0 ? 16 : 0);
      }
    }
  };

  // this warp's slice of chunk c -> f16 rows of the KV tile; empty FP4 rows become zeros
  auto convert = [&](int c, int buf) {
    uint8_t* kvb = reinterpret_cast<uint8_t*>(sm.kv[buf]);
    if (c < nfp4) {
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int task = it * 32 + lane, r = task >> 1, piece = 2 * warp + (task & 1);
        uint4 o[4];
        if (sm.pos[c * kCH + r] >= 0) {
          const uint4 cb = *reinterpret_cast<const uint4*>(sm.raw_codes[buf] + r * CSA2_CODE_BYTES +
                                                           ((piece ^ (r & 7)) << 4));
          const uint16_t s2 = *reinterpret_cast<const uint16_t*>(sm.raw_scales[buf] + r * CSA2_SCALE_BYTES + 2 * piece);
          const __half2 sab = bits_h2(e4m3x2_to_f16x2(s2));
          const __half2 sA = __low2half2(sab), sB = __high2half2(sab);
          const uint32_t words[4] = {cb.x, cb.y, cb.z, cb.w};
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            const __half2 sc = wi < 2 ? sA : sB;
            uint32_t f0, f1, f2, f3;
            e2m1x8_to_f16x2x4(words[wi], f0, f1, f2, f3);
            o[wi].x = h2_bits(__hmul2(bits_h2(f0), sc));
            o[wi].y = h2_bits(__hmul2(bits_h2(f1), sc));
            o[wi].z = h2_bits(__hmul2(bits_h2(f2), sc));
            o[wi].w = h2_bits(__hmul2(bits_h2(f3), sc));
          }
        } else {
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) o[wi] = make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) *reinterpret_cast<uint4*>(kvb + swz(r, 4 * piece + wi)) = o[wi];
      }
    } else {
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int task = it * 32 + lane, r = task >> 3, cc = 8 * warp + (task & 7);
        uint4* p = reinterpret_cast<uint4*>(kvb + swz(r, cc));
        uint4 v = *p;
        v.x = bf16x2_to_f16x2(v.x);
        v.y = bf16x2_to_f16x2(v.y);
        v.z = bf16x2_to_f16x2(v.z);
        v.w = bf16x2_to_f16x2(v.w);
        *p = v;
      }
    }
  };

  float oacc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.0f;
  float m_run = -INFINITY, l_run = 0.0f;  // softmax state of head (t >> 4), same in its 16 threads
  const int sh = t >> 4, sc2 = (t & 15) * 2;

  uint32_t qa[4][4];  // this warp's Q slice (16 heads x 64 channels) as four f16 A fragments
  if (c_begin < c_end) {
    // Q slice of this warp: 16 rows x 128 B of bf16, staged in kv[1] (free until chunk c_begin+1
    // is issued, and each warp touches only its own channel slice), converted to f16, then loaded
    // into registers
    const uint16_t* qrow = q + int64_t(inst) * CSA2_H * CSA2_D;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int task = it * 32 + lane, r = task >> 3, cc = 8 * warp + (task & 7);
      cp_async16(kv_addr(1) + swz(r, cc), qrow + r * CSA2_D + 8 * cc, 16);
    }
    cp_async_commit();
    issue(c_begin, 0);
    cp_async_commit();
    cp_async_wait<1>();
    __syncwarp();
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int task = it * 32 + lane, r = task >> 3, cc = 8 * warp + (task & 7);
      uint4* p = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(sm.kv[1]) + swz(r, cc));
      uint4 v = *p;
      v.x = bf16x2_to_f16x2(v.x);
      v.y = bf16x2_to_f16x2(v.y);
      v.z = bf16x2_to_f16x2(v.z);
      v.w = bf16x2_to_f16x2(v.w);
      *p = v;
    }
    __syncwarp();
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const int r = mrow + ((mat & 1) << 3);
      ldmatrix_x4(qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], kv_addr(1) + swz(r, 8 * warp + 2 * kk + (mat >> 1)));
    }
    __syncwarp();

    for (int c = c_begin; c < c_end; ++c) {
      const int buf = (c - c_begin) & 1;
      if (c + 1 < c_end) {
        issue(c + 1, buf ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncwarp();
      convert(c, buf);
      __syncwarp();
      // ---- S_w = Q[:, slice] K[:, slice]^T for the 32 rows ------------------------------------
      float sacc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.0f;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          const int kr = 16 * np + mrow + ((mat >> 1) << 3);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(b0, b1, b2, b3, kv_addr(buf) + swz(kr, 8 * warp + 2 * kk + (mat & 1)));
          mma_f16_16816(sacc[2 * np], qa[kk], b0, b1);
          mma_f16_16816(sacc[2 * np + 1], qa[kk], b2, b3);
        }
      }
      float* sw = sm.s[warp];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        *reinterpret_cast<float2*>(sw + g * kPitchS + 8 * nt + 2 * tq) = make_float2(sacc[nt][0], sacc[nt][1]);
        *reinterpret_cast<float2*>(sw + (g + 8) * kPitchS + 8 * nt + 2 * tq) = make_float2(sacc[nt][2], sacc[nt][3]);
      }
      __syncthreads();
      // ---- online softmax: thread t owns head sh, columns sc2, sc2+1 ---------------------------
      {
        float v[2];
        float vmax = -INFINITY;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int o = sh * kPitchS + sc2 + e;
          float x = sm.s[0][o];
#pragma unroll
          for (int w2 = 1; w2 < kWarps; ++w2) x += sm.s[w2][o];
          v[e] = row_valid(c, sc2 + e) ? x * scale_log2 : -INFINITY;
          vmax = fmaxf(vmax, v[e]);
        }
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
        const float m_new = fmaxf(m_run, vmax);
        float corr = 1.0f, p0 = 0.0f, p1 = 0.0f;
        if (m_new != -INFINITY) {
          corr = exp2f(m_run - m_new);
          p0 = exp2f(v[0] - m_new);
          p1 = exp2f(v[1] - m_new);
        }
        float rs = p0 + p1;
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) rs += __shfl_xor_sync(0xffffffffu, rs, off);
        l_run = l_run * corr + rs;
        m_run = m_new;
        *reinterpret_cast<uint32_t*>(sm.p + sh * kPitchP + sc2) = pack_f16x2(p0, p1);
        if ((t & 15) == 0) sm.corr[sh] = corr;
      }
      __syncthreads();
      // ---- O[:, slice] = corr * O + P V[:, slice] ---------------------------------------------
      {
        const float cr0 = sm.corr[g], cr1 = sm.corr[g + 8];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          oacc[nt][0] *= cr0;
          oacc[nt][1] *= cr0;
          oacc[nt][2] *= cr1;
          oacc[nt][3] *= cr1;
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          uint32_t pa[4];
          {
            const int r = mrow + ((mat & 1) << 3);
            ldmatrix_x4(pa[0], pa[1], pa[2], pa[3], smem_u32(sm.p + r * kPitchP + 16 * kk + ((mat >> 1) << 3)));
          }
#pragma unroll
          for (int np = 0; np < 4; ++np) {
            const int kr = 16 * kk + mrow + ((mat & 1) << 3);
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4_trans(b0, b1, b2, b3, kv_addr(buf) + swz(kr, 8 * warp + 2 * np + (mat >> 1)));
            mma_f16_16816(oacc[2 * np], pa, b0, b1);
            mma_f16_16816(oacc[2 * np + 1], pa, b2, b3);
          }
        }
      }
    }
  }

  if ((t & 15) == 0) {
    sm.m_fin[sh] = m_run;
    sm.l_fin[sh] = l_run;
  }
  __syncthreads();

  if (n_split == 1) {
    const float l0 = sm.l_fin[g], l1 = sm.l_fin[g + 8];
    const float i0 = l0 > 0.0f ? 1.0f / l0 : 0.0f, i1 = l1 > 0.0f ? 1.0f / l1 : 0.0f;
    uint16_t* orow = out + int64_t(inst) * CSA2_H * CSA2_D;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int ch = 64 * warp + 8 * nt + 2 * tq;
      *reinterpret_cast<uint32_t*>(orow + g * CSA2_D + ch) = pack_bf16x2(oacc[nt][0] * i0, oacc[nt][1] * i0);
      *reinterpret_cast<uint32_t*>(orow + (g + 8) * CSA2_D + ch) = pack_bf16x2(oacc[nt][2] * i1, oacc[nt][3] * i1);
    }
    if (lse && t < CSA2_H) {
      const float l = sm.l_fin[t];
      lse[int64_t(inst) * CSA2_H + t] = l > 0.0f ? (sm.m_fin[t] + log2f(l)) * kLn2 : -INFINITY;
    }
    return;
  }
  // ---- split partials, then the last CTA of this query merges them ------------------------------
  const int64_t instances = gridDim.y;
  float* po = ws + (int64_t(inst) * n_split + split) * (CSA2_H * CSA2_D);
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int ch = 64 * warp + 8 * nt + 2 * tq;
    *reinterpret_cast<float2*>(po + g * CSA2_D + ch) = make_float2(oacc[nt][0], oacc[nt][1]);
    *reinterpret_cast<float2*>(po + (g + 8) * CSA2_D + ch) = make_float2(oacc[nt][2], oacc[nt][3]);
  }
  float* mlb = ws + instances * n_split * (CSA2_H * CSA2_D);
  if (t < CSA2_H) {
    float* ml = mlb + (int64_t(inst) * n_split + split) * (2 * CSA2_H);
    ml[2 * t] = sm.m_fin[t];
    ml[2 * t + 1] = sm.l_fin[t];
  }
  __threadfence();
  __syncthreads();
  if (t == 0) sm.is_last = (atomicAdd(tickets + inst, 1u) == unsigned(n_split - 1));
  __syncthreads();
  if (!sm.is_last) return;
  __threadfence();
  // o = sum_j 2^(m_j - M) O_j / sum_j 2^(m_j - M) l_j, splits in order; thread: head t>>4, 32 channels
  {
    const int h = t >> 4, c0 = (t & 15) * 32;
    const float* ml = mlb + int64_t(inst) * n_split * (2 * CSA2_H);
    float M = -INFINITY;
    for (int j = 0; j < n_split; ++j) M = fmaxf(M, __ldcg(ml + j * 2 * CSA2_H + 2 * h));
    float L = 0.0f;
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
    if (M != -INFINITY) {
      for (int j = 0; j < n_split; ++j) {
        const float a = exp2f(__ldcg(ml + j * 2 * CSA2_H + 2 * h) - M);
        L += a * __ldcg(ml + j * 2 * CSA2_H + 2 * h + 1);
        const float4* pj = reinterpret_cast<const float4*>(ws + (int64_t(inst) * n_split + j) * (CSA2_H * CSA2_D) +
                                                           h * CSA2_D + c0);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const float4 x = __ldcg(pj + v);
          acc[4 * v] += a * x.x;
          acc[4 * v + 1] += a * x.y;
          acc[4 * v + 2] += a * x.z;
          acc[4 * v + 3] += a * x.w;
        }
      }
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    uint4* dst = reinterpret_cast<uint4*>(out + (int64_t(inst) * CSA2_H + h) * CSA2_D + c0);
#pragma unroll
    for (int v = 0; v < 4; ++v)
      dst[v] = make_uint4(pack_bf16x2(acc[8 * v] * inv, acc[8 * v + 1] * inv),
                          pack_bf16x2(acc[8 * v + 2] * inv, acc[8 * v + 3] * inv),
                          pack_bf16x2(acc[8 * v + 4] * inv, acc[8 * v + 5] * inv),
                          pack_bf16x2(acc[8 * v + 6] * inv, acc[8 * v + 7] * inv));
    if (lse && (t & 15) == 0) lse[int64_t(inst) * CSA2_H + h] = L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY;
  }
  if (t == 0) tickets[inst] = 0u;  // ready for the next launch
}

}  // namespace

// partial O and (m, l) of every split, then one ticket per query (zeroed before each launch)
size_t attn_ws_bytes(int64_t instances, int n_split) {
  if (n_split <= 1) return 0;
  return size_t(instances) * size_t(n_split) * (CSA2_H * CSA2_D + 2 * CSA2_H) * sizeof(float) +
         size_t(instances) * sizeof(unsigned int);
}

int attn_auto_split(int64_t instances, int k, int W) {
  const int nch = (k + kCH - 1) / kCH + (W + kCH - 1) / kCH;
  if (instances <= 0 || nch <= 0) return 1;
  const int64_t target = 2 * 152;  // two resident CTAs per SM
  int64_t s = (target + instances - 1) / instances;
  s = std::min<int64_t>(s, std::min(nch, kMaxSplit));
  return int(std::max<int64_t>(s, 1));
}

cudaError_t launch_sparse_attn(const uint16_t* q, int B, int Nq, const uint8_t* codes,
                               const uint8_t* scales, int64_t cap, const int32_t* idx,
                               const int32_t* n_valid, int k, const uint16_t* swa,
                               const int32_t* swa_len, int W, float softmax_scale, uint16_t* out,
                               float* lse, int n_split, float* ws, cudaStream_t st) {
  const int64_t instances = int64_t(B) * Nq;
  if (instances == 0) return cudaSuccess;
  unsigned int* flags = device_flags_ptr();
  if (!flags) return cudaErrorUnknown;
  const size_t smem = sizeof(AttnSmem);
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  unsigned int* tickets = nullptr;
  if (n_split > 1) {
    tickets = reinterpret_cast<unsigned int*>(ws + instances * n_split * (CSA2_H * CSA2_D + 2 * CSA2_H));
    cudaError_t e = cudaMemsetAsync(tickets, 0, size_t(instances) * sizeof(unsigned int), st);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid{unsigned(n_split), unsigned(instances), 1u};
  sparse_attn_kernel<<<grid, kThreads, smem, st>>>(q, Nq, codes, scales, cap, idx, n_valid, k, swa, swa_len,
                                                   W, scale_log2, out, lse, n_split, ws, tickets, flags);
  return cudaGetLastError();
}

}  // namespace csa2

extern "C" csa2_status csa2_sparse_attn_decode(const uint16_t* q, int B, int Nq, const uint8_t* codes,
                                               const uint8_t* scales, int64_t cap, const int32_t* idx,
                                               const int32_t* n_valid, int k, const uint16_t* swa,
                                               const int32_t* swa_len, int W, float softmax_scale,
                                               uint16_t* out, float* lse, int n_split, void* ws,
                                               size_t ws_bytes, csa2_stream_t stream) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (B < 0 || Nq < 0 || cap < 0 || k < 0 || k > CSA2_MAX_ATTN_K || n_split < 0 || n_split > csa2::kMaxSplit)
    return CSA2_ERR_INVALID_ARG;
  if (swa && (W < 1 || W > CSA2_MAX_W || !swa_len)) return CSA2_ERR_INVALID_ARG;
  if (!swa) W = 0;
  const int64_t instances = int64_t(B) * Nq;
  if (instances == 0) return CSA2_OK;
  if (instances > 65535) return CSA2_ERR_UNSUPPORTED;
  if (!q || !out || !al16(q) || !al16(out)) return CSA2_ERR_INVALID_ARG;
  if (k > 0 && (!codes || !scales || !idx || !al16(codes) || !al16(scales))) return CSA2_ERR_INVALID_ARG;
  if (swa && !al16(swa)) return CSA2_ERR_INVALID_ARG;
  const int ns = n_split ? n_split : csa2::attn_auto_split(instances, k, W);
  const size_t need = csa2::attn_ws_bytes(instances, ns);
  if (need && (!ws || ws_bytes < need || !al16(ws))) return CSA2_ERR_WORKSPACE;
  return csa2::launch_sparse_attn(q, B, Nq, codes, scales, cap, idx, n_valid, k, swa, swa_len, W,
                                  softmax_scale, out, lse, ns, static_cast<float*>(ws),
                                  reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? CSA2_OK
             : CSA2_ERR_CUDA;
}

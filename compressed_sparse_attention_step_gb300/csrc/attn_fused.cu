// Sparse attention of L layers (2..4) that attend the same selected rows, in one pass over those
// rows ("Reuse: takes the most recent Full layer's indices and skips the indexer", ai-maestro.online
// "DeepSeek AI released DeepSeek-V4.1-Flash with 1M context, FP4", section "Compressed Sparse
// Attention 2"; every layer keeps its own main Q and 128-token window: same section and "Causal
// Encoder-Decoder architecture").  K = V = the dequantised row; softmax over the union of a layer's
// selected rows and its window rows.
//
// The Full (or Reindex) layer and the Reuse layers after it read the same FP4 rows, so each 64-row
// FP4 tile is gathered and dequantised once for all L layers: S^T = K [Q_0; ..; Q_{L-1}]^T with
// N = 16 L columns (layer-major, 16 heads each), and O^T += V^T P^T with the same N.  Window tiles
// belong to one layer each (every layer has its own window cache) and run at N = 16 on that
// layer's columns.  Per CTA:
//   - a contiguous range of the instance's tiles: every layer's window tiles, then the FP4 tiles;
//   - the next FP4 tile's bytes are copied (cp.async) into a staging buffer while the current tile
//     is processed; window rows are loaded into registers before the operand buffer frees up;
//   - S^T on the tensor core (tcgen05.mma, M = 64 rows) split over kP issuing warps, each summing a
//     slice of the 512 channels into its own tensor-memory partial (independent chains);
//   - an online softmax per (layer, head) column on the summed partials, with lazy rescaling (a
//     column's offset moves only when a tile's maximum exceeds it by more than 2^8);
//   - O^T for all L layers stays in tensor memory (4 channel blocks x 16 L columns), zeroed once,
//     so every PV accumulates.
// Splits of an instance are merged by the last CTA to finish (one ticket per instance, all L
// layers), in split order.  Tensor memory (4 S partials or 8, plus O^T) takes all 512 columns for
// L = 4, so one CTA runs per SM.
//
// Operand types as in the single-layer kernel (attn.cu): FP4 tiles and 8-bit window tiles in f16
// (both exact), bf16 window tiles in bf16, fp32 accumulation; P rounded to the tile's type.
#include <cuda_fp16.h>

#include <algorithm>

#include "attn_common.cuh"

namespace csa2 {
namespace {
using namespace attn;

constexpr int kWinTiles = (CSA2_MAX_W + kRows - 1) / kRows;       // 2
constexpr int kFp4Tiles = (CSA2_MAX_ATTN_K + kRows - 1) / kRows;  // 8
constexpr int kMaxL = 4;
constexpr int kMaxTilesF = kMaxL * kWinTiles + kFp4Tiles;        // 16
constexpr uint32_t kTmemColsF = 512;
constexpr float kLazyF = 8.0f;

template <int L>
struct Cfg {
  static constexpr int kN = 16 * L;                     // columns of an FP4 tile: L layers x 16 heads
  static constexpr int kP = (L <= 2) ? 8 : 4;           // S^T partials (issuing warps)
  static constexpr uint32_t kOCol = uint32_t(kP * kN);  // O^T block i at kOCol + i kN
  static constexpr uint32_t kTileGroup = kRows * 128;   // 8 KiB per 64-channel group of a tile
  static constexpr uint32_t kTileOff = 0;
  static constexpr uint32_t kQGroup = uint32_t(kN) * 128u;  // Q: 8 groups x 16 L rows x 128 B
  static constexpr uint32_t kQOff = kTileOff + 8 * kTileGroup;
  static constexpr uint32_t kPOff = kQOff + 8 * kQGroup;     // P^T: 16 L rows x 128 B
  static constexpr uint32_t kRawOff = kPOff + uint32_t(kN) * 128u;
  static constexpr uint32_t kRawScOff = kRawOff + kRows * CSA2_CODE_BYTES;
  static constexpr uint32_t kMiscOff = kRawScOff + kRows * CSA2_SCALE_BYTES;
  static_assert(kOCol + 4 * kN <= kTmemColsF, "tensor memory");
};

struct MiscF {
  unsigned long long mbar_s, mbar_o;
  uint32_t tmem_base;
  int is_last;
  int32_t pos[kMaxTilesF][kRows];       // source row of each row of the CTA's tiles, -1 if empty
  float red[4][16 * kMaxL];             // per-quarter tile maxima, then (at the end) partial sums
  float m_run[2][16 * kMaxL];           // running offset per column, by parity
  float corr[16 * kMaxL];               // rescale factor of a column whose offset moved
  float l_fin[16 * kMaxL];              // final sum per column
};

template <int L>
constexpr size_t fused_smem() { return 1024 + Cfg<L>::kMiscOff + sizeof(MiscF); }

// 8 columns at column offset `off` of each of the P partials (stride `stride` columns), one wait.
template <int P>
__device__ __forceinline__ void tmem_ld8_parts(uint32_t taddr, uint32_t stride, float (&v)[P][8]) {
  uint32_t r[P][8];
#pragma unroll
  for (int p = 0; p < P; ++p)
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n"
                 : "=r"(r[p][0]), "=r"(r[p][1]), "=r"(r[p][2]), "=r"(r[p][3]), "=r"(r[p][4]), "=r"(r[p][5]),
                   "=r"(r[p][6]), "=r"(r[p][7])
                 : "r"(taddr + uint32_t(p) * stride)
                 : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int p = 0; p < P; ++p)
#pragma unroll
    for (int i = 0; i < 8; ++i) v[p][i] = __uint_as_float(r[p][i]);
}
// 16 columns of this warp's lane quarter (one wait), and their store back (one wait).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};\n\t"
      "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}

template <int L>
__global__ void __launch_bounds__(kThreads, 1) sparse_attn_fused_kernel(
    const __grid_constant__ AttnLayers layers, int Nq, const uint8_t* __restrict__ codes,
    const uint8_t* __restrict__ scales, int64_t cap, const int32_t* __restrict__ idx, int k,
    const int32_t* __restrict__ swa_len, int W, float scale_log2, int n_split, float* __restrict__ ws,
    unsigned int* __restrict__ tickets, unsigned int* flags, int win_fp8) {
  using C = Cfg<L>;
  constexpr int kN = C::kN, kP = C::kP;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // the selected positions may come from the kernel right before this one
  pdl_wait();
  pdl_trigger();
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  unsigned char* base = smem_raw + (base_s - raw_s);
  MiscF& ms = *reinterpret_cast<MiscF*>(base + C::kMiscOff);
  const uint32_t tile_s = base_s + C::kTileOff, q_s = base_s + C::kQOff, p_s = base_s + C::kPOff;
  const uint32_t mbar_s = smem_u32(&ms.mbar_s), mbar_o = smem_u32(&ms.mbar_o);

  const int inst = blockIdx.y, split = blockIdx.x;
  const int b = inst / Nq, qi = inst - b * Nq;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int quarter = warp & 3, half = warp >> 2;

  // ---- this split's tiles: layer l's window tiles at l nwin .. l nwin + nwin - 1, then FP4 tiles ----
  const bool has_win = layers.swa[0] != nullptr;
  const int nwin = has_win ? (W + kRows - 1) / kRows : 0;
  const int nwin_all = L * nwin;
  const int ntiles = nwin_all + (k + kRows - 1) / kRows;
  // splits cut the tiles by cost: a window tile (N = 16) is 4 units, an FP4 tile (N = 16 L) 4 + L; a
  // tile goes to the split its cost-prefix falls in
  auto cost = [&](int tile) { return tile < nwin_all ? 4 : 4 + L; };
  int total = 0;
  for (int tile = 0; tile < ntiles; ++tile) total += cost(tile);
  int t_begin = ntiles, t_end = ntiles;
  {
    int pre = 0;
    for (int tile = 0; tile < ntiles; ++tile) {
      const int s_of = int(int64_t(pre) * n_split / total);
      if (s_of == split && t_begin == ntiles) t_begin = tile;
      if (s_of > split) {
        t_end = tile;
        break;
      }
      pre += cost(tile);
    }
    if (t_begin > t_end) t_begin = t_end;
  }
  const int n_fp4_valid = k;
  const int SW = W - 1 + Nq;
  const int swa_lo = has_win ? SW - min(max(swa_len[b], 0), SW) : SW;
  auto live = [&](int tile) {
    if (tile < nwin_all) {
      const int wt = tile % nwin;
      return qi + min((wt + 1) * kRows, W) - 1 >= swa_lo;
    }
    return (tile - nwin_all) * kRows < n_fp4_valid;
  };
  int first_live = -1, last_live = -1;
  for (int tile = t_begin; tile < t_end; ++tile)
    if (live(tile)) {
      if (first_live < 0) first_live = tile;
      last_live = tile;
    }

  const int32_t* irow = idx + int64_t(inst) * k;
  const uint8_t* cbase = codes + int64_t(b) * cap * CSA2_CODE_BYTES;
  const uint8_t* sbase = scales + int64_t(b) * cap * CSA2_SCALE_BYTES;
  // window row of tile row r of window tile wt, or -1
  auto win_row = [&](int wt, int r) {
    const int wr = wt * kRows + r;
    return (wr < W && qi + wr >= swa_lo) ? qi + wr : -1;
  };
  auto swb16 = [&](int l) { return layers.swa[l] + int64_t(b) * SW * CSA2_D; };  // bf16 rows
  auto swb8 = [&](int l) {  // E4M3 rows of 512 B
    return reinterpret_cast<const uint8_t*>(layers.swa[l]) + int64_t(b) * SW * CSA2_D;
  };

  if (t < kN) {
    ms.m_run[0][t] = -INFINITY;
    ms.l_fin[t] = 0.0f;
  }
  if (first_live >= 0) {
    if (t == 0) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(mbar_s), "r"(kP) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(mbar_o), "r"(4) : "memory");
      asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 0) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(&ms.tmem_base)),
                   "r"(kTmemColsF)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
  }
  // ---- source rows of every tile of the split; FP4 rows and window rows pulled into L2 --------------
  for (int e = t; e < (t_end - t_begin) * kRows; e += kThreads) {
    const int tile = t_begin + e / kRows, r = e % kRows;
    int32_t p = -1;
    if (tile >= nwin_all) {
      const int slot = (tile - nwin_all) * kRows + r;
      if (slot < n_fp4_valid) {
        p = __ldg(irow + slot);
        if (int64_t(p) >= cap) {
          atomicOr(flags, CSA2_FLAG_INDEX_OOB);
          p = -1;
        }
        if (p >= 0) {
          const uint8_t* cr = cbase + int64_t(p) * CSA2_CODE_BYTES;
          asm volatile("prefetch.global.L2 [%0];" ::"l"(cr));
          asm volatile("prefetch.global.L2 [%0];" ::"l"(cr + 128));
          asm volatile("prefetch.global.L2 [%0];" ::"l"(sbase + int64_t(p) * CSA2_SCALE_BYTES));
        }
      }
    } else {
      const int l = tile / nwin, wt = tile % nwin;
      p = win_row(wt, r);
      if (p >= 0) {
        if (win_fp8) {
          const uint8_t* sr = swb8(l) + int64_t(p) * CSA2_D;
#pragma unroll
          for (int c = 0; c < 4; ++c) asm volatile("prefetch.global.L2 [%0];" ::"l"(sr + 128 * c));
        } else {
          const uint16_t* sr = swb16(l) + int64_t(p) * CSA2_D;
#pragma unroll
          for (int c = 0; c < 8; ++c) asm volatile("prefetch.global.L2 [%0];" ::"l"(sr + 64 * c));
        }
      }
    }
    ms.pos[tile - t_begin][r] = p < 0 ? -1 : p;
  }
  tc_fence_before();
  __syncthreads();

  // FP4 tile -> staging buffer (cp.async; empty rows zero-filled), as in the single-layer kernel
  auto stage_fp4 = [&](int tile) {
    const int32_t* pos = ms.pos[tile - t_begin];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = (t & 7) + 8 * ((t >> 7) + 2 * i), piece = (t >> 3) & 15;
      const int32_t p = pos[r];
      const uint8_t* src = p >= 0 ? cbase + int64_t(p) * CSA2_CODE_BYTES + 16 * piece : codes;
      cp_async16(base_s + C::kRawOff + raw_off(r, piece), src, p >= 0 ? 16 : 0);
    }
    if (t < 2 * kRows) {
      const int r = t >> 1, h2 = t & 1;
      const int32_t p = pos[r];
      const uint8_t* src = p >= 0 ? sbase + int64_t(p) * CSA2_SCALE_BYTES + 16 * h2 : scales;
      cp_async16(base_s + C::kRawScOff + r * CSA2_SCALE_BYTES + 16 * h2, src, p >= 0 ? 16 : 0);
    }
    cp_async_commit();
  };
  auto next_live = [&](int tile) {
    while (tile <= last_live && !live(tile)) ++tile;
    return tile;
  };

  bool ok = true;
  int par = 0;
  if (first_live >= 0) {
    tc_fence_after();
    const uint32_t tmem = ms.tmem_base;
    const uint32_t t_lane = tmem + (uint32_t(32 * quarter) << 16);
    // O^T of all layers starts at zero (every PV accumulates): this warp's lane quarter, blocks
    // 2 half and 2 half + 1
    {
      float z[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) z[i] = 0.0f;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int c = 0; c < kN; c += 16) tmem_st16(t_lane + C::kOCol + uint32_t(2 * half + j) * kN + uint32_t(c), z);
    }
    const int first_fp4 = next_live(max(first_live, nwin_all));
    if (first_fp4 <= last_live) stage_fp4(first_fp4);
    uint32_t ph_s = 0, ph_o = 0;
    int q_kind = -1;  // -1: none; 0: every layer's Q in f16; 1 + l: layer l's Q in bf16
    bool first = true;
    float l_w[L];     // running sums of this lane's head (8 half + lane / 4), per layer, over the warp's rows
#pragma unroll
    for (int l = 0; l < L; ++l) l_w[l] = 0.0f;

    for (int tile = first_live; tile <= last_live; ++tile) {
      if (!live(tile)) continue;
      const bool is_fp4 = tile >= nwin_all;
      const int wl = is_fp4 ? 0 : tile / nwin;         // the window tile's layer
      const int c0 = is_fp4 ? 0 : 16 * wl;             // first column of the tile
      const int nc = is_fp4 ? kN : 16;                 // columns of the tile
      const int32_t* pos = ms.pos[tile - t_begin];
      const bool f16_tile = is_fp4 || win_fp8;
      const bool win16 = !is_fp4 && !win_fp8;
      // -- window rows into registers before the operand tile is free (thread t: rows (t & 7) + 8 j,
      //    16-byte chunk (t >> 3) + 32 (j >> 3) for bf16; 16 E4M3 channels at piece t >> 3 for 8-bit)
      uint4 wv[16];
      if (!is_fp4) {
        if (win16) {
          const uint16_t* sw = swb16(wl);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = (t & 7) + 8 * (j & 7), cc = (t >> 3) + 32 * (j >> 3);
            const int32_t br = pos[r];
            wv[j] = br >= 0 ? __ldg(reinterpret_cast<const uint4*>(sw + int64_t(br) * CSA2_D + 8 * cc))
                            : make_uint4(0, 0, 0, 0);
          }
        } else {
          const uint8_t* sw = swb8(wl);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int32_t br = pos[(t & 7) + 8 * j];
            wv[j] = br >= 0 ? __ldg(reinterpret_cast<const uint4*>(sw + int64_t(br) * CSA2_D + 16 * (t >> 3)))
                            : make_uint4(0, 0, 0, 0);
          }
        }
      }
      // -- the previous tile's O^T MMAs read the operand tile and P^T: wait for them
      if (!first) {
        ok = ok && mbar_wait(mbar_o, ph_o);
        ph_o ^= 1u;
      }
      // -- Q in the tile's operand type: every layer in f16, or the window layer in bf16
      const int kind = f16_tile ? 0 : 1 + wl;
      if (kind != q_kind) {
        const int l0 = kind == 0 ? 0 : wl, nl = kind == 0 ? L : 1;
        for (int e = t; e < nl * 16 * 64; e += kThreads) {  // 16-byte chunks: (layer, head, chunk)
          const int l = l0 + e / (16 * 64), h = (e / 64) % 16, cc = e % 64;
          uint4 v = __ldg(reinterpret_cast<const uint4*>(layers.q[l] + (int64_t(inst) * CSA2_H + h) * CSA2_D + 8 * cc));
          if (kind == 0) {
            v.x = bf16x2_to_f16x2(v.x);
            v.y = bf16x2_to_f16x2(v.y);
            v.z = bf16x2_to_f16x2(v.z);
            v.w = bf16x2_to_f16x2(v.w);
          }
          *reinterpret_cast<uint4*>(base + C::kQOff + sw128(C::kQGroup, 16 * l + h, cc)) = v;
        }
        q_kind = kind;
      }
      // -- rows -> operand tile
      if (is_fp4) {
        cp_async_wait<0>();
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = (t & 7) + 8 * ((t >> 7) + 2 * i), piece = (t >> 3) & 15;
          const uint4 cw = *reinterpret_cast<const uint4*>(base + C::kRawOff + raw_off(r, piece));
          const uint16_t s2 = *reinterpret_cast<const uint16_t*>(base + C::kRawScOff + r * CSA2_SCALE_BYTES + 2 * piece);
          const __half2 sab = bits_h2(e4m3x2_to_f16x2(s2));
          const __half2 sA = __low2half2(sab), sB = __high2half2(sab);
          const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            const __half2 sc = wi < 2 ? sA : sB;
            uint32_t f0, f1, f2, f3;
            e2m1x8_to_f16x2x4(words[wi], f0, f1, f2, f3);
            uint4 o;
            o.x = h2_bits(__hmul2(bits_h2(f0), sc));
            o.y = h2_bits(__hmul2(bits_h2(f1), sc));
            o.z = h2_bits(__hmul2(bits_h2(f2), sc));
            o.w = h2_bits(__hmul2(bits_h2(f3), sc));
            *reinterpret_cast<uint4*>(base + C::kTileOff + sw128(C::kTileGroup, r, 4 * piece + wi)) = o;
          }
        }
      } else if (win16) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int r = (t & 7) + 8 * (j & 7), cc = (t >> 3) + 32 * (j >> 3);
          *reinterpret_cast<uint4*>(base + C::kTileOff + sw128(C::kTileGroup, r, cc)) = wv[j];
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = (t & 7) + 8 * j, cc = 2 * (t >> 3);
          const uint32_t bw[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
          uint32_t h[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            h[2 * e] = e4m3x2_to_f16x2(uint16_t(bw[e] & 0xFFFFu));
            h[2 * e + 1] = e4m3x2_to_f16x2(uint16_t(bw[e] >> 16));
          }
          *reinterpret_cast<uint4*>(base + C::kTileOff + sw128(C::kTileGroup, r, cc)) = make_uint4(h[0], h[1], h[2], h[3]);
          *reinterpret_cast<uint4*>(base + C::kTileOff + sw128(C::kTileGroup, r, cc + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
      }
      fence_async_smem();
      __syncthreads();

      // -- S^T = K Q^T: warp p < kP issues channels [512 p / kP, 512 (p + 1) / kP) into partial p,
      //    columns [c0, c0 + nc) (Q rows 16 wl .. for a window tile)
      if (lane == 0 && warp < kP) {
        tc_fence_after();
        const uint32_t id = instr_desc(kRows, !f16_tile, false, nc);
        constexpr int kSteps = CSA2_D / 16 / kP;
#pragma unroll
        for (int s = 0; s < kSteps; ++s) {
          const int kk = warp * kSteps + s;
          const uint32_t off = uint32_t(kk & 3) * 32u;
          const uint64_t a = smem_desc(tile_s + uint32_t(kk >> 2) * C::kTileGroup + off, 0, 1024);
          const uint64_t bq = smem_desc(q_s + uint32_t(kk >> 2) * C::kQGroup + uint32_t(c0) * 128u + off, 0, 1024);
          umma_f16(tmem + uint32_t(warp * kN + c0), a, bq, id, s > 0 ? 1u : 0u);
        }
        umma_commit(mbar_s);
      }
      if (is_fp4) {
        const int nxt = next_live(tile + 1);
        if (nxt <= last_live) stage_fp4(nxt);
      }
      ok = ok && mbar_wait(mbar_s, ph_s);
      ph_s ^= 1u;
      tc_fence_after();

      // -- online softmax over the tile's columns: warp (quarter, half) holds rows 16 quarter + lane
      //    (lanes < 16) and, in each 16-column chunk j, heads 8 half .. 8 half + 7
      const int row = 16 * quarter + (lane & 15);
      const bool row_ok = lane < 16 && pos[row] >= 0;
      const int nchunk = nc / 16;
      float x[L][8];
#pragma unroll
      for (int j = 0; j < L; ++j) {
        if (j < nchunk) {
          float sp[kP][8];
          tmem_ld8_parts<kP>(t_lane + uint32_t(c0 + 16 * j + 8 * half), uint32_t(kN), sp);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float v;
            if (kP == 8)
              v = ((sp[0][i] + sp[1 % kP][i]) + (sp[2 % kP][i] + sp[3 % kP][i])) +
                  ((sp[4 % kP][i] + sp[5 % kP][i]) + (sp[6 % kP][i] + sp[7 % kP][i]));
            else
              v = (sp[0][i] + sp[1 % kP][i]) + (sp[2 % kP][i] + sp[3 % kP][i]);
            x[j][i] = row_ok ? v * scale_log2 : -INFINITY;
          }
          const float mx = reduce_scatter8<true>(x[j], lane);
          if ((lane & 3) == 0) ms.red[quarter][c0 + 16 * j + 8 * half + (lane >> 2)] = mx;
        }
      }
      tc_fence_before();
      __syncthreads();
      const float* m_old = ms.m_run[par];
      float* m_new = ms.m_run[par ^ 1];
      if (t < nc) {  // column c0 + t: new offset and correction factor
        const int c = c0 + t;
        const float mt = fmaxf(fmaxf(ms.red[0][c], ms.red[1][c]), fmaxf(ms.red[2][c], ms.red[3][c]));
        const float mo = m_old[c], mn = mt > mo + kLazyF ? mt : mo;
        m_new[c] = mn;
        ms.corr[c] = (mn != mo && mo != -INFINITY) ? exp2f(mo - mn) : 1.0f;
      } else if (t >= 64 && t - 64 < kN && (t - 64 < c0 || t - 64 >= c0 + nc)) {
        m_new[t - 64] = m_old[t - 64];  // columns outside the tile keep their offsets
        ms.corr[t - 64] = 1.0f;
      }
#pragma unroll
      for (int j = 0; j < L; ++j) {
        if (j < nchunk) {
          float pr[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int c = c0 + 16 * j + 8 * half + i;
            const float mt = fmaxf(fmaxf(ms.red[0][c], ms.red[1][c]), fmaxf(ms.red[2][c], ms.red[3][c]));
            const float mj = mt > m_old[c] + kLazyF ? mt : m_old[c];
            pr[i] = mj == -INFINITY ? 0.0f : exp2f(x[j][i] - mj);
          }
          // P^T row = the column's index within the tile, K-major with a 128-byte swizzle
          if (lane < 16) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int n = 16 * j + 8 * half + i;
              const uint32_t off = uint32_t(n) * 128u + uint32_t(((row >> 3) ^ (n & 7)) << 4) + uint32_t(row & 7) * 2u;
              const uint16_t bits = f16_tile ? __half_as_ushort(__float2half_rn(pr[i])) : uint16_t(f2bf_bits(pr[i]));
              *reinterpret_cast<uint16_t*>(base + C::kPOff + off) = bits;
            }
          }
          const float sum = reduce_scatter8<false>(pr, lane);
          const int c = c0 + 16 * j + 8 * half + (lane >> 2);
          const float mt = fmaxf(fmaxf(ms.red[0][c], ms.red[1][c]), fmaxf(ms.red[2][c], ms.red[3][c]));
          const float mo = m_old[c], mn = mt > mo + kLazyF ? mt : mo;
          const float cr = (mn != mo && mo != -INFINITY) ? exp2f(mo - mn) : 1.0f;
          const int lay = c / 16;
#pragma unroll
          for (int l = 0; l < L; ++l)
            if (l == lay) l_w[l] = l_w[l] * cr + sum;
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();
      par ^= 1;
      bool moved = false;
      for (int c = c0; c < c0 + nc; ++c) moved |= ms.corr[c] != 1.0f;
      if (moved) {
        // rescale the tile's columns of the O^T accumulated so far (blocks 2 half, 2 half + 1)
        tc_fence_after();
        for (int j = 0; j < 2; ++j)
          for (int cc = c0; cc < c0 + nc; cc += 16) {
            const uint32_t ta = t_lane + C::kOCol + uint32_t(2 * half + j) * kN + uint32_t(cc);
            float o[16];
            tmem_ld16(ta, o);
#pragma unroll
            for (int h = 0; h < 16; ++h) o[h] *= ms.corr[cc + h];
            tmem_st16(ta, o);
          }
        tc_fence_before();
        __syncthreads();
      }

      // -- O^T[:, c0 .. c0 + nc) += V^T P^T: warp i < 4 issues channel block i in 4 steps of 16 rows
      if (lane == 0 && warp < 4) {
        tc_fence_after();
        const uint32_t id = instr_desc(128, !f16_tile, true, nc);
        const int i = warp;
#pragma unroll
        for (int s = 0; s < kRows / 16; ++s) {
          const uint64_t a = smem_desc(tile_s + uint32_t(2 * i) * C::kTileGroup + uint32_t(s) * 2048u, C::kTileGroup, 1024);
          const uint64_t bp = smem_desc(p_s + uint32_t(s) * 32u, 0, 1024);
          umma_f16(tmem + C::kOCol + uint32_t(i * kN + c0), a, bp, id, 1u);
        }
        umma_commit(mbar_o);
      }
      first = false;
    }
    // ---- the last tile's MMAs, the sums per column, then O^T out of tensor memory ------------------
    ok = ok && mbar_wait(mbar_o, ph_o);
    tc_fence_after();
#pragma unroll
    for (int l = 0; l < L; ++l)
      if ((lane & 3) == 0) ms.red[quarter][16 * l + 8 * half + (lane >> 2)] = l_w[l];
    __syncthreads();
    if (t < kN) ms.l_fin[t] = (ms.red[0][t] + ms.red[1][t]) + (ms.red[2][t] + ms.red[3][t]);
    __syncthreads();
#pragma unroll
    for (int l = 0; l < L; ++l) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float o[16];
        tmem_ld16(t_lane + C::kOCol + uint32_t(2 * half + j) * kN + uint32_t(16 * l), o);
        const int ch = 128 * (2 * half + j) + 32 * quarter + lane;
        if (n_split == 1) {
          uint16_t* orow = layers.out[l] + int64_t(inst) * CSA2_H * CSA2_D + ch;
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            const float lv = ms.l_fin[16 * l + h];
            orow[h * CSA2_D] = uint16_t(f2bf_bits(o[h] * (lv > 0.0f ? 1.0f / lv : 0.0f)));
          }
        } else {
          const int64_t ginst = int64_t(l) * gridDim.y + inst;
          float* po = ws + (ginst * n_split + split) * (CSA2_H * CSA2_D) + ch;
#pragma unroll
          for (int h = 0; h < 16; ++h) po[h * CSA2_D] = o[h];
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
      tc_fence_after();
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemColsF) : "memory");
    }
    if (!ok && t == 0) atomicOr(flags, CSA2_FLAG_TIMEOUT);
  } else if (n_split == 1) {
    for (int l = 0; l < L; ++l) {
      uint16_t* orow = layers.out[l] + int64_t(inst) * CSA2_H * CSA2_D;
      for (int e = t; e < CSA2_H * CSA2_D; e += kThreads) orow[e] = 0;
    }
  }

  if (n_split == 1) {
    if (t < kN) {
      const int l = t / 16, h = t % 16;
      if (layers.lse[l]) {
        const float lv = ms.l_fin[t];
        layers.lse[l][int64_t(inst) * CSA2_H + h] = lv > 0.0f ? (ms.m_run[par][t] + log2f(lv)) * kLn2 : -INFINITY;
      }
    }
    return;
  }
  // ---- split partials of every layer, then the last CTA of this instance merges them ---------------
  const int64_t instances = int64_t(gridDim.y) * L;
  float* mlb = ws + instances * n_split * (CSA2_H * CSA2_D);
  if (t < kN) {
    const int l = t / 16, h = t % 16;
    const int64_t ginst = int64_t(l) * gridDim.y + inst;
    float* ml = mlb + (ginst * n_split + split) * (2 * CSA2_H);
    ml[2 * h] = ms.m_run[par][t];
    ml[2 * h + 1] = ms.l_fin[t];
  }
  __threadfence();
  __syncthreads();
  if (t == 0) ms.is_last = (atomicAdd(tickets + inst, 1u) == unsigned(n_split - 1));
  __syncthreads();
  if (!ms.is_last) return;
  __threadfence();
  float* wgt = reinterpret_cast<float*>(base + C::kTileOff);
  for (int l = 0; l < L; ++l) {
    const int64_t ginst = int64_t(l) * gridDim.y + inst;
    const float* ml = mlb + ginst * n_split * (2 * CSA2_H);
    for (int e = t; e < n_split * CSA2_H; e += kThreads) {
      wgt[e] = __ldcg(ml + 2 * e);
      wgt[kMaxSplit * CSA2_H + e] = __ldcg(ml + 2 * e + 1);
    }
    __syncthreads();
    if (t < CSA2_H) {
      float M = -INFINITY;
      for (int j = 0; j < n_split; ++j)
        if (wgt[kMaxSplit * CSA2_H + j * CSA2_H + t] > 0.0f) M = fmaxf(M, wgt[j * CSA2_H + t]);
      float Ls = 0.0f;
      for (int j = 0; j < n_split; ++j) {
        const float lj = wgt[kMaxSplit * CSA2_H + j * CSA2_H + t];
        const float a = (lj > 0.0f && M != -INFINITY) ? exp2f(wgt[j * CSA2_H + t] - M) : 0.0f;
        Ls += a * lj;
        wgt[j * CSA2_H + t] = a;
      }
      wgt[2 * kMaxSplit * CSA2_H + t] = Ls > 0.0f ? 1.0f / Ls : 0.0f;
      wgt[2 * kMaxSplit * CSA2_H + CSA2_H + t] = Ls > 0.0f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
    }
    __syncthreads();
    const float4* p0 = reinterpret_cast<const float4*>(ws + ginst * n_split * (CSA2_H * CSA2_D)) + t;
    float4 acc[8];
#pragma unroll
    for (int v = 0; v < 8; ++v) acc[v] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int j = 0; j < n_split; ++j) {
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const int h = (t >> 7) + 2 * v;
        const float a = wgt[j * CSA2_H + h];
        if (a != 0.0f) {
          const float4 xv = __ldcg(p0 + int64_t(j) * (CSA2_H * CSA2_D / 4) + kThreads * v);
          acc[v].x += a * xv.x;
          acc[v].y += a * xv.y;
          acc[v].z += a * xv.z;
          acc[v].w += a * xv.w;
        }
      }
    }
    uint16_t* orow = layers.out[l] + int64_t(inst) * CSA2_H * CSA2_D;
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const int h = (t >> 7) + 2 * v;
      const float inv = wgt[2 * kMaxSplit * CSA2_H + h];
      *reinterpret_cast<uint2*>(orow + 4 * (t + kThreads * v)) =
          make_uint2(pack_bf16x2(acc[v].x * inv, acc[v].y * inv), pack_bf16x2(acc[v].z * inv, acc[v].w * inv));
    }
    if (layers.lse[l] && t < CSA2_H) layers.lse[l][int64_t(inst) * CSA2_H + t] = wgt[2 * kMaxSplit * CSA2_H + CSA2_H + t];
    __syncthreads();  // wgt is reused by the next layer
  }
  if (t == 0) tickets[inst] = 0u;  // ready for the next launch
}

template <int L>
cudaError_t launch_fused_l(const AttnLayers& layers, int B, int Nq, const uint8_t* codes, const uint8_t* scales,
                           int64_t cap, const int32_t* idx, int k, const int32_t* swa_len, int W, float scale_log2,
                           int n_split, float* partials, unsigned int* tickets, unsigned int* flags, bool win_fp8,
                           cudaStream_t st) {
  static std::atomic<bool> attr_set[64];  // per device; set once, by any host thread
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(sparse_attn_fused_kernel<L>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               int(fused_smem<L>()));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const dim3 grid{unsigned(n_split), unsigned(int64_t(B) * Nq), 1u};
  return launch_pdl(sparse_attn_fused_kernel<L>, grid, dim3(kThreads), fused_smem<L>(), st, layers, Nq, codes, scales,
                    cap, idx, k, swa_len, W, scale_log2, n_split, partials, tickets, flags, int(win_fp8));
}

}  // namespace

int attn_fused_tiles(int L, int k, int W) {
  return (k + kRows - 1) / kRows + (W > 0 ? L * ((W + kRows - 1) / kRows) : 0);
}

// Split of a fused launch: one CTA per SM, at most one split per tile.
int attn_fused_split(int64_t instances, int L, int k, int W) {
  const int nt = attn_fused_tiles(L, k, W);
  if (instances <= 0 || nt <= 0) return 1;
  int64_t s = std::max<int64_t>(152 / instances, 1);
  s = std::min<int64_t>(s, std::min(nt, kMaxSplit));
  return int(std::max<int64_t>(s, 1));
}

cudaError_t launch_sparse_attn_fused(const AttnLayers& layers, int n_layers, int B, int Nq, const uint8_t* codes,
                                     const uint8_t* scales, int64_t cap, const int32_t* idx, int k,
                                     const int32_t* swa_len, int W, float softmax_scale, int n_split, float* ws,
                                     cudaStream_t st, bool tickets_zeroed, bool win_fp8) {
  const int64_t instances = int64_t(B) * Nq;
  if (instances == 0) return cudaSuccess;
  if (n_layers < 2 || n_layers > kMaxL || instances > 65535 || k < 1) return cudaErrorInvalidValue;
  if (!layers.swa[0]) W = 0;
  n_split = std::max(1, std::min(n_split, attn_fused_tiles(n_layers, k, W)));
  unsigned int* flags = device_flags_ptr();
  if (!flags) return cudaErrorUnknown;
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  unsigned int* tickets = nullptr;
  float* partials = nullptr;
  if (n_split > 1) {
    tickets = reinterpret_cast<unsigned int*>(ws);
    partials = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + attn_ticket_bytes(instances * n_layers));
    if (!tickets_zeroed) {
      const cudaError_t e = cudaMemsetAsync(tickets, 0, size_t(instances) * sizeof(unsigned int), st);
      if (e != cudaSuccess) return e;
    }
  }
  switch (n_layers) {
    case 2: return launch_fused_l<2>(layers, B, Nq, codes, scales, cap, idx, k, swa_len, W, scale_log2, n_split,
                                     partials, tickets, flags, win_fp8, st);
    case 3: return launch_fused_l<3>(layers, B, Nq, codes, scales, cap, idx, k, swa_len, W, scale_log2, n_split,
                                     partials, tickets, flags, win_fp8, st);
    default: return launch_fused_l<4>(layers, B, Nq, codes, scales, cap, idx, k, swa_len, W, scale_log2, n_split,
                                      partials, tickets, flags, win_fp8, st);
  }
}

}  // namespace csa2

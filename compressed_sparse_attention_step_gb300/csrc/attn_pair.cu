// Sparse attention of a pair of layers that attend the same selected FP4 rows ("Every layer retains
// its own main Q and sliding-window key-value cache", ai-maestro.online "DeepSeek AI released
// DeepSeek-V4.1-Flash with 1M context, FP4", section "Compressed Sparse Attention 2": a Full or
// Reindex layer selects rows and the Reuse layers after it attend the same rows; E2M1 codes with an
// E4M3 scale per 16 channels: section "FP4 KV, Bounded Replay, and other extensions").
//
// The per-layer kernels gather and dequantise the shared rows once per layer and run the tensor core
// at N = 16 heads.  Here a CTA takes one query's tiles for two layers: an FP4 tile is dequantised
// once and its S^T = K Q^T and O^T += V^T P^T run at N = 32 (the two layers' heads, layer-major);
// a window tile (each layer has its own window rows) runs at N = 16 in its layer's columns.  The
// tensor-memory budget (256 columns: four 128-channel O^T blocks and four K-slice partials of S^T,
// 32 columns each) and about 104 KB of shared memory keep two CTAs on an SM, so one CTA's loads and
// conversions overlap the other's tensor-core work, as in the per-layer kernel:
//   - the next FP4 tile's code and scale bytes are loaded into registers while the current tile is
//     computed (kept as loaded: a thread that combined them at once would wait for the loads), and
//     dequantised (E2M1 -> f16x2 and E4M3 -> f16x2 conversions, one exact f16 multiply) into a
//     64 x 512 operand tile in the 128-byte-swizzled layout;
//   - a window tile's first 256 channels per row are loaded into registers before the previous
//     tile's O^T products release the operand tile, the other 256 go there by cp.async while the
//     first half is stored; the warps of the other layer's columns skip the tile's softmax;
//   - four warps issue a 128-channel quarter each of S^T into their own partial; the softmax warps
//     add the four partials, run the online softmax per column (two warps per tensor-memory lane
//     quarter, 16 columns each) with lazy offsets (an offset moves only when a score passes it by
//     more than 2^12; one block barrier with an OR tells whether any did) and write P^T;
//   - four warps issue one 128-channel block of O^T each.
// The FP4 tiles come first (Q as f16), then the window tiles (Q rewritten as bf16, or kept as f16
// for 8-bit windows); one CTA per (query, pair) writes the outputs.  The kernel serves launches of
// at least one full wave of such CTAs (prefill chunks): smaller ones would have to split a query
// over CTAs and merge partials, which measured slower than the per-layer kernel.
//
// Operand types: FP4 tiles and 8-bit window tiles run in f16 (exact for the dequantised rows), bf16
// window tiles in bf16; Q is converted from bf16 for the f16 tiles, P is rounded to the tile's
// type; accumulation is fp32.  Tensor-memory layouts: S^T (M = 64) row r in lane 32 (r / 16) +
// r % 16; O^T (M = 128) channel c of a block in lane c; column n is column n.
#include <cuda_fp16.h>

#include <algorithm>
#include <type_traits>

#include "attn_common.cuh"

namespace csa2 {
namespace {
using namespace attn;

constexpr int kPairTiles = (CSA2_MAX_ATTN_K + kRows - 1) / kRows;
constexpr float kLazyPair = 12.0f;  // log2 units, as in the per-layer kernels
constexpr int N = 32;               // columns: the pair's heads, layer-major
constexpr int NC = 16;              // columns per thread in the softmax
constexpr int P = 4;                // S^T partials (K slices of 128 channels)
constexpr uint32_t kOCol = 0;       // O^T block i: columns [32 i, 32 i + 32)
constexpr uint32_t kSCol = 4 * N;   // S^T partial p: columns [128 + 32 p, ...)
constexpr uint32_t kTmemCols = 256;
// shared memory (offsets from a 1024-byte aligned base)
constexpr uint32_t kTileGroup = kRows * 128;            // 8 KiB per 64-channel group
constexpr uint32_t kTileOff = 0;                        // 8 groups x 64 rows x 128 B
constexpr uint32_t kQGroup = N * 128;                   // 4 KiB
constexpr uint32_t kQOff = kTileOff + 8 * kTileGroup;   // Q: 8 groups x 32 rows x 128 B
constexpr uint32_t kPOff = kQOff + 8 * kQGroup;         // P^T: 32 rows x 64 (128 B)
constexpr uint32_t kMiscOff = kPOff + N * 128;

struct PairMisc {
  unsigned long long mbar_s;  // S^T of a tile complete (one arrival per S issuer)
  unsigned long long mbar_o;  // O^T of a tile complete (one arrival per O issuer)
  uint32_t tmem_base;
  int32_t pos[kPairTiles][kRows];  // source row of each row of the FP4 tiles, -1 if empty
  float red[4][N];                 // per-quarter column maxima, then partial sums
  float mj[N];                     // running offset per column (log2 units)
  float corr[N];                   // factor rescaling what came before, per column, after a move
  float m_fin[N];
  float l_fin[N];
};
constexpr size_t kPairSmem = 1024 + kMiscOff + sizeof(PairMisc);
static_assert(2 * (kPairSmem + 1024) <= 232448, "two CTAs per SM");

// Sixteen consecutive columns of this warp's 32 lanes, one wait.
__device__ __forceinline__ void tmem_ld16c(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// Eight consecutive columns of this warp's 32 lanes, one wait.
__device__ __forceinline__ void tmem_ld8c(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16c(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};\n\t"
      "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}

// grid (queries, pairs).  Layers [2 y, 2 y + 2) of the launch's n_layers share the selected rows.
// The CTA of query x takes its FP4 tiles (both layers, N = 32), then its window tiles (layer l,
// tile w: that layer's 16 columns, N = 16), and writes the outputs.
__global__ void __launch_bounds__(kThreads, 2) sparse_attn_pair_kernel(
    const __grid_constant__ AttnLayers layers, int n_layers, const uint8_t* __restrict__ codes,
    const uint8_t* __restrict__ scales, int64_t cap, const int32_t* __restrict__ idx,
    const int32_t* __restrict__ n_valid, int k, const int32_t* __restrict__ swa_len, int W, int Nq,
    float scale_log2, int win_fp8, unsigned int* flags) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  pdl_wait();  // the selected positions come from the kernels before this one
  pdl_trigger();
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  unsigned char* base = smem_raw + (base_s - raw_s);
  PairMisc& ms = *reinterpret_cast<PairMisc*>(base + kMiscOff);
  const uint32_t tile_s = base_s + kTileOff, q_s = base_s + kQOff, p_s = base_s + kPOff;
  const uint32_t mbar_s = smem_u32(&ms.mbar_s), mbar_o = smem_u32(&ms.mbar_o);

  const int inst = blockIdx.x;
  const int l0 = 2 * blockIdx.y, gv = min(2, n_layers - l0);  // this pair's layers
  const int b = inst / Nq, qi = inst - b * Nq;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int quarter = warp & 3, half = warp >> 2;

  // ---- this CTA's tiles ----------------------------------------------------------------------------
  const int n_fp4_valid = min(k, n_valid ? max(n_valid[inst], 0) : k);
  const int n_my_fp4 = (n_fp4_valid + kRows - 1) / kRows;  // FP4 tiles holding a row
  const bool has_win = layers.swa[l0] != nullptr && W > 0;
  const int nwin = has_win ? (W + kRows - 1) / kRows : 0;
  const int SW = W - 1 + Nq;
  const int swa_lo = has_win ? SW - min(max(swa_len[b], 0), SW) : SW;
  auto win_live = [&](int w) { return qi + min((w + 1) * kRows, W) - 1 >= swa_lo; };
  int n_my_win = 0;  // window items w < gv nwin: layer w / nwin, tile w % nwin
  for (int w = 0; w < gv * nwin; ++w) n_my_win += win_live(w % nwin) ? 1 : 0;
  const bool any = n_my_fp4 + n_my_win > 0;

  const int32_t* irow = (layers.idx[l0] ? layers.idx[l0] : idx) + int64_t(inst) * k;
  const uint8_t* cbase = codes + int64_t(b) * cap * CSA2_CODE_BYTES;
  const uint8_t* sbase = scales + int64_t(b) * cap * CSA2_SCALE_BYTES;
  // window row of tile row r of window tile w, or -1
  auto win_row = [&](int w, int r) {
    const int wr = w * kRows + r;
    return (wr < W && qi + wr >= swa_lo) ? qi + wr : -1;
  };
  // Q of the pair's layers into the Q buffer (row 16 l + h; absent layers zero), as f16 or as bf16
  auto load_q = [&](bool as_f16) {
#pragma unroll
    for (int l = 0; l < 2; ++l) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = u * kThreads + t;  // (h, cc) = (e >> 6, e & 63)
        v[u] = l < gv ? __ldg(reinterpret_cast<const uint4*>(layers.q[l0 + l] + int64_t(inst) * CSA2_H * CSA2_D) + e)
                      : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = u * kThreads + t, row = 16 * l + (e >> 6), cc = e & 63;
        uint4 w = v[u];
        if (as_f16) {
          w.x = bf16x2_to_f16x2(w.x);
          w.y = bf16x2_to_f16x2(w.y);
          w.z = bf16x2_to_f16x2(w.z);
          w.w = bf16x2_to_f16x2(w.w);
        }
        *reinterpret_cast<uint4*>(base + kQOff + sw128(kQGroup, row, cc)) = w;
      }
    }
  };

  if (t < N) {
    ms.m_fin[t] = -INFINITY;
    ms.l_fin[t] = 0.0f;
    ms.mj[t] = -INFINITY;
  }
  if (any) {
    if (t == 0) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(mbar_s), "r"(P) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(mbar_o), "r"(4) : "memory");
      asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 0) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                       smem_u32(&ms.tmem_base)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    load_q(n_my_fp4 > 0 || win_fp8);
    // source rows of the CTA's FP4 tiles, pulled into L2
    for (int e = t; e < n_my_fp4 * kRows; e += kThreads) {
      const int tile = e / kRows, r = e % kRows;
      const int slot = tile * kRows + r;
      int32_t p = -1;
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
      ms.pos[tile][r] = p < 0 ? -1 : p;
    }
  }
  tc_fence_before();
  __syncthreads();

  // an FP4 tile's bytes into registers: thread t takes 16-byte piece (t >> 3) & 15 of rows
  // (t & 7) + 8 ((t >> 7) + 2 i), i < 4, and the two scale bytes of each piece (empty rows: zeros)
  // (the loads are not used until the tile is converted, so the thread does not wait for them)
  uint4 cw[4];
  uint32_t sw[4];  // the two scale bytes of each row's piece
  auto load_fp4 = [&](int tile) {
    const int32_t* pos = ms.pos[tile];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = (t & 7) + 8 * ((t >> 7) + 2 * i), piece = (t >> 3) & 15;
      const int32_t p = pos[r];
      cw[i] = p >= 0 ? __ldg(reinterpret_cast<const uint4*>(cbase + int64_t(p) * CSA2_CODE_BYTES) + piece)
                     : make_uint4(0, 0, 0, 0);
      sw[i] = p >= 0 ? uint32_t(__ldg(reinterpret_cast<const unsigned short*>(sbase + int64_t(p) * CSA2_SCALE_BYTES) + piece))
                     : 0u;
    }
  };

  // ls[c]: this lane's row's running sum for column half NC + c (the columns' running offsets are
  // in shared memory, ms.mj)
  float ls[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) ls[c] = 0.0f;
  bool ok = true;
  if (any) {
    tc_fence_after();
    const uint32_t tmem = ms.tmem_base;
    const uint32_t t_lane = tmem + (uint32_t(32 * quarter) << 16);  // this warp's lane quarter
    {
      // O^T starts at zero (window tiles accumulate into their layer's columns only)
      float z[NC];
#pragma unroll
      for (int c = 0; c < NC; ++c) z[c] = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) tmem_st16c(t_lane + kOCol + uint32_t(i * N + half * NC), z);
    }
    if (n_my_fp4 > 0) load_fp4(0);
    uint32_t ph_s = 0, ph_o = 0;
    bool first = true;
    bool q_f16 = n_my_fp4 > 0 || win_fp8;  // the Q buffer's type
    // one tile: FP4 tile `tile` (fp4_c true; next: the CTA's next FP4 tile, or -1), or window tile wt
    // of layer wl; compiled separately for the two kinds
    auto tile_step = [&](auto fp4_c, int tile, int next, int wl, int wt) {
      constexpr bool is_fp4 = decltype(fp4_c)::value;
      const bool win8 = !is_fp4 && win_fp8;
      const bool f16_tile = is_fp4 || win_fp8;
      const int c0 = is_fp4 ? 0 : 16 * wl;  // the tile's columns [c0, c0 + nc)
      const int nc = is_fp4 ? N : 16;
      const uint16_t* swbase = is_fp4 ? nullptr : layers.swa[l0 + wl] + int64_t(b) * SW * CSA2_D;
      const uint8_t* sw8 =
          is_fp4 ? nullptr : reinterpret_cast<const uint8_t*>(layers.swa[l0 + wl]) + int64_t(b) * SW * CSA2_D;
      // -- window rows into registers before the operand tile is free: bf16 rows, thread t 16 B
      //    chunks (t >> 3) + 32 (j >> 3) of rows (t & 7) + 8 (j & 7) (the first eight now, the rest
      //    after the first are stored); 8-bit rows, 16 B (16 channels) of rows (t & 7) + 8 j
      uint4 wv[8];
      if (!is_fp4) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int br = win_row(wt, (t & 7) + 8 * j);
          if (win8)
            wv[j] = br >= 0 ? __ldg(reinterpret_cast<const uint4*>(sw8 + int64_t(br) * CSA2_D + 16 * (t >> 3)))
                            : make_uint4(0, 0, 0, 0);
          else
            wv[j] = br >= 0 ? __ldg(reinterpret_cast<const uint4*>(swbase + int64_t(br) * CSA2_D + 8 * (t >> 3)))
                            : make_uint4(0, 0, 0, 0);
        }
      }
      // -- the previous tile's O^T MMAs read the operand tile and P^T: wait for them
      if (!first) {
        ok = ok && mbar_wait(mbar_o, ph_o);
        ph_o ^= 1u;
      }
      // -- rows -> operand tile
      if (is_fp4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = (t & 7) + 8 * ((t >> 7) + 2 * i), piece = (t >> 3) & 15;
          const __half2 sab = bits_h2(e4m3x2_to_f16x2(uint16_t(sw[i])));
          const __half2 sA = __low2half2(sab), sB = __high2half2(sab);
          const uint32_t words[4] = {cw[i].x, cw[i].y, cw[i].z, cw[i].w};
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
            *reinterpret_cast<uint4*>(base + kTileOff + sw128(kTileGroup, r, 4 * piece + wi)) = o;
          }
        }
      } else if (win8) {
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
          *reinterpret_cast<uint4*>(base + kTileOff + sw128(kTileGroup, r, cc)) = make_uint4(h[0], h[1], h[2], h[3]);
          *reinterpret_cast<uint4*>(base + kTileOff + sw128(kTileGroup, r, cc + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
      } else {
        // the second half of the rows' channels straight into the tile (cp.async; empty rows are
        // zero-filled), and at the first bf16 window tile the pair's Q as bf16 (the previous tile's
        // S^T products are complete); the first half, already in registers, is stored meanwhile
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = (t & 7) + 8 * j, cc = (t >> 3) + 32;
          const int br = win_row(wt, r);
          cp_async16(tile_s + sw128(kTileGroup, r, cc), swbase + (br >= 0 ? int64_t(br) * CSA2_D + 8 * cc : 0),
                     br >= 0 ? 16 : 0);
        }
        if (q_f16) {
#pragma unroll
          for (int l = 0; l < 2; ++l)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int e = u * kThreads + t, row = 16 * l + (e >> 6), cc = e & 63;
              const uint16_t* src = layers.q[l0] + int64_t(inst) * CSA2_H * CSA2_D;
              if (l < gv) src = layers.q[l0 + l] + int64_t(inst) * CSA2_H * CSA2_D + 8 * e;
              cp_async16(q_s + sw128(kQGroup, row, cc), src, l < gv ? 16 : 0);
            }
          q_f16 = false;
        }
        cp_async_commit();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = (t & 7) + 8 * j, cc = t >> 3;
          *reinterpret_cast<uint4*>(base + kTileOff + sw128(kTileGroup, r, cc)) = wv[j];
        }
        cp_async_wait<0>();
      }
      fence_async_smem();
      __syncthreads();

      // -- S^T = K Q^T (tensor core): warp p < 4 issues channel groups 2 p, 2 p + 1 into partial p's
      //    columns [c0, c0 + nc)
      if (lane == 0 && warp < P) {
        tc_fence_after();
        const uint32_t id = instr_desc(kRows, !f16_tile, false, nc);
#pragma unroll
        for (int gi = 0; gi < 2; ++gi) {
          const int grp = 2 * warp + gi;
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const uint32_t off = uint32_t(k4) * 32u;  // 16 channels = 32 B inside the swizzle atom
            const uint64_t a = smem_desc(tile_s + uint32_t(grp) * kTileGroup + off, 0, 1024);
            const uint64_t bq = smem_desc(q_s + uint32_t(grp) * kQGroup + uint32_t(c0) * 128u + off, 0, 1024);
            umma_f16(tmem + kSCol + uint32_t(warp * N + c0), a, bq, id, (gi > 0 || k4 > 0) ? 1u : 0u);
          }
        }
        umma_commit(mbar_s);
      }
      // -- the CTA's next FP4 tile into registers while this one is computed
      if (is_fp4 && next >= 0) load_fp4(next);
      ok = ok && mbar_wait(mbar_s, ph_s);
      ph_s ^= 1u;
      tc_fence_after();

      // -- online softmax: warp (quarter, half) holds rows 16 quarter + lane (lanes < 16) and
      //    columns 16 half .. 16 half + 15 (those outside [c0, c0 + nc) take no part); S^T is the sum
      //    of the four partials
      const int row = 16 * quarter + (lane & 15);
      const bool row_ok = lane < 16 && (is_fp4 ? ms.pos[tile][row] >= 0 : win_row(wt, row) >= 0);
      const bool cols_in = half * NC >= c0 && half * NC < c0 + nc;  // a half's columns are all in or all out
      float x[NC];
      if (cols_in) {  // (warp-uniform; the warps of the other layer's columns skip a window tile)
        tmem_ld16c(t_lane + kSCol + uint32_t(half * NC), x);
#pragma unroll
        for (int p = 1; p < P; ++p)
#pragma unroll
          for (int h8 = 0; h8 < 2; ++h8) {
            float part[8];
            tmem_ld8c(t_lane + kSCol + uint32_t(p * N + half * NC + 8 * h8), part);
#pragma unroll
            for (int c = 0; c < 8; ++c) x[8 * h8 + c] += part[c];
          }
#pragma unroll
        for (int c = 0; c < NC; ++c) x[c] = row_ok ? x[c] * scale_log2 : -INFINITY;
      } else {
#pragma unroll
        for (int c = 0; c < NC; ++c) x[c] = -INFINITY;
      }
      const float* mjh = ms.mj + half * NC;  // this half's offsets (the same for every lane: a broadcast)
      const float* crh = ms.corr + half * NC;
      bool rescale = false;  // (warp-uniform) O^T must be rescaled before this tile's products
      bool jump = false;
#pragma unroll
      for (int c = 0; c < NC; ++c) jump |= x[c] > mjh[c] + kLazyPair;
      tc_fence_before();
      if (__syncthreads_or(jump)) {
        // the tile's maximum per column over the 64 rows, then the offsets that move (one thread per
        // column), then the sums and O^T rescaled by the factors
#pragma unroll
        for (int g8 = 0; g8 < NC / 8; ++g8) {
          float v8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) v8[i] = x[8 * g8 + i];
          const float mx = reduce_scatter8<true>(v8, lane);
          if ((lane & 3) == 0) ms.red[quarter][half * NC + 8 * g8 + (lane >> 2)] = mx;
        }
        __syncthreads();
        if (t < N) {
          const float mt = fmaxf(fmaxf(ms.red[0][t], ms.red[1][t]), fmaxf(ms.red[2][t], ms.red[3][t]));
          const float mo = ms.mj[t];
          const float mn = mt > mo + kLazyPair ? mt : mo;
          ms.corr[t] = (mn != mo && mo != -INFINITY) ? ex2(mo - mn) : 1.0f;
          ms.mj[t] = mn;
        }
        __syncthreads();
        bool moved = false;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          ls[c] *= crh[c];
          moved |= crh[c] != 1.0f;
        }
        rescale = __any_sync(0xffffffffu, moved);
      }
      // P^T (columns x rows, K-major, 128-byte swizzle): element (col, row); columns outside the
      // tile's range are not written (its O^T products do not read them)
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        if (!cols_in) break;
        // an empty row (x = -inf) gives 0; a finite x has a finite offset
        const float pr = x[c] == -INFINITY ? 0.0f : ex2(x[c] - mjh[c]);
        ls[c] += pr;
        if (lane < 16) {
          const int col = half * NC + c;
          const uint32_t off = uint32_t(col) * 128u + uint32_t(((row >> 3) ^ (col & 7)) << 4) + uint32_t(row & 7) * 2u;
          const uint16_t bits = f16_tile ? __half_as_ushort(__float2half_rn(pr)) : uint16_t(f2bf_bits(pr));
          *reinterpret_cast<uint16_t*>(base + kPOff + off) = bits;
        }
      }
      if (rescale) {
        // O^T accumulated so far (complete: its MMAs were waited for above), this half's columns of
        // this lane quarter's channels of each block, before this tile's products add to it
        tc_fence_after();
#pragma unroll 1
        for (int i = 0; i < 4; ++i) {
          float o[NC];
          const uint32_t ta = t_lane + kOCol + uint32_t(i * N + half * NC);
          tmem_ld16c(ta, o);
#pragma unroll
          for (int c = 0; c < NC; ++c) o[c] *= crh[c];
          tmem_st16c(ta, o);
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();

      // -- O^T += V^T P^T (tensor core): warp i < 4 issues channel block i in 4 steps of 16 rows,
      //    into the tile's columns [c0, c0 + nc)
      if (lane == 0 && warp < 4) {
        tc_fence_after();
        const uint32_t id = instr_desc(128, !f16_tile, true, nc);
        const int i = warp;
#pragma unroll
        for (int s = 0; s < kRows / 16; ++s) {
          const uint64_t a = smem_desc(tile_s + uint32_t(2 * i) * kTileGroup + uint32_t(s) * 2048u, kTileGroup, 1024);
          const uint64_t bp = smem_desc(p_s + uint32_t(c0) * 128u + uint32_t(s) * 32u, 0, 1024);
          umma_f16(tmem + kOCol + uint32_t(i * N + c0), a, bp, id, 1u);
        }
        umma_commit(mbar_o);
      }
      first = false;
    };
    for (int tile = 0; tile < n_my_fp4; ++tile)
      tile_step(std::true_type{}, tile, tile + 1 < n_my_fp4 ? tile + 1 : -1, 0, 0);
    for (int w = 0; w < gv * nwin; ++w)
      if (win_live(w % nwin)) tile_step(std::false_type{}, 0, -1, w / nwin, w % nwin);
    // ---- the last tile's MMAs, the sums per column, then O^T out of tensor memory -------------------
    if (!first) {
      ok = ok && mbar_wait(mbar_o, ph_o);
    }
    tc_fence_after();
#pragma unroll
    for (int g8 = 0; g8 < NC / 8; ++g8) {
      float v8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v8[i] = ls[8 * g8 + i];
      const float lw = reduce_scatter8<false>(v8, lane);
      if ((lane & 3) == 0) ms.red[quarter][half * NC + 8 * g8 + (lane >> 2)] = lw;
    }
    if (t < N) ms.m_fin[t] = ms.mj[t];
    __syncthreads();
    if (t < N) ms.l_fin[t] = (ms.red[0][t] + ms.red[1][t]) + (ms.red[2][t] + ms.red[3][t]);
    __syncthreads();
    // O^T out: this warp's lane quarter (channel 32 quarter + lane of each block) and its half's
    // columns, which are layer `half`'s 16 heads
    if (half < gv) {
      uint16_t* obase = layers.out[l0 + half] + int64_t(inst) * CSA2_H * CSA2_D;
#pragma unroll 1
      for (int i = 0; i < 4; ++i) {
        float o[NC];
        tmem_ld16c(t_lane + kOCol + uint32_t(i * N + half * NC), o);
        const int ch = 128 * i + 32 * quarter + lane;
#pragma unroll
        for (int h = 0; h < NC; ++h) {
          const float lf = ms.l_fin[half * NC + h];
          obase[h * CSA2_D + ch] = uint16_t(f2bf_bits(o[h] * (lf > 0.0f ? 1.0f / lf : 0.0f)));
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
      tc_fence_after();
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
    if (!ok && t == 0) atomicOr(flags, CSA2_FLAG_TIMEOUT);
  } else {
    for (int l = 0; l < gv; ++l)
      for (int e = t; e < CSA2_H * CSA2_D; e += kThreads) layers.out[l0 + l][int64_t(inst) * CSA2_H * CSA2_D + e] = 0;
  }
  if (t < N && (t >> 4) < gv && layers.lse[l0 + (t >> 4)]) {
    const float l = ms.l_fin[t];
    layers.lse[l0 + (t >> 4)][int64_t(inst) * CSA2_H + (t & 15)] = l > 0.0f ? (ms.m_fin[t] + log2f(l)) * kLn2 : -INFINITY;
  }
}

}  // namespace

// A run of layers that share their selected rows, two layers per CTA, one CTA per (query, pair).
cudaError_t launch_sparse_attn_pairs(const AttnLayers& layers, int n_layers, int per_layer, int Nq,
                                     const uint8_t* codes, const uint8_t* scales, int64_t cap, const int32_t* idx,
                                     const int32_t* n_valid, int k, const int32_t* swa_len, int W, float scale_log2,
                                     bool win_fp8, unsigned int* flags, cudaStream_t st) {
  static std::atomic<bool> attr_set[64];  // per device; set once, by any host thread
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(sparse_attn_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kPairSmem));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const dim3 grid{unsigned(per_layer), unsigned((n_layers + 1) / 2), 1u};
  return launch_pdl(sparse_attn_pair_kernel, grid, dim3(kThreads), kPairSmem, st, layers, n_layers, codes, scales, cap,
                    idx, n_valid, k, swa_len, W, Nq, scale_log2, int(win_fp8), flags);
}

}  // namespace csa2

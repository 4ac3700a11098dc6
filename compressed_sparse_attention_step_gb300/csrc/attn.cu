// Sparse attention of each query's 16 heads over its selected FP4 main-KV rows plus its
// sliding-window rows ("Every layer retains its own main Q and sliding-window key-value cache",
// ai-maestro.online "DeepSeek AI released DeepSeek-V4.1-Flash with 1M context, FP4", section
// "Compressed Sparse Attention 2"; the 128-token window: section "Causal Encoder-Decoder
// architecture"; E2M1 codes with an E4M3 scale per 16 channels: section "FP4 KV, Bounded Replay,
// and other extensions").  K = V = the dequantised row.
//
// A query's rows form 64-row tiles: the window rows (ceil(W/64) tiles), then the selected FP4 rows
// (ceil(k/64) tiles).  A CTA takes a contiguous range of one query's tiles (the split); two CTAs
// fit on an SM so that one's loads and conversions overlap the other's tensor-core work.  Per CTA:
//   - the first window tile is copied straight into the operand buffer while the source rows of
//     the other tiles are resolved and pulled into L2;
//   - the next FP4 tile's bytes are copied (cp.async) into a staging buffer while the current tile
//     is processed; window rows are loaded into registers before the operand buffer frees up;
//   - per tile, the rows are written to shared memory as a 64 x 512 operand in the 128-byte-swizzled
//     layout the tensor core reads (FP4 rows dequantised to f16 with the E2M1 -> f16x2 and
//     E4M3 -> f16x2 hardware conversions and one exact f16 multiply; window rows as bf16);
//   - eight warps each issue an eighth of S^T = K Q^T on the 5th-generation tensor core
//     (tcgen05.mma, M = 64 rows, N = 16 heads, 64 of the 512 channels each) into their own
//     tensor-memory accumulator; a chain of N = 16 MMAs is bound by per-instruction latency, so
//     independent chains from several warps run side by side;
//   - the warps read the eight partial S^T back (one row per lane), add them, run the online
//     softmax and write P^T.  A running offset moves only when a score passes it by more than 2^12
//     (one block barrier with an OR tells every warp whether any did; only then the tile's maxima);
//   - four warps each issue one 128-channel block of O^T += V^T P^T (M = 128 channels, N = 16
//     heads, K = 64 rows), V^T being the same shared-memory tile read channel-major; O^T stays in
//     tensor memory across the CTA's tiles and is rescaled there when an offset moves.
// Splits of a query are merged by the last CTA to finish (an atomic ticket), in split order, so
// the result does not depend on which CTA finishes last.
//
// This kernel runs every launch of more than one CTA per SM (the decode group's 256 queries, prefill
// chunks), where the second CTA on an SM hides each CTA's setup and tail; launches that fit in one
// wave (a Full layer's split query, the hierarchical step's 40 queries) go to the warp-specialised
// kernel of attn_ws.cu, whose pipeline overlaps the tiles of one query.
//
// Operand types: a tile's MMA operands share one type.  FP4 tiles run in f16: the dequantised row
// is exact in f16 (at most 6 significant bits, magnitudes in [2^-10, 2688]), Q is converted from
// bf16 (exact for magnitudes in [2^-14, 65504]) and P is rounded to f16.  Window tiles run in bf16
// with Q and the rows as given and P rounded to bf16.  Accumulation is fp32.
//
// Tensor-memory layouts used: for M = 128 accumulator row r is lane r; for M = 64 row r is lane
// 32 (r / 16) + r % 16; column n is column n in both.
#include <cuda_fp16.h>

#include <algorithm>

#include "attn_common.cuh"

namespace csa2 {
namespace {
using namespace attn;

constexpr int kMaxTiles = (CSA2_MAX_ATTN_K + kRows - 1) / kRows + (CSA2_MAX_W + kRows - 1) / kRows;
constexpr int kSIssuers = 8;         // warps whose lane 0 issues a 64-channel eighth of S^T (independent chains)
constexpr int kOIssuers = 4;         // warps whose lane 0 issues a 128-channel block of O^T
constexpr uint32_t kOCol = 16 * kSIssuers;  // S^T partial i in columns [16 i, 16 i + 16); O^T block i at kOCol + 16 i
constexpr uint32_t kTmemCols = 256;
// Lazy rescaling: a head's running offset moves only when a tile's maximum exceeds it by more than
// this many (log2 units), so P = 2^(x - m) stays below 2^12 (f16 P stays far from its 65504 limit)
// and the accumulated O^T and sums are rescaled only on such a jump.
constexpr float kLazy = 12.0f;

// Shared-memory map (offsets from a 1024-byte aligned base).
constexpr uint32_t kTileGroup = kRows * 128;                 // 8 KiB per 64-channel group
constexpr uint32_t kTileOff = 0;                             // 8 groups x 64 rows x 128 B
constexpr uint32_t kQGroup = CSA2_H * 128;                   // 2 KiB
constexpr uint32_t kQOff = kTileOff + 8 * kTileGroup;        // Q: 8 groups x 16 heads x 128 B
constexpr uint32_t kPOff = kQOff + 8 * kQGroup;              // P^T: 16 heads x 64 rows (128 B)
constexpr uint32_t kRawOff = kPOff + kQGroup;                // staged FP4 codes: 64 rows x 256 B
constexpr uint32_t kRawScOff = kRawOff + kRows * CSA2_CODE_BYTES;  // staged scales: 64 rows x 32 B
constexpr uint32_t kMiscOff = kRawScOff + kRows * CSA2_SCALE_BYTES;

struct Misc {
  unsigned long long mbar_s;      // S^T of a tile complete (one arrival per S issuer)
  unsigned long long mbar_o;      // O^T of a tile complete (one arrival per O issuer)
  uint32_t tmem_base;
  int is_last;
  int32_t pos[kMaxTiles][kRows];  // source row of each row of the CTA's tiles, -1 if empty
  float red[4][CSA2_H];           // per-quarter tile maximum, then (at the end) partial sums
  float m_fin[CSA2_H];            // final offset per head (log2 units)
  float l_fin[CSA2_H];            // final sum per head
};
constexpr size_t kSmemBytes = 1024 + kMiscOff + sizeof(Misc);

__global__ void __launch_bounds__(kThreads, 2) sparse_attn_kernel(
    const __grid_constant__ AttnLayers layers, int Nq, const uint8_t* __restrict__ codes,
    const uint8_t* __restrict__ scales, int64_t cap, const int32_t* __restrict__ idx,
    const int32_t* __restrict__ n_valid, int k, const int32_t* __restrict__ swa_len, int W, float scale_log2,
    int n_split, float* __restrict__ ws, unsigned int* __restrict__ tickets, unsigned int* flags, int win_fp8) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // the selected positions may come from the kernel right before this one
  pdl_wait();
  pdl_trigger();
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  unsigned char* base = smem_raw + (base_s - raw_s);
  Misc& ms = *reinterpret_cast<Misc*>(base + kMiscOff);
  const uint32_t tile_s = base_s + kTileOff, q_s = base_s + kQOff, p_s = base_s + kPOff;
  const uint32_t mbar_s = smem_u32(&ms.mbar_s), mbar_o = smem_u32(&ms.mbar_o);

  // blockIdx.z: the layer; blockIdx.y: the query (its selected rows are the same in every layer);
  // ginst: the instance's slot in the split workspace and tickets
  const int inst = blockIdx.y, split = blockIdx.x;
  const int64_t ginst = int64_t(blockIdx.z) * gridDim.y + inst;
  const uint16_t* __restrict__ q = layers.q[blockIdx.z];
  const uint16_t* __restrict__ swa = layers.swa[blockIdx.z];
  uint16_t* __restrict__ out = layers.out[blockIdx.z];
  float* __restrict__ lse = layers.lse[blockIdx.z];
  const int b = inst / Nq, qi = inst - b * Nq;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int quarter = warp & 3, half = warp >> 2;  // TMEM lane quarter; heads / channel blocks half

  // ---- this split's tiles: window tiles first, then FP4 tiles ---------------------------------------
  const int nwin = swa ? (W + kRows - 1) / kRows : 0;
  const int ntiles = nwin + (k + kRows - 1) / kRows;
  const int t_begin = split * ntiles / n_split, t_end = (split + 1) * ntiles / n_split;
  const int n_fp4_valid = min(k, n_valid ? max(n_valid[inst], 0) : k);
  const int SW = W - 1 + Nq;
  const int swa_lo = swa ? SW - min(max(swa_len[b], 0), SW) : SW;
  // a tile can hold a row: window tiles reaching a stored row, FP4 tiles below n_fp4_valid
  auto live = [&](int tile) {
    if (tile < nwin) return qi + min((tile + 1) * kRows, W) - 1 >= swa_lo;
    return (tile - nwin) * kRows < n_fp4_valid;
  };
  int first_live = -1, last_live = -1;
  for (int tile = t_begin; tile < t_end; ++tile)
    if (live(tile)) {
      if (first_live < 0) first_live = tile;
      last_live = tile;
    }

  const int32_t* irow = (layers.idx[blockIdx.z] ? layers.idx[blockIdx.z] : idx) + int64_t(inst) * k;
  const uint8_t* cbase = codes + int64_t(b) * cap * CSA2_CODE_BYTES;
  const uint8_t* sbase = scales + int64_t(b) * cap * CSA2_SCALE_BYTES;
  const uint16_t* swbase = swa ? swa + int64_t(b) * SW * CSA2_D : nullptr;
  // 8-bit window: E4M3 bytes, rows of 512 B
  const uint8_t* sw8 = swa ? reinterpret_cast<const uint8_t*>(swa) + int64_t(b) * SW * CSA2_D : nullptr;
  const uint16_t* qrow = q + int64_t(inst) * CSA2_H * CSA2_D;

  // window row of tile row r of window tile `tile`, or -1
  auto win_row = [&](int tile, int r) {
    const int wr = tile * kRows + r;
    return (wr < W && qi + wr >= swa_lo) ? qi + wr : -1;
  };
  // window tile -> operand tile (cp.async; empty rows are zero-filled)
  // thread t: rows (t & 7) + 8 (j & 7), 16-byte chunks (t >> 3) + 32 (j >> 3), j = 0..15
  auto copy_window = [&](int tile) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int r = (t & 7) + 8 * (j & 7), cc = (t >> 3) + 32 * (j >> 3);
      const int br = win_row(tile, r);
      const uint16_t* src = br >= 0 ? swbase + int64_t(br) * CSA2_D + 8 * cc : swa;
      cp_async16(tile_s + sw128(kTileGroup, r, cc), src, br >= 0 ? 16 : 0);
    }
    cp_async_commit();
  };

  if (t < CSA2_H) {
    ms.m_fin[t] = -INFINITY;
    ms.l_fin[t] = 0.0f;
  }
  if (first_live >= 0) {
    // tensor memory, the MMA barriers, and the first window tile's rows, before anything waits
    if (t == 0) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(mbar_s), "r"(kSIssuers) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(mbar_o), "r"(kOIssuers) : "memory");
      asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 0) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(&ms.tmem_base)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    if (first_live < nwin && !win_fp8) copy_window(first_live);
  }
  // ---- source rows of every tile of the split; FP4 and later window rows pulled into L2 ------------
  for (int e = t; e < (t_end - t_begin) * kRows; e += kThreads) {
    const int tile = t_begin + e / kRows, r = e % kRows;
    int32_t p = -1;
    if (tile >= nwin) {
      const int slot = (tile - nwin) * kRows + r;
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
      p = win_row(tile, r);
      if (p >= 0 && win_fp8) {
        const uint8_t* sr = sw8 + int64_t(p) * CSA2_D;
#pragma unroll
        for (int l = 0; l < 4; ++l) asm volatile("prefetch.global.L2 [%0];" ::"l"(sr + 128 * l));
      } else if (p >= 0 && tile != first_live) {
        const uint16_t* sr = swbase + int64_t(p) * CSA2_D;
#pragma unroll
        for (int l = 0; l < 8; ++l) asm volatile("prefetch.global.L2 [%0];" ::"l"(sr + 64 * l));
      }
    }
    ms.pos[tile - t_begin][r] = p < 0 ? -1 : p;
  }
  tc_fence_before();
  __syncthreads();

  // FP4 tile -> staging buffer (cp.async; empty rows are zero-filled).  Thread t copies 16-byte
  // piece (t >> 3) & 15 of rows (t & 7) + 8 ((t >> 7) + 2 i), i < 4, and one half of row t >> 1's
  // scale bytes.
  auto stage_fp4 = [&](int tile) {
    const int32_t* pos = ms.pos[tile - t_begin];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = (t & 7) + 8 * ((t >> 7) + 2 * i), piece = (t >> 3) & 15;
      const int32_t p = pos[r];
      const uint8_t* src = p >= 0 ? cbase + int64_t(p) * CSA2_CODE_BYTES + 16 * piece : codes;
      cp_async16(base_s + kRawOff + raw_off(r, piece), src, p >= 0 ? 16 : 0);
    }
    if (t < 2 * kRows) {
      const int r = t >> 1, h2 = t & 1;
      const int32_t p = pos[r];
      const uint8_t* src = p >= 0 ? sbase + int64_t(p) * CSA2_SCALE_BYTES + 16 * h2 : scales;
      cp_async16(base_s + kRawScOff + r * CSA2_SCALE_BYTES + 16 * h2, src, p >= 0 ? 16 : 0);
    }
    cp_async_commit();
  };
  auto next_live = [&](int tile) {
    while (tile <= last_live && !live(tile)) ++tile;
    return tile;
  };

  bool ok = true;
  if (first_live >= 0) {
    tc_fence_after();
    const uint32_t tmem = ms.tmem_base;
    const uint32_t t_lane = tmem + (uint32_t(32 * quarter) << 16);  // this warp's lane quarter
    const int first_fp4 = next_live(max(first_live, nwin));
    if (first_fp4 <= last_live) stage_fp4(first_fp4);  // first FP4 tile, behind any window tile's copy
    uint32_t ph_s = 0, ph_o = 0;
    int q_kind = -1;  // 0: Q staged as f16, 1: as bf16
    bool first = true;
    // mj[j]: the running offset of head 8 half + j (the same in every thread of the half); ls[j]: this
    // lane's row's running sum for that head; lanes 0..15 also keep the offset of head `lane` in m_h
    float mj[8], ls[8], m_h = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      mj[j] = -INFINITY;
      ls[j] = 0.0f;
    }

    for (int tile = first_live; tile <= last_live; ++tile) {
      if (!live(tile)) continue;
      const bool is_fp4 = tile >= nwin;
      const int32_t* pos = ms.pos[tile - t_begin];
      // -- a later window tile: half of its rows into registers before the operand tile is free
      auto win_load = [&](int j) -> uint4 {
        const int r = (t & 7) + 8 * (j & 7), cc = (t >> 3) + 32 * (j >> 3);
        const int32_t br = pos[r];
        return br >= 0 ? __ldg(reinterpret_cast<const uint4*>(swbase + int64_t(br) * CSA2_D + 8 * cc))
                       : make_uint4(0, 0, 0, 0);
      };
      auto win_store = [&](int j, uint4 v) {
        const int r = (t & 7) + 8 * (j & 7), cc = (t >> 3) + 32 * (j >> 3);
        *reinterpret_cast<uint4*>(base + kTileOff + sw128(kTileGroup, r, cc)) = v;
      };
      const bool f16_tile = is_fp4 || win_fp8;  // operands in f16 (FP4 rows, 8-bit window rows)
      const bool win8 = !is_fp4 && win_fp8;
      const bool win_regs = !is_fp4 && !win_fp8 && !first;
      uint4 wv[8];
      if (win_regs) {
#pragma unroll
        for (int j = 0; j < 8; ++j) wv[j] = win_load(j);
      } else if (win8) {
        // 8-bit window tile: thread t loads 16 channels (16 B, piece t >> 3) of rows (t & 7) + 8 j
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int32_t br = pos[(t & 7) + 8 * j];
          wv[j] = br >= 0 ? __ldg(reinterpret_cast<const uint4*>(sw8 + int64_t(br) * CSA2_D + 16 * (t >> 3)))
                          : make_uint4(0, 0, 0, 0);
        }
      }
      // -- the previous tile's O^T MMAs read the operand tile and P^T: wait for them
      if (!first) {
        ok = ok && mbar_wait(mbar_o, ph_o);
        ph_o ^= 1u;
      }
      // -- Q in the tile's operand type
      const int kind = f16_tile ? 0 : 1;
      if (kind != q_kind) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int h = (t & 7) + 8 * (j & 1), cc = (t >> 3) + 32 * (j >> 1);
          uint4 v = __ldg(reinterpret_cast<const uint4*>(qrow + h * CSA2_D + 8 * cc));
          if (kind == 0) {
            v.x = bf16x2_to_f16x2(v.x);
            v.y = bf16x2_to_f16x2(v.y);
            v.z = bf16x2_to_f16x2(v.z);
            v.w = bf16x2_to_f16x2(v.w);
          }
          *reinterpret_cast<uint4*>(base + kQOff + sw128(kQGroup, h, cc)) = v;
        }
        q_kind = kind;
      }
      // -- rows -> operand tile
      if (is_fp4) {
        cp_async_wait<0>();
        __syncthreads();  // every thread's staged pieces are visible
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = (t & 7) + 8 * ((t >> 7) + 2 * i), piece = (t >> 3) & 15;
          const uint4 cw = *reinterpret_cast<const uint4*>(base + kRawOff + raw_off(r, piece));
          const uint16_t s2 = *reinterpret_cast<const uint16_t*>(base + kRawScOff + r * CSA2_SCALE_BYTES + 2 * piece);
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
      } else if (win_regs) {
        // the second half of the rows' channels by cp.async (empty rows zero-filled) while the first
        // half, already in registers, is stored; the FP4 tile staged before it is older and done
#pragma unroll
        for (int j = 8; j < 16; ++j) {
          const int r = (t & 7) + 8 * (j & 7), cc = (t >> 3) + 32 * (j >> 3);
          const int32_t br = pos[r];
          cp_async16(tile_s + sw128(kTileGroup, r, cc), br >= 0 ? swbase + int64_t(br) * CSA2_D + 8 * cc : swa,
                     br >= 0 ? 16 : 0);
        }
        cp_async_commit();
#pragma unroll
        for (int j = 0; j < 8; ++j) win_store(j, wv[j]);
        cp_async_wait<0>();
      } else if (first_fp4 <= last_live) {
        cp_async_wait<1>();  // the window copy; the staged FP4 tile may still be in flight
      } else {
        cp_async_wait<0>();
      }
      fence_async_smem();
      __syncthreads();

      // -- S^T = K Q^T (tensor core): warp i < 8 issues the 64 channels [64 i, 64 i + 64) in 4 steps
      if (lane == 0 && warp < kSIssuers) {
        tc_fence_after();
        const uint32_t id = instr_desc(kRows, !f16_tile, false);
#pragma unroll
        for (int k4 = 0; k4 < CSA2_D / 16 / kSIssuers; ++k4) {
          const uint32_t off = uint32_t(k4) * 32u;  // 16 channels = 32 B inside the swizzle atom
          const uint64_t a = smem_desc(tile_s + uint32_t(warp) * kTileGroup + off, 0, 1024);
          const uint64_t bq = smem_desc(q_s + uint32_t(warp) * kQGroup + off, 0, 1024);
          umma_f16(tmem + uint32_t(16 * warp), a, bq, id, k4 > 0 ? 1u : 0u);
        }
        umma_commit(mbar_s);
      }
      ok = ok && mbar_wait(mbar_s, ph_s);
      ph_s ^= 1u;
      tc_fence_after();
      // -- the staging buffer is free again: copy the next FP4 tile while this one is computed
      if (is_fp4) {
        const int nxt = next_live(tile + 1);
        if (nxt <= last_live) stage_fp4(nxt);
      }

      // -- online softmax: warp (quarter, half) holds rows 16 quarter + lane (lanes < 16) and
      //    heads 8 half .. 8 half + 7; S^T is the sum of the eight channel-eighth partials
      const int row = 16 * quarter + (lane & 15);
      float x[8];
      {
        // ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7)), the first half summed before the second loads
        float sp[4][8], lo4[8];
        tmem_ld8x4(t_lane + uint32_t(8 * half), sp);  // partials 0..3
#pragma unroll
        for (int j = 0; j < 8; ++j) lo4[j] = (sp[0][j] + sp[1][j]) + (sp[2][j] + sp[3][j]);
        tmem_ld8x4(t_lane + 64u + uint32_t(8 * half), sp);  // partials 4..7
        const bool row_ok = lane < 16 && pos[row] >= 0;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          x[j] = row_ok ? (lo4[j] + ((sp[0][j] + sp[1][j]) + (sp[2][j] + sp[3][j]))) * scale_log2 : -INFINITY;
      }
      // Does any score pass its head's offset by more than kLazy?  Usually not, and then the offsets
      // stay and no maximum is needed (one block barrier with an OR); otherwise the tile's maxima set
      // the offsets that move, and the O^T accumulated so far (complete: its MMAs were waited for
      // above) and the sums are rescaled.
      bool jump = false;
#pragma unroll
      for (int j = 0; j < 8; ++j) jump |= x[j] > mj[j] + kLazy;
      tc_fence_before();
      if (__syncthreads_or(jump)) {
        const float mx = reduce_scatter8<true>(x, lane);
        if ((lane & 3) == 0) ms.red[quarter][8 * half + (lane >> 2)] = mx;
        __syncthreads();
        // lanes 0..15: head `lane`'s new offset and the factor that rescales what came before
        float mn = m_h, corr = 1.0f;
        if (lane < 16) {
          const float mt = fmaxf(fmaxf(ms.red[0][lane], ms.red[1][lane]), fmaxf(ms.red[2][lane], ms.red[3][lane]));
          mn = mt > m_h + kLazy ? mt : m_h;
          corr = (mn != m_h && m_h != -INFINITY) ? ex2(m_h - mn) : 1.0f;
          m_h = mn;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          mj[j] = __shfl_sync(0xffffffffu, mn, 8 * half + j);
          ls[j] *= __shfl_sync(0xffffffffu, corr, 8 * half + j);
        }
        if (__any_sync(0xffffffffu, corr != 1.0f)) {
          // channel blocks 2 half, 2 half + 1 of this lane quarter
          tc_fence_after();
          float cr[16];
#pragma unroll
          for (int h = 0; h < 16; ++h) cr[h] = __shfl_sync(0xffffffffu, corr, h);
          const uint32_t ta = t_lane + kOCol + uint32_t(32 * half);
          float o[2][16];
          tmem_ld16x2(ta, o);
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int h = 0; h < 16; ++h) o[j][h] *= cr[h];
          tmem_st16x2(ta, o);
        }
      }
      float pr[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        // an empty row (x = -inf) gives 0; a finite x has a finite offset (the tile that first held a
        // finite score for the head took the slow path)
        pr[j] = x[j] == -INFINITY ? 0.0f : ex2(x[j] - mj[j]);
        ls[j] += pr[j];
      }
      // P^T (heads x rows, K-major, 128-byte swizzle): element (h, row)
      if (lane < 16) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int h = 8 * half + j;
          const uint32_t off = uint32_t(h) * 128u + uint32_t(((row >> 3) ^ (h & 7)) << 4) + uint32_t(row & 7) * 2u;
          const uint16_t bits = f16_tile ? __half_as_ushort(__float2half_rn(pr[j])) : uint16_t(f2bf_bits(pr[j]));
          *reinterpret_cast<uint16_t*>(base + kPOff + off) = bits;
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();

      // -- O^T += V^T P^T (tensor core): warp i < 4 issues channel block i in 4 steps of 16 rows
      if (lane == 0 && warp < kOIssuers) {
        tc_fence_after();
        const uint32_t id = instr_desc(128, !f16_tile, true);
        const int i = warp;
#pragma unroll
        for (int s = 0; s < kRows / 16; ++s) {
          const uint64_t a = smem_desc(tile_s + uint32_t(2 * i) * kTileGroup + uint32_t(s) * 2048u, kTileGroup, 1024);
          const uint64_t bp = smem_desc(p_s + uint32_t(s) * 32u, 0, 1024);
          umma_f16(tmem + kOCol + uint32_t(16 * i), a, bp, id, (first && s == 0) ? 0u : 1u);
        }
        umma_commit(mbar_o);
      }
      first = false;
    }
    // ---- last tile's MMAs, the sums per head, then O^T out of tensor memory -------------------------
    ok = ok && mbar_wait(mbar_o, ph_o);
    tc_fence_after();
    const float l_w = reduce_scatter8<false>(ls, lane);  // this warp's rows, head 8 half + lane / 4
    if ((lane & 3) == 0) ms.red[quarter][8 * half + (lane >> 2)] = l_w;
    __syncthreads();
    if (t < CSA2_H) {
      ms.l_fin[t] = (ms.red[0][t] + ms.red[1][t]) + (ms.red[2][t] + ms.red[3][t]);
      ms.m_fin[t] = m_h;
    }
    __syncthreads();
    float o[2][16];
    tmem_ld16x2(t_lane + kOCol + uint32_t(32 * half), o);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int ch = 128 * (2 * half + j) + 32 * quarter + lane;
      if (n_split == 1) {
        uint16_t* orow = out + int64_t(inst) * CSA2_H * CSA2_D + ch;
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const float l = ms.l_fin[h];
          orow[h * CSA2_D] = uint16_t(f2bf_bits(o[j][h] * (l > 0.0f ? 1.0f / l : 0.0f)));
        }
      } else {
        float* po = ws + (ginst * n_split + split) * (CSA2_H * CSA2_D) + ch;
#pragma unroll
        for (int h = 0; h < 16; ++h) po[h * CSA2_D] = o[j][h];
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
    if (n_split == 1) {
      uint16_t* orow = out + int64_t(inst) * CSA2_H * CSA2_D;
      for (int e = t; e < CSA2_H * CSA2_D; e += kThreads) orow[e] = 0;
    }
  }

  if (n_split == 1) {
    if (lse && t < CSA2_H) {
      const float l = ms.l_fin[t];
      lse[int64_t(inst) * CSA2_H + t] = l > 0.0f ? (ms.m_fin[t] + log2f(l)) * kLn2 : -INFINITY;
    }
    return;
  }
  // ---- split partials, then the last CTA of this query merges them ------------------------------
  const int64_t instances = int64_t(gridDim.y) * gridDim.z;
  float* mlb = ws + instances * n_split * (CSA2_H * CSA2_D);
  if (t < CSA2_H) {
    float* ml = mlb + (ginst * n_split + split) * (2 * CSA2_H);
    ml[2 * t] = ms.m_fin[t];
    ml[2 * t + 1] = ms.l_fin[t];
  }
  __threadfence();
  __syncthreads();
  if (t == 0) ms.is_last = (atomicAdd(tickets + ginst, 1u) == unsigned(n_split - 1));
  __syncthreads();
  if (!ms.is_last) return;
  __threadfence();
  // o = sum_j 2^(m_j - M) O_j / sum_j 2^(m_j - M) l_j over the splits with rows, in split order.
  // The per-head weights go through shared memory (the operand tile is free now): wgt[j][h] holds
  // m_j then the weight, wgt[kMaxSplit + j][h] holds l_j, then 1 / L and the lse per head.  The
  // partials are read coalesced: thread t takes float4 t + 256 v (v < 8) of the 16 x 512 block,
  // i.e. head (t >> 7) + 2 v, channels 4 (t & 127) .. + 3.
  float* wgt = reinterpret_cast<float*>(base + kTileOff);
  {
    const float* ml = mlb + ginst * n_split * (2 * CSA2_H);
    for (int e = t; e < n_split * CSA2_H; e += kThreads) {
      wgt[e] = __ldcg(ml + 2 * e);                            // m_j, e = j * 16 + h
      wgt[kMaxSplit * CSA2_H + e] = __ldcg(ml + 2 * e + 1);   // l_j
    }
    __syncthreads();
    if (t < CSA2_H) {
      float M = -INFINITY;
      for (int j = 0; j < n_split; ++j)
        if (wgt[kMaxSplit * CSA2_H + j * CSA2_H + t] > 0.0f) M = fmaxf(M, wgt[j * CSA2_H + t]);
      float L = 0.0f;
      for (int j = 0; j < n_split; ++j) {
        const float lj = wgt[kMaxSplit * CSA2_H + j * CSA2_H + t];
        const float a = (lj > 0.0f && M != -INFINITY) ? exp2f(wgt[j * CSA2_H + t] - M) : 0.0f;
        L += a * lj;
        wgt[j * CSA2_H + t] = a;
      }
      wgt[2 * kMaxSplit * CSA2_H + t] = L > 0.0f ? 1.0f / L : 0.0f;
      wgt[2 * kMaxSplit * CSA2_H + CSA2_H + t] = L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
    __syncthreads();
  }
  {
    const float4* p0 = reinterpret_cast<const float4*>(ws + ginst * n_split * (CSA2_H * CSA2_D)) + t;
    float4 acc[8];
#pragma unroll
    for (int v = 0; v < 8; ++v) acc[v] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int j0 = 0; j0 < n_split; j0 += 2) {
      const int j1 = min(j0 + 1, n_split - 1);
      float4 x0[8], x1[8];
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        x0[v] = __ldcg(p0 + int64_t(j0) * (CSA2_H * CSA2_D / 4) + kThreads * v);
        x1[v] = __ldcg(p0 + int64_t(j1) * (CSA2_H * CSA2_D / 4) + kThreads * v);
      }
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const int h = (t >> 7) + 2 * v;
        // a split without rows wrote no partial: its (zero-weight) slot is never read into acc
        const float a0 = wgt[j0 * CSA2_H + h], a1 = j1 > j0 ? wgt[j1 * CSA2_H + h] : 0.0f;
        if (a0 != 0.0f) {
          acc[v].x += a0 * x0[v].x;
          acc[v].y += a0 * x0[v].y;
          acc[v].z += a0 * x0[v].z;
          acc[v].w += a0 * x0[v].w;
        }
        if (a1 != 0.0f) {
          acc[v].x += a1 * x1[v].x;
          acc[v].y += a1 * x1[v].y;
          acc[v].z += a1 * x1[v].z;
          acc[v].w += a1 * x1[v].w;
        }
      }
    }
    uint16_t* orow = out + int64_t(inst) * CSA2_H * CSA2_D;
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const int h = (t >> 7) + 2 * v;
      const float inv = wgt[2 * kMaxSplit * CSA2_H + h];
      *reinterpret_cast<uint2*>(orow + 4 * (t + kThreads * v)) =
          make_uint2(pack_bf16x2(acc[v].x * inv, acc[v].y * inv), pack_bf16x2(acc[v].z * inv, acc[v].w * inv));
    }
    if (lse && t < CSA2_H) lse[int64_t(inst) * CSA2_H + t] = wgt[2 * kMaxSplit * CSA2_H + CSA2_H + t];
  }
  if (t == 0) tickets[ginst] = 0u;  // ready for the next launch
}

int attn_tiles(int k, int W) { return (k + kRows - 1) / kRows + (W > 0 ? (W + kRows - 1) / kRows : 0); }

}  // namespace

// Splits actually launched: at most one per tile.
int attn_effective_split(int k, int W, int n_split) {
  return std::max(1, std::min(n_split, std::max(attn_tiles(k, W), 1)));
}

// one ticket per query (zero before a launch; every launch leaves them zero), padded to 256 B,
// then the partial O and (m, l) of every split
size_t attn_ticket_bytes(int64_t instances) { return (size_t(instances) * sizeof(unsigned int) + 255) & ~size_t(255); }
size_t attn_ws_bytes(int64_t instances, int n_split) {
  if (n_split <= 1) return 0;
  return attn_ticket_bytes(instances) +
         size_t(instances) * size_t(n_split) * (CSA2_H * CSA2_D + 2 * CSA2_H) * sizeof(float);
}

// SMs of the current device, looked up once per device.
int sm_count() {
  static std::atomic<int> count[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  int c = count[dev].load();
  if (c <= 0) {
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0) c = 152;
    count[dev] = c;
  }
  return c;
}

// Launches of at most this many CTAs per SM run the warp-specialised kernel (one CTA per SM, so one
// wave); larger ones this kernel, whose second CTA per SM hides each CTA's setup.
constexpr int kWsMaxCtasPerSm = 1;

int attn_auto_split(int64_t instances, int k, int W) {
  const int nt = attn_tiles(k, W);
  if (instances <= 0 || nt <= 0) return 1;
  const int64_t slots = sm_count();  // one CTA per SM for the launches that split
  int64_t s = std::max<int64_t>(slots / instances, 1);
  s = std::min<int64_t>(s, std::min(nt, kMaxSplit));
  return int(std::max<int64_t>(s, 1));
}

// The pair path (attn_pair.cu) for a run of layers that attend the same selected rows: two layers per
// CTA, one CTA per (query, pair), two CTAs per SM.  Taken when those CTAs fill at least one wave;
// smaller runs keep the per-layer kernels, which split a query over CTAs.
bool attn_pair_path(int64_t per_layer, int n_layers) {
  if (n_layers < 2 || per_layer <= 0) return false;
  return per_layer * ((n_layers + 1) / 2) >= 2 * int64_t(sm_count());
}

cudaError_t launch_sparse_attn_layers(const AttnLayers& layers, int n_layers, int B, int Nq, const uint8_t* codes,
                                      const uint8_t* scales, int64_t cap, const int32_t* idx,
                                      const int32_t* n_valid, int k, const int32_t* swa_len, int W,
                                      float softmax_scale, int n_split, float* ws, cudaStream_t st,
                                      bool tickets_zeroed, bool win_fp8, bool allow_pairs) {
  const int64_t per_layer = int64_t(B) * Nq, instances = per_layer * n_layers;
  if (instances == 0) return cudaSuccess;
  if (n_layers < 1 || n_layers > CSA2_MAX_LAYERS || per_layer > 65535) return cudaErrorInvalidValue;
  if (!layers.swa[0]) W = 0;
  n_split = attn_effective_split(k, W, n_split);
  unsigned int* flags = device_flags_ptr();
  if (!flags) return cudaErrorUnknown;
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  unsigned int* tickets = nullptr;
  float* partials = nullptr;
  // the pair path, when every layer of the run attends the same rows
  bool shared_rows = true;
  for (int l = 1; l < n_layers; ++l) shared_rows = shared_rows && layers.idx[l] == layers.idx[0];
  if (allow_pairs && shared_rows && attn_pair_path(per_layer, n_layers))
    return launch_sparse_attn_pairs(layers, n_layers, int(per_layer), Nq, codes, scales, cap, idx, n_valid, k, swa_len,
                                    W, scale_log2, win_fp8, flags, st);
  if (n_split > 1) {
    tickets = reinterpret_cast<unsigned int*>(ws);
    partials = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + attn_ticket_bytes(instances));
    if (!tickets_zeroed) {
      cudaError_t e = cudaMemsetAsync(tickets, 0, size_t(instances) * sizeof(unsigned int), st);
      if (e != cudaSuccess) return e;
    }
  }
  if (instances * n_split <= int64_t(kWsMaxCtasPerSm) * sm_count())
    return launch_sparse_attn_ws(layers, n_layers, int(per_layer), Nq, codes, scales, cap, idx, n_valid, k, swa_len,
                                 W, scale_log2, n_split, partials, tickets, flags, win_fp8, st);
  static std::atomic<bool> attr_set[64];  // per device; set once, by any host thread
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const dim3 grid{unsigned(n_split), unsigned(per_layer), unsigned(n_layers)};
  return launch_pdl(sparse_attn_kernel, grid, dim3(kThreads), kSmemBytes, st, layers, Nq, codes, scales, cap, idx,
                    n_valid, k, swa_len, W, scale_log2, n_split, partials, tickets, flags, int(win_fp8));
}

cudaError_t launch_sparse_attn(const uint16_t* q, int B, int Nq, const uint8_t* codes,
                               const uint8_t* scales, int64_t cap, const int32_t* idx,
                               const int32_t* n_valid, int k, const uint16_t* swa,
                               const int32_t* swa_len, int W, float softmax_scale, uint16_t* out,
                               float* lse, int n_split, float* ws, cudaStream_t st, bool tickets_zeroed) {
  AttnLayers layers{};
  layers.q[0] = q;
  layers.swa[0] = swa;
  layers.out[0] = out;
  layers.lse[0] = lse;
  return launch_sparse_attn_layers(layers, 1, B, Nq, codes, scales, cap, idx, n_valid, k, swa_len, W, softmax_scale,
                                   n_split, ws, st, tickets_zeroed, false, false);
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
  const int ns = csa2::attn_effective_split(k, W, n_split ? n_split : csa2::attn_auto_split(instances, k, W));
  const size_t need = csa2::attn_ws_bytes(instances, ns);
  if (need && (!ws || ws_bytes < need || !al16(ws))) return CSA2_ERR_WORKSPACE;
  return csa2::launch_sparse_attn(q, B, Nq, codes, scales, cap, idx, n_valid, k, swa, swa_len, W,
                                  softmax_scale, out, lse, ns, static_cast<float*>(ws),
                                  reinterpret_cast<cudaStream_t>(stream), false) == cudaSuccess
             ? CSA2_OK
             : CSA2_ERR_CUDA;
}

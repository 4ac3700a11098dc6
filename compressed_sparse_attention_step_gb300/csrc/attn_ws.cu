// Sparse attention of each query's 16 heads over its selected FP4 main-KV rows plus its
// sliding-window rows ("Every layer retains its own main Q and sliding-window key-value cache",
// ai-maestro.online "DeepSeek AI released DeepSeek-V4.1-Flash with 1M context, FP4", section
// "Compressed Sparse Attention 2"; the 128-token window: section "Causal Encoder-Decoder
// architecture"; E2M1 codes with an E4M3 scale per 16 channels: section "FP4 KV, Bounded Replay,
// and other extensions").  K = V = the dequantised row.
//
// The warp-specialised kernel, for launches of at most one CTA per SM (one wave; larger launches run
// the kernel of attn.cu, whose two CTAs per SM hide each other's setup).  A
// query's rows form 64-row tiles: the selected FP4 rows (ceil(k/64) tiles), then the window rows
// (ceil(W/64) tiles).  A CTA takes a contiguous range of one query's tiles (the split) and runs its
// live tiles through a pipeline of warp roles, one CTA per SM:
//   - eight converter warps, one per 64-channel eighth, write their eighth of each tile into one of
//     three operand buffers (64 rows x 512 channels in the 128-byte-swizzled layout the tensor core
//     reads): FP4 rows (32 code bytes and two scale bytes of the eighth per row, loaded into
//     registers one tile ahead) dequantised to f16 with the E2M1 -> f16x2 and E4M3 -> f16x2
//     hardware conversions and one exact f16 multiply; window rows copied as bf16 (cp.async) or
//     converted from E4M3.  Each then issues its eighth of S^T = K Q^T on the 5th-generation
//     tensor core (tcgen05.mma, M = 64 rows, N = 16 heads, K = 64 channels) into its own
//     tensor-memory partial, in one of three S^T buffers;
//   - eight softmax warps read a tile's eight S^T partials (one row per lane), add them, run the
//     online softmax and write P^T.  A running offset moves only when a score exceeds it by more
//     than 2^12 (one barrier-reduction tells every softmax warp whether any did), and then the
//     tile's maxima set the offsets that move and the accumulated O^T is rescaled in tensor memory;
//   - four warps each issue one 128-channel block of O^T += V^T P^T (M = 128 channels, N = 16
//     heads, K = 64 rows), V^T being the operand tile read channel-major; O^T stays in tensor
//     memory.
// One thread issuing tcgen05.mma waits about 150 cycles per instruction while independent issuers
// overlap, so each tile's 48 MMAs come from 12 warps.  With three operand, S^T and P^T buffers the
// dependent chain convert -> S^T -> softmax -> O^T of a tile overlaps those of the two tiles after
// it.  Splits of a query are merged by the last CTA to finish (an atomic ticket), in split order,
// so the result does not depend on which CTA finishes last.
//
// Operand types: a tile's MMA operands share one type.  FP4 tiles run in f16: the dequantised row
// is exact in f16 (at most 6 significant bits, magnitudes in [2^-10, 2688]), Q is converted from
// bf16 (exact for magnitudes in [2^-14, 65504]) and P is rounded to f16.  Window tiles run in bf16
// with Q and the rows as given and P rounded to bf16 (8-bit window rows: f16, exact).  Accumulation
// is fp32.  One Q buffer serves both: each converter warp rewrites its eighth of Q as bf16 before
// the first bf16 window tile, once its own earlier S^T products are complete.
//
// Tensor-memory layouts used: for M = 128 accumulator row r is lane r; for M = 64 row r is lane
// 32 (r / 16) + r % 16; column n is column n in both.
//
// Synchronisation (mbarriers; n is a live tile's position in the CTA's range, b = n % 3; every wait
// is bounded and a wait that gives up raises CSA2_FLAG_TIMEOUT):
//   s_full[b]    S^T of tile n complete (8 commits)            s_free[b]  S^T of tile n read (8 warps)
//   p_full[b]    P^T of tile n written, O^T rescaled (8 softmax warps) -> O^T issuers
//   op_empty[b]  O^T of tile n complete (4 commits): its operand buffer and P^T buffer are free
//                again, and O^T may be rescaled or read out.
// No waiter falls two phases behind a barrier: each barrier's next phase needs the waiter's own
// progress first.
#include <cuda_fp16.h>

#include <algorithm>

#include "attn_common.cuh"

namespace csa2 {
namespace {
using namespace attn;

constexpr int kMaxTiles = (CSA2_MAX_ATTN_K + kRows - 1) / kRows + (CSA2_MAX_W + kRows - 1) / kRows;
constexpr int kNBuf = 3;                             // operand, S^T and P^T buffers
constexpr int kSoftWarps = 8;                        // softmax, epilogue and merge
constexpr int kConvWarps = 8;                        // operand eighths and S^T issue
constexpr int kOWarp0 = kSoftWarps + kConvWarps;     // four O^T issuers, one channel block each
constexpr int kWsThreads = 32 * (kOWarp0 + 4);       // 640: five warps per SM sub-partition
static_assert(kThreads == 32 * kSoftWarps, "the softmax warps run the epilogue and the merge");
constexpr uint32_t kSCols = 16 * kConvWarps;         // one S^T buffer: eight partials of 16 heads
constexpr uint32_t kOCol = kNBuf * kSCols;           // O^T block i at kOCol + 16 i
constexpr uint32_t kTmemCols = 512;
static_assert(kOCol + 4 * CSA2_H <= kTmemCols, "tensor memory");
// Lazy rescaling: a head's running offset moves only when a tile's maximum exceeds it by more than
// this many (log2 units), so P = 2^(x - m) stays below 2^12 (f16 P stays far from its 65504 limit)
// and the accumulated O^T and sums are rescaled only on such a jump.
constexpr float kLazy = 12.0f;

// Shared-memory map (offsets from a 1024-byte aligned base).
constexpr uint32_t kTileGroup = kRows * 128;             // 8 KiB per 64-channel group
constexpr uint32_t kOpBytes = 8 * kTileGroup;            // one operand tile
constexpr uint32_t kQGroup = CSA2_H * 128;               // 2 KiB
constexpr uint32_t kOpOff = 0;                           // three operand tiles
constexpr uint32_t kQOff = kOpOff + kNBuf * kOpBytes;    // Q: 8 groups x 16 heads x 128 B
constexpr uint32_t kPOff = kQOff + 8 * kQGroup;          // three P^T: 16 heads x 64 rows (128 B)
constexpr uint32_t kMiscOff = kPOff + kNBuf * kQGroup;

struct Misc {
  unsigned long long s_full[kNBuf], s_free[kNBuf], p_full[kNBuf], op_empty[kNBuf];
  uint32_t tmem_base;
  int is_last;
  int32_t pos[kMaxTiles][kRows];  // source row of each row of the CTA's tiles, -1 if empty
  float red[2][4][CSA2_H];        // per-quarter tile maximum, by the parity of the slow-path count
  float lsum[4][CSA2_H];          // per-quarter sums at the end
  float m_fin[CSA2_H];            // final offset per head (log2 units)
  float l_fin[CSA2_H];            // final sum per head
};
constexpr size_t kSmemBytes = 1024 + kMiscOff + sizeof(Misc);
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
// Barrier of the eight softmax warps only.
__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, 256;\n" ::: "memory"); }
// The same barrier, returning whether `v` holds on any of the eight warps' threads.
__device__ __forceinline__ bool softmax_any(bool v) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, 256, pi;\n\t"
      "selp.u32 %0, 1, 0, po; }\n"
      : "=r"(r)
      : "r"(uint32_t(v))
      : "memory");
  return r != 0;
}
// Waits for the completion of use n / 3 of barrier bars[n % 3].
__device__ __forceinline__ bool wait_use(const unsigned long long* bars, int n) {
  return mbar_wait(smem_u32(&bars[n % kNBuf]), uint32_t(n / kNBuf) & 1u);
}

// 640 threads = five warps per SM sub-partition, at most 96 registers each (one CTA per SM).
__global__ void __launch_bounds__(kWsThreads, 1) sparse_attn_ws_kernel(
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

  // ---- this split's tiles: FP4 tiles [0, nfp4), then window tiles [nfp4, ntiles) -------------------
  const int nfp4 = (k + kRows - 1) / kRows;
  const int nwin = swa ? (W + kRows - 1) / kRows : 0;
  const int ntiles = nfp4 + nwin;
  const int t_begin = split * ntiles / n_split, t_end = (split + 1) * ntiles / n_split;
  const int n_fp4_valid = min(k, n_valid ? max(n_valid[inst], 0) : k);
  const int SW = W - 1 + Nq;
  const int swa_lo = swa ? SW - min(max(swa_len[b], 0), SW) : SW;
  // live tiles: FP4 tiles holding a selected slot (a prefix of the FP4 tiles), window tiles reaching
  // a stored row (a suffix of the window tiles); the range's live tiles are [fa, fb) then [wa, wb)
  int w_first = nwin;  // first window tile reaching a stored row
  for (int w = nwin - 1; w >= 0 && qi + min((w + 1) * kRows, W) - 1 >= swa_lo; --w) w_first = w;
  const int fa = t_begin, fb = min(t_end, min(nfp4, (n_fp4_valid + kRows - 1) / kRows));
  const int wa = max(t_begin, nfp4 + w_first), wb = t_end;
  const int nf = max(fb - fa, 0), n_live = nf + max(wb - wa, 0);
  auto tile_of = [&](int n) { return n < nf ? fa + n : wa + (n - nf); };

  const int32_t* irow = (layers.idx[blockIdx.z] ? layers.idx[blockIdx.z] : idx) + int64_t(inst) * k;
  const uint8_t* cbase = codes + int64_t(b) * cap * CSA2_CODE_BYTES;
  const uint8_t* sbase = scales + int64_t(b) * cap * CSA2_SCALE_BYTES;
  const uint16_t* swbase = swa ? swa + int64_t(b) * SW * CSA2_D : nullptr;
  // 8-bit window: E4M3 bytes, rows of 512 B
  const uint8_t* sw8 = swa ? reinterpret_cast<const uint8_t*>(swa) + int64_t(b) * SW * CSA2_D : nullptr;
  const uint16_t* qrow = q + int64_t(inst) * CSA2_H * CSA2_D;

  // window row of tile row r of window tile w (0-based among the window tiles), or -1
  auto win_row = [&](int w, int r) {
    const int wr = w * kRows + r;
    return (wr < W && qi + wr >= swa_lo) ? qi + wr : -1;
  };

  if (t == 0) {
    for (int i = 0; i < kNBuf; ++i) {
      mbar_init(smem_u32(&ms.s_full[i]), kConvWarps);
      mbar_init(smem_u32(&ms.s_free[i]), kSoftWarps);
      mbar_init(smem_u32(&ms.p_full[i]), kSoftWarps);
      mbar_init(smem_u32(&ms.op_empty[i]), 4);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0 && n_live > 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(&ms.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  if (t < CSA2_H) {
    ms.m_fin[t] = -INFINITY;
    ms.l_fin[t] = 0.0f;
  }
  // the first live tile's Q type: f16 for FP4 and 8-bit window tiles, bf16 for window tiles
  const bool q_f16_first = n_live > 0 && (nf > 0 || win_fp8);
  // ---- Q (softmax warps: thread t, 16-byte chunk (t >> 4) + 16 i of head t & 15) and the source
  // rows of the range's tiles, with their bytes pulled into L2 (O^T issuer warps) ------------------
  if (n_live > 0 && warp < kSoftWarps) {
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      v[i] = __ldg(reinterpret_cast<const uint4*>(qrow + (t & 15) * CSA2_D + 8 * ((t >> 4) + 16 * i)));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 w = v[i];
      if (q_f16_first) {
        w.x = bf16x2_to_f16x2(w.x);
        w.y = bf16x2_to_f16x2(w.y);
        w.z = bf16x2_to_f16x2(w.z);
        w.w = bf16x2_to_f16x2(w.w);
      }
      *reinterpret_cast<uint4*>(base + kQOff + sw128(kQGroup, t & 15, (t >> 4) + 16 * i)) = w;
    }
  }
  for (int e = t - 32 * kOWarp0; e >= 0 && e < (t_end - t_begin) * kRows; e += 128) {
    const int tile = t_begin + e / kRows, r = e % kRows;
    int32_t p = -1;
    if (tile < nfp4) {
      const int slot = tile * kRows + r;
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
      p = win_row(tile - nfp4, r);
      if (p >= 0) {
        const uint8_t* sr = win_fp8 ? sw8 + int64_t(p) * CSA2_D : reinterpret_cast<const uint8_t*>(swbase + int64_t(p) * CSA2_D);
        for (int l = 0; l < (win_fp8 ? 4 : 8); ++l) asm volatile("prefetch.global.L2 [%0];" ::"l"(sr + 128 * l));
      }
    }
    ms.pos[tile - t_begin][r] = p < 0 ? -1 : p;
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;
  bool ok = true;

  if (warp >= kSoftWarps) {
    if (n_live > 0 && warp < kOWarp0) {
      // ======== converter warp e: channels [64 e, 64 e + 64) of every tile, then its S^T eighth ====
      const int e = warp - kSoftWarps;
      // FP4 rows of the eighth, one tile ahead in registers.  Lane: 16-byte code piece
      // 2 e + ((lane >> 3) & 1) (32 channels, two scale groups) of rows (lane & 7) + 8 ((lane >> 4) + 2 i)
      const int pl = (lane >> 3) & 1, pp = 2 * e + pl;
      uint4 cw[4];
      uint16_t sc[4];
      auto load_fp4 = [&](int tile) {
        const int32_t* pos = ms.pos[tile - t_begin];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int32_t p = pos[(lane & 7) + 8 * ((lane >> 4) + 2 * i)];
          cw[i] = p >= 0 ? __ldg(reinterpret_cast<const uint4*>(cbase + int64_t(p) * CSA2_CODE_BYTES + 16 * pp))
                         : make_uint4(0, 0, 0, 0);
          sc[i] = p >= 0 ? __ldg(reinterpret_cast<const uint16_t*>(sbase + int64_t(p) * CSA2_SCALE_BYTES + 2 * pp))
                         : uint16_t(0);
        }
      };
      if (nf > 0) load_fp4(fa);
      bool q_f16 = q_f16_first;
      for (int n = 0; n < n_live; ++n) {
        const int tile = tile_of(n), buf = n % kNBuf;
        const bool is_fp4 = tile < nfp4;
        const bool f16 = is_fp4 || win_fp8;
        const int32_t* pos = ms.pos[tile - t_begin];
        unsigned char* op = base + kOpOff + uint32_t(buf) * kOpBytes;
        // the operand buffer was last read by O^T of tile n - 3
        if (n >= kNBuf) ok = ok && wait_use(ms.op_empty, n - kNBuf);
        if (is_fp4) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = (lane & 7) + 8 * ((lane >> 4) + 2 * i);
            const __half2 sab = bits_h2(e4m3x2_to_f16x2(sc[i]));
            const __half2 sA = __low2half2(sab), sB = __high2half2(sab);
            const uint32_t words[4] = {cw[i].x, cw[i].y, cw[i].z, cw[i].w};
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
              const __half2 s2 = wi < 2 ? sA : sB;
              uint32_t f0, f1, f2, f3;
              e2m1x8_to_f16x2x4(words[wi], f0, f1, f2, f3);
              *reinterpret_cast<uint4*>(op + sw128(kTileGroup, r, 4 * pp + wi)) =
                  make_uint4(h2_bits(__hmul2(bits_h2(f0), s2)), h2_bits(__hmul2(bits_h2(f1), s2)),
                             h2_bits(__hmul2(bits_h2(f2), s2)), h2_bits(__hmul2(bits_h2(f3), s2)));
            }
          }
          // the next FP4 tile's rows, in flight while this tile's S^T is issued
          if (n + 1 < nf) load_fp4(tile_of(n + 1));
        } else if (win_fp8) {
          // 8-bit window tile: lane converts 16 channels (piece 4 e + (lane >> 3)) of rows
          // (lane & 7) + 8 j
          const int pc = 4 * e + (lane >> 3);
          uint4 v[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int32_t br = pos[(lane & 7) + 8 * j];
            v[j] = br >= 0 ? __ldg(reinterpret_cast<const uint4*>(sw8 + int64_t(br) * CSA2_D + 16 * pc))
                           : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int r = (lane & 7) + 8 * j;
            const uint32_t bw[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
            uint32_t h[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              h[2 * i] = e4m3x2_to_f16x2(uint16_t(bw[i] & 0xFFFFu));
              h[2 * i + 1] = e4m3x2_to_f16x2(uint16_t(bw[i] >> 16));
            }
            *reinterpret_cast<uint4*>(op + sw128(kTileGroup, r, 2 * pc)) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(op + sw128(kTileGroup, r, 2 * pc + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
          }
        } else {
          // bf16 window tile: rows (lane & 7) + 8 (j & 7), 16-byte chunk 8 e + (lane >> 3) + 4 (j >> 3)
          const uint32_t ops = base_s + kOpOff + uint32_t(buf) * kOpBytes;
#pragma unroll 4
          for (int j = 0; j < 16; ++j) {
            const int r = (lane & 7) + 8 * (j & 7), cc = 8 * e + (lane >> 3) + 4 * (j >> 3);
            const int32_t br = pos[r];
            const uint16_t* src = br >= 0 ? swbase + int64_t(br) * CSA2_D + 8 * cc : swa;
            cp_async16(ops + sw128(kTileGroup, r, cc), src, br >= 0 ? 16 : 0);
          }
          cp_async_commit();
          // Q's eighth as bf16 once this warp's earlier S^T products (which read it as f16) are done
          if (q_f16) {
            if (n >= 1) ok = ok && wait_use(ms.s_full, n - 1);
            uint4 v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int h = (lane & 15) , cc = 8 * e + (lane >> 4) + 2 * i;
              v[i] = __ldg(reinterpret_cast<const uint4*>(qrow + h * CSA2_D + 8 * cc));
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
              *reinterpret_cast<uint4*>(base + kQOff + sw128(kQGroup, lane & 15, 8 * e + (lane >> 4) + 2 * i)) = v[i];
            q_f16 = false;
          }
          cp_async_wait<0>();
        }
        fence_async_smem();
        __syncwarp();
        // S^T buffer n % 3 was last read by the softmax of tile n - 3
        if (n >= kNBuf) ok = ok && wait_use(ms.s_free, n - kNBuf);
        if (lane == 0) {
          tc_fence_after();
          const uint32_t id = instr_desc(kRows, !f16, false);
          const uint32_t a0 = base_s + kOpOff + uint32_t(buf) * kOpBytes + uint32_t(e) * kTileGroup;
          const uint32_t b0 = base_s + kQOff + uint32_t(e) * kQGroup;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_f16(tmem + uint32_t(buf) * kSCols + uint32_t(16 * e), smem_desc(a0 + 32u * kk, 0, 1024),
                     smem_desc(b0 + 32u * kk, 0, 1024), id, kk > 0 ? 1u : 0u);
          umma_commit(smem_u32(&ms.s_full[buf]));
        }
        __syncwarp();
      }
    } else if (n_live > 0) {
      // ======== O^T issuer i: O^T += V^T P^T for channel block i once P^T of the tile is written ===
      const int i = warp - kOWarp0;
      if (lane == 0) {
        for (int n = 0; n < n_live && ok; ++n) {
          const int buf = n % kNBuf;
          ok = wait_use(ms.p_full, n);
          if (!ok) break;
          tc_fence_after();
          const bool f16 = tile_of(n) < nfp4 || win_fp8;
          const uint32_t id = instr_desc(128, !f16, true);
          const uint32_t op = base_s + kOpOff + uint32_t(buf) * kOpBytes + uint32_t(2 * i) * kTileGroup;
          const uint32_t pb = base_s + kPOff + uint32_t(buf) * kQGroup;
#pragma unroll
          for (int s = 0; s < kRows / 16; ++s)
            umma_f16(tmem + kOCol + uint32_t(16 * i), smem_desc(op + uint32_t(s) * 2048u, kTileGroup, 1024),
                     smem_desc(pb + uint32_t(s) * 32u, 0, 1024), id, (n == 0 && s == 0) ? 0u : 1u);
          umma_commit(smem_u32(&ms.op_empty[buf]));
        }
      }
      __syncwarp();
    }
    if (!ok && lane == 0) atomicOr(flags, CSA2_FLAG_TIMEOUT);
    return;
  }

  // ======== softmax warps ==============================================================================
  const int quarter = warp & 3, half = warp >> 2;  // TMEM lane quarter; heads / channel blocks half
  if (n_live > 0) {
    const uint32_t t_lane = tmem + (uint32_t(32 * quarter) << 16);  // this warp's lane quarter
    const int row = 16 * quarter + (lane & 15);
    // mj[j]: the running offset of head 8 half + j (the same in every thread of the half); ls[j]: this
    // lane's row's running sum for that head; lanes 0..15 also keep the offset of head `lane` in m_h
    float mj[8], ls[8], m_h = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      mj[j] = -INFINITY;
      ls[j] = 0.0f;
    }
    int n_slow = 0;
    for (int n = 0; n < n_live; ++n) {
      const int tile = tile_of(n), buf = n % kNBuf;
      const bool f16_tile = tile < nfp4 || win_fp8;
      const bool row_ok = lane < 16 && ms.pos[tile - t_begin][row] >= 0;
      ok = ok && wait_use(ms.s_full, n);
      tc_fence_after();
      // warp (quarter, half): rows 16 quarter + lane (lanes < 16), heads 8 half .. 8 half + 7;
      // S^T = ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7)) over the eight partials
      float x[8];
      {
        float sp[4][8], lo4[8];
        const uint32_t sa = t_lane + uint32_t(buf) * kSCols + uint32_t(8 * half);
        tmem_ld8x4(sa, sp);  // partials 0..3
#pragma unroll
        for (int j = 0; j < 8; ++j) lo4[j] = (sp[0][j] + sp[1][j]) + (sp[2][j] + sp[3][j]);
        tmem_ld8x4(sa + 64u, sp);  // partials 4..7
#pragma unroll
        for (int j = 0; j < 8; ++j)
          x[j] = row_ok ? (lo4[j] + ((sp[0][j] + sp[1][j]) + (sp[2][j] + sp[3][j]))) * scale_log2 : -INFINITY;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ms.s_free[buf]));
      // Does any score pass its head's offset by more than kLazy?  Usually not, and then the offsets
      // stay and no maximum is needed; otherwise the tile's maxima set the offsets that move.
      bool jump = false;
#pragma unroll
      for (int j = 0; j < 8; ++j) jump |= x[j] > mj[j] + kLazy;
      if (softmax_any(jump)) {
        float(&red)[4][CSA2_H] = ms.red[n_slow & 1];
        ++n_slow;
        const float mx = reduce_scatter8<true>(x, lane);
        if ((lane & 3) == 0) red[quarter][8 * half + (lane >> 2)] = mx;
        softmax_sync();
        // lanes 0..15: head `lane`'s new offset and the factor that rescales what came before
        float mn = m_h, corr = 1.0f;
        if (lane < 16) {
          const float mt = fmaxf(fmaxf(red[0][lane], red[1][lane]), fmaxf(red[2][lane], red[3][lane]));
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
          // rescale the O^T accumulated so far (this lane quarter's channels of blocks 2 half and
          // 2 half + 1) once O^T of tile n - 1 is complete
          ok = ok && wait_use(ms.op_empty, n - 1);
          tc_fence_after();
          float cr[16];
#pragma unroll
          for (int h = 0; h < 16; ++h) cr[h] = __shfl_sync(0xffffffffu, corr, h);
          const uint32_t ta = t_lane + kOCol + uint32_t(32 * half);
          float o[2][16];
          tmem_ld16x2(ta, o);
#pragma unroll
          for (int g = 0; g < 2; ++g)
#pragma unroll
            for (int h = 0; h < 16; ++h) o[g][h] *= cr[h];
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
      // P^T buffer n % 3 was last read by O^T of tile n - 3
      if (n >= kNBuf) ok = ok && wait_use(ms.op_empty, n - kNBuf);
      // P^T (heads x rows, K-major, 128-byte swizzle): element (h, row)
      if (lane < 16) {
        unsigned char* pbuf = base + kPOff + uint32_t(buf) * kQGroup;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int h = 8 * half + j;
          const uint32_t off = uint32_t(h) * 128u + uint32_t(((row >> 3) ^ (h & 7)) << 4) + uint32_t(row & 7) * 2u;
          const uint16_t bits = f16_tile ? __half_as_ushort(__float2half_rn(pr[j])) : uint16_t(f2bf_bits(pr[j]));
          *reinterpret_cast<uint16_t*>(pbuf + off) = bits;
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ms.p_full[buf]));
    }
    const float l_w = reduce_scatter8<false>(ls, lane);  // this warp's rows, head 8 half + lane / 4
    // ---- the last tile's O^T, the sums per head, then O^T out of tensor memory ----------------------
    ok = ok && wait_use(ms.op_empty, n_live - 1);
    tc_fence_after();
    if ((lane & 3) == 0) ms.lsum[quarter][8 * half + (lane >> 2)] = l_w;
    softmax_sync();
    if (t < CSA2_H) {
      ms.l_fin[t] = (ms.lsum[0][t] + ms.lsum[1][t]) + (ms.lsum[2][t] + ms.lsum[3][t]);
      ms.m_fin[t] = m_h;
    }
    softmax_sync();
    // channel 128 (2 half + g) + 32 quarter + lane
    float o[2][16];
    tmem_ld16x2(t_lane + kOCol + uint32_t(32 * half), o);
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const int ch = 128 * (2 * half + g) + 32 * quarter + lane;
      if (n_split == 1) {
        uint16_t* orow = out + int64_t(inst) * CSA2_H * CSA2_D + ch;
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const float l = ms.l_fin[h];
          orow[h * CSA2_D] = uint16_t(f2bf_bits(o[g][h] * (l > 0.0f ? 1.0f / l : 0.0f)));
        }
      } else {
        float* po = ws + (ginst * n_split + split) * (CSA2_H * CSA2_D) + ch;
#pragma unroll
        for (int h = 0; h < 16; ++h) po[h * CSA2_D] = o[g][h];
      }
    }
    tc_fence_before();
    softmax_sync();
    if (warp == 0) {
      tc_fence_after();
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
    if (!ok && lane == 0) atomicOr(flags, CSA2_FLAG_TIMEOUT);
  } else if (n_split == 1) {
    uint16_t* orow = out + int64_t(inst) * CSA2_H * CSA2_D;
    for (int e = t; e < CSA2_H * CSA2_D; e += kThreads) orow[e] = 0;
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
  softmax_sync();
  if (t == 0) ms.is_last = (atomicAdd(tickets + ginst, 1u) == unsigned(n_split - 1));
  softmax_sync();
  if (!ms.is_last) return;
  __threadfence();
  // o = sum_j 2^(m_j - M) O_j / sum_j 2^(m_j - M) l_j over the splits with rows, in split order.
  // The per-head weights go through shared memory (the operand tile is free now): wgt[j][h] holds
  // m_j then the weight, wgt[kMaxSplit + j][h] holds l_j, then 1 / L and the lse per head.  The
  // partials are read coalesced: thread t takes float4 t + 256 v (v < 8) of the 16 x 512 block,
  // i.e. head (t >> 7) + 2 v, channels 4 (t & 127) .. + 3.
  float* wgt = reinterpret_cast<float*>(base + kOpOff);
  {
    const float* ml = mlb + ginst * n_split * (2 * CSA2_H);
    for (int e = t; e < n_split * CSA2_H; e += kThreads) {
      wgt[e] = __ldcg(ml + 2 * e);                            // m_j, e = j * 16 + h
      wgt[kMaxSplit * CSA2_H + e] = __ldcg(ml + 2 * e + 1);   // l_j
    }
    softmax_sync();
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
    softmax_sync();
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

}  // namespace

// The warp-specialised kernel for launches of at most one CTA per SM.  The split is already
// effective (attn_effective_split) and the tickets are zero.
cudaError_t launch_sparse_attn_ws(const AttnLayers& layers, int n_layers, int per_layer, int Nq,
                                  const uint8_t* codes, const uint8_t* scales, int64_t cap, const int32_t* idx,
                                  const int32_t* n_valid, int k, const int32_t* swa_len, int W, float scale_log2,
                                  int n_split, float* partials, unsigned int* tickets, unsigned int* flags,
                                  bool win_fp8, cudaStream_t st) {
  static std::atomic<bool> attr_set[64];  // per device; set once, by any host thread
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(sparse_attn_ws_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const dim3 grid{unsigned(n_split), unsigned(per_layer), unsigned(n_layers)};
  return launch_pdl(sparse_attn_ws_kernel, grid, dim3(kWsThreads), kSmemBytes, st, layers, Nq, codes, scales, cap,
                    idx, n_valid, k, swa_len, W, scale_log2, n_split, partials, tickets, flags, int(win_fp8));
}

}  // namespace csa2

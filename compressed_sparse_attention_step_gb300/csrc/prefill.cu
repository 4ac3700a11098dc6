// Indexer scoring for prefill chunks on the 5th-generation tensor cores, with an exact result.
//
// A prefill chunk scores every query of the chunk against every visible cached indexer key
// (ai-maestro.online "DeepSeek AI released DeepSeek-V4.1-Flash with 1M context, FP4", section
// "Compressed Sparse Attention 2": the indexer scans the sequence for each query; section "Causal
// Encoder-Decoder architecture": ratio-2 compressed entries under a causal mask).  That is a dense
// [queries x 4 heads, 128] x [128, keys] product, so it runs on tcgen05, but the selection must be
// the exact Top-K of the canonical fp32 scores.  The scheme ("filter, then rescore"):
//   1. pass A: tensor-core scores a(q, t) = sum_h w_h relu(qI_h . KI_t) (bf16 operands, fp32
//      accumulate in tensor memory); for every query the maximum of a over each aligned group of 32
//      keys is kept;
//   2. the 512th largest group maximum L(q) bounds the 512th largest a(q, .) from below (the 512
//      largest maxima are 512 distinct keys); with delta(q) a rigorous bound on |a - canonical|,
//      every key of the exact Top-512 has a >= L - 2 delta;
//   3. pass B: the same product again, marking every visible key with a >= L - 2 delta in a bitmap;
//   4. the marked keys are rescored in the canonical order on CUDA cores and the exact Top-512 is
//      selected among them (topk.cu).
// delta(q) = C * sum_h |w_h| ||qI_h||_2 * max_t ||KI_t||_2 (Cauchy-Schwarz on the dot-product
// error of both summation orders, with a safety factor), see prefill_delta_coef().
//
// The product: M = 128 keys (A, streamed), N = 256 = 64 queries x 4 heads (B, resident per item),
// K = 128 channels; both operands are bf16, K-major, 128-byte swizzled, loaded by TMA.  Keys on M
// put the four heads of a query in one thread's accumulator columns.  A persistent CTA per SM:
// warp 0 issues the TMA loads, warp 1 the MMAs (two accumulator buffers of 256 TMEM columns),
// warps 2..9 run the epilogue.
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <type_traits>

#include "common.cuh"

namespace csa2 {
namespace {

constexpr int kKeyTile = 128;                 // MMA M: keys per tile
constexpr int kQPerTile = 64;                 // queries per item (N = 4 x 64 = 256)
constexpr int kTilesPerItem = 32;             // key tiles per work item (4096 keys)
constexpr int kStages = 4;                    // A (key) stages
constexpr int kEpiWarps = 16;               // four per scheduler: one per (lane quarter, 64 columns)
constexpr int kPfThreads = (2 + kEpiWarps) * 32;
constexpr uint32_t kATileBytes = kKeyTile * CSA2_DI * 2;        // 32 KiB
constexpr uint32_t kBTileBytes = 4 * kQPerTile * CSA2_DI * 2;   // 64 KiB
constexpr size_t kPfSmem = 1024 + size_t(kStages) * kATileBytes + kBTileBytes;
constexpr int kGroup = 32;                    // keys per group maximum

__device__ __forceinline__ uint64_t pf_time() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool pf_wait(uint32_t bar, uint32_t parity) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p; }\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if ((it & 63u) == 0u) {
      const uint64_t now = pf_time();
      if (it == 0u) t0 = now;
      else if (now - t0 > 1000000000ull) return false;
    }
  }
}
__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void bar_expect(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
// 2-D TMA tile load (x = channel, y = row) completing on an mbarrier
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ uint64_t sdesc(uint32_t addr) {  // K-major, 128-byte swizzle, 8-row atoms
  return uint64_t((addr >> 4) & 0x3FFFu) | (uint64_t(1024 >> 4) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}
__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar) : "memory");
}
// 16 accumulator columns of this warp's lane quarter into r, asynchronously: r is valid only after
// a wait that names r (tmem_wait4), so that no use of it moves above the wait.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_wait4(uint32_t (&a)[16], uint32_t (&b)[16], uint32_t (&c)[16],
                                           uint32_t (&d)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]), "+r"(b[14]), "+r"(b[15]), "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3]), "+r"(c[4]), "+r"(c[5]), "+r"(c[6]), "+r"(c[7]), "+r"(c[8]), "+r"(c[9]), "+r"(c[10]), "+r"(c[11]), "+r"(c[12]), "+r"(c[13]), "+r"(c[14]), "+r"(c[15]), "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3]), "+r"(d[4]), "+r"(d[5]), "+r"(d[6]), "+r"(d[7]), "+r"(d[8]), "+r"(d[9]), "+r"(d[10]), "+r"(d[11]), "+r"(d[12]), "+r"(d[13]), "+r"(d[14]), "+r"(d[15])
               :
               : "memory");
}

// Visible cache entries of query row `row` (as in the CUDA-core scan).
__device__ __forceinline__ int64_t pf_visible(int64_t row, int Nq, const int32_t* lens, int64_t cap, int ratio,
                                              const int32_t* q_pos) {
  const int64_t b = row / Nq, qi = row - b * Nq;
  const int64_t T = min(max(int64_t(lens[b]), int64_t(0)), cap);
  const int64_t p = q_pos ? int64_t(q_pos[row]) : int64_t(ratio) * T - Nq + qi;
  return (p + 1 < 0) ? 0 : min((p + 1) / ratio, T);
}

// Work item i: sequence b, query tile qt (64 queries), key tiles [kt0, kt1).
struct PfItems {
  int Nq, q_tiles, chunks;
  int64_t n_items;
};

// Pass A (kMark = false): group maxima of the tensor-core scores (float bits).  Pass B (kMark =
// true): bitmap of the keys with score >= thr[row].
template <bool kMark>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_score_kernel(
    const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_q,
    const float* __restrict__ w, const int32_t* __restrict__ lens, int64_t cap, int ratio,
    const int32_t* __restrict__ q_pos, PfItems it, int64_t n_groups, uint32_t* __restrict__ out,
    const float* __restrict__ thr, unsigned int* flags) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ __align__(8) unsigned long long fullA[kStages], emptyA[kStages], fullB, emptyB, accF[2], accE[2];
  __shared__ uint32_t tmem_base;
  __shared__ float4 s_w[kQPerTile];     // the current item's queries: halved head weights,
  __shared__ int32_t s_vis[kQPerTile];  // visible entries (0 past the chunk's end),
  __shared__ float s_thr[kQPerTile];    // and pass-B thresholds
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  const uint32_t a_s = base_s, b_s = base_s + kStages * kATileBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Nq = it.Nq;

  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      bar_init(smem_u32(&fullA[s]), 1);
      bar_init(smem_u32(&emptyA[s]), 1);
    }
    bar_init(smem_u32(&fullB), 1);
    bar_init(smem_u32(&emptyB), 1);
    for (int a = 0; a < 2; ++a) {
      bar_init(smem_u32(&accF[a]), 1);
      bar_init(smem_u32(&accE[a]), kEpiWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(smem_u32(&tmem_base))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
  const uint32_t tmem = tmem_base;

  // the key-tile range of an item (tiles past every query's visible prefix are skipped)
  auto item_range = [&](int64_t i, int& b, int& qt, int& kt0, int& kt1) {
    const int64_t per_seq = int64_t(it.q_tiles) * it.chunks;
    b = int(i / per_seq);
    const int64_t r = i - int64_t(b) * per_seq;
    qt = int(r / it.chunks);
    const int ch = int(r - int64_t(qt) * it.chunks);
    const int q1 = min((qt + 1) * kQPerTile, Nq);
    // the largest visible prefix of the tile's queries: a query's prefix does not shrink as its
    // position grows, so it is the prefix of the tile's last (or largest explicit) position
    int64_t vis = 0;
    if (!q_pos) {
      vis = pf_visible(int64_t(b) * Nq + q1 - 1, Nq, lens, cap, ratio, q_pos);
    } else {
      const int32_t* qp = q_pos + int64_t(b) * Nq;
      int32_t pm = qp[qt * kQPerTile];
#pragma unroll 8
      for (int qq = qt * kQPerTile + 1; qq < q1; ++qq) pm = max(pm, __ldg(qp + qq));
      const int64_t T = min(max(int64_t(lens[b]), int64_t(0)), cap);
      vis = (int64_t(pm) + 1 < 0) ? 0 : min((int64_t(pm) + 1) / ratio, T);
    }
    const int n_kt = int((vis + kKeyTile - 1) / kKeyTile);
    kt0 = min(ch * kTilesPerItem, n_kt);
    kt1 = min(kt0 + kTilesPerItem, n_kt);
  };

  bool ok = true;
  if (warp == 0) {
    // ---- TMA producer ------------------------------------------------------------------------------
    if (lane == 0) {
      uint32_t tile = 0, nitem = 0;
      for (int64_t i = blockIdx.x; i < it.n_items; i += gridDim.x) {
        int b, qt, kt0, kt1;
        item_range(i, b, qt, kt0, kt1);
        if (kt0 >= kt1) continue;
        if (nitem > 0) ok = ok && pf_wait(smem_u32(&emptyB), (nitem - 1) & 1u);
        const uint32_t fb = smem_u32(&fullB);
        bar_expect(fb, kBTileBytes);
        const int qrow = (b * Nq + qt * kQPerTile) * 4;
        tma_load_2d(b_s, &map_q, 0, qrow, fb);
        tma_load_2d(b_s + kBTileBytes / 2, &map_q, 64, qrow, fb);
        for (int kt = kt0; kt < kt1; ++kt, ++tile) {
          const int s = int(tile % kStages);
          if (tile >= uint32_t(kStages)) ok = ok && pf_wait(smem_u32(&emptyA[s]), ((tile / kStages) - 1) & 1u);
          const uint32_t fa = smem_u32(&fullA[s]);
          bar_expect(fa, kATileBytes);
          const int krow = int(int64_t(b) * cap + int64_t(kt) * kKeyTile);
          tma_load_2d(a_s + s * kATileBytes, &map_k, 0, krow, fa);
          tma_load_2d(a_s + s * kATileBytes + kATileBytes / 2, &map_k, 64, krow, fa);
        }
        ++nitem;
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer --------------------------------------------------------------------------------
    if (lane == 0) {
      // kind::f16, bf16 A and B, fp32 accumulator, both K-major, N = 256, M = 128
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((256u >> 3) << 17) | ((128u >> 4) << 24);
      uint32_t tile = 0, nitem = 0;
      for (int64_t i = blockIdx.x; i < it.n_items; i += gridDim.x) {
        int b, qt, kt0, kt1;
        item_range(i, b, qt, kt0, kt1);
        if (kt0 >= kt1) continue;
        ok = ok && pf_wait(smem_u32(&fullB), nitem & 1u);
        for (int kt = kt0; kt < kt1; ++kt, ++tile) {
          const int s = int(tile % kStages), a = int(tile & 1u);
          ok = ok && pf_wait(smem_u32(&fullA[s]), (tile / kStages) & 1u);
          if (tile >= 2) ok = ok && pf_wait(smem_u32(&accE[a]), ((tile >> 1) - 1) & 1u);
          asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
#pragma unroll
          for (int kk = 0; kk < CSA2_DI / 16; ++kk) {
            const uint32_t off = uint32_t(kk >> 2) * (kATileBytes / 2) + uint32_t(kk & 3) * 32u;
            const uint32_t offb = uint32_t(kk >> 2) * (kBTileBytes / 2) + uint32_t(kk & 3) * 32u;
            mma_bf16(tmem + uint32_t(256 * a), sdesc(a_s + s * kATileBytes + off), sdesc(b_s + offb), idesc,
                     kk > 0 ? 1u : 0u);
          }
          mma_commit(smem_u32(&emptyA[s]));
          mma_commit(smem_u32(&accF[a]));
        }
        mma_commit(smem_u32(&emptyB));
        ++nitem;
      }
    }
  } else {
    // ---- epilogue: warp e covers lane quarter warp % 4 and accumulator columns [64 (e / 4), +64) ----
    const int e = warp - 2, quarter = warp & 3, colq = e >> 2, et = int(threadIdx.x) - 64;
    uint32_t tile = 0;
    for (int64_t i = blockIdx.x; i < it.n_items; i += gridDim.x) {
      int b, qt, kt0, kt1;
      item_range(i, b, qt, kt0, kt1);
      if (kt0 >= kt1) continue;
      const int64_t row0 = int64_t(b) * Nq + int64_t(qt) * kQPerTile;  // the item's first query row
      const int qlim = Nq - qt * kQPerTile;                               // queries of the item: q < qlim
      asm volatile("bar.sync 1, %0;\n" ::"n"(kEpiWarps * 32) : "memory");  // the last item's readers are done
      if (et < kQPerTile) {
        const bool qv = et < qlim;
        const int64_t row = qv ? row0 + et : row0;
        const float4 wq = qv ? __ldg(reinterpret_cast<const float4*>(w + row * 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
        s_w[et] = make_float4(0.5f * wq.x, 0.5f * wq.y, 0.5f * wq.z, 0.5f * wq.w);
        s_vis[et] = qv ? int32_t(pf_visible(row, Nq, lens, cap, ratio, q_pos)) : 0;
        s_thr[et] = (kMark && qv) ? __ldg(thr + row) : 0.0f;
      }
      asm volatile("bar.sync 1, %0;\n" ::"n"(kEpiWarps * 32) : "memory");
      int32_t vmin = 0x7FFFFFFF;  // the fewest entries any of the warp's 16 queries sees
#pragma unroll
      for (int qi = 0; qi < 16; ++qi) vmin = min(vmin, s_vis[16 * colq + qi]);
      for (int kt = kt0; kt < kt1; ++kt, ++tile) {
        const int a = int(tile & 1u);
        ok = ok && pf_wait(smem_u32(&accF[a]), (tile >> 1) & 1u);
        asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
        const int32_t key = kt * kKeyTile + 32 * quarter + lane;  // this lane's key
        const int64_t grp = (int64_t(kt) * kKeyTile + 32 * quarter) / kGroup;
        // four chunks of 16 columns (4 queries each), loaded together; query qi's result (pass A: the
        // group's largest score, pass B: its mask) ends in lane qi.  On a tile that every key of is
        // visible to all 16 queries (all of them in the chunk) no per-query test remains.  The score
        // is sum_h w_h relu(d_h), with w_h relu(d) computed as (w_h / 2) (d + |d|): the same product
        // (halving and doubling are exact), on the FMA pipe rather than the ALU.
        const uint32_t tq = tmem + (uint32_t(32 * quarter) << 16) + uint32_t(256 * a + 64 * colq);
        uint32_t res = 0u;
        auto tile_body = [&](auto full_c) {
          constexpr bool kFull = decltype(full_c)::value;  // every key of the tile visible to all 16
          uint32_t da[16], db[16], dc[16], dd[16];
          auto use = [&](const uint32_t (&d)[16], int c) {
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              const int qi = 4 * c + qq;     // query within the warp's 16
              const int q = 16 * colq + qi;  // query within the item
              const float4 hw = s_w[q];
              auto r2 = [&](int h) {  // 2 relu(d_h), exactly
                const float x = __uint_as_float(d[4 * qq + h]);
                return __fadd_rn(x, fabsf(x));
              };
              const float s = fmaf(hw.w, r2(3), fmaf(hw.z, r2(2), fmaf(hw.y, r2(1), hw.x * r2(0))));
              const bool v = kFull || key < s_vis[q];
              uint32_t m;
              if (kMark) {
                m = __ballot_sync(0xffffffffu, v && s >= s_thr[q]);
              } else {
                float mf;
                asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(mf) : "f"(v ? s : -INFINITY));
                m = __float_as_uint(mf);
              }
              res = lane == qi ? m : res;
            }
          };
          tmem_ld16(tq, da);
          tmem_ld16(tq + 16u, db);
          tmem_ld16(tq + 32u, dc);
          tmem_ld16(tq + 48u, dd);
          tmem_wait4(da, db, dc, dd);
          use(da, 0);
          use(db, 1);
          use(dc, 2);
          use(dd, 3);
        };
        if ((kt + 1) * kKeyTile <= vmin) tile_body(std::true_type{});
        else tile_body(std::false_type{});
        if (lane < 16 && 16 * colq + lane < qlim && grp < n_groups)  // pass A: float bits of the maximum
          out[(row0 + 16 * colq + lane) * n_groups + grp] = res;
        asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
        __syncwarp();
        if (lane == 0) bar_arrive(smem_u32(&accE[a]));
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem) : "memory");
  }
  if (!ok) atomicOr(flags, CSA2_FLAG_TIMEOUT);
}

// Per sequence and chunk of kNormChunk entries: the largest sum of squares of KI_t over the visible
// part of the chunk (kmax_part[b][chunk]; the threshold kernel takes the maximum over chunks).
constexpr int kNormChunk = 256;  // entries per CTA: about three CTAs per SM at 131072 entries
__global__ void __launch_bounds__(256) prefill_key_norm_kernel(const uint16_t* __restrict__ KI,
                                                               const int32_t* __restrict__ lens, int64_t cap,
                                                               float* __restrict__ kmax_part) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[8];
  const int b = blockIdx.y;
  const int64_t T = min(max(int64_t(lens[b]), int64_t(0)), cap);
  const int64_t t0 = int64_t(blockIdx.x) * kNormChunk, t1 = min(t0 + kNormChunk, T);
  float m = 0.0f;
  // eight threads per entry, 16 channels each; a warp takes four consecutive entries per step.  The
  // loop runs on the warp's first entry, so every lane of a warp makes the same trips and the
  // shuffles below always see the full warp (lanes past the chunk's end add nothing).
#pragma unroll 4
  for (int64_t tw = t0 + ((threadIdx.x >> 5) << 2); tw < t1; tw += blockDim.x >> 3) {
    const int64_t t = tw + ((threadIdx.x & 31) >> 3);
    const bool valid = t < t1;
    float acc = 0.0f;
    if (valid) {
      const uint4* kp = reinterpret_cast<const uint4*>(KI + (int64_t(b) * cap + t) * CSA2_DI) + 2 * (threadIdx.x & 7);
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        const uint4 x = __ldg(kp + v);
        const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc = fmaf(bf16lo(u[e]), bf16lo(u[e]), acc);
          acc = fmaf(bf16hi(u[e]), bf16hi(u[e]), acc);
        }
      }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    m = fmaxf(m, acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float mm = 0.0f;
    for (int i = 0; i < int(blockDim.x >> 5); ++i) mm = fmaxf(mm, red[i]);
    kmax_part[int64_t(b) * gridDim.x + blockIdx.x] = mm;
  }
}

// Per query row: thr = L - 2 delta, rounded down, with L at most the k-th largest group maximum of
// the tensor-core scores; -inf when fewer than k groups are visible (every visible key is then kept).  Also the row's
// score bound ub (as a score key): every canonical score is <= (largest tensor-core score) + 2 delta,
// and <= -0 when all four head weights are negative (each product w_h relu(.) is then <= -0).  One
// CTA of 256 threads per row: the row's group maxima (keys) go to shared memory, and two radix
// rounds of 11 bits bound the k-th largest from below (its top 22 bits, the rest zero).
constexpr int kThThreads = 256;
constexpr int64_t kMaxGroups = 49152;  // group maxima of one row held in shared memory (cap <= 1.5 Mi)
constexpr int kThBins = 2048;
__global__ void __launch_bounds__(kThThreads) prefill_threshold_kernel(
    const uint32_t* __restrict__ gmax, int64_t n_groups, const uint16_t* __restrict__ qI, const float* __restrict__ w,
    const int32_t* __restrict__ lens, int64_t cap, int Nq, int ratio, const int32_t* __restrict__ q_pos, int k,
    const float* __restrict__ kmax_part, int n_chunks, float delta_coef, float* __restrict__ thr,
    uint32_t* __restrict__ ubound) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint32_t keys[];  // n_groups
  __shared__ uint32_t hist[kThBins];
  __shared__ uint32_t scan_tmp[32];
  __shared__ float part[4];
  __shared__ float kred[kThThreads / 32];
  __shared__ uint32_t res_bin, res_before;
  const int t = threadIdx.x;
  const int64_t row = blockIdx.x;
  const int64_t vis = pf_visible(row, Nq, lens, cap, ratio, q_pos);
  const int64_t ng = min((vis + kGroup - 1) / kGroup, n_groups);
  const float4 wq = __ldg(reinterpret_cast<const float4*>(w + row * 4));
  const bool all_neg = wq.x < 0.0f && wq.y < 0.0f && wq.z < 0.0f && wq.w < 0.0f;
  if (ng < k) {
    if (t == 0) {
      thr[row] = -INFINITY;
      ubound[row] = all_neg ? score_key(-0.0f) : 0xFFFFFFFFu;
    }
    return;
  }
  uint32_t kmx = 0u;
  for (int64_t i = t; i < ng; i += kThThreads) {  // group maxima: float bits -> score keys
    keys[i] = score_key(__uint_as_float(__ldg(gmax + row * n_groups + i)));
    kmx = max(kmx, keys[i]);
  }
  kmx = __reduce_max_sync(0xffffffffu, kmx);
  __shared__ uint32_t kmx_w[kThThreads / 32];
  if ((t & 31) == 0) kmx_w[t >> 5] = kmx;
  // delta = coef * sum_h |w_h| ||qI_h||_2 * max_t ||KI_t||_2 (norms rounded up)
  {
    float km = 0.0f;
    for (int i = t; i < n_chunks; i += kThThreads) km = fmaxf(km, __ldg(kmax_part + (row / Nq) * n_chunks + i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, o));
    if ((t & 31) == 0) kred[t >> 5] = km;
    const int h = t >> 6, c = (t & 63) * 2;  // 4 heads x 64 threads x 2 channels
    const uint32_t pr = *reinterpret_cast<const uint32_t*>(qI + row * (CSA2_HI * CSA2_DI) + h * CSA2_DI + c);
    float a = fmaf(bf16lo(pr), bf16lo(pr), bf16hi(pr) * bf16hi(pr));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if ((t & 31) == 0) scan_tmp[t >> 5] = __float_as_uint(a);
    __syncthreads();
    if (t < 4) part[t] = __uint_as_float(scan_tmp[2 * t]) + __uint_as_float(scan_tmp[2 * t + 1]);
    __syncthreads();
  }
  // two radix rounds resolve the top 22 key bits of the k-th largest group maximum; the key with the
  // low 10 bits zero is at most that maximum, so L below stays a lower bound on the k-th largest
  // filter score (about 2^-13 lower, relative, than the exact value)
  uint32_t prefix = 0, mask = 0, need = uint32_t(k);
  const int shifts[2] = {21, 10}, widths[2] = {11, 11};
  for (int r = 0; r < 2; ++r) {
    const int nb = 1 << widths[r];
    for (int i = t; i < nb; i += kThThreads) hist[i] = 0u;
    __syncthreads();
    for (int64_t i = t; i < ng; i += kThThreads) {
      const uint32_t key = keys[i];
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shifts[r]) & uint32_t(nb - 1)], 1u);
    }
    __syncthreads();
    // walk from the top bin: thread t owns bins [nb - per (t + 1), nb - per t)
    const int per = nb / kThThreads;
    const int lo_bin = nb - (t + 1) * per;
    uint32_t local = 0;
    for (int e = 0; e < per; ++e) local += hist[lo_bin + e];
    const uint32_t excl = block_exclusive_scan(local, scan_tmp, nullptr);
    if (excl < need && excl + local >= need) {
      uint32_t cum = excl;
      for (int e = per - 1; e >= 0; --e) {
        if (cum + hist[lo_bin + e] >= need) {
          res_bin = uint32_t(lo_bin + e);
          res_before = cum;
          break;
        }
        cum += hist[lo_bin + e];
      }
    }
    __syncthreads();
    prefix |= res_bin << shifts[r];
    mask |= uint32_t(nb - 1) << shifts[r];
    need -= res_before;
    __syncthreads();
  }
  if (t == 0) {
    const float qn = fabsf(wq.x) * (__fsqrt_ru(part[0]) * 1.001f) + fabsf(wq.y) * (__fsqrt_ru(part[1]) * 1.001f) +
                     fabsf(wq.z) * (__fsqrt_ru(part[2]) * 1.001f) + fabsf(wq.w) * (__fsqrt_ru(part[3]) * 1.001f);
    float km = 0.0f;
    for (int i = 0; i < kThThreads / 32; ++i) km = fmaxf(km, kred[i]);
    // a sum of 128 squares in fp32 is within a relative 2^-16 of exact; sqrt rounded up, then a margin
    const float kmax = __fsqrt_ru(km) * 1.001f;
    const float delta = delta_coef * qn * kmax * 1.001f;
    auto key_score = [](uint32_t key) {
      return (key & 0x80000000u) ? __uint_as_float(key & 0x7FFFFFFFu) : __uint_as_float(~key);
    };
    thr[row] = __fsub_rd(key_score(prefix), 2.0f * delta);
    uint32_t top = 0u;
    for (int i = 0; i < kThThreads / 32; ++i) top = max(top, kmx_w[i]);
    uint32_t ub = score_key(__fadd_ru(key_score(top), 2.0f * delta));
    if (all_neg) ub = min(ub, score_key(-0.0f));
    ubound[row] = ub;
  }
}

// Marked keys per query row: the visible words of the row's bitmap, one CTA per row.
__global__ void __launch_bounds__(256) prefill_count_kernel(const uint32_t* __restrict__ bitmap, int64_t n_words,
                                                            const int32_t* __restrict__ lens, int64_t cap, int Nq,
                                                            int ratio, const int32_t* __restrict__ q_pos,
                                                            uint32_t* __restrict__ counts) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint32_t red[8];
  const int64_t row = blockIdx.x;
  const int64_t vis = pf_visible(row, Nq, lens, cap, ratio, q_pos);
  const int64_t nw = min((vis + 31) / 32, n_words);
  const uint32_t* bm = bitmap + row * n_words;
  uint32_t c = 0;
  for (int64_t i = threadIdx.x; i < nw; i += blockDim.x) {
    uint32_t v = bm[i];
    const int64_t valid = vis - 32 * i;
    if (valid < 32) v &= (1u << valid) - 1u;
    c += __popc(v);
  }
  c = __reduce_add_sync(0xffffffffu, c);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t tot = 0;
    for (int i = 0; i < int(blockDim.x >> 5); ++i) tot += red[i];
    counts[row] = tot;
  }
}

// The rows in selection order: first the n_top rows with the most rescoring work (the selection
// splits each of them over several CTAs), then the rows with more than `heavy` marked keys (they
// take several list rounds and would otherwise finish last), then the rest, each class in row
// order.  A row's work is its marked keys, or only the first chunk of `lim` when the list
// overflows and its bound is <= 0 (it stops after that chunk).  Zeroes the sliced rows' tickets.
// One CTA.
constexpr int kOrdThreads = 1024;
constexpr int64_t kOrderMaxRows = 16384;  // longer launches keep the natural order
constexpr int kSliceRows = 4;             // rows split over several CTAs
constexpr int kSlices = 8;                // CTAs per split row
__global__ void __launch_bounds__(kOrdThreads) prefill_order_kernel(const uint32_t* __restrict__ counts,
                                                                    const uint32_t* __restrict__ ubound, int rows,
                                                                    uint32_t heavy, uint32_t lim, int n_top,
                                                                    int32_t* __restrict__ order,
                                                                    unsigned int* __restrict__ tickets) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint32_t scan_tmp[32];
  __shared__ uint32_t run_h, run_l, n_heavy;
  __shared__ unsigned long long wmax[kOrdThreads / 32];
  __shared__ int top[kSliceRows];
  const int t = threadIdx.x;
  auto work = [&](int r) -> uint32_t {
    const uint32_t c = counts[r];
    return (c > heavy && ubound[r] <= score_key(0.0f)) ? min(c, lim) : c;
  };
  auto picked = [&](int r, int n) {
    bool p = false;
    for (int i = 0; i < n; ++i) p = p || top[i] == r;
    return p;
  };
  // the n_top rows of most work (ties: the lower row), one block maximum each
  for (int i = 0; i < n_top; ++i) {
    unsigned long long best = 0;
    for (int r = t; r < rows; r += kOrdThreads)
      if (!picked(r, i)) best = max(best, (static_cast<unsigned long long>(work(r)) << 32) | (0xFFFFFFFFu - uint32_t(r)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
    if ((t & 31) == 0) wmax[t >> 5] = best;
    __syncthreads();
    if (t == 0) {
      unsigned long long m = 0;
      for (int j = 0; j < kOrdThreads / 32; ++j) m = max(m, wmax[j]);
      top[i] = int(0xFFFFFFFFu - uint32_t(m & 0xFFFFFFFFull));
      order[i] = top[i];
      tickets[i] = 0u;
    }
    __syncthreads();
  }
  uint32_t h = 0;
  for (int r = t; r < rows; r += kOrdThreads) h += (counts[r] > heavy && !picked(r, n_top)) ? 1u : 0u;
  uint32_t tot;
  block_exclusive_scan(h, scan_tmp, &tot);
  if (t == 0) {
    n_heavy = uint32_t(n_top) + tot;
    run_h = uint32_t(n_top);
    run_l = 0;
  }
  __syncthreads();
  for (int base = 0; base < rows; base += kOrdThreads) {
    const int r = base + t;
    const bool pk = r < rows && picked(r, n_top);
    const bool hv = r < rows && !pk && counts[r] > heavy;
    const bool lt = r < rows && !pk && !hv;
    uint32_t th;
    const uint32_t ph = block_exclusive_scan((hv ? 1u : 0u) | ((lt ? 1u : 0u) << 16), scan_tmp, &th);
    if (hv) order[run_h + (ph & 0xFFFFu)] = r;
    if (lt) order[n_heavy + run_l + (ph >> 16)] = r;
    __syncthreads();
    if (t == 0) {
      run_h += th & 0xFFFFu;
      run_l += th >> 16;
    }
    __syncthreads();
  }
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static std::mutex mu;
  std::lock_guard<std::mutex> guard(mu);
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiled>(p);
  }
  return fn;
}

// [rows][128] bf16 rows, boxes of 64 channels x box_rows rows, 128-byte swizzle
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int box_rows) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cuuint64_t(CSA2_DI), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(CSA2_DI * 2)};
  const cuuint32_t box[2] = {64u, cuuint32_t(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// The bound on |tensor-core score - canonical score| per unit of sum_h |w_h| ||qI_h|| ||KI_t||:
// both dot products are within gamma_n * sum |qI_c KI_c| of the exact one (n = 19 roundings on the
// canonical path; 2 x 128 allowed for the tensor core, which may truncate), relu does not widen a
// difference, and the two 4-term weighted sums add gamma_3 + gamma_4 of sum |w_h r_h|; a safety
// factor of 8 covers the tensor core's internal alignment.
float prefill_delta_coef() {
  const double u = std::ldexp(1.0, -24);
  auto gamma = [&](double n) { return n * u / (1.0 - n * u); };
  const double c = gamma(2.0 * 128.0) + gamma(19.0) + gamma(3.0) + gamma(4.0);
  return float(8.0 * c * (1.0 + 1e-3));
}

// The split rows' candidates (keys, columns, counts) and tickets, at the end of the workspace.
constexpr size_t kSliceCand = size_t(kSliceRows) * kSlices * CSA2_MAX_K;
size_t slice_ws_bytes() {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  return 2 * al(kSliceCand * 4) + al(size_t(kSliceRows) * kSlices * 4) + al(size_t(kSliceRows) * 4);
}

size_t prefill_ws_bytes(int64_t rows, int64_t cap, int B) {
  const int64_t ng = (cap + 31) / 32;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const int64_t nch = (cap + kNormChunk - 1) / kNormChunk;
  return 2 * al(size_t(rows) * size_t(ng) * 4) + 4 * al(size_t(rows) * 4) + al(size_t(B) * size_t(nch) * 4) +
         slice_ws_bytes();
}

int64_t prefill_max_groups() { return kMaxGroups; }

// Exact Top-k indices for every query row of a prefill chunk via the tensor-core filter.
cudaError_t launch_prefill_select(const uint16_t* qI, const float* w, int B, int Nq, const uint16_t* KI,
                                  int64_t cap, const int32_t* lens, int ratio, const int32_t* q_pos, int k,
                                  int32_t* idx, int32_t* n_sel, void* ws, cudaStream_t st) {
  const int64_t rows = int64_t(B) * Nq;
  if (rows == 0) return cudaSuccess;
  unsigned int* flags = device_flags_ptr();
  if (!flags) return cudaErrorUnknown;
  const int64_t ng = (cap + 31) / 32;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  char* p = static_cast<char*>(ws);
  uint32_t* gmax = reinterpret_cast<uint32_t*>(p);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(p + al(size_t(rows) * ng * 4));
  float* thr = reinterpret_cast<float*>(p + 2 * al(size_t(rows) * ng * 4));
  uint32_t* ubound = reinterpret_cast<uint32_t*>(p + 2 * al(size_t(rows) * ng * 4) + al(size_t(rows) * 4));
  uint32_t* counts = reinterpret_cast<uint32_t*>(p + 2 * al(size_t(rows) * ng * 4) + 2 * al(size_t(rows) * 4));
  int32_t* order = reinterpret_cast<int32_t*>(p + 2 * al(size_t(rows) * ng * 4) + 3 * al(size_t(rows) * 4));
  float* kmax = reinterpret_cast<float*>(p + 2 * al(size_t(rows) * ng * 4) + 4 * al(size_t(rows) * 4));
  char* ps = p + 2 * al(size_t(rows) * ng * 4) + 4 * al(size_t(rows) * 4) +
             al(size_t(B) * size_t((cap + kNormChunk - 1) / kNormChunk) * 4);
  BmSlices sl;
  sl.n_slices = kSlices;
  sl.key = reinterpret_cast<uint32_t*>(ps);
  sl.col = reinterpret_cast<int32_t*>(ps + al(kSliceCand * 4));
  sl.cnt = reinterpret_cast<uint32_t*>(ps + 2 * al(kSliceCand * 4));
  sl.tickets = reinterpret_cast<unsigned int*>(ps + 2 * al(kSliceCand * 4) + al(size_t(kSliceRows) * kSlices * 4));

  CUtensorMap map_k, map_q;
  if (!make_map(&map_k, KI, int64_t(B) * cap, kKeyTile) || !make_map(&map_q, qI, rows * 4, 4 * kQPerTile))
    return cudaErrorUnknown;
  static std::atomic<bool> attr_set[64];  // per device; set once, by any host thread
  static int n_sm[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prefill_score_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kPfSmem));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(prefill_score_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kPfSmem));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(prefill_threshold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kMaxGroups * 4));
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&n_sm[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  PfItems items;
  items.Nq = Nq;
  items.q_tiles = (Nq + kQPerTile - 1) / kQPerTile;
  items.chunks = int((cap + int64_t(kKeyTile) * kTilesPerItem - 1) / (int64_t(kKeyTile) * kTilesPerItem));
  items.n_items = int64_t(B) * items.q_tiles * items.chunks;
  const int grid = int(std::min<int64_t>(items.n_items, dev < 64 ? n_sm[dev] : 148));

  const int64_t nch = (cap + kNormChunk - 1) / kNormChunk;
  cudaError_t e = launch_pdl(prefill_key_norm_kernel, dim3(unsigned(nch), unsigned(B)), dim3(256), 0, st, KI, lens,
                             cap, kmax);
  if (e != cudaSuccess) return e;
  e = launch_pdl(prefill_score_kernel<false>, dim3(grid), dim3(kPfThreads), kPfSmem, st, map_k, map_q, w, lens, cap,
                 ratio, q_pos, items, ng, gmax, static_cast<const float*>(nullptr), flags);
  if (e != cudaSuccess) return e;
  e = launch_pdl(prefill_threshold_kernel, dim3(unsigned(rows)), dim3(kThThreads), size_t(ng) * 4, st,
                 static_cast<const uint32_t*>(gmax), ng, qI, w, lens, cap, Nq, ratio, q_pos, k,
                 static_cast<const float*>(kmax), int(nch), prefill_delta_coef(), thr, ubound);
  if (e != cudaSuccess) return e;
  e = launch_pdl(prefill_score_kernel<true>, dim3(grid), dim3(kPfThreads), kPfSmem, st, map_k, map_q, w, lens, cap,
                 ratio, q_pos, items, ng, bitmap, static_cast<const float*>(thr), flags);
  if (e != cudaSuccess) return e;
  const bool ordered = rows <= kOrderMaxRows;
  sl.n_rows = ordered ? int(std::min<int64_t>(rows, kSliceRows)) : 0;
  if (ordered) {
    e = launch_pdl(prefill_count_kernel, dim3(unsigned(rows)), dim3(256), 0, st, static_cast<const uint32_t*>(bitmap),
                   ng, lens, cap, Nq, ratio, q_pos, counts);
    if (e != cudaSuccess) return e;
    e = launch_pdl(prefill_order_kernel, dim3(1), dim3(kOrdThreads), 0, st, static_cast<const uint32_t*>(counts),
                   static_cast<const uint32_t*>(ubound), int(rows), uint32_t(bitmap_list_cap()),
                   uint32_t(std::max(2 * k, 1024)), sl.n_rows, order, sl.tickets);
    if (e != cudaSuccess) return e;
  }
  return launch_bitmap_select(qI, w, B, Nq, KI, cap, lens, ratio, q_pos, k, bitmap, ng,
                              static_cast<const uint32_t*>(ubound), ordered ? order : nullptr, sl, idx, n_sel, st);
}

}  // namespace csa2

extern "C" csa2_status csa2_index_select_prefill(const uint16_t* qI, const float* w, int B, int Nq,
                                                 const uint16_t* KI, int64_t cap, const int32_t* lens, int ratio,
                                                 const int32_t* q_pos, int k, int32_t* idx, int32_t* n_sel,
                                                 void* ws, size_t ws_bytes, csa2_stream_t stream) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (B < 0 || Nq < 0 || cap < 0 || ratio < 1 || k < 1 || k > CSA2_MAX_K) return CSA2_ERR_INVALID_ARG;
  const int64_t rows = int64_t(B) * Nq;
  if (rows == 0) return CSA2_OK;
  if (rows > (int64_t(1) << 28) || B > 65535 || int64_t(B) * cap >= (int64_t(1) << 31) ||
      (cap + 31) / 32 > csa2::prefill_max_groups())
    return CSA2_ERR_UNSUPPORTED;
  if (!qI || !w || !KI || !lens || !idx || !al16(qI) || !al16(w) || !al16(KI) || !al16(idx))
    return CSA2_ERR_INVALID_ARG;
  const size_t need = csa2::prefill_ws_bytes(rows, cap, B);
  if (!ws || ws_bytes < need || !al16(ws)) return CSA2_ERR_WORKSPACE;
  return csa2::launch_prefill_select(qI, w, B, Nq, KI, cap, lens, ratio, q_pos, k, idx, n_sel, ws,
                                     reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? CSA2_OK
             : CSA2_ERR_CUDA;
}

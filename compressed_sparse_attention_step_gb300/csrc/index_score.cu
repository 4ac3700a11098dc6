// Lightning-indexer scoring: s_t = sum_h w_h * relu(qI_h . KI_t) for every visible cached
// indexer key (or every position of a candidate pool).  Full layers select with it, Reindex
// layers rescore with their own indexer Q (ai-maestro.online "DeepSeek AI released
// DeepSeek-V4.1-Flash with 1M context, FP4", section "Compressed Sparse Attention 2").
//
// HBM-bound streaming kernels (256 B of indexer K per position, ~2 FMA per byte): eight lanes
// share one position, each lane owning 16 consecutive channels (32 bytes), so a warp covers four
// whole 256-byte rows per step.  The indexer query slice (4 heads x 16 channels) stays in
// registers for the whole CTA.  Contiguous keys (a sequence's cache or its block keys) stream
// through shared memory by bulk asynchronous copies (index_score_stream_kernel, below); so do
// candidate pools, whose gathered rows arrive as one bulk copy each.  The register-loaded form
// (index_score_kernel, four steps in flight per lane) serves keys that are not 16-byte aligned.
//
// The fp32 result is bit-identical to the canonical order: per head, lane j computes the
// fused-multiply-add chain p_j over channels 16j..16j+15 from +0; the 8-lane reduction is a
// reduce-scatter whose additions are exactly ((p0+p1)+(p2+p3))+((p4+p5)+(p6+p7)) (IEEE addition
// is commutative, so either operand order gives the same bits); then relu, w_h * r_h, and
// (m0 + m1) + (m2 + m3).  Only _rn intrinsics (and the packed fma.rn.f32x2, whose two lanes each
// round like one fmaf) are used, so nothing is contracted or reordered.
#include "common.cuh"

namespace csa2 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kU = 4;                                // 4-position groups in flight per lane
constexpr int kPosPerWarpIt = 4 * kU;                // 16
constexpr int kPosPerCtaIt = kWarps * kPosPerWarpIt; // 128
constexpr int kPrefetch = 2;                         // sweeps of L2 prefetch ahead of the loads

template <bool kCand>
__global__ void __launch_bounds__(kThreads, 2) index_score_kernel(
    const uint16_t* __restrict__ qI, const float* __restrict__ w, int Nq,
    const uint16_t* __restrict__ KI, int64_t key_stride_rows, const int32_t* __restrict__ lens,
    int64_t cap_entries, int block_div, const int32_t* __restrict__ cand,
    const int32_t* __restrict__ cand_len, int64_t n_cand, int ratio,
    const int32_t* __restrict__ q_pos, float* __restrict__ scores, int64_t ld,
    int32_t* __restrict__ n_valid_out, int64_t chunk, unsigned int* flags) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.y;
  const int b = row / Nq, qi = row - b * Nq;
  const int64_t T = min(max(int64_t(lens[b]), int64_t(0)), cap_entries);
  const int64_t p = q_pos ? int64_t(q_pos[row]) : int64_t(ratio) * T - Nq + qi;
  const int64_t nvis = (p + 1 < 0) ? 0 : min((p + 1) / ratio, T);   // visible cache entries

  int64_t nv;  // scored prefix of this row
  const int32_t* crow = nullptr;
  if (kCand) {
    crow = cand + int64_t(row) * n_cand;
    const int64_t cl = min(max(int64_t(cand_len[row]), int64_t(0)), n_cand);
    int64_t lo = 0, hi = cl;  // first pool entry not visible (the pool is ascending)
    if (cl > 0 && int64_t(crow[cl - 1]) < nvis) lo = hi;  // all visible (every decode query): no search
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if (int64_t(crow[mid]) < nvis) lo = mid + 1;
      else hi = mid;
    }
    nv = lo;
  } else {
    nv = nvis / block_div;
  }
  if (n_valid_out && blockIdx.x == 0 && threadIdx.x == 0) n_valid_out[row] = int32_t(nv);

  const int64_t c0 = int64_t(blockIdx.x) * chunk;
  const int64_t c1 = min(c0 + chunk, ld);
  if (c0 >= c1) return;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane >> 3;  // position within the warp's group of four
  const int j = lane & 7;     // channel chunk 16j .. 16j+15

  float qf[4][16];
  const uint16_t* qrow = qI + int64_t(row) * (CSA2_HI * CSA2_DI);
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const uint4 a = *reinterpret_cast<const uint4*>(qrow + h * CSA2_DI + 16 * j);
    const uint4 c = *reinterpret_cast<const uint4*>(qrow + h * CSA2_DI + 16 * j + 8);
    const uint32_t v[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      qf[h][2 * e] = bf16lo(v[e]);
      qf[h][2 * e + 1] = bf16hi(v[e]);
    }
  }
  // head held by this lane after the reduce-scatter
  const int my_head = 2 * (j & 1) + ((j >> 1) & 1);
  const float wh = w[int64_t(row) * CSA2_HI + my_head];
  const bool odd = (j & 1) != 0, second = (j & 2) != 0;

  const uint16_t* kbase = KI + int64_t(b) * key_stride_rows * CSA2_DI + 16 * j;
  float* srow = scores + int64_t(row) * ld;

  for (int64_t base = c0 + warp * kPosPerWarpIt; base < c1; base += kPosPerCtaIt) {
    if (!kCand) {
      // pull this warp's rows of PF sweeps ahead into L2 (one 128-byte line per lane)
      const int64_t tp = base + int64_t(kPrefetch) * kPosPerCtaIt + (lane >> 1);
      if (tp < nv && tp < c1) asm volatile("prefetch.global.L2 [%0];" ::"l"(kbase - 16 * j + tp * CSA2_DI + 64 * (lane & 1)));
    }
    uint4 kv[kU][2];
    bool ok[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t t = base + u * 4 + sub;
      const int64_t pos = (t < nv && t < c1) ? (kCand ? int64_t(crow[t]) : t) : -1;
      ok[u] = pos >= 0 && pos < key_stride_rows;
      if (kCand && t < nv && t < c1 && !ok[u] && j == 0) atomicOr(flags, CSA2_FLAG_INDEX_OOB);
      if (ok[u]) {
        const uint16_t* kp = kbase + pos * CSA2_DI;
        kv[u][0] = ld_stream16(kp);
        kv[u][1] = ld_stream16(kp + 8);
      } else {
        kv[u][0] = make_uint4(0, 0, 0, 0);
        kv[u][1] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const uint32_t kw[8] = {kv[u][0].x, kv[u][0].y, kv[u][0].z, kv[u][0].w,
                              kv[u][1].x, kv[u][1].y, kv[u][1].z, kv[u][1].w};
      float P[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float acc = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          acc = __fmaf_rn(qf[h][2 * e], bf16lo(kw[e]), acc);
          acc = __fmaf_rn(qf[h][2 * e + 1], bf16hi(kw[e]), acc);
        }
        P[h] = acc;
      }
      // step 1 (lanes j, j^1): even lanes keep heads 0,1, odd lanes keep heads 2,3
      const float s0 = odd ? P[0] : P[2], s1 = odd ? P[1] : P[3];
      const float k0 = odd ? P[2] : P[0], k1 = odd ? P[3] : P[1];
      const float A0 = __fadd_rn(k0, __shfl_xor_sync(0xffffffffu, s0, 1));
      const float A1 = __fadd_rn(k1, __shfl_xor_sync(0xffffffffu, s1, 1));
      // step 2 (lanes j, j^2): keep one head of the pair
      const float sendB = second ? A0 : A1, keepB = second ? A1 : A0;
      const float Bv = __fadd_rn(keepB, __shfl_xor_sync(0xffffffffu, sendB, 2));
      // step 3 (lanes j, j^4): the two halves of the channels
      const float dot = __fadd_rn(Bv, __shfl_xor_sync(0xffffffffu, Bv, 4));
      const float r = dot > 0.0f ? dot : 0.0f;
      const float m = __fmul_rn(wh, r);
      const float m2 = __fadd_rn(m, __shfl_xor_sync(0xffffffffu, m, 2));  // heads (0,1) / (2,3)
      const float s = __fadd_rn(m2, __shfl_xor_sync(0xffffffffu, m2, 1));
      const int64_t t = base + u * 4 + sub;
      if (j == 0 && t < c1) srow[t] = ok[u] ? s : -INFINITY;
    }
  }
}

// ---- contiguous keys (a sequence's cache or its block keys): staged by bulk asynchronous copies --
// Each warp streams its own 16-position steps (4 KiB of contiguous keys) through a ring of
// kStages shared-memory buffers: lane 0 issues one cp.async.bulk per step, completing on the
// stage's mbarrier, kStages steps ahead of the arithmetic.  The copies in flight hold no registers,
// so an SM keeps 2 CTAs x 8 warps x kStages x 4 KiB of keys requested, far more than the
// register-staged loads allow at this kernel's occupancy.  The arithmetic (the same lanes, order
// and rounding as above) reads each position's 32 bytes per lane from shared memory.
constexpr int kStages = 3;
constexpr uint32_t kStepBytes = uint32_t(kPosPerWarpIt) * CSA2_DI * 2;  // 4096
constexpr size_t kStreamSmem = size_t(kWarps) * kStages * kStepBytes + size_t(kWarps) * kStages * 8;

// (x, y) <- (a * k + x, b * k + y), each rounded once to nearest (one packed fp32 FMA).
__device__ __forceinline__ void fma2_rn(float& x, float& y, float a, float b, float k) {
  asm("{ .reg .b64 ab, kk, xy;\n\t"
      "mov.b64 ab, {%2, %3};\n\t"
      "mov.b64 kk, {%4, %4};\n\t"
      "mov.b64 xy, {%0, %1};\n\t"
      "fma.rn.f32x2 xy, ab, kk, xy;\n\t"
      "mov.b64 {%0, %1}, xy; }\n"
      : "+f"(x), "+f"(y)
      : "f"(a), "f"(b), "f"(k));
}

// Waits for phase `parity` of a shared-memory mbarrier, for at most about one second.
__device__ __forceinline__ bool stage_wait(uint32_t bar, uint32_t parity) {
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
      uint64_t now;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
      if (it == 0u) t0 = now;
      else if (now - t0 > 1000000000ull) return false;
    }
  }
}

// kCand: the positions are gathered from a candidate pool (ascending cache positions, cand_len[row]
// valid): each step's 16 key rows arrive by bulk copies issued by lanes 0..15, one per run of
// consecutive positions (a pool expanded from blocks of 8 holds such runs).
template <bool kCand>
__global__ void __launch_bounds__(kThreads, 2) index_score_stream_kernel(
    const uint16_t* __restrict__ qI, const float* __restrict__ w, int Nq,
    const uint16_t* __restrict__ KI, int64_t key_stride_rows, const int32_t* __restrict__ lens,
    int64_t cap_entries, int block_div, const int32_t* __restrict__ cand, const int32_t* __restrict__ cand_len,
    int64_t n_cand, int ratio, const int32_t* __restrict__ q_pos,
    float* __restrict__ scores, int64_t ld, int32_t* __restrict__ n_valid_out, int64_t chunk,
    unsigned int* flags) {
  extern __shared__ __align__(128) unsigned char smem[];
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.y;
  const int b = row / Nq, qi = row - b * Nq;
  const int64_t T = min(max(int64_t(lens[b]), int64_t(0)), cap_entries);
  const int64_t p = q_pos ? int64_t(q_pos[row]) : int64_t(ratio) * T - Nq + qi;
  const int64_t nvis = (p + 1 < 0) ? 0 : min((p + 1) / ratio, T);
  int64_t nv;  // scored prefix of this row
  const int32_t* crow = nullptr;
  if (kCand) {
    crow = cand + int64_t(row) * n_cand;
    const int64_t cl = min(max(int64_t(cand_len[row]), int64_t(0)), n_cand);
    int64_t lo = 0, hi = cl;  // first pool entry not visible (the pool is ascending)
    if (cl > 0 && int64_t(crow[cl - 1]) < nvis) lo = hi;  // all visible (every decode query): no search
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if (int64_t(crow[mid]) < nvis) lo = mid + 1;
      else hi = mid;
    }
    nv = lo;
  } else {
    nv = nvis / block_div;
  }
  if (n_valid_out && blockIdx.x == 0 && threadIdx.x == 0) n_valid_out[row] = int32_t(nv);

  const int64_t c0 = int64_t(blockIdx.x) * chunk;
  const int64_t c1 = min(c0 + chunk, ld);
  if (c0 >= c1) return;
  // positions below this are read (contiguous keys: also inside the cache)
  const int64_t lend = kCand ? min(nv, c1) : min(min(nv, c1), key_stride_rows);
  // a gathered position that can be read
  auto readable = [&](int64_t t) {
    if (t >= lend) return false;
    if (!kCand) return true;
    const int32_t q = crow[t];
    return q >= 0 && int64_t(q) < key_stride_rows;
  };

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane >> 3;
  const int j = lane & 7;
  const uint32_t ring = smem_u32(smem) + uint32_t(warp) * kStages * kStepBytes;
  const uint32_t bars = smem_u32(smem) + uint32_t(kWarps) * kStages * kStepBytes + uint32_t(warp) * kStages * 8u;
  const unsigned char* ring_p = smem + size_t(warp) * kStages * kStepBytes;
  if (lane == 0) {
    for (int st = 0; st < kStages; ++st)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(bars + 8u * st) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncwarp();

  const uint16_t* kseq = KI + int64_t(b) * key_stride_rows * CSA2_DI;
  uint64_t stream_policy = 0;
  if (!kCand) asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(stream_policy));
  const int64_t first = c0 + int64_t(warp) * kPosPerWarpIt;
  const int n_steps = first < c1 ? int((c1 - first + kPosPerCtaIt - 1) / kPosPerCtaIt) : 0;
  // step i covers positions first + i * kPosPerCtaIt + [0, 16); the keys of those below lend.
  // Called by the whole warp: contiguous keys are one copy by lane 0; gathered keys one copy per
  // readable position by lanes 0..15 (row slot = position - base), after lane 0 has announced
  // their bytes.  An unreadable gathered position below lend is flagged.
  auto issue = [&](int i) {
    const int64_t base = first + int64_t(i) * kPosPerCtaIt;
    const int64_t cnt = min(max(lend - base, int64_t(0)), int64_t(kPosPerWarpIt));
    const uint32_t bar = bars + 8u * uint32_t(i % kStages);
    const uint32_t dst = ring + uint32_t(i % kStages) * kStepBytes;
    if (!kCand) {
      const uint32_t bytes = uint32_t(cnt) * CSA2_DI * 2u;
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
        // the keys are read once: first out of L2, so that the scores written beside them stay
        // there for the selection that reads them next
        if (bytes)
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
              "%4;\n" ::"r"(dst),
              "l"(kseq + base * CSA2_DI), "r"(bytes), "r"(bar), "l"(stream_policy)
              : "memory");
      }
      return;
    }
    const bool mine = lane < cnt;
    const int32_t q = mine ? crow[base + lane] : -1;
    const bool rd = mine && q >= 0 && int64_t(q) < key_stride_rows;
    if (mine && !rd) atomicOr(flags, CSA2_FLAG_INDEX_OOB);
    const uint32_t n_rd = __popc(__ballot_sync(0xffffffffu, rd));
    // runs of consecutive readable positions (a pool expanded from blocks holds runs of 8): the
    // lane that starts a run copies the whole run's rows in one bulk copy
    const int32_t q_prev = __shfl_up_sync(0xffffffffu, q, 1);
    const bool rd_prev = __shfl_up_sync(0xffffffffu, rd, 1);
    const bool cont = rd && lane > 0 && rd_prev && q_prev + 1 == q;  // continues lane - 1's run
    const uint32_t cont_mask = __ballot_sync(0xffffffffu, cont);
    if (lane == 0) {
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar),
                   "r"(n_rd * uint32_t(CSA2_DI * 2))
                   : "memory");
    }
    __syncwarp();
    if (rd && !cont) {
      // lanes lane + 1 .. continue the run while their bits of cont_mask are set (lanes < 16 only)
      const uint32_t run = uint32_t(__ffs(~(cont_mask >> (lane + 1))));
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
              dst + uint32_t(lane) * uint32_t(CSA2_DI * 2)),
          "l"(kseq + int64_t(q) * CSA2_DI), "r"(run * uint32_t(CSA2_DI * 2)), "r"(bar)
          : "memory");
    }
  };
  for (int i = 0; i < min(n_steps, kStages); ++i) issue(i);

  float qf[4][16];
  const uint16_t* qrow = qI + int64_t(row) * (CSA2_HI * CSA2_DI);
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const uint4 a = *reinterpret_cast<const uint4*>(qrow + h * CSA2_DI + 16 * j);
    const uint4 c = *reinterpret_cast<const uint4*>(qrow + h * CSA2_DI + 16 * j + 8);
    const uint32_t v[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      qf[h][2 * e] = bf16lo(v[e]);
      qf[h][2 * e + 1] = bf16hi(v[e]);
    }
  }
  const int my_head = 2 * (j & 1) + ((j >> 1) & 1);
  const float wh = w[int64_t(row) * CSA2_HI + my_head];
  const bool odd = (j & 1) != 0, second = (j & 2) != 0;
  float* srow = scores + int64_t(row) * ld;

  int done = n_steps;
  for (int i = 0; i < n_steps; ++i) {
    const int64_t base = first + int64_t(i) * kPosPerCtaIt;
    // the whole warp agrees on the outcome (the copies it issues next are warp-collective)
    if (!__all_sync(0xffffffffu, stage_wait(bars + 8u * uint32_t(i % kStages), uint32_t(i / kStages) & 1u))) {
      if (lane == 0) atomicOr(flags, CSA2_FLAG_TIMEOUT);
      done = i;
      break;
    }
    const unsigned char* stg = ring_p + size_t(i % kStages) * kStepBytes;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t t = base + u * 4 + sub;
      const bool ok = readable(t);
      const uint4* kp = reinterpret_cast<const uint4*>(stg + (u * 4 + sub) * (CSA2_DI * 2) + 32 * j);
      const uint4 k0 = kp[0], k1 = kp[1];
      const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
      // the four heads' chains two at a time (packed fp32 FMA: each lane of the pair rounds as one
      // fmaf would), channels in the same order
      float P[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float klo = bf16lo(kw[e]), khi = bf16hi(kw[e]);
#pragma unroll
        for (int hp = 0; hp < 2; ++hp) {
          fma2_rn(P[2 * hp], P[2 * hp + 1], qf[2 * hp][2 * e], qf[2 * hp + 1][2 * e], klo);
          fma2_rn(P[2 * hp], P[2 * hp + 1], qf[2 * hp][2 * e + 1], qf[2 * hp + 1][2 * e + 1], khi);
        }
      }
      const float s0 = odd ? P[0] : P[2], s1 = odd ? P[1] : P[3];
      const float k0f = odd ? P[2] : P[0], k1f = odd ? P[3] : P[1];
      const float A0 = __fadd_rn(k0f, __shfl_xor_sync(0xffffffffu, s0, 1));
      const float A1 = __fadd_rn(k1f, __shfl_xor_sync(0xffffffffu, s1, 1));
      const float sendB = second ? A0 : A1, keepB = second ? A1 : A0;
      const float Bv = __fadd_rn(keepB, __shfl_xor_sync(0xffffffffu, sendB, 2));
      const float dot = __fadd_rn(Bv, __shfl_xor_sync(0xffffffffu, Bv, 4));
      const float r = dot > 0.0f ? dot : 0.0f;
      const float m = __fmul_rn(wh, r);
      const float m2 = __fadd_rn(m, __shfl_xor_sync(0xffffffffu, m, 2));
      const float sc = __fadd_rn(m2, __shfl_xor_sync(0xffffffffu, m2, 1));
      if (j == 0 && t < c1) srow[t] = ok ? sc : -INFINITY;
    }
    __syncwarp();  // every lane has read the stage before it is refilled
    if (i + kStages < n_steps) issue(i + kStages);
  }
  if (done < n_steps) {
    // gave up waiting: wait (bounded) for the copies still in flight before the CTA leaves
    for (int i = done; i < min(n_steps, done + kStages); ++i)
      stage_wait(bars + 8u * uint32_t(i % kStages), uint32_t(i / kStages) & 1u);
  }
}

}  // namespace

cudaError_t launch_index_score(const uint16_t* qI, const float* w, int B, int Nq, const uint16_t* KI,
                               int64_t key_stride_rows, const int32_t* lens, int64_t cap_entries,
                               int block_div, const int32_t* cand, const int32_t* cand_len,
                               int64_t n_cand, int ratio, const int32_t* q_pos, float* scores,
                               int64_t ld, int32_t* n_valid, cudaStream_t st) {
  const int64_t rows = int64_t(B) * Nq;
  if (rows == 0 || ld == 0) return cudaSuccess;
  // chunk: a multiple of the CTA step.  Contiguous keys: sized for at least ~8 CTAs per SM over the
  // grid, at most 2048 positions.  Gathered keys (a pool, a few MB in all): one wave of two CTAs per
  // SM, so that every warp keeps its whole ring of copies in flight.
  const int64_t per = cand ? 152 * 2 : 152 * 8;
  int64_t chunk = (rows * ld + per - 1) / per;
  chunk = ((chunk + kPosPerCtaIt - 1) / kPosPerCtaIt) * kPosPerCtaIt;
  chunk = max(int64_t(kPosPerCtaIt), min(chunk, int64_t(2048)));
  const dim3 grid(unsigned((ld + chunk - 1) / chunk), unsigned(rows));
  unsigned int* flags = device_flags_ptr();
  if (!flags) return cudaErrorUnknown;
  static std::atomic<bool> attr_set[2][64];  // per kernel and device; set once, by any host thread
  int dev = 0;
  cudaGetDevice(&dev);
  const int kind = cand ? 1 : 0;
  if (dev < 64 && !attr_set[kind][dev]) {
    const cudaError_t e = cudaFuncSetAttribute(cand ? index_score_stream_kernel<true> : index_score_stream_kernel<false>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, int(kStreamSmem));
    if (e != cudaSuccess) return e;
    attr_set[kind][dev] = true;
  }
  // keys are read by bulk copies, which need 16-byte aligned sources (every 256-byte row of an
  // aligned KI is)
  if ((reinterpret_cast<uintptr_t>(KI) & 15u) == 0) {
    if (cand)
      return launch_pdl(index_score_stream_kernel<true>, grid, dim3(kThreads), kStreamSmem, st, qI, w, Nq, KI,
                        key_stride_rows, lens, cap_entries, block_div, cand, cand_len, n_cand, ratio, q_pos, scores,
                        ld, n_valid, chunk, flags);
    return launch_pdl(index_score_stream_kernel<false>, grid, dim3(kThreads), kStreamSmem, st, qI, w, Nq, KI,
                      key_stride_rows, lens, cap_entries, block_div, nullptr, nullptr, int64_t(0), ratio, q_pos,
                      scores, ld, n_valid, chunk, flags);
  }
  if (cand)
    return launch_pdl(index_score_kernel<true>, grid, dim3(kThreads), 0, st, qI, w, Nq, KI, key_stride_rows, lens,
                      cap_entries, block_div, cand, cand_len, n_cand, ratio, q_pos, scores, ld, n_valid, chunk, flags);
  return launch_pdl(index_score_kernel<false>, grid, dim3(kThreads), 0, st, qI, w, Nq, KI, key_stride_rows, lens,
                    cap_entries, block_div, nullptr, nullptr, int64_t(0), ratio, q_pos, scores, ld, n_valid, chunk,
                    flags);
}

}  // namespace csa2

extern "C" csa2_status csa2_index_score(const uint16_t* qI, const float* w, int B, int Nq,
                                        const uint16_t* KI, int64_t cap, const int32_t* lens,
                                        const int32_t* cand, const int32_t* cand_len, int64_t n_cand,
                                        int ratio, const int32_t* q_pos, float* scores,
                                        int32_t* n_valid, csa2_stream_t stream) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (B < 0 || Nq < 0 || cap < 0 || ratio < 1) return CSA2_ERR_INVALID_ARG;
  if (int64_t(B) * Nq > 65535) return CSA2_ERR_UNSUPPORTED;  // grid.y limit
  if (int64_t(B) * Nq == 0) return CSA2_OK;
  if (!qI || !w || !KI || !lens || !scores || !al16(qI) || !al16(KI)) return CSA2_ERR_INVALID_ARG;
  if (cand && (!cand_len || n_cand < 0)) return CSA2_ERR_INVALID_ARG;
  const int64_t ld = cand ? n_cand : cap;
  return csa2::launch_index_score(qI, w, B, Nq, KI, cap, lens, cap, 1, cand, cand_len, n_cand, ratio,
                                  q_pos, scores, ld, n_valid,
                                  reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? CSA2_OK
             : CSA2_ERR_CUDA;
}

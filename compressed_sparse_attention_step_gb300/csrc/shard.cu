// Context split of one sequence's cache over G shards (one per GPU, or G logical shards on one GPU).
//
// The Hierarchical Sparse Indexer exists so that a query at 1M context touches a bounded set of
// positions (ai-maestro.online "DeepSeek AI released DeepSeek-V4.1-Flash with 1M context, FP4",
// section "Compressed Sparse Attention 2": a candidate pool of up to 16,384 positions); at that
// length one sequence's cache can also be spread over several GPUs.  Shard g holds the cache
// entries [lo_g, hi_g) with lo_0 = 0 and hi_g = lo_{g+1}.  A step then needs two exchanges:
//   1. every shard scores its own entries and keeps its local Top-k as (score, position) pairs;
//      the union of the G local Top-k sets contains the global Top-k (a key of the global Top-k
//      is beaten by fewer than k keys overall, so by fewer than k keys of its own shard), so the
//      exact global Top-k (larger score first, equal scores by lower position) is the Top-k of the
//      G x k pairs;
//   2. every shard attends to the selected rows it holds (the shard holding the newest entries
//      also to the window rows) and the per-shard results are combined by their log-sum-exp:
//      o = sum_g exp(lse_g - L) o_g with L = log sum_g exp(lse_g), which is softmax attention over
//      the union of the rows.
// This file holds the kernels around the exchanges; the exchanges themselves are collectives of
// the caller (or, for logical shards, plain copies).
#include <algorithm>
#include <cmath>

#include "common.cuh"

namespace csa2 {
namespace {

// Local Top-k columns -> (score, global position) pairs, in place on the positions.
__global__ void __launch_bounds__(256) shard_pairs_kernel(const float* __restrict__ scores, int64_t ld, int64_t total,
                                                          int k, const int32_t* __restrict__ map, int64_t map_ld,
                                                          int64_t pos_offset, int32_t* __restrict__ pos,
                                                          float* __restrict__ pair_score) {
  pdl_wait();
  pdl_trigger();
  const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= total) return;
  const int64_t r = e / k;
  const int32_t col = pos[e];
  if (col < 0) {
    pair_score[e] = -INFINITY;
    return;
  }
  pair_score[e] = scores[r * ld + col];
  pos[e] = map ? map[r * map_ld + col] : int32_t(pos_offset + col);
}

// The valid pairs of each row, shard after shard, packed into one row of G * k entries: pairs
// [G][rows][k] with pair_n [G][rows] valid entries each (NULL: k) -> packed score and position
// [rows][G * k] and the row's count.  Shards cover ascending position ranges and each shard's
// pairs are ascending, so a packed row is ascending in position and a column tie-break is a
// position tie-break.
__global__ void __launch_bounds__(256) pack_pairs_kernel(const float* __restrict__ pair_score,
                                                         const int32_t* __restrict__ pair_pos,
                                                         const int32_t* __restrict__ pair_n, int G, int rows, int k,
                                                         float* __restrict__ pscore, int32_t* __restrict__ ppos,
                                                         int32_t* __restrict__ pcount) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const int64_t ld = int64_t(G) * k;
  int base = 0;
  for (int g = 0; g < G; ++g) {
    const int n = pair_n ? min(max(pair_n[int64_t(g) * rows + r], 0), k) : k;
    const int64_t src = (int64_t(g) * rows + r) * k;
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
      pscore[int64_t(r) * ld + base + j] = pair_score[src + j];
      ppos[int64_t(r) * ld + base + j] = pair_pos[src + j];
    }
    base += n;
  }
  if (threadIdx.x == 0) pcount[r] = base;
}

// Global selected positions -> the shard's local rows: p in [lo, hi) becomes p - lo, others -1.
__global__ void __launch_bounds__(256) shard_indices_kernel(const int32_t* __restrict__ idx, int64_t total, int64_t lo,
                                                            int64_t hi, int32_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= total) return;
  const int32_t p = idx[e];
  out[e] = (p >= lo && p < hi) ? int32_t(p - lo) : -1;
}

// Per-shard attention results -> their combination: one CTA of 128 threads per (row, head), four
// channels per thread.  Shards are combined in shard order; a shard with lse = -inf (no rows)
// weighs nothing, and a row no shard attended gets out = 0, lse = -inf.
__global__ void __launch_bounds__(128) merge_shards_kernel(const uint16_t* __restrict__ out_g,
                                                           const float* __restrict__ lse_g, int G, int rows,
                                                           uint16_t* __restrict__ out, float* __restrict__ lse) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x, h = blockIdx.y;
  const int64_t rh = int64_t(r) * CSA2_H + h;
  float M = -INFINITY;
  for (int g = 0; g < G; ++g) M = fmaxf(M, lse_g[int64_t(g) * rows * CSA2_H + rh]);
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f}, L = 0.0f;
  const int c0 = 4 * threadIdx.x;
  if (M != -INFINITY) {
    for (int g = 0; g < G; ++g) {
      const float lg = lse_g[int64_t(g) * rows * CSA2_H + rh];
      if (lg == -INFINITY) continue;
      const float wgt = expf(lg - M);
      L += wgt;
      const uint2 v = *reinterpret_cast<const uint2*>(out_g + (int64_t(g) * rows * CSA2_H + rh) * CSA2_D + c0);
      acc[0] += wgt * bf16lo(v.x);
      acc[1] += wgt * bf16hi(v.x);
      acc[2] += wgt * bf16lo(v.y);
      acc[3] += wgt * bf16hi(v.y);
    }
  }
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  *reinterpret_cast<uint2*>(out + rh * CSA2_D + c0) =
      make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv));
  if (lse && threadIdx.x == 0) lse[rh] = L > 0.0f ? M + logf(L) : -INFINITY;
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

size_t merge_pairs_ws_bytes(int rows, int G, int k) {
  const int64_t n = int64_t(G) * k;
  return 2 * align256(size_t(rows) * size_t(n) * 4) + align256(size_t(rows) * 4) + topk_ws_bytes(rows, n);
}

}  // namespace csa2

using csa2::al16;

extern "C" csa2_status csa2_shard_topk_pairs(const float* scores, int rows, int64_t n, int64_t ld,
                                             const int32_t* n_valid, int k, const int32_t* map, int64_t map_ld,
                                             int64_t pos_offset, float* pair_score, int32_t* pair_pos,
                                             int32_t* pair_n, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  if (rows < 0 || n < 0 || ld < n || k < 1 || k > CSA2_MAX_K || n >= (int64_t(1) << 31) || pos_offset < 0 ||
      pos_offset + n >= (int64_t(1) << 31))
    return CSA2_ERR_INVALID_ARG;
  if (rows == 0) return CSA2_OK;
  if (rows > 65535) return CSA2_ERR_UNSUPPORTED;
  if (!scores || !pair_score || !pair_pos || (map && map_ld < n)) return CSA2_ERR_INVALID_ARG;
  const size_t need = csa2::topk_ws_bytes(rows, n);
  if (need && (!ws || ws_bytes < need || !al16(ws))) return CSA2_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (csa2::launch_topk(scores, rows, n, ld, n_valid, k, nullptr, 0, pair_pos, pair_n, 0, nullptr, ws, st) !=
      cudaSuccess)
    return CSA2_ERR_CUDA;
  const int64_t total = int64_t(rows) * k;
  return csa2::launch_pdl(csa2::shard_pairs_kernel, dim3(unsigned((total + 255) / 256)), dim3(256), 0, st, scores, ld,
                          total, k, map, map_ld, pos_offset, pair_pos, pair_score) == cudaSuccess
             ? CSA2_OK
             : CSA2_ERR_CUDA;
}

extern "C" csa2_status csa2_merge_topk_pairs(const float* pair_score, const int32_t* pair_pos, const int32_t* pair_n,
                                             int G, int rows, int k, int32_t* idx, int32_t* n_sel, void* ws,
                                             size_t ws_bytes, csa2_stream_t stream) {
  if (G < 1 || G > 64 || rows < 0 || k < 1 || k > CSA2_MAX_K) return CSA2_ERR_INVALID_ARG;
  if (rows == 0) return CSA2_OK;
  if (rows > 65535) return CSA2_ERR_UNSUPPORTED;
  if (!pair_score || !pair_pos || !idx) return CSA2_ERR_INVALID_ARG;
  const size_t need = csa2::merge_pairs_ws_bytes(rows, G, k);
  if (!ws || ws_bytes < need || !al16(ws)) return CSA2_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t n = int64_t(G) * k;
  char* w = static_cast<char*>(ws);
  float* pscore = reinterpret_cast<float*>(w);
  int32_t* ppos = reinterpret_cast<int32_t*>(w + csa2::align256(size_t(rows) * size_t(n) * 4));
  int32_t* pcount = reinterpret_cast<int32_t*>(w + 2 * csa2::align256(size_t(rows) * size_t(n) * 4));
  void* tws = w + 2 * csa2::align256(size_t(rows) * size_t(n) * 4) + csa2::align256(size_t(rows) * 4);
  if (csa2::launch_pdl(csa2::pack_pairs_kernel, dim3(unsigned(rows)), dim3(256), 0, st, pair_score, pair_pos, pair_n,
                       G, rows, k, pscore, ppos, pcount) != cudaSuccess)
    return CSA2_ERR_CUDA;
  return csa2::launch_topk(pscore, rows, n, n, pcount, k, ppos, n, idx, n_sel, 0, nullptr, tws, st) == cudaSuccess
             ? CSA2_OK
             : CSA2_ERR_CUDA;
}

extern "C" csa2_status csa2_shard_indices(const int32_t* idx, int rows, int k, int64_t lo, int64_t hi,
                                          int32_t* idx_local, csa2_stream_t stream) {
  if (rows < 0 || k < 1 || lo < 0 || hi < lo) return CSA2_ERR_INVALID_ARG;
  if (rows == 0) return CSA2_OK;
  if (!idx || !idx_local) return CSA2_ERR_INVALID_ARG;
  const int64_t total = int64_t(rows) * k;
  return csa2::launch_pdl(csa2::shard_indices_kernel, dim3(unsigned((total + 255) / 256)), dim3(256), 0,
                          reinterpret_cast<cudaStream_t>(stream), idx, total, lo, hi, idx_local) == cudaSuccess
             ? CSA2_OK
             : CSA2_ERR_CUDA;
}

extern "C" csa2_status csa2_attn_merge_shards(const uint16_t* out_g, const float* lse_g, int G, int rows,
                                              uint16_t* out, float* lse, csa2_stream_t stream) {
  if (G < 1 || rows < 0) return CSA2_ERR_INVALID_ARG;
  if (rows == 0) return CSA2_OK;
  if (rows > 65535) return CSA2_ERR_UNSUPPORTED;
  if (!out_g || !lse_g || !out || !al16(out_g) || !al16(out)) return CSA2_ERR_INVALID_ARG;
  return csa2::launch_pdl(csa2::merge_shards_kernel, dim3(unsigned(rows), unsigned(CSA2_H)), dim3(128), 0,
                          reinterpret_cast<cudaStream_t>(stream), out_g, lse_g, G, rows, out, lse) == cudaSuccess
             ? CSA2_OK
             : CSA2_ERR_CUDA;
}

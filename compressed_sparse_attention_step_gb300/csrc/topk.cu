// Exact Top-K selection ("selects fresh Top-512 indices", ai-maestro.online "DeepSeek AI released
// DeepSeek-V4.1-Flash with 1M context, FP4", section "Compressed Sparse Attention 2"; Top-2,048
// blocks for the hierarchical pool).  Order: larger score first, equal scores by lower column.
//
// One CTA of 1024 threads per row, radix select on ordered 32-bit score keys:
//  1. histogram of the top 12 key bits over the row (shared-memory atomics);
//  2. the bin b1 holding the k-th largest key is found with a block scan; every key above b1 is
//     selected outright (fewer than k of them);
//  3. fast path (bin b1 holds <= 8192 keys, the common case): one more pass over the row
//     collects the selected columns and the (key, column) candidates of bin b1 in shared
//     memory; radix rounds on the low 20 key bits then on the column bits (ascending, so equal
//     keys go to the lower column) find the exact threshold; the k columns are sorted with a
//     bitonic network and written ascending;
//  4. fallback (bin b1 larger, e.g. massive ties): the same radix rounds run over the row in
//     global memory, and a final ordered pass with a block scan writes the selected columns in
//     ascending order directly.
// All counts are integers and the output is a pure function of the scores: deterministic.
#include "common.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 1024;
constexpr int kCap = 8192;  // candidates kept in shared memory

struct SelSmem {
  uint32_t hist[4096];
  uint32_t cand_key[kCap];
  int32_t cand_col[kCap];
  int32_t sel[CSA2_MAX_K];
  uint32_t scan_tmp[32];
  uint32_t nsel, ncand;
  uint32_t res_bin, res_before;
  uint32_t run_g, run_e;
};

__device__ __forceinline__ uint32_t load_key(const float* s, int64_t i) { return score_key(__ldg(s + i)); }

// Find the bin where the cumulative count, walking from the highest bin down (from_top) or from
// the lowest bin up, first reaches `need` (1 <= need <= total).  Writes sm.res_bin and
// sm.res_before (count strictly before that bin in walking order).  All threads call it.
__device__ void find_bin(SelSmem& sm, int nbins, uint32_t need, bool from_top) {
  const int t = threadIdx.x;
  const int per = (nbins + kThreads - 1) / kThreads;  // 1..4
  // thread t owns walk positions [t*per, t*per + per)
  uint32_t local = 0;
  for (int e = 0; e < per; ++e) {
    const int wpos = t * per + e;
    if (wpos < nbins) local += sm.hist[from_top ? nbins - 1 - wpos : wpos];
  }
  const uint32_t excl = block_exclusive_scan(local, sm.scan_tmp, nullptr);
  if (excl < need && excl + local >= need) {
    uint32_t cum = excl;
    for (int e = 0; e < per; ++e) {
      const int wpos = t * per + e;
      const int bin = from_top ? nbins - 1 - wpos : wpos;
      const uint32_t h = sm.hist[bin];
      if (cum + h >= need) {
        sm.res_bin = uint32_t(bin);
        sm.res_before = cum;
        break;
      }
      cum += h;
    }
  }
  __syncthreads();
}

__device__ __forceinline__ void zero_hist(SelSmem& sm, int nbins) {
  for (int i = threadIdx.x; i < nbins; i += kThreads) sm.hist[i] = 0;
  __syncthreads();
}

__device__ __forceinline__ int32_t out_value(const int32_t* mrow, int32_t col) {
  return mrow ? __ldg(mrow + col) : col;
}

__global__ void __launch_bounds__(kThreads, 1) topk_select_kernel(
    const float* __restrict__ scores, int64_t n, int64_t ld, const int32_t* __restrict__ n_valid,
    int k, const int32_t* __restrict__ map, int64_t map_ld, int32_t* __restrict__ idx,
    int32_t* __restrict__ n_sel, int expand8, int32_t* __restrict__ pool_len) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  const int row = blockIdx.x;
  const int t = threadIdx.x;
  const float* s = scores + int64_t(row) * ld;
  const int32_t* mrow = map ? map + int64_t(row) * map_ld : nullptr;
  const int64_t nv = n_valid ? min(max(int64_t(n_valid[row]), int64_t(0)), n) : n;
  __syncthreads();  // every thread has read n_valid before pool_len (possibly the same array) is written
  const int out_w = expand8 ? k * CSA2_BLOCK : k;
  int32_t* out = idx + int64_t(row) * out_w;

  auto emit = [&](int slot, int32_t col) {
    const int32_t v = out_value(mrow, col);
    if (expand8) {
#pragma unroll
      for (int r = 0; r < CSA2_BLOCK; ++r) out[slot * CSA2_BLOCK + r] = v * CSA2_BLOCK + r;
    } else {
      out[slot] = v;
    }
  };
  auto finish = [&](int64_t cnt) {
    if (t == 0) {
      if (n_sel) n_sel[row] = int32_t(cnt);
      if (pool_len) pool_len[row] = int32_t(cnt * (expand8 ? CSA2_BLOCK : 1));
    }
    for (int i = int(cnt) * (expand8 ? CSA2_BLOCK : 1) + t; i < out_w; i += kThreads) out[i] = -1;
  };

  if (nv <= k) {  // everything valid is selected, already ascending
    for (int i = t; i < nv; i += kThreads) emit(i, i);
    finish(nv);
    return;
  }

  // ---- pass 0: histogram of the top 12 key bits --------------------------------------------
  zero_hist(sm, 4096);
  for (int64_t i = t; i < nv; i += kThreads) atomicAdd(&sm.hist[load_key(s, i) >> 20], 1u);
  __syncthreads();
  find_bin(sm, 4096, uint32_t(k), true);
  const uint32_t b1 = sm.res_bin;
  uint32_t need = uint32_t(k) - sm.res_before;  // still to take from bin b1 (>= 1)
  const uint32_t cnt1 = sm.hist[b1];
  __syncthreads();

  if (cnt1 <= uint32_t(kCap)) {
    // ---- fast path ---------------------------------------------------------------------------
    if (t == 0) { sm.nsel = 0; sm.ncand = 0; }
    __syncthreads();
    for (int64_t i = t; i < nv; i += kThreads) {
      const uint32_t key = load_key(s, i);
      const uint32_t bin = key >> 20;
      if (bin > b1) {
        sm.sel[atomicAdd(&sm.nsel, 1u)] = int32_t(i);
      } else if (bin == b1) {
        const uint32_t c = atomicAdd(&sm.ncand, 1u);
        sm.cand_key[c] = key;
        sm.cand_col[c] = int32_t(i);
      }
    }
    __syncthreads();
    const int nc = int(sm.ncand);
    // rounds on key bits [19:10] and [9:0] (largest first)
    zero_hist(sm, 1024);
    for (int c = t; c < nc; c += kThreads) atomicAdd(&sm.hist[(sm.cand_key[c] >> 10) & 1023u], 1u);
    __syncthreads();
    find_bin(sm, 1024, need, true);
    const uint32_t d1 = sm.res_bin;
    need -= sm.res_before;
    __syncthreads();
    zero_hist(sm, 1024);
    for (int c = t; c < nc; c += kThreads) {
      const uint32_t key = sm.cand_key[c];
      if (((key >> 10) & 1023u) == d1) atomicAdd(&sm.hist[key & 1023u], 1u);
    }
    __syncthreads();
    find_bin(sm, 1024, need, true);
    const uint32_t tau = (b1 << 20) | (d1 << 10) | sm.res_bin;
    need -= sm.res_before;            // ties at tau to take, lowest columns first
    const uint32_t nties = sm.hist[sm.res_bin];
    __syncthreads();
    int32_t col_cut = 0x7FFFFFFF;     // take ties with column <= col_cut
    if (need < nties) {
      // rounds on column bits [30:20], [19:10], [9:0] (smallest first)
      uint32_t prefix = 0;
      const int shifts[3] = {20, 10, 0};
      const int widths[3] = {11, 10, 10};
      for (int r = 0; r < 3; ++r) {
        const int nb = 1 << widths[r];
        zero_hist(sm, nb);
        const uint32_t hi_mask = (r == 0) ? 0u : (0xFFFFFFFFu << (shifts[r] + widths[r]));
        for (int c = t; c < nc; c += kThreads) {
          const uint32_t col = uint32_t(sm.cand_col[c]);
          if (sm.cand_key[c] == tau && (col & hi_mask) == prefix)
            atomicAdd(&sm.hist[(col >> shifts[r]) & uint32_t(nb - 1)], 1u);
        }
        __syncthreads();
        find_bin(sm, nb, need, false);
        prefix |= sm.res_bin << shifts[r];
        need -= sm.res_before;
        __syncthreads();
      }
      col_cut = int32_t(prefix);
    }
    for (int c = t; c < nc; c += kThreads) {
      const uint32_t key = sm.cand_key[c];
      if (key > tau || (key == tau && sm.cand_col[c] <= col_cut)) sm.sel[atomicAdd(&sm.nsel, 1u)] = sm.cand_col[c];
    }
    __syncthreads();
    // bitonic sort of the k selected columns (padded to a power of two)
    int P = 1;
    while (P < k) P <<= 1;
    for (int i = k + t; i < P; i += kThreads) sm.sel[i] = 0x7FFFFFFF;
    __syncthreads();
    for (int size = 2; size <= P; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = t; i < P / 2; i += kThreads) {
          const int lo = 2 * i - (i & (stride - 1));
          const int hi = lo + stride;
          const bool up = ((lo & size) == 0);
          const int32_t a = sm.sel[lo], b = sm.sel[hi];
          if ((a > b) == up) { sm.sel[lo] = b; sm.sel[hi] = a; }
        }
        __syncthreads();
      }
    }
    for (int i = t; i < k; i += kThreads) emit(i, sm.sel[i]);
    finish(k);
    return;
  }

  // ---- fallback: radix rounds over the row in global memory ------------------------------------
  zero_hist(sm, 1024);
  for (int64_t i = t; i < nv; i += kThreads) {
    const uint32_t key = load_key(s, i);
    if ((key >> 20) == b1) atomicAdd(&sm.hist[(key >> 10) & 1023u], 1u);
  }
  __syncthreads();
  find_bin(sm, 1024, need, true);
  const uint32_t d1 = sm.res_bin;
  need -= sm.res_before;
  __syncthreads();
  zero_hist(sm, 1024);
  const uint32_t pre22 = (b1 << 10) | d1;
  for (int64_t i = t; i < nv; i += kThreads) {
    const uint32_t key = load_key(s, i);
    if ((key >> 10) == pre22) atomicAdd(&sm.hist[key & 1023u], 1u);
  }
  __syncthreads();
  find_bin(sm, 1024, need, true);
  const uint32_t tau = (pre22 << 10) | sm.res_bin;
  need -= sm.res_before;  // ties at tau to take, in column order
  if (t == 0) { sm.run_g = 0; sm.run_e = 0; }
  __syncthreads();
  // ordered output: slot(i) = #(key > tau before i) + min(#(key == tau before i), need)
  constexpr int kItems = 4;
  for (int64_t base = 0; base < nv; base += int64_t(kThreads) * kItems) {
    uint32_t keys[kItems];
    uint32_t g = 0, e = 0;
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      const int64_t i = base + int64_t(t) * kItems + it;
      keys[it] = (i < nv) ? load_key(s, i) : 0u;
      if (i < nv) { g += keys[it] > tau; e += keys[it] == tau; }
    }
    uint32_t tot;
    const uint32_t pre = block_exclusive_scan((g << 16) | e, sm.scan_tmp, &tot);
    uint32_t G = sm.run_g + (pre >> 16), E = sm.run_e + (pre & 0xFFFFu);
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      const int64_t i = base + int64_t(t) * kItems + it;
      if (i >= nv) break;
      if (keys[it] > tau) {
        emit(int(G + min(E, need)), int32_t(i));
        ++G;
      } else if (keys[it] == tau) {
        if (E < need) emit(int(G + E), int32_t(i));
        ++E;
      }
    }
    __syncthreads();
    if (t == 0) { sm.run_g += tot >> 16; sm.run_e += tot & 0xFFFFu; }
    __syncthreads();
  }
  finish(k);
}

}  // namespace

cudaError_t launch_topk(const float* scores, int rows, int64_t n, int64_t ld, const int32_t* n_valid,
                        int k, const int32_t* map, int64_t map_ld, int32_t* idx, int32_t* n_sel,
                        int expand8, int32_t* pool_len, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const size_t smem = sizeof(SelSmem);
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  topk_select_kernel<<<rows, kThreads, smem, st>>>(scores, n, ld, n_valid, k, map, map_ld, idx, n_sel,
                                                   expand8, pool_len);
  return cudaGetLastError();
}

}  // namespace csa2

extern "C" csa2_status csa2_topk(const float* scores, int rows, int64_t n, int64_t ld,
                                 const int32_t* n_valid, int k, const int32_t* map, int64_t map_ld,
                                 int32_t* idx, int32_t* n_sel, void* ws, size_t ws_bytes,
                                 csa2_stream_t stream) {
  (void)ws;
  (void)ws_bytes;
  if (rows < 0 || n < 0 || ld < n || k < 1 || k > CSA2_MAX_K || n >= (int64_t(1) << 31))
    return CSA2_ERR_INVALID_ARG;
  if (rows == 0) return CSA2_OK;
  if (!scores || !idx || (map && map_ld < n)) return CSA2_ERR_INVALID_ARG;
  return csa2::launch_topk(scores, rows, n, ld, n_valid, k, map, map_ld, idx, n_sel, 0, nullptr,
                           reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? CSA2_OK
             : CSA2_ERR_CUDA;
}

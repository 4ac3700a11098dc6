// Exact Top-K selection ("selects fresh Top-512 indices", ai-maestro.online "DeepSeek AI released
// DeepSeek-V4.1-Flash with 1M context, FP4", section "Compressed Sparse Attention 2"; Top-2,048
// blocks for the hierarchical pool).  Order: larger score first, equal scores by lower column;
// the k selected columns are returned in ascending order.
//
// Radix select on ordered 32-bit score keys (-0 and +0 share a key):
//  * rows up to 8192 columns (topk_kernel): one CTA per row histograms the top 12 key bits, lists
//    the keys in and above the bin of the k-th largest key, and selects among them;
//  * rows of 8193 to 131072 columns (topk_cluster_kernel): one thread-block cluster of two, four or
//    eight CTAs per row, in one launch.  The CTAs histogram the maxima of their 16-key groups, sum the
//    histograms through distributed shared memory, take the bin of the k-th largest group maximum
//    as a lower bound on the k-th largest key (those k maxima are k distinct keys) and append the
//    keys at or above it to the first CTA's list, which selects among them;
//  * longer rows, the same bound over three launches of (slices x rows) CTAs and then one CTA per
//    row: topk_hist_kernel histograms the rows' 16-key group maxima and keeps every group's key;
//    topk_filter_kernel takes the bin of the k-th largest group maximum as a lower bound on the
//    k-th largest key (those k maxima are k distinct keys) and lists the keys at or above it,
//    reading only the groups whose key reaches it; topk_select_kernel selects among the list.
// Among the candidates, a list of one key takes its k lowest columns directly; otherwise radix
// rounds on the key bits, then on the column bits (ascending, so equal keys go to the lower
// column), find the exact k-th (key, column).  The winners are written in column order by rank,
// each found by a binary search over the per-word prefix counts of the winners' column bitmap (a
// bitonic sort for very long rows).  A row whose candidates overflow the list (massive ties) is
// selected by one CTA with the same rounds over the row in global memory and an ordered,
// scan-based output.  Counts are integers and every decision is a pure function of the scores,
// so the result is deterministic.
#include <algorithm>

#include "common.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 512;          // CTA size of the one-CTA-per-row selections
constexpr int kCandCap = 10240;        // candidates per row
constexpr int kBins = 4096;            // first-level bins (top 12 key bits)
constexpr int64_t kBitmapCols = 262144;   // rows up to this long are ordered through a bitmap

struct SelSmem {
  static constexpr int kNT = kThreads;
  static constexpr int kCap = kCandCap;
  static constexpr int kHistBins = kBins;
  uint32_t hist[kBins];
  uint32_t cand_key[kCandCap];
  int32_t cand_col[kCandCap];
  union {
    int32_t sel[CSA2_MAX_K];
    uint32_t bits[kBitmapCols / 32];
  };
  int32_t stage[CSA2_MAX_K];  // the winners' columns by output slot
  uint32_t scan_tmp[32];
  uint32_t nsel, ncand, base;
  uint32_t res_bin, res_before;
  uint32_t run_g, run_e;
  int is_last;
  __device__ __forceinline__ int phys(int c) const { return c; }
  __device__ __forceinline__ int32_t* out_stage() { return stage; }
};

// The prefill rows' selection (bitmap_select_kernel): a shorter candidate list (marked keys beyond
// it stream through keep_top), kept in column order, so that two CTAs share an SM.
constexpr int kBmThreads = 256;
constexpr int kBmCap = 4096;  // > CSA2_MAX_K
struct BmSmem {
  static constexpr int kNT = kBmThreads;
  static constexpr int kHistBins = 2048;
  uint32_t hist[2048];
  uint32_t cand_key[kBmCap];
  int32_t cand_col[kBmCap];  // always in column order
  uint32_t scan_tmp[32];
  uint32_t nsel, ncand, base;
  uint32_t res_bin, res_before;
  uint32_t run_g, run_e;
  uint32_t is_last;
  __device__ __forceinline__ int phys(int c) const { return c; }
};

// Visit keys [lo, hi) of a row in tiles of 4 * U * blockDim.x (each thread takes U groups of 4
// consecutive keys, with 16-byte loads when aligned).  Every thread makes the same number of
// calls (valid = false past hi), so warp collectives inside f are safe.
template <int U, class F>
__device__ __forceinline__ void for_each_key(const float* s, int64_t lo, int64_t hi, F&& f) {
  const int nt = blockDim.x;
  for (int64_t base = lo; base < hi; base += int64_t(4) * nt * U) {
    float v[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i0 = base + (int64_t(u) * nt + threadIdx.x) * 4;
      if (i0 + 3 < hi && ((reinterpret_cast<uintptr_t>(s + i0) & 15u) == 0)) {
        const float4 x = __ldg(reinterpret_cast<const float4*>(s + i0));
        v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) v[u][e] = (i0 + e < hi) ? __ldg(s + i0 + e) : 0.0f;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i0 = base + (int64_t(u) * nt + threadIdx.x) * 4;
#pragma unroll
      for (int e = 0; e < 4; ++e) f(i0 + e, score_key(v[u][e]), i0 + e < hi);
    }
  }
}

// The 16 scores thread t reads in one sweep step starting at b0: float4 number u * kThreads + t
// (u < 4) of the step, i.e. v[4 u + e] = s[b0 + 4 (u kThreads + t) + e]; past hi they are NaN,
// which every comparison rejects and fmaxf ignores.
template <int NT = kThreads>
__device__ __forceinline__ void load16(const float* s, int64_t b0, int64_t hi, float (&v)[16]) {
  const int t = threadIdx.x;
  const bool full = b0 + int64_t(16) * NT <= hi && ((reinterpret_cast<uintptr_t>(s + b0) & 15u) == 0);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int64_t i0 = b0 + (int64_t(u) * NT + t) * 4;
    if (full) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(s + i0));
      v[4 * u] = x.x; v[4 * u + 1] = x.y; v[4 * u + 2] = x.z; v[4 * u + 3] = x.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) v[4 * u + e] = (i0 + e < hi) ? __ldg(s + i0 + e) : __int_as_float(0x7FC00000);
    }
  }
}

template <int NB, int NT>
__device__ void find_bin_n(const uint32_t* hist, uint32_t need, bool from_top, uint32_t* scan_tmp,
                           uint32_t* res_bin, uint32_t* res_before) {
  constexpr int per = NB / NT;   // 2 .. 16 bins per thread (NT threads in the block)
  static_assert(per * NT == NB && (per == 16 || per == 8 || per == 4 || per == 2), "bin count");
  const int t = threadIdx.x;
  // the run of walk positions [t*per, t*per + per) covers bins [lo_bin, lo_bin + per)
  const int lo_bin = from_top ? NB - (t + 1) * per : t * per;
  uint32_t h[per];
  if constexpr (per >= 4) {
#pragma unroll
    for (int v = 0; v < per / 4; ++v) {
      const uint4 a = reinterpret_cast<const uint4*>(hist + lo_bin)[v];
      h[4 * v] = a.x; h[4 * v + 1] = a.y; h[4 * v + 2] = a.z; h[4 * v + 3] = a.w;
    }
  } else {
    const uint2 a = *reinterpret_cast<const uint2*>(hist + lo_bin);
    h[0] = a.x; h[1] = a.y;
  }
  uint32_t local = 0;
#pragma unroll
  for (int e = 0; e < per; ++e) local += h[e];
  const uint32_t excl = block_exclusive_scan(local, scan_tmp, nullptr);
  if (excl < need && excl + local >= need) {
    uint32_t cum = excl;
    bool done = false;
#pragma unroll
    for (int e = 0; e < per; ++e) {
      const int i = from_top ? per - 1 - e : e;   // walk order within the run
      if (!done && cum + h[i] >= need) {
        *res_bin = uint32_t(lo_bin + i);
        *res_before = cum;
        done = true;
      }
      cum += h[i];
    }
  }
  __syncthreads();
}

// Bin where the cumulative count, walking from the highest bin down (from_top) or from the lowest
// bin up, first reaches need (1 <= need <= total).  Result in *res_bin / *res_before (count
// strictly before that bin in walking order).  All NT threads of the block call it.  Each thread
// reads its run of bins with vector loads (a strided scalar walk would hit one bank per warp).
template <int NT = kThreads>
__device__ __forceinline__ void find_bin(const uint32_t* hist, int nbins, uint32_t need, bool from_top,
                                         uint32_t* scan_tmp, uint32_t* res_bin, uint32_t* res_before) {
  if constexpr (4096 / NT <= 16) {
    if (nbins == 4096) {
      find_bin_n<4096, NT>(hist, need, from_top, scan_tmp, res_bin, res_before);
      return;
    }
  }
  if (nbins == 2048) find_bin_n<2048, NT>(hist, need, from_top, scan_tmp, res_bin, res_before);
  else find_bin_n<1024, NT>(hist, need, from_top, scan_tmp, res_bin, res_before);
}

__device__ __forceinline__ void zero(uint32_t* h, int n) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) h[i] = 0;
  __syncthreads();
}

// Histogram of the top 12 key bits of keys [lo, hi) into h (shared memory).
__device__ __forceinline__ void hist12(const float* s, int64_t lo, int64_t hi, uint32_t* h) {
  for_each_key<8>(s, lo, hi, [&](int64_t, uint32_t key, bool valid) {
    if (valid) atomicAdd(&h[key >> 20], 1u);
  });
}

// Output of one row (optionally through a column -> position map, optionally expanded to the
// eight positions of each selected block).
static_assert(CSA2_BLOCK == 8, "a block's positions are written as two 16-byte stores");
struct RowOut {
  const int32_t* mrow;
  int32_t* out;
  int out_w, expand8;
  __device__ __forceinline__ void emit(int slot, int32_t col) const {
    const int32_t v = mrow ? __ldg(mrow + col) : col;
    if (expand8) {
#pragma unroll
      for (int r = 0; r < CSA2_BLOCK; ++r) out[slot * CSA2_BLOCK + r] = v * CSA2_BLOCK + r;
    } else {
      out[slot] = v;
    }
  }
  // Slots [0, cnt) from stage[slot] = column, consecutive threads writing consecutive outputs.
  __device__ __forceinline__ void emit_staged(const int32_t* stage, int cnt) const {
    if (expand8 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0) {  // a slot's eight positions: two 16-byte stores
      for (int sl = threadIdx.x; sl < cnt; sl += blockDim.x) {
        const int32_t col = stage[sl];
        const int32_t v = (mrow ? __ldg(mrow + col) : col) * CSA2_BLOCK;
        int4* o4 = reinterpret_cast<int4*>(out + int64_t(sl) * CSA2_BLOCK);
        o4[0] = make_int4(v, v + 1, v + 2, v + 3);
        o4[1] = make_int4(v + 4, v + 5, v + 6, v + 7);
      }
    } else if (expand8) {
      for (int i = threadIdx.x; i < cnt * CSA2_BLOCK; i += blockDim.x) {
        const int32_t col = stage[i / CSA2_BLOCK];
        out[i] = (mrow ? __ldg(mrow + col) : col) * CSA2_BLOCK + i % CSA2_BLOCK;
      }
    } else {
      for (int i = threadIdx.x; i < cnt; i += blockDim.x) {
        const int32_t col = stage[i];
        out[i] = mrow ? __ldg(mrow + col) : col;
      }
    }
  }
};

__device__ void finish_row(const RowOut& o, int64_t cnt, int row, int32_t* n_sel, int32_t* pool_len) {
  if (threadIdx.x == 0) {
    if (n_sel) n_sel[row] = int32_t(cnt);
    if (pool_len) pool_len[row] = int32_t(cnt * (o.expand8 ? CSA2_BLOCK : 1));
  }
  for (int i = int(cnt) * (o.expand8 ? CSA2_BLOCK : 1) + threadIdx.x; i < o.out_w; i += blockDim.x) o.out[i] = -1;
}

// The cut of the k largest of the nc candidates in shared memory (nc >= k) by (key desc, column
// asc): a candidate is among them iff key > tau, or key == tau and column <= col_cut.
// kmin / kmax: bounds of the candidates' keys (the bits they share need no round).
template <class S>
__device__ __forceinline__ void candidate_cut(S& sm, int nc, int k, uint32_t& tau_out, int32_t& cut_out,
                                              uint32_t kmin = 0u, uint32_t kmax = 0xFFFFFFFFu) {
  const int t = threadIdx.x;
  const uint32_t diff = kmin ^ kmax;
  int top = diff ? 32 - __clz(diff) : 0;  // key bits [0, top) differ among the candidates
  uint32_t need = uint32_t(k);
  uint32_t mask = top >= 32 ? 0u : 0xFFFFFFFFu << top;
  uint32_t prefix = kmin & mask;
  uint32_t nties = uint32_t(nc);  // candidates equal to tau (all of them when no round runs)
  while (top > 0) {  // rounds of up to 12 bits (11 with a 2048-bin histogram), from the highest differing bit down
    const int w = min(S::kHistBins >= 4096 ? 12 : 11, top), sh = top - w;
    const uint32_t wmask = (1u << w) - 1u;
    const int nb = max(1 << w, 1024);  // find_bin's smallest width
    zero(sm.hist, nb);
    for (int c = t; c < nc; c += blockDim.x) {
      const uint32_t key = sm.cand_key[sm.phys(c)];
      if ((key & mask) == prefix) atomicAdd(&sm.hist[(key >> sh) & wmask], 1u);
    }
    __syncthreads();
    find_bin<S::kNT>(sm.hist, nb, need, true, sm.scan_tmp, &sm.res_bin, &sm.res_before);
    prefix |= sm.res_bin << sh;
    mask |= wmask << sh;
    need -= sm.res_before;
    nties = sm.hist[sm.res_bin];
    __syncthreads();
    top = sh;
  }
  const uint32_t tau = prefix;                       // the k-th largest key
  int32_t col_cut = 0x7FFFFFFF;                       // take ties at tau with column <= col_cut
  if (need < nties) {
    uint32_t cpre = 0;
    const int cshift[3] = {20, 10, 0}, cwidth[3] = {11, 10, 10};
    for (int r = 0; r < 3; ++r) {
      const int nb = 1 << cwidth[r];
      zero(sm.hist, nb);
      const uint32_t hi_mask = (r == 0) ? 0u : (0xFFFFFFFFu << (cshift[r] + cwidth[r]));
      for (int c = t; c < nc; c += blockDim.x) {
        const uint32_t col = uint32_t(sm.cand_col[sm.phys(c)]);
        if (sm.cand_key[sm.phys(c)] == tau && (col & hi_mask) == cpre)
          atomicAdd(&sm.hist[(col >> cshift[r]) & uint32_t(nb - 1)], 1u);
      }
      __syncthreads();
      find_bin<S::kNT>(sm.hist, nb, need, false, sm.scan_tmp, &sm.res_bin, &sm.res_before);
      cpre |= sm.res_bin << cshift[r];
      need -= sm.res_before;
      __syncthreads();
    }
    col_cut = int32_t(cpre);
  }
  tau_out = tau;
  cut_out = col_cut;
}

// Writes each winner (key > tau, or key == tau and column <= col_cut) of the nc candidates whose
// rank among the set bits of the bitmap sm.bits (the winners' columns; nwords words, zero up to
// per * NT words, per a power of two <= 8) is below cnt to out slot = that rank.  Each thread owns
// a run of per words; the words' exclusive prefix counts go to sm.hist, and a winner's rank is its
// word's prefix plus the set bits below it in the word.  The columns are placed by rank in shared
// memory first (sm.out_stage()), so that the output is written in order.
template <class S>
__device__ __forceinline__ void emit_by_column(S& sm, int nc, int per, int cnt, uint32_t tau, int32_t col_cut,
                                               const RowOut& o) {
  const int t = threadIdx.x;
  uint32_t wv[8];
  const uint32_t* run = sm.bits + t * per;
  if (per >= 4) {
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (4 * q < per) {
        const uint4 a = reinterpret_cast<const uint4*>(run)[q];
        wv[4 * q] = a.x; wv[4 * q + 1] = a.y; wv[4 * q + 2] = a.z; wv[4 * q + 3] = a.w;
      }
  } else {
#pragma unroll
    for (int e = 0; e < 2; ++e)
      if (e < per) wv[e] = run[e];
  }
  uint32_t local = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e)
    if (e < per) local += __popc(wv[e]);
  uint32_t pre = block_exclusive_scan(local, sm.scan_tmp, nullptr);
  uint32_t* pw = sm.hist;
#pragma unroll
  for (int e = 0; e < 8; ++e)
    if (e < per) {
      pw[t * per + e] = pre;
      pre += __popc(wv[e]);
    }
  __syncthreads();
  int32_t* stage = sm.out_stage();
  for (int c = t; c < nc; c += blockDim.x) {
    const uint32_t key = sm.cand_key[sm.phys(c)];
    const int32_t col = sm.cand_col[sm.phys(c)];
    if (key > tau || (key == tau && col <= col_cut)) {
      const int w = col >> 5;
      const uint32_t r = pw[w] + __popc(sm.bits[w] & ((1u << (col & 31)) - 1u));
      if (r < uint32_t(cnt)) stage[r] = col;
    }
  }
  __syncthreads();
  o.emit_staged(stage, cnt);
}

// The k largest of the nc candidates in shared memory (nc >= k) by (key desc, column asc), emitted
// in column order; columns are < ncols.
template <class S>
__device__ __noinline__ void select_candidates(S& sm, int nc, int k, int64_t ncols, const RowOut o) {
  const int t = threadIdx.x, lane = t & 31;
  // A list of one key (all candidates tie, as the exact zeros of a row whose head weights are all
  // negative do): the k lowest columns win, with no radix rounds.
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  for (int c = t; c < nc; c += blockDim.x) {
    const uint32_t key = sm.cand_key[sm.phys(c)];
    kmin = min(kmin, key);
    kmax = max(kmax, key);
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (t == 0) {
    sm.run_g = 0xFFFFFFFFu;
    sm.run_e = 0u;
  }
  __syncthreads();
  if (lane == 0) {
    atomicMin(&sm.run_g, kmin);
    atomicMax(&sm.run_e, kmax);
  }
  __syncthreads();
  const uint32_t kmin_all = sm.run_g, kmax_all = sm.run_e;
  const bool one_key = kmin_all == kmax_all;
  uint32_t tau = kmin_all;
  int32_t col_cut = 0x7FFFFFFF;
  __syncthreads();
  const int nwords = int((ncols + 31) / 32);
  int per = 1;
  while (per * int(blockDim.x) < nwords) per <<= 1;
  const bool rank_emit = per <= 8 && per * int(blockDim.x) <= kBins;
  if (!(one_key && rank_emit)) candidate_cut(sm, nc, k, tau, col_cut, kmin_all, kmax_all);
  if (rank_emit) {
    // bitmap of the winners (of every candidate for one key); each winner of column rank below k
    // goes to that slot
    for (int i = t; i < per * int(blockDim.x); i += blockDim.x) sm.bits[i] = 0u;
    __syncthreads();
    for (int c = t; c < nc; c += blockDim.x) {
      const uint32_t key = sm.cand_key[sm.phys(c)];
      const int32_t col = sm.cand_col[sm.phys(c)];
      if (key > tau || (key == tau && col <= col_cut)) atomicOr(&sm.bits[col >> 5], 1u << (col & 31));
    }
    __syncthreads();
    emit_by_column(sm, nc, per, k, tau, col_cut, o);
    return;
  }
  if (ncols <= kBitmapCols) {
    // slot of a winner = number of winners in lower columns: bitmap + prefix popcounts
    for (int i = t; i < nwords; i += blockDim.x) sm.bits[i] = 0u;
    __syncthreads();
    for (int c = t; c < nc; c += blockDim.x) {
      const uint32_t key = sm.cand_key[sm.phys(c)];
      const int32_t col = sm.cand_col[sm.phys(c)];
      if (key > tau || (key == tau && col <= col_cut)) atomicOr(&sm.bits[col >> 5], 1u << (col & 31));
    }
    __syncthreads();
    const int per2 = (nwords + int(blockDim.x) - 1) / int(blockDim.x);
    uint32_t local = 0;
    for (int e = 0; e < per2; ++e) {
      const int wi = t * per2 + e;
      if (wi < nwords) local += __popc(sm.bits[wi]);
    }
    uint32_t slot = block_exclusive_scan(local, sm.scan_tmp, nullptr);
    for (int e = 0; e < per2; ++e) {
      const int wi = t * per2 + e;
      if (wi >= nwords) break;
      uint32_t wv = sm.bits[wi];
      while (wv) {
        const int b = __ffs(wv) - 1;
        o.emit(int(slot++), int32_t(wi * 32 + b));
        wv &= wv - 1u;
      }
    }
    return;
  }
  if (t == 0) sm.nsel = 0;
  __syncthreads();
  for (int c = t; c < nc; c += blockDim.x) {
    const uint32_t key = sm.cand_key[sm.phys(c)];
    if (key > tau || (key == tau && sm.cand_col[sm.phys(c)] <= col_cut)) sm.sel[atomicAdd(&sm.nsel, 1u)] = sm.cand_col[sm.phys(c)];
  }
  __syncthreads();
  int P = 1;
  while (P < k) P <<= 1;
  for (int i = k + t; i < P; i += blockDim.x) sm.sel[i] = 0x7FFFFFFF;
  __syncthreads();
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = t; i < P / 2; i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool up = ((lo & size) == 0);
        const int32_t a = sm.sel[lo], b = sm.sel[hi];
        if ((a > b) == up) { sm.sel[lo] = b; sm.sel[hi] = a; }
      }
      __syncthreads();
    }
  }
  for (int i = t; i < k; i += blockDim.x) o.emit(i, sm.sel[i]);
}

// Visits the winners (key > tau, or key == tau and column <= col_cut) of the nc listed candidates in
// list order: f(slot, key, col) with slot = the number of winners before it.  All threads call it.
template <class S, class F>
__device__ __forceinline__ void for_each_winner(S& sm, int nc, uint32_t tau, int32_t col_cut, F&& f) {
  const int t = threadIdx.x;
  if (t == 0) sm.run_g = 0;
  __syncthreads();
  for (int base = 0; base < nc; base += blockDim.x) {
    const int c = base + t;
    uint32_t key = 0;
    int32_t col = 0;
    bool win = false;
    if (c < nc) {
      key = sm.cand_key[c];
      col = sm.cand_col[c];
      win = key > tau || (key == tau && col <= col_cut);
    }
    uint32_t tot;
    const uint32_t slot = sm.run_g + block_exclusive_scan(win ? 1u : 0u, sm.scan_tmp, &tot);  // reads done
    if (win) f(slot, key, col);
    __syncthreads();
    if (t == 0) sm.run_g += tot;
    __syncthreads();
  }
}

// Keeps the k largest of the nc candidates (nc >= k) by (key desc, column asc) at the front of the
// list, in their list order (a stable compaction); returns the k-th largest key.
template <class S>
__device__ __noinline__ uint32_t keep_top(S& sm, int nc, int k) {
  uint32_t tau;
  int32_t col_cut;
  candidate_cut(sm, nc, k, tau, col_cut);
  for_each_winner(sm, nc, tau, col_cut, [&](uint32_t slot, uint32_t key, int32_t col) {
    sm.cand_key[slot] = key;
    sm.cand_col[slot] = col;
  });
  return tau;
}

// The k largest of the nc listed candidates (nc >= k), emitted in list order (the list is in
// column order).
template <class S>
__device__ __noinline__ void select_listed(S& sm, int nc, int k, const RowOut o) {
  uint32_t tau;
  int32_t col_cut;
  candidate_cut(sm, nc, k, tau, col_cut);
  for_each_winner(sm, nc, tau, col_cut, [&](uint32_t slot, uint32_t, int32_t col) { o.emit(int(slot), col); });
}

// Whole-row selection by one CTA (short rows, and rows whose candidates overflow).
template <class S>
__device__ __noinline__ void select_row(S& sm, const float* s, int64_t nv, int k, const RowOut o) {
  const int t = threadIdx.x;
  if (nv <= int64_t(16) * S::kNT) {
    // the whole row in registers, 16 keys per thread: one read serves the histogram and the list
    float v[16];
    load16<S::kNT>(s, 0, nv, v);  // NaN past nv: neither counted nor listed
    zero(sm.hist, kBins);
#pragma unroll
    for (int e = 0; e < 16; ++e)
      if (v[e] == v[e]) atomicAdd(&sm.hist[score_key(v[e]) >> 20], 1u);
    __syncthreads();
    find_bin(sm.hist, kBins, uint32_t(k), true, sm.scan_tmp, &sm.res_bin, &sm.res_before);
    const uint32_t b1 = sm.res_bin;  // the list (keys in bins >= b1) holds at most nv <= S::kCap keys
    __syncthreads();
    uint32_t take = 0;
#pragma unroll
    for (int e = 0; e < 16; ++e) take |= (v[e] == v[e] && (score_key(v[e]) >> 20) >= b1) ? 1u << e : 0u;
    uint32_t listed;
    uint32_t slot = block_exclusive_scan(uint32_t(__popc(take)), sm.scan_tmp, &listed);
#pragma unroll
    for (int e = 0; e < 16; ++e)
      if ((take >> e) & 1u) {
        sm.cand_key[slot] = score_key(v[e]);
        sm.cand_col[slot] = int32_t(4 * ((e >> 2) * S::kNT + t) + (e & 3));
        ++slot;
      }
    __syncthreads();
    select_candidates(sm, int(listed), k, nv, o);
    return;
  }
  zero(sm.hist, kBins);
  hist12(s, 0, nv, sm.hist);
  __syncthreads();
  find_bin(sm.hist, kBins, uint32_t(k), true, sm.scan_tmp, &sm.res_bin, &sm.res_before);
  const uint32_t b1 = sm.res_bin;
  const uint32_t ncand = sm.res_before + sm.hist[b1];   // keys in bins >= b1
  uint32_t need = uint32_t(k) - sm.res_before;
  __syncthreads();
  if (ncand <= uint32_t(S::kCap)) {
    // the keys in bins >= b1, listed one tile of 16 keys per thread at a time: one block scan of the
    // threads' counts per tile places them (one counter shared by every warp would serialise)
    uint32_t listed = 0;
    for (int64_t b0 = 0; b0 < nv; b0 += int64_t(16) * blockDim.x) {  // the same trip count for every thread
      float v[16];
      load16<S::kNT>(s, b0, nv, v);  // NaN past nv: never listed
      uint32_t take = 0;
#pragma unroll
      for (int e = 0; e < 16; ++e) take |= (v[e] == v[e] && (score_key(v[e]) >> 20) >= b1) ? 1u << e : 0u;
      uint32_t tot;
      uint32_t slot = listed + block_exclusive_scan(uint32_t(__popc(take)), sm.scan_tmp, &tot);
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if ((take >> e) & 1u) {
          sm.cand_key[slot] = score_key(v[e]);
          sm.cand_col[slot] = int32_t(b0 + 4 * ((e >> 2) * int64_t(S::kNT) + t) + (e & 3));
          ++slot;
        }
      listed += tot;
    }
    __syncthreads();
    select_candidates(sm, int(listed), k, nv, o);
    return;
  }
  // rounds on key bits [19:10] and [9:0] over the row, then an ordered pass
  zero(sm.hist, 1024);
  for_each_key<8>(s, 0, nv, [&](int64_t, uint32_t key, bool valid) {
    if (valid && (key >> 20) == b1) atomicAdd(&sm.hist[(key >> 10) & 1023u], 1u);
  });
  __syncthreads();
  find_bin(sm.hist, 1024, need, true, sm.scan_tmp, &sm.res_bin, &sm.res_before);
  const uint32_t pre22 = (b1 << 10) | sm.res_bin;
  need -= sm.res_before;
  __syncthreads();
  zero(sm.hist, 1024);
  for_each_key<8>(s, 0, nv, [&](int64_t, uint32_t key, bool valid) {
    if (valid && (key >> 10) == pre22) atomicAdd(&sm.hist[key & 1023u], 1u);
  });
  __syncthreads();
  find_bin(sm.hist, 1024, need, true, sm.scan_tmp, &sm.res_bin, &sm.res_before);
  const uint32_t tau = (pre22 << 10) | sm.res_bin;
  need -= sm.res_before;  // ties at tau to take, in column order
  if (t == 0) { sm.run_g = 0; sm.run_e = 0; }
  __syncthreads();
  // slot(i) = #(key > tau before i) + min(#(key == tau before i), need)
  constexpr int kItems = 4;
  for (int64_t base = 0; base < nv; base += int64_t(blockDim.x) * kItems) {
    uint32_t keys[kItems];
    uint32_t g = 0, e = 0;
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      const int64_t i = base + int64_t(t) * kItems + it;
      keys[it] = (i < nv) ? score_key(__ldg(s + i)) : 0u;
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
        o.emit(int(G + min(E, need)), int32_t(i));
        ++G;
      } else if (keys[it] == tau) {
        if (E < need) o.emit(int(G + E), int32_t(i));
        ++E;
      }
    }
    __syncthreads();
    if (t == 0) { sm.run_g += tot >> 16; sm.run_e += tot & 0xFFFFu; }
    __syncthreads();
  }
}

// The smallest score whose key is >= key (the -0/+0 key gives -0, which +0 also passes).
__device__ __forceinline__ float key_floor_score(uint32_t key) {
  if (key <= 0x00800000u) return -INFINITY;  // at or below the key of -FLT_MAX: every finite score
  if (key & 0x80000000u) return __uint_as_float(key & 0x7FFFFFFFu) == 0.0f ? -0.0f : __uint_as_float(key & 0x7FFFFFFFu);
  return __uint_as_float(~key);
}

__device__ __forceinline__ int64_t row_valid(const int32_t* n_valid, int row, int64_t n) {
  return n_valid ? min(max(int64_t(n_valid[row]), int64_t(0)), n) : n;
}

// Rows up to kSmallRow entries: one CTA selects over the whole row.
__global__ void __launch_bounds__(kThreads, 1) topk_kernel(
    const float* __restrict__ scores, int64_t n, int64_t ld, const int32_t* __restrict__ n_valid, int k,
    const int32_t* __restrict__ map, int64_t map_ld, int32_t* __restrict__ idx, int32_t* __restrict__ n_sel,
    int expand8, int32_t* __restrict__ pool_len) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.y, t = threadIdx.x;
  const float* s = scores + int64_t(row) * ld;
  const int64_t nv = row_valid(n_valid, row, n);
  __syncthreads();  // every thread has read n_valid before pool_len (possibly the same array) is written
  RowOut o{map ? map + int64_t(row) * map_ld : nullptr, idx + int64_t(row) * (expand8 ? k * CSA2_BLOCK : k),
           expand8 ? k * CSA2_BLOCK : k, expand8};
  if (nv <= k) {  // everything valid is selected, already ascending
    for (int i = t; i < nv; i += kThreads) o.emit(i, i);
    finish_row(o, nv, row, n_sel, pool_len);
    return;
  }
  select_row(sm, s, nv, k, o);
  finish_row(o, k, row, n_sel, pool_len);
}

// ---- rows longer than kSmallRow: the row's bound first, then only the keys above it are listed -----
// 1. topk_hist_kernel: every CTA of a row adds the maxima of its slice's 16-key groups (the 16 keys a
//    thread reads in one sweep step) to the row's histogram of the top 12 key bits;
// 2. topk_filter_kernel: every CTA of the row takes the bin of the k-th largest group maximum (a
//    lower bound on the k-th largest key: those k maxima are k distinct keys) from the complete
//    histogram and appends the keys of its slice at or above that bin to the row's list, a superset
//    of the Top-k.  It reads the scores of only the groups whose maximum (kept by the histogram
//    kernel) reaches the bound: every key at or above it lies in one of them;
// 3. topk_select_kernel: one CTA per row selects among them (the whole row instead, should they
//    overflow the list) and clears the histogram and counters for the next launch.
constexpr int kHThreads = 256;
constexpr int64_t kSmallRow = 8192;  // rows up to this long: one CTA selects over the whole row
constexpr int64_t kSweep = int64_t(16) * kHThreads;  // keys of one sweep step of a slice CTA
constexpr int kFSweeps = 4;          // sweeps whose groups the filter lists at once (4 * kHThreads <= kBins)

__global__ void __launch_bounds__(kHThreads) topk_hist_kernel(const float* __restrict__ scores, int64_t n, int64_t ld,
                                                              const int32_t* __restrict__ n_valid, int k,
                                                              int64_t slice_len, uint32_t* __restrict__ row_hist,
                                                              uint32_t* __restrict__ gkey, int64_t gld) {
  __shared__ uint32_t h[kBins];
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.y, t = threadIdx.x, lane = t & 31;
  const int64_t nv = row_valid(n_valid, row, n);
  const int64_t lo = int64_t(blockIdx.x) * slice_len, hi = min(lo + slice_len, nv);
  if (nv <= k || lo >= hi) return;
  for (int i = t; i < kBins; i += kHThreads) h[i] = 0u;
  __syncthreads();
  const float* s = scores + int64_t(row) * ld;
  for (int64_t b0 = lo; b0 < hi; b0 += int64_t(16) * kHThreads) {  // the same trip count for every thread
    float v[16];
    load16<kHThreads>(s, b0, hi, v);  // NaN past hi: fmaxf skips it
    float gm = v[0];
#pragma unroll
    for (int e = 1; e < 16; ++e) gm = fmaxf(gm, v[e]);
    const bool has = b0 + 4 * t < hi;
    const uint32_t gmk = score_key(gm);
    if (has) gkey[int64_t(row) * gld + (b0 / kSweep) * kHThreads + t] = gmk;
    const uint32_t bin = has ? gmk >> 20 : 0xFFFFFFFFu;
    const unsigned peers = __match_any_sync(0xffffffffu, bin);
    if (has && (__ffs(peers) - 1) == lane) atomicAdd(&h[bin], uint32_t(__popc(peers)));
  }
  __syncthreads();
  uint32_t* gh = row_hist + int64_t(row) * kBins;
  for (int i = t; i < kBins; i += kHThreads)
    if (h[i]) atomicAdd(gh + i, h[i]);
}

__global__ void __launch_bounds__(kHThreads) topk_filter_kernel(const float* __restrict__ scores, int64_t n,
                                                                int64_t ld, const int32_t* __restrict__ n_valid, int k,
                                                                int64_t slice_len, const uint32_t* __restrict__ row_hist,
                                                                const uint32_t* __restrict__ gkey, int64_t gld,
                                                                uint32_t* __restrict__ cand_key,
                                                                int32_t* __restrict__ cand_col,
                                                                uint32_t* __restrict__ row_ctl) {
  __shared__ __align__(16) uint32_t h[kBins];  // the row histogram, then the chunk's group list
  __shared__ uint32_t scan_tmp[32];
  __shared__ uint32_t res_bin, res_before, s_base;
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.y, t = threadIdx.x, lane = t & 31;
  const int64_t nv = row_valid(n_valid, row, n);
  const int64_t lo = int64_t(blockIdx.x) * slice_len, hi = min(lo + slice_len, nv);
  if (nv <= k || lo >= hi) return;
  // the row's histogram: four 16-byte loads per thread, all in flight together
  const uint4* gh4 = reinterpret_cast<const uint4*>(row_hist + int64_t(row) * kBins);
  uint4 hv[kBins / 4 / kHThreads];
#pragma unroll
  for (int u = 0; u < kBins / 4 / kHThreads; ++u) hv[u] = __ldcg(gh4 + u * kHThreads + t);
  uint32_t groups = 0;
#pragma unroll
  for (int u = 0; u < kBins / 4 / kHThreads; ++u) {
    reinterpret_cast<uint4*>(h)[u * kHThreads + t] = hv[u];
    groups += hv[u].x + hv[u].y + hv[u].z + hv[u].w;
  }
  groups = __reduce_add_sync(0xffffffffu, groups);
  if (lane == 0) scan_tmp[t >> 5] = groups;
  __syncthreads();
  groups = 0;
  for (int w = 0; w < kHThreads / 32; ++w) groups += scan_tmp[w];
  __syncthreads();
  uint32_t bound = 0;  // keys >= bound: a superset of the row's Top-k
  if (groups >= uint32_t(k)) {
    find_bin<kHThreads>(h, kBins, uint32_t(k), true, scan_tmp, &res_bin, &res_before);
    bound = res_bin << 20;
  }
  const float fb = key_floor_score(bound);
  const float* s = scores + int64_t(row) * ld;
  const bool vec = (reinterpret_cast<uintptr_t>(s) & 15u) == 0;  // slices start at multiples of kSweep keys
  const uint32_t* gk = gkey + int64_t(row) * gld;
  uint32_t* ctl = row_ctl + 2 * int64_t(row);
  uint32_t* ck = cand_key + int64_t(row) * kCandCap;
  int32_t* cc = cand_col + int64_t(row) * kCandCap;
  for (int64_t c0 = lo; c0 < hi; c0 += int64_t(kFSweeps) * kSweep) {  // the same trip count for every thread
    // 1. the chunk's groups whose key reaches the bound (group q * kHThreads + t: the 16 keys thread t
    //    of the histogram kernel took in sweep q), listed in shared memory
    uint32_t take = 0;
#pragma unroll
    for (int q = 0; q < kFSweeps; ++q) {
      const int64_t b0 = c0 + int64_t(q) * kSweep;
      if (b0 + 4 * t < hi && __ldcg(gk + (b0 / kSweep) * kHThreads + t) >= bound) take |= 1u << q;
    }
    uint32_t nlist;
    uint32_t slot = block_exclusive_scan(uint32_t(__popc(take)), scan_tmp, &nlist);
#pragma unroll
    for (int q = 0; q < kFSweeps; ++q)
      if ((take >> q) & 1u) h[slot++] = uint32_t(q * kHThreads + t);
    __syncthreads();
    // 2. their keys, a quarter group (four consecutive keys) per item and four items per thread in
    //    flight; one reservation per CTA and batch
    const int items = int(nlist) * 4;
    for (int i0 = 0; i0 < items; i0 += 4 * kHThreads) {
      float v[4][4];
      int64_t col[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int it = i0 + u * kHThreads + t;
        col[u] = hi;
        if (it < items) {
          const uint32_t g = h[it >> 2];
          col[u] = c0 + int64_t(g / kHThreads) * kSweep + 4 * (int64_t(it & 3) * kHThreads + (g % kHThreads));
        }
        if (vec && col[u] + 3 < hi) {
          const float4 x = __ldcg(reinterpret_cast<const float4*>(s + col[u]));
          v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) v[u][e] = (col[u] + e < hi) ? __ldcg(s + col[u] + e) : __int_as_float(0x7FC00000);
        }
      }
      uint32_t m = 0;  // bit 4u+e: key v[u][e] is listed (NaN, past hi, fails)
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int e = 0; e < 4; ++e) m |= (v[u][e] >= fb) ? 1u << (4 * u + e) : 0u;
      uint32_t tot;
      uint32_t base = block_exclusive_scan(uint32_t(__popc(m)), scan_tmp, &tot);
      if (tot == 0) continue;
      if (t == 0) s_base = atomicAdd(ctl, tot);
      __syncthreads();
      base += s_base;
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if ((m >> (4 * u + e)) & 1u) {
            if (base < uint32_t(kCandCap)) {
              ck[base] = score_key(v[u][e]);
              cc[base] = int32_t(col[u] + e);
            }
            ++base;
          }
      __syncthreads();  // s_base is read by every thread before the next reservation
    }
    __syncthreads();  // the group list is rewritten by the next chunk
  }
}

__global__ void __launch_bounds__(kThreads, 1) topk_select_kernel(
    const float* __restrict__ scores, int64_t n, int64_t ld, const int32_t* __restrict__ n_valid, int k,
    const int32_t* __restrict__ map, int64_t map_ld, int32_t* __restrict__ idx, int32_t* __restrict__ n_sel,
    int expand8, int32_t* __restrict__ pool_len, uint32_t* __restrict__ row_hist,
    const uint32_t* __restrict__ cand_key, const int32_t* __restrict__ cand_col, uint32_t* __restrict__ row_ctl) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x, t = threadIdx.x;
  const float* s = scores + int64_t(row) * ld;
  const int64_t nv = row_valid(n_valid, row, n);
  __syncthreads();  // every thread has read n_valid before pool_len (possibly the same array) is written
  RowOut o{map ? map + int64_t(row) * map_ld : nullptr, idx + int64_t(row) * (expand8 ? k * CSA2_BLOCK : k),
           expand8 ? k * CSA2_BLOCK : k, expand8};
  if (nv <= k) {  // everything valid is selected, already ascending
    for (int i = t; i < nv; i += kThreads) o.emit(i, i);
    finish_row(o, nv, row, n_sel, pool_len);
    return;
  }
  const uint32_t total = __ldcg(row_ctl + 2 * int64_t(row));
  if (total <= uint32_t(kCandCap)) {
    const uint32_t* ck = cand_key + int64_t(row) * kCandCap;
    const int32_t* cc = cand_col + int64_t(row) * kCandCap;
    // the list in 16-byte pieces, all of a thread's loads in flight together (rows start 16-byte
    // aligned: kCandCap is a multiple of 4)
    constexpr int kPieces = (kCandCap / 4 + kThreads - 1) / kThreads;
    const uint32_t np = (total + 3) / 4;
    uint4 pa[kPieces], pb[kPieces];
#pragma unroll
    for (int u = 0; u < kPieces; ++u) {
      const uint32_t pi = u * kThreads + t;
      if (pi < np) {
        pa[u] = __ldcg(reinterpret_cast<const uint4*>(ck) + pi);
        pb[u] = __ldcg(reinterpret_cast<const uint4*>(cc) + pi);
      }
    }
#pragma unroll
    for (int u = 0; u < kPieces; ++u) {
      const uint32_t pi = u * kThreads + t;
      if (pi < np) {
        reinterpret_cast<uint4*>(sm.cand_key)[pi] = pa[u];
        reinterpret_cast<uint4*>(sm.cand_col)[pi] = pb[u];
      }
    }
    __syncthreads();
    select_candidates(sm, int(total), k, nv, o);
  } else {
    select_row(sm, s, nv, k, o);
  }
  finish_row(o, k, row, n_sel, pool_len);
  // the next launch finds the histogram and the counters zero
  uint32_t* gh = row_hist + int64_t(row) * kBins;
  for (int i = t; i < kBins; i += kThreads) gh[i] = 0u;
  if (t == 0) {
    row_ctl[2 * int64_t(row)] = 0u;
    row_ctl[2 * int64_t(row) + 1] = 0u;
  }
}

// ---- rows of 8193 to 131072 columns: one thread-block cluster per row, one launch ------------------
// The C CTAs of a cluster (C = 2, 4 or 8) split the row into C runs of whole sweeps (8192 columns).  In a
// sweep, thread t's group is the 16 keys at columns 4 (u kThreads + t) + e (u, e < 4), so that a warp's
// loads are contiguous.  Each CTA keeps its groups' largest keys (and how many keys equal them) in
// shared memory and histograms them by the top 12 key bits; the C histograms are summed through
// distributed shared memory (each CTA sums a C-th of the bins and writes the sums into every CTA).
// Then the bin of the k-th largest group maximum bounds the k-th largest key from below (those k
// maxima are k distinct keys), and every CTA lists its keys at or above the bound, read again from
// only its groups that reach it: the first CTA at the front of its list, the others in their own
// shared memory and then, behind one reservation each, at the back of the first CTA's list, which
// selects among the whole list.  When at least k keys equal the row's largest key, those k with the
// lowest columns are the answer, and every CTA writes its share in column order without a list.
constexpr int kClCap = 8192;        // candidates the first CTA of a cluster holds
constexpr int kClSweep = 16 * kThreads;
constexpr int kClGroups = 2048;     // groups per CTA: four sweeps
static_assert(kClGroups >= CSA2_MAX_K, "the group maxima's space stages the output");
constexpr int64_t kClMaxCols = 131072;

struct ClSmem {
  static constexpr int kNT = kThreads;
  static constexpr int kCap = kClCap;
  static constexpr int kHistBins = kBins;
  uint32_t hist[kBins];          // this CTA's histogram of its group maxima; later the selection's
  union {
    uint32_t hsum[kBins];        // the row's histogram (every CTA holds all of it)
    uint32_t bits[kBins];        // the first CTA's winner bitmap (columns < 131072)
    int32_t sel[CSA2_MAX_K];
  };
  uint32_t gmax[kClGroups];      // largest key of each of this CTA's groups
  uint8_t gcnt[kClGroups];       // how many of the group's keys equal it (0: an empty group)
  uint32_t cand_key[kClCap];     // the list: the first CTA's keys at the front, the others' at the back
  int32_t cand_col[kClCap];
  uint32_t scan_tmp[32];
  uint32_t peer_max[8], peer_cnt[8], peer_ng[8];  // every CTA's largest key, its count, its groups
  uint32_t nsel, ncand, base, tail, ngrp;
  uint32_t res_bin, res_before;
  uint32_t run_g, run_e;
  int n0, gap;                   // list entry c lies at c (c < n0) or c + gap
  __device__ __forceinline__ int phys(int c) const { return c < n0 ? c : c + gap; }
  // the winners' columns by output slot (the group maxima are no longer needed then)
  __device__ __forceinline__ int32_t* out_stage() { return reinterpret_cast<int32_t*>(gmax); }
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
// The address of the same shared-memory word in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t dsmem_ld(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];\n" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void dsmem_st(uint32_t a, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;\n" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t dsmem_add(uint32_t a, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;\n" : "=r"(old) : "r"(a), "r"(v) : "memory");
  return old;
}
// Every thread of every CTA of the cluster; what any of them wrote before it is visible after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// Group t of the sweep at column c0: key[4 u + e] = column c0 + 4 (u kThreads + t) + e, below hi;
// bit 4 u + e of the returned mask: that key exists.
__device__ __forceinline__ uint32_t load_sweep_group(const float* s, int64_t c0, int64_t hi, int t,
                                                     uint32_t (&key)[16]) {
  const bool full = c0 + kClSweep <= hi && ((reinterpret_cast<uintptr_t>(s + c0) & 15u) == 0);
  uint32_t m = 0u;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int64_t i0 = c0 + 4 * (int64_t(u) * kThreads + t);
    if (full) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(s + i0));
      key[4 * u] = score_key(x.x); key[4 * u + 1] = score_key(x.y);
      key[4 * u + 2] = score_key(x.z); key[4 * u + 3] = score_key(x.w);
      m |= 0xFu << (4 * u);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool in = i0 + e < hi;
        key[4 * u + e] = in ? score_key(__ldg(s + i0 + e)) : 0u;
        m |= in ? 1u << (4 * u + e) : 0u;
      }
    }
  }
  return m;
}

template <int C>
__global__ void __launch_bounds__(kThreads, 2) topk_cluster_kernel(
    const float* __restrict__ scores, int64_t n, int64_t ld, const int32_t* __restrict__ n_valid, int k,
    const int32_t* __restrict__ map, int64_t map_ld, int32_t* __restrict__ idx, int32_t* __restrict__ n_sel,
    int expand8, int32_t* __restrict__ pool_len) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ClSmem& sm = *reinterpret_cast<ClSmem*>(smem_raw);
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.y, t = threadIdx.x, lane = t & 31, wid = t >> 5;
  const uint32_t rank = cluster_rank();
  const float* s = scores + int64_t(row) * ld;
  const int64_t nv = row_valid(n_valid, row, n);  // read by every CTA before the first CTA writes pool_len
  const RowOut o{map ? map + int64_t(row) * map_ld : nullptr, idx + int64_t(row) * (expand8 ? k * CSA2_BLOCK : k),
                 expand8 ? k * CSA2_BLOCK : k, expand8};
  const bool all = nv <= k;  // the same in every CTA of the cluster
  // this CTA's sweeps [q0, q0 + nq) of the row's ceil(nv / kClSweep)
  const int64_t sweeps = (nv + kClSweep - 1) / kClSweep, spc = (sweeps + C - 1) / C;
  const int64_t q0 = int64_t(rank) * spc;
  const int nq = all ? 0 : int(max(min(spc, sweeps - q0), int64_t(0)));
  const int ng = nq * kThreads;  // group q kThreads + t: thread t's group of sweep q0 + q
  auto sweep_col = [&](int q) { return (q0 + q) * int64_t(kClSweep); };

  // ---- 1. group maxima, their histogram, this CTA's largest key and its count ---------------------
  for (int i = t; i < kBins; i += kThreads) sm.hist[i] = 0u;
  if (t == 0) {
    sm.nsel = 0u;
    sm.base = 0u;
    sm.tail = 0u;
    sm.ngrp = 0u;
  }
  __syncthreads();
  uint32_t lmax = 0u, lng = 0u;
  for (int q = 0; q < nq; q += 2) {  // two sweeps' loads in flight
    uint32_t key[2][16], m[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      m[u] = 0u;
      if (q + u < nq) m[u] = load_sweep_group(s, sweep_col(q + u), nv, t, key[u]);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (q + u >= nq) break;
      uint32_t gm = 0u, gc = 0u;
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if ((m[u] >> e) & 1u) gm = max(gm, key[u][e]);
#pragma unroll
      for (int e = 0; e < 16; ++e) gc += ((m[u] >> e) & 1u) && key[u][e] == gm;
      const bool has = m[u] != 0u;
      const int gi = (q + u) * kThreads + t;
      sm.gmax[gi] = gm;
      sm.gcnt[gi] = uint8_t(gc);
      lmax = max(lmax, gm);
      lng += has;
      const uint32_t bin = has ? gm >> 20 : 0xFFFFFFFFu;
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      if (has && (__ffs(peers) - 1) == lane) atomicAdd(&sm.hist[bin], uint32_t(__popc(peers)));
    }
  }
  lmax = __reduce_max_sync(0xffffffffu, lmax);
  lng = __reduce_add_sync(0xffffffffu, lng);
  if (lane == 0) {
    sm.scan_tmp[wid] = lmax;
    if (lng) atomicAdd(&sm.ngrp, lng);
  }
  __syncthreads();
  lmax = 0u;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) lmax = max(lmax, sm.scan_tmp[w]);
  uint32_t lcnt = 0u;
  for (int gi = t; gi < ng; gi += kThreads)
    if (sm.gmax[gi] == lmax) lcnt += sm.gcnt[gi];
  lcnt = __reduce_add_sync(0xffffffffu, lcnt);
  if (lane == 0 && lcnt) atomicAdd(&sm.base, lcnt);
  cluster_sync_all();  // 1: every CTA has started, and its histogram and counts are complete

  if (all) {  // everything valid is selected, already ascending
    if (rank == 0) {
      for (int i = t; i < nv; i += kThreads) o.emit(i, i);
      finish_row(o, nv, row, n_sel, pool_len);
    }
    return;
  }
  // ---- 2. the row's histogram in every CTA; every CTA's largest key, its count, its groups --------
  constexpr int kPer = kBins / C;
  for (int b = t; b < kPer; b += kThreads) {
    const int bin = int(rank) * kPer + b;
    uint32_t sum = 0u;
#pragma unroll
    for (int r = 0; r < C; ++r) sum += dsmem_ld(dsmem_addr(&sm.hist[bin], uint32_t(r)));
#pragma unroll
    for (int r = 0; r < C; ++r) dsmem_st(dsmem_addr(&sm.hsum[bin], uint32_t(r)), sum);
  }
  if (t < C) {
    dsmem_st(dsmem_addr(&sm.peer_max[rank], uint32_t(t)), lmax);
    dsmem_st(dsmem_addr(&sm.peer_cnt[rank], uint32_t(t)), sm.base);
    dsmem_st(dsmem_addr(&sm.peer_ng[rank], uint32_t(t)), sm.ngrp);
  }
  cluster_sync_all();  // 2

  uint32_t M = 0u, cnt_m = 0u, before_m = 0u, groups = 0u;  // the row's largest key, its count, its
#pragma unroll                                               // count in lower CTAs; non-empty groups
  for (int r = 0; r < C; ++r) {
    M = max(M, sm.peer_max[r]);
    groups += sm.peer_ng[r];
  }
#pragma unroll
  for (int r = 0; r < C; ++r)
    if (sm.peer_max[r] == M) {
      cnt_m += sm.peer_cnt[r];
      before_m += r < int(rank) ? sm.peer_cnt[r] : 0u;
    }
  if (cnt_m >= uint32_t(k)) {
    // ---- at least k keys equal the largest: the k lowest columns holding it, in column order ------
    if (lmax == M && before_m < uint32_t(k)) {
      uint32_t done = before_m;
      for (int q = 0; q < nq && done < uint32_t(k); ++q) {
        const int gi = q * kThreads + t;
        uint32_t key[16], m = 0u;
        if (sm.gmax[gi] == M) m = load_sweep_group(s, sweep_col(q), nv, t, key);
#pragma unroll
        for (int u = 0; u < 4; ++u) {  // the sweep's columns in order: by u, then thread, then e
          uint32_t c = 0u;
#pragma unroll
          for (int e = 0; e < 4; ++e) c += ((m >> (4 * u + e)) & 1u) && key[4 * u + e] == M;
          uint32_t tot;
          uint32_t slot = done + block_exclusive_scan(c, sm.scan_tmp, &tot);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (((m >> (4 * u + e)) & 1u) && key[4 * u + e] == M) {
              if (slot < uint32_t(k)) o.emit(int(slot), int32_t(sweep_col(q) + 4 * (u * kThreads + t) + e));
              ++slot;
            }
          done += tot;
        }
      }
    }
    if (rank == 0) finish_row(o, k, row, n_sel, pool_len);
    return;
  }
  // ---- 3. the bound; this CTA's keys at or above it listed -----------------------------------------
  uint32_t bound = 0u;  // keys >= bound: a superset of the row's Top-k
  if (groups >= uint32_t(k)) {
    find_bin<kThreads>(sm.hsum, kBins, uint32_t(k), true, sm.scan_tmp, &sm.res_bin, &sm.res_before);
    bound = sm.res_bin << 20;
  }
  // the groups that reach the bound, listed (the row histogram's space is free now), so that each
  // thread loads at most one group per round and all of a round's loads are in flight together
  uint32_t* glist = sm.hsum;
  if (t == 0) sm.ncand = 0u;
  __syncthreads();
  {
    uint32_t hits = 0u;  // bit q: this thread's group of sweep q0 + q reaches the bound
    for (int q = 0; q < nq; ++q) {
      const int gi = q * kThreads + t;
      if (sm.gcnt[gi] && sm.gmax[gi] >= bound) hits |= 1u << q;
    }
    const uint32_t hc = __popc(hits);
    uint32_t incl = hc;  // the warp's inclusive prefix of the counts, one reservation per warp
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += y;
    }
    const uint32_t wtot = __shfl_sync(0xffffffffu, incl, 31);
    uint32_t wb = 0u;
    if (lane == 31 && wtot) wb = atomicAdd(&sm.ncand, wtot);
    uint32_t slot = __shfl_sync(0xffffffffu, wb, 31) + incl - hc;
    for (int q = 0; q < nq; ++q)
      if ((hits >> q) & 1u) glist[slot++] = uint32_t(q * kThreads + t);
  }
  __syncthreads();
  const int nlist = int(sm.ncand);
  for (int i0 = 0; i0 < nlist; i0 += kThreads) {  // the same trip count for every thread of the CTA
    const int i = i0 + t;
    const int gi = i < nlist ? int(glist[i]) : 0, q = gi / kThreads, gt = gi % kThreads;
    uint32_t key[16], m = 0u;
    if (i < nlist) m = load_sweep_group(s, sweep_col(q), nv, gt, key);
    uint32_t take = 0u;
#pragma unroll
    for (int e = 0; e < 16; ++e) take |= (((m >> e) & 1u) && key[e] >= bound) ? 1u << e : 0u;
    const uint32_t cnt = __popc(take);
    uint32_t incl = cnt;  // the warp's inclusive prefix of the counts
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += y;
    }
    const uint32_t wtot = __shfl_sync(0xffffffffu, incl, 31);
    uint32_t wbase = 0u;
    if (lane == 31 && wtot) wbase = atomicAdd(&sm.nsel, wtot);
    wbase = __shfl_sync(0xffffffffu, wbase, 31);
    uint32_t slot = wbase + incl - cnt;
#pragma unroll
    for (int e = 0; e < 16; ++e)
      if ((take >> e) & 1u) {
        if (slot < uint32_t(kClCap)) {
          sm.cand_key[slot] = key[e];
          sm.cand_col[slot] = int32_t(sweep_col(q) + 4 * ((e >> 2) * kThreads + gt) + (e & 3));
        }
        ++slot;
      }
  }
  __syncthreads();
  const uint32_t mine = sm.nsel;  // may exceed kClCap: then the row falls back to the whole-row path
  if (rank != 0 && mine) {
    // behind one reservation, at the back of the first CTA's list
    if (t == 0) sm.base = dsmem_add(dsmem_addr(&sm.tail, 0u), mine > uint32_t(kClCap) ? uint32_t(kClCap) + 1u : mine);
    __syncthreads();
    const uint32_t end = uint32_t(kClCap) - sm.base;  // this CTA's entries end here
    if (sm.base + mine <= uint32_t(kClCap)) {
      const uint32_t key_at = dsmem_addr(sm.cand_key, 0u), col_at = dsmem_addr(sm.cand_col, 0u);
      for (uint32_t i = t; i < mine; i += kThreads) {
        const uint32_t d = end - mine + i;
        dsmem_st(key_at + 4u * d, sm.cand_key[i]);
        dsmem_st(col_at + 4u * d, uint32_t(sm.cand_col[i]));
      }
    }
  }
  cluster_sync_all();  // 3: the list is complete; no CTA touches another's shared memory after this
  if (rank != 0) return;
  // ---- 4. the first CTA selects among the list (the whole row should it have overflowed) -----------
  const uint32_t back = sm.tail;  // the other CTAs' entries, [kClCap - back, kClCap)
  const uint32_t nc = mine + back;
  if (nc <= uint32_t(kClCap)) {
    sm.n0 = int(mine);
    sm.gap = kClCap - int(back) - int(mine);
    select_candidates(sm, int(nc), k, nv, o);
  } else {
    sm.n0 = kClCap;
    sm.gap = 0;
    select_row(sm, s, nv, k, o);
  }
  finish_row(o, k, row, n_sel, pool_len);
}

// Prefill rows: the keys marked in the tensor-core filter's bitmap are rescored in the canonical
// order (eight lanes per key, the query slice in registers) and the exact Top-k is selected among
// them.  One CTA per query row, except that the first n_sliced rows of the order (those with the
// most marked keys) take n_slices CTAs each: CTA s rescores the marked keys of ranks
// [s total / n_slices, (s + 1) total / n_slices), keeps its k best (in column order) in the
// workspace, and the last of them to finish (an atomic ticket) merges the slices in order and
// selects among them.  The k best of the row are among the slices' k best, so this is exact.
__global__ void __launch_bounds__(kBmThreads, 2) bitmap_select_kernel(
    const uint16_t* __restrict__ qI, const float* __restrict__ w, int Nq, const uint16_t* __restrict__ KI,
    int64_t cap, const int32_t* __restrict__ lens, int ratio, const int32_t* __restrict__ q_pos, int k,
    const uint32_t* __restrict__ bitmap, int64_t n_words, const uint32_t* __restrict__ ubound,
    const int32_t* __restrict__ order, int n_sliced, int n_slices, uint32_t* __restrict__ sl_key,
    int32_t* __restrict__ sl_col, uint32_t* __restrict__ sl_cnt, unsigned int* __restrict__ tickets,
    int32_t* __restrict__ idx, int32_t* __restrict__ n_sel) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  BmSmem& sm = *reinterpret_cast<BmSmem*>(smem_raw);
  pdl_wait();
  pdl_trigger();
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  // this CTA's place in the order, and its slice (-1: the whole row)
  const int n_sl_ctas = n_sliced * n_slices;
  int pos = int(blockIdx.x), slice = -1;
  if (pos < n_sl_ctas) {
    slice = pos % n_slices;
    pos /= n_slices;
  } else {
    pos -= n_sl_ctas - n_sliced;
  }
  const int64_t row = order ? int64_t(__ldg(order + pos)) : int64_t(pos), b = row / Nq, qi = row - b * Nq;
  const int64_t T = min(max(int64_t(lens[b]), int64_t(0)), cap);
  const int64_t p = q_pos ? int64_t(q_pos[row]) : int64_t(ratio) * T - Nq + qi;
  const int64_t vis = (p + 1 < 0) ? 0 : min((p + 1) / ratio, T);
  RowOut o{nullptr, idx + row * k, k, 0};
  if (vis <= k) {
    if (slice > 0) return;
    for (int64_t i = t; i < vis; i += kBmThreads) o.emit(int(i), int32_t(i));
    finish_row(o, vis, int(row), n_sel, nullptr);
    return;
  }
  const uint32_t* bm = bitmap + row * n_words;
  const uint16_t* qrow = qI + row * (CSA2_HI * CSA2_DI);
  const uint16_t* kseq = KI + b * cap * CSA2_DI;
  const int64_t nw = min((vis + 31) / 32, n_words);
  const int per = int((nw + kBmThreads - 1) / kBmThreads);
  auto word = [&](int64_t wi) -> uint32_t {
    uint32_t v = __ldg(bm + wi);
    const int64_t valid = vis - 32 * wi;  // bits of this word that are visible positions
    if (valid < 32) v &= (1u << valid) - 1u;
    return v;
  };
  uint32_t local = 0;
  for (int e = 0; e < per; ++e) {
    const int64_t wi = int64_t(t) * per + e;
    if (wi < nw) local += __popc(word(wi));
  }
  uint32_t total;
  const uint32_t first = block_exclusive_scan(local, sm.scan_tmp, &total);  // rank of this thread's first key
  const int j = lane & 7, sub = lane >> 3;  // eight lanes per candidate, four candidates per warp step
  float qf[4][16];
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
  const float wh = w[row * CSA2_HI + 2 * (j & 1) + ((j >> 1) & 1)];
  // Marked keys in rank (= position) order, a chunk at a time: the chunk is appended to the list
  // and rescored; while keys remain, the list is cut back to its k best (in position order), so
  // any number of marked keys (ties at the threshold) is selected exactly.  Once the k-th best key
  // reaches the row's score bound ubound[row] no later key can enter (a later tie loses on
  // position).  A row whose marked keys overflow the list and whose bound is <= 0 (all head
  // weights negative: typically thousands of exact zeros tie) takes chunks of max(2k, 1024) keys
  // and stops after the first.
  const uint32_t ub = ubound ? __ldg(ubound + row) : 0xFFFFFFFFu;
  const uint32_t lim = (total > uint32_t(kBmCap) && ub <= score_key(0.0f)) ? uint32_t(max(2 * k, 1024))
                                                                          : uint32_t(kBmCap);
  // the ranks this CTA rescores
  const uint32_t r_lo = slice < 0 ? 0u : uint32_t(uint64_t(total) * uint32_t(slice) / uint32_t(n_slices));
  const uint32_t r_hi = slice < 0 ? total : uint32_t(uint64_t(total) * uint32_t(slice + 1) / uint32_t(n_slices));
  uint32_t n = 0;
  for (uint32_t lo = r_lo; lo < r_hi;) {
    const uint32_t hi = min(r_hi, lo + min(uint32_t(kBmCap) - n, lim));
    uint32_t slot = first;
    for (int e = 0; e < per && slot < hi; ++e) {
      const int64_t wi = int64_t(t) * per + e;
      if (wi >= nw) break;
      uint32_t v = word(wi);
      const uint32_t pc = __popc(v);
      if (slot + pc <= lo) {  // the whole word lies before this chunk
        slot += pc;
        continue;
      }
      while (v && slot < hi) {
        const int bit = __ffs(v) - 1;
        if (slot >= lo) sm.cand_col[n + slot - lo] = int32_t(wi * 32 + bit);
        ++slot;
        v &= v - 1u;
      }
    }
    __syncthreads();
    const uint32_t n_end = n + (hi - lo);
    // the next step's key rows load while this step's are scored
    constexpr uint32_t kStep = 4 * (kBmThreads / 32);
    auto load_key = [&](uint32_t c, uint4& k0, uint4& k1) {
      k0 = make_uint4(0, 0, 0, 0);
      k1 = k0;
      if (c < n_end) {
        const uint4* kp = reinterpret_cast<const uint4*>(kseq + int64_t(sm.cand_col[c]) * CSA2_DI + 16 * j);
        k0 = __ldg(kp);
        k1 = __ldg(kp + 1);
      }
    };
    uint4 k0, k1;
    load_key(n + uint32_t(warp) * 4 + sub, k0, k1);
    for (uint32_t c0 = n + uint32_t(warp) * 4; c0 < n_end; c0 += kStep) {
      const uint32_t c = c0 + sub;
      uint4 n0, n1;
      load_key(c + kStep, n0, n1);
      const float sc = canon_score_lane8(qf, wh, k0, k1, j);
      if (j == 0 && c < n_end) sm.cand_key[c] = score_key(sc);
      k0 = n0;
      k1 = n1;
    }
    __syncthreads();
    n = n_end;
    lo = hi;
    if (lo < r_hi) {
      const uint32_t tau = keep_top(sm, int(n), k);
      n = uint32_t(k);
      if (tau >= ub) break;
    }
  }
  if (slice >= 0) {
    // this slice's k best into the workspace; the last slice of the row merges them in order
    if (n > uint32_t(k)) {
      keep_top(sm, int(n), k);
      n = uint32_t(k);
    }
    const int64_t sbase = (int64_t(pos) * n_slices + slice) * k;
    for (uint32_t i = t; i < n; i += kBmThreads) {
      sl_key[sbase + i] = sm.cand_key[i];
      sl_col[sbase + i] = sm.cand_col[i];
    }
    if (t == 0) sl_cnt[pos * n_slices + slice] = n;
    __threadfence();
    __syncthreads();
    if (t == 0) sm.is_last = atomicAdd(tickets + pos, 1u) == unsigned(n_slices - 1) ? 1u : 0u;
    __syncthreads();
    if (!sm.is_last) return;
    __threadfence();
    n = 0;
    for (int s2 = 0; s2 < n_slices; ++s2) {
      const uint32_t c = __ldcg(sl_cnt + pos * n_slices + s2);
      if (n + c > uint32_t(kBmCap)) {  // then n > kBmCap - k >= k
        keep_top(sm, int(n), k);
        n = uint32_t(k);
      }
      const int64_t b2 = (int64_t(pos) * n_slices + s2) * k;
      for (uint32_t i = t; i < c; i += kBmThreads) {
        sm.cand_key[n + i] = __ldcg(sl_key + b2 + i);
        sm.cand_col[n + i] = __ldcg(sl_col + b2 + i);
      }
      __syncthreads();
      n += c;
    }
    if (t == 0) tickets[pos] = 0u;  // ready for the next launch
  }
  if (n < uint32_t(k)) {  // not reached: at least k groups hold a key at or above the threshold
    for (uint32_t i = t; i < n; i += kBmThreads) o.emit(int(i), sm.cand_col[i]);
    finish_row(o, n, int(row), n_sel, nullptr);
    return;
  }
  select_listed(sm, int(n), k, o);
  finish_row(o, k, int(row), n_sel, nullptr);
}

}  // namespace

size_t topk_counters_offset(int rows) { return size_t(rows) * kCandCap * (sizeof(uint32_t) + sizeof(int32_t)); }
// (count, ticket) per row, padded to a multiple of four words so that the histograms after them
// start on a 16-byte boundary
inline size_t topk_ctl_words(int rows) { return (size_t(rows) * 2 + 3) / 4 * 4; }

// group keys per row: one per thread and sweep step
inline int64_t topk_group_ld(int64_t n) { return (n + kSweep - 1) / kSweep * kHThreads; }

// workspace (rows longer than kSmallRow): candidate keys and columns per row, then (count, ticket)
// per row, then the row histograms of group maxima (the last two zero before each launch; every
// launch leaves them zero), then the group keys (written before they are read in every launch)
size_t topk_ws_bytes(int rows, int64_t n) {
  if (n <= kSmallRow) return 0;
  return size_t(rows) * (kCandCap * (sizeof(uint32_t) + sizeof(int32_t)) + kBins * sizeof(uint32_t)) +
         topk_ctl_words(rows) * sizeof(uint32_t) + size_t(rows) * size_t(topk_group_ld(n)) * sizeof(uint32_t);
}

// One cluster of C CTAs per row (rows of kSmallRow + 1 to kClMaxCols columns).
template <int C>
cudaError_t launch_topk_cluster(const float* scores, int rows, int64_t n, int64_t ld, const int32_t* n_valid, int k,
                                const int32_t* map, int64_t map_ld, int32_t* idx, int32_t* n_sel, int expand8,
                                int32_t* pool_len, cudaStream_t st) {
  const size_t smem = sizeof(ClSmem);
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(C), unsigned(rows), 1u);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = unsigned(C);
  attr[1].val.clusterDim.y = 1u;
  attr[1].val.clusterDim.z = 1u;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, topk_cluster_kernel<C>, scores, n, ld, n_valid, k, map, map_ld, idx, n_sel, expand8,
                            pool_len);
}

cudaError_t launch_topk(const float* scores, int rows, int64_t n, int64_t ld, const int32_t* n_valid,
                        int k, const int32_t* map, int64_t map_ld, int32_t* idx, int32_t* n_sel,
                        int expand8, int32_t* pool_len, void* ws, cudaStream_t st, bool counters_zeroed) {
  if (rows == 0) return cudaSuccess;
  const size_t smem = sizeof(SelSmem);
  static std::atomic<bool> attr_set[64];  // per device; set once, by any host thread
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  if (topk_ws_bytes(rows, n) == 0)  // one CTA per row over the whole row
    return launch_pdl(topk_kernel, dim3(1u, unsigned(rows), 1u), dim3(kThreads), smem, st, scores, n, ld, n_valid, k,
                      map, map_ld, idx, n_sel, expand8, pool_len);
  if (n <= kClMaxCols) {
    // one cluster per row: eight CTAs when every row's cluster fits in one wave of two CTAs per SM
    // and each CTA keeps at least 8192 columns; two for rows of at most two sweeps; else four
    if (int64_t(rows) * 8 <= 2 * int64_t(sm_count()) && n >= 8 * 8192)
      return launch_topk_cluster<8>(scores, rows, n, ld, n_valid, k, map, map_ld, idx, n_sel, expand8, pool_len, st);
    if (n <= 2 * kClSweep)
      return launch_topk_cluster<2>(scores, rows, n, ld, n_valid, k, map, map_ld, idx, n_sel, expand8, pool_len, st);
    return launch_topk_cluster<4>(scores, rows, n, ld, n_valid, k, map, map_ld, idx, n_sel, expand8, pool_len, st);
  }
  if (!ws) return cudaErrorInvalidValue;
  uint32_t* ckey = static_cast<uint32_t*>(ws);
  int32_t* ccol = reinterpret_cast<int32_t*>(ckey + size_t(rows) * kCandCap);
  uint32_t* ctl = reinterpret_cast<uint32_t*>(ccol + size_t(rows) * kCandCap);
  uint32_t* hist = ctl + topk_ctl_words(rows);
  uint32_t* gkey = hist + size_t(rows) * kBins;
  const int64_t gld = topk_group_ld(n);
  if (!counters_zeroed) {
    cudaError_t e = cudaMemsetAsync(ctl, 0, (topk_ctl_words(rows) + size_t(rows) * kBins) * sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
  }
  static std::atomic<bool> sel_attr[64];
  if (dev < 64 && !sel_attr[dev]) {
    cudaError_t e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    sel_attr[dev] = true;
  }
  // slices: about four CTAs of 256 threads per SM over all rows, whole sweep steps of kSweep keys
  const int64_t want = std::max<int64_t>(1, (4 * 152 + rows - 1) / rows);
  const int64_t sweeps = (n + kSweep - 1) / kSweep;
  const int64_t slice_len = (sweeps + want - 1) / want * kSweep;
  const int64_t nsl = (n + slice_len - 1) / slice_len;
  const dim3 grid{unsigned(nsl), unsigned(rows), 1u};
  cudaError_t e = launch_pdl(topk_hist_kernel, grid, dim3(kHThreads), 0, st, scores, n, ld, n_valid, k, slice_len, hist,
                             gkey, gld);
  if (e != cudaSuccess) return e;
  e = launch_pdl(topk_filter_kernel, grid, dim3(kHThreads), 0, st, scores, n, ld, n_valid, k, slice_len,
                 static_cast<const uint32_t*>(hist), static_cast<const uint32_t*>(gkey), gld, ckey, ccol, ctl);
  if (e != cudaSuccess) return e;
  return launch_pdl(topk_select_kernel, dim3(unsigned(rows)), dim3(kThreads), smem, st, scores, n, ld, n_valid, k, map,
                    map_ld, idx, n_sel, expand8, pool_len, hist, static_cast<const uint32_t*>(ckey),
                    static_cast<const int32_t*>(ccol), ctl);
}

cudaError_t launch_bitmap_select(const uint16_t* qI, const float* w, int B, int Nq, const uint16_t* KI,
                                 int64_t cap, const int32_t* lens, int ratio, const int32_t* q_pos, int k,
                                 const uint32_t* bitmap, int64_t n_words, const uint32_t* ubound,
                                 const int32_t* order, const BmSlices& sl, int32_t* idx, int32_t* n_sel,
                                 cudaStream_t st) {
  const int64_t rows = int64_t(B) * Nq;
  if (rows == 0) return cudaSuccess;
  const int n_sliced = order ? sl.n_rows : 0;
  if (n_sliced < 0 || n_sliced > rows || (n_sliced > 0 && (sl.n_slices < 1 || !sl.key || !sl.col || !sl.cnt ||
                                                          !sl.tickets)))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(BmSmem);
  static std::atomic<bool> attr_set[64];  // per device; set once, by any host thread
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(bitmap_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int64_t grid = rows + int64_t(n_sliced) * (sl.n_slices - 1);
  return launch_pdl(bitmap_select_kernel, dim3(unsigned(grid)), dim3(kBmThreads), smem, st, qI, w, Nq, KI, cap,
                    lens, ratio, q_pos, k, bitmap, n_words, ubound, order, n_sliced, sl.n_slices, sl.key, sl.col,
                    sl.cnt, sl.tickets, idx, n_sel);
}

int bitmap_list_cap() { return kBmCap; }

}  // namespace csa2

extern "C" csa2_status csa2_topk(const float* scores, int rows, int64_t n, int64_t ld,
                                 const int32_t* n_valid, int k, const int32_t* map, int64_t map_ld,
                                 int32_t* idx, int32_t* n_sel, void* ws, size_t ws_bytes,
                                 csa2_stream_t stream) {
  if (rows < 0 || n < 0 || ld < n || k < 1 || k > CSA2_MAX_K || n >= (int64_t(1) << 31))
    return CSA2_ERR_INVALID_ARG;
  if (rows == 0) return CSA2_OK;
  if (rows > 65535) return CSA2_ERR_UNSUPPORTED;
  if (!scores || !idx || (map && map_ld < n)) return CSA2_ERR_INVALID_ARG;
  const size_t need = csa2::topk_ws_bytes(rows, n);
  if (need && (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 15u))) return CSA2_ERR_WORKSPACE;
  return csa2::launch_topk(scores, rows, n, ld, n_valid, k, map, map_ld, idx, n_sel, 0, nullptr, ws,
                           reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? CSA2_OK
             : CSA2_ERR_CUDA;
}

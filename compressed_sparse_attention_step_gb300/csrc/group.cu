// CSA2 layer-group driver, hierarchical pool entry point, workspace sizing and status helpers.
//
// A group runs its layers in order (ai-maestro.online "DeepSeek AI released
// DeepSeek-V4.1-Flash with 1M context, FP4", section "Compressed Sparse Attention 2"):
//   Full     [append new rows] -> [block scores -> Top-keep blocks -> pool] -> scores -> Top-K
//   Reindex  scores (pool or all visible entries) with its own indexer Q -> Top-K
//   Reuse    nothing: the latest indices are used as they are
// and every layer then runs split-KV sparse attention with its own Q and window.  Scores live in
// the caller's workspace; the selection kernels read them while they are still in L2.
#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace csa2 {

__device__ unsigned int g_device_flags = 0;

unsigned int* device_flags_ptr() {
  static unsigned int* ptrs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  if (dev >= 64) return nullptr;
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_flags) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned int*>(p);
  }
  return ptrs[dev];
}

DeviceStreams* device_streams() {
  static DeviceStreams res[64];
  static std::mutex init_mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return nullptr;
  DeviceStreams& r = res[dev];
  std::lock_guard<std::mutex> guard(init_mu);
  if (!r.ready) {
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return nullptr;
    if (cudaStreamCreateWithPriority(&r.aux, cudaStreamNonBlocking, greatest) != cudaSuccess) return nullptr;
    for (auto& e : r.fork)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&r.join, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    if (cudaStreamCreateWithPriority(&r.aux2, cudaStreamNonBlocking, greatest) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&r.pool_ready, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&r.sel_done, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    r.ready = true;
  }
  return &r;
}

namespace {

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Prefill chunks of at least 64 queries per sequence select on the tensor cores without
// materialising scores (flat selection only; TMA row coordinates are 32-bit, and a row's group
// maxima must fit in shared memory).
constexpr int kPrefillMinQueries = 64;
inline bool prefill_path(int B, int Nq, int hierarchical, int64_t cap) {
  return Nq >= kPrefillMinQueries && !hierarchical && B <= 65535 && int64_t(B) * cap < (int64_t(1) << 31) &&
         (cap + 31) / 32 <= prefill_max_groups();
}

// Attention workspace of a group step.  One launch serves a run of L' layers that share their
// selected rows, L' * rows instances at a split.  Tickets: for rows * max(ns, CSA2_MAX_LAYERS)
// instances (ns: one layer's split).  Partials: with the automatic split, enough for a run of any
// length L' <= CSA2_MAX_LAYERS at its own automatic split (about max(152, L' rows) instance-splits,
// a few MB); with a forced split, for one layer's rows at that split (a longer run takes the
// largest split that fits).
size_t group_attn_ticket_bytes(int64_t rows, int K, int W, int n_split) {
  const int ns = attn_effective_split(K, W, n_split ? n_split : attn_auto_split(rows, K, W));
  return attn_ticket_bytes(rows * std::max(ns, CSA2_MAX_LAYERS));
}
size_t group_attn_ws_bytes(int64_t rows, int K, int W, int n_split) {
  auto partials = [&](int64_t inst, int ns) { return ns <= 1 ? size_t(0) : attn_ws_bytes(inst, ns) - attn_ticket_bytes(inst); };
  size_t part = 0;
  if (n_split) {
    part = partials(rows, attn_effective_split(K, W, n_split));
  } else {
    for (int l = 1; l <= CSA2_MAX_LAYERS; ++l)
      part = std::max(part, partials(l * rows, attn_effective_split(K, W, attn_auto_split(l * rows, K, W))));
  }
  return group_attn_ticket_bytes(rows, K, W, n_split) + part;
}

struct GroupWs {
  size_t scores_off, nv_off, topk_off, attn_off, pf_off, topk2_off, nv2_off, total;
  int64_t score_ld;
};

GroupWs group_ws_layout(int B, int Nq, int64_t cap, int K, int W, int hierarchical, int keep, int n_split) {
  GroupWs L{};
  const int64_t rows = int64_t(B) * Nq;
  const bool pf = prefill_path(B, Nq, hierarchical, cap);
  int64_t ld = pf ? 0 : cap;
  if (hierarchical) ld = std::max<int64_t>(cap / CSA2_BLOCK, int64_t(keep) * CSA2_BLOCK);
  L.score_ld = ld;
  L.scores_off = 0;
  L.nv_off = align256(size_t(rows) * size_t(ld) * sizeof(float));
  L.topk_off = L.nv_off + align256(size_t(rows) * sizeof(int32_t));
  L.attn_off = L.topk_off + align256(topk_ws_bytes(int(rows), ld));
  L.pf_off = L.attn_off + align256(group_attn_ws_bytes(rows, K, W, n_split));
  L.total = L.pf_off + (pf ? align256(prefill_ws_bytes(rows, cap, B)) : 0);
  // hierarchical: the Top-K workspace and valid counts of a Reindex selection that runs beside the
  // Full layer's (its pool scores take the second pool-sized region of the score buffer)
  L.topk2_off = L.nv2_off = L.total;
  if (hierarchical) {
    const int64_t pool_w = int64_t(keep) * CSA2_BLOCK;
    L.topk2_off = L.total;
    L.nv2_off = L.topk2_off + align256(topk_ws_bytes(int(rows), pool_w));
    L.total = L.nv2_off + align256(size_t(rows) * sizeof(int32_t));
  }
  return L;
}

}  // namespace
}  // namespace csa2

using csa2::al16;

extern "C" size_t csa2_workspace_size(int op, const csa2_dims* d) {
  if (!d) return 0;
  const int64_t rows = int64_t(d->B) * d->Nq;
  switch (op) {
    case CSA2_OP_TOPK:
      return csa2::topk_ws_bytes(int(rows), d->n);
    case CSA2_OP_BLOCK_POOL: {
      const int64_t nb = std::max<int64_t>(d->cap / CSA2_BLOCK, 1);
      return csa2::align256(size_t(rows) * size_t(nb) * sizeof(float)) + csa2::topk_ws_bytes(int(rows), nb);
    }
    case CSA2_OP_SPARSE_ATTN: {
      const int W = d->W;
      const int ns = csa2::attn_effective_split(d->k, W, d->n_split ? d->n_split : csa2::attn_auto_split(rows, d->k, W));
      return csa2::attn_ws_bytes(rows, ns);
    }
    case CSA2_OP_INDEX_SELECT_PREFILL:
      return csa2::prefill_ws_bytes(rows, d->cap, d->B);
    case CSA2_OP_MERGE_PAIRS:
      return (d->n >= 1 && d->n <= 64 && d->k >= 1 && d->k <= CSA2_MAX_K)
                 ? csa2::merge_pairs_ws_bytes(int(rows), int(d->n), d->k)
                 : 0;
    case CSA2_OP_GROUP_STEP:
      return csa2::group_ws_layout(d->B, d->Nq, d->cap, d->k, d->W, d->hierarchical, d->n_blocks_keep,
                                   d->n_split)
          .total;
    default:
      return 0;
  }
}

extern "C" int csa2_attn_auto_split(int64_t instances, int k, int W) {
  return csa2::attn_auto_split(instances, k, W);
}

extern "C" const char* csa2_status_string(csa2_status s) {
  switch (s) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_INVALID_ARG: return "invalid argument";
    case CSA2_ERR_UNSUPPORTED: return "unsupported dimension";
    case CSA2_ERR_CUDA: return "CUDA error";
    case CSA2_ERR_WORKSPACE: return "workspace missing or too small";
    case CSA2_ERR_TOO_LARGE: return "problem exceeds the library's built-in scratch";
  }
  return "unknown status";
}

extern "C" csa2_status csa2_device_flags(uint32_t* flags, int clear, csa2_stream_t stream) {
  if (!flags) return CSA2_ERR_INVALID_ARG;
  unsigned int* dptr = csa2::device_flags_ptr();
  if (!dptr) return CSA2_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return CSA2_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, dptr, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return CSA2_ERR_CUDA;
  *flags = v;
  if (clear && cudaMemset(dptr, 0, sizeof(unsigned int)) != cudaSuccess) return CSA2_ERR_CUDA;
  if (clear && cudaDeviceSynchronize() != cudaSuccess) return CSA2_ERR_CUDA;
  return CSA2_OK;
}

extern "C" csa2_status csa2_block_pool(const uint16_t* qI, const float* w, int B, int Nq,
                                       const uint16_t* block_keys, int64_t cap, const int32_t* lens,
                                       int ratio, const int32_t* q_pos, int keep, int32_t* pool,
                                       int32_t* pool_len, void* ws, size_t ws_bytes,
                                       csa2_stream_t stream) {
  if (B < 0 || Nq < 0 || cap < 0 || ratio < 1 || keep < 1 || keep > CSA2_MAX_K) return CSA2_ERR_INVALID_ARG;
  const int64_t rows = int64_t(B) * Nq;
  if (rows == 0) return CSA2_OK;
  if (rows > 65535) return CSA2_ERR_UNSUPPORTED;
  if (!qI || !w || !block_keys || !lens || !pool || !pool_len || !al16(qI) || !al16(block_keys))
    return CSA2_ERR_INVALID_ARG;
  const int64_t nb = cap / CSA2_BLOCK;
  csa2_dims d{};
  d.B = B;
  d.Nq = Nq;
  d.cap = cap;
  const size_t need = csa2_workspace_size(CSA2_OP_BLOCK_POOL, &d);
  if (!ws || ws_bytes < need || !al16(ws)) return CSA2_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  float* sc = static_cast<float*>(ws);
  if (nb == 0) {
    // no complete block can exist: empty pools
    if (cudaMemsetAsync(pool_len, 0, size_t(rows) * sizeof(int32_t), st) != cudaSuccess) return CSA2_ERR_CUDA;
    if (cudaMemsetAsync(pool, 0xFF, size_t(rows) * keep * CSA2_BLOCK * sizeof(int32_t), st) != cudaSuccess)
      return CSA2_ERR_CUDA;
    return CSA2_OK;
  }
  // the visible block count of each row is returned through pool_len, then consumed
  if (csa2::launch_index_score(qI, w, B, Nq, block_keys, nb, lens, cap, CSA2_BLOCK, nullptr, nullptr, 0,
                               ratio, q_pos, sc, nb, pool_len, st) != cudaSuccess)
    return CSA2_ERR_CUDA;
  void* tws = static_cast<char*>(ws) + csa2::align256(size_t(rows) * size_t(nb) * sizeof(float));
  if (csa2::launch_topk(sc, int(rows), nb, nb, pool_len, keep, nullptr, 0, pool, nullptr, 1, pool_len, tws, st) !=
      cudaSuccess)
    return CSA2_ERR_CUDA;
  return CSA2_OK;
}

extern "C" size_t csa2_group_desc_size(void) { return sizeof(csa2_group_desc); }

namespace {
// The argument checks of a group step, made before anything is launched.  *empty: the step has no
// queries (nothing to launch; the remaining checks are skipped).
csa2_status group_check(const csa2_group_desc* g, const void* ws, size_t ws_bytes, bool* empty) {
  *empty = false;
  if (!g) return CSA2_ERR_INVALID_ARG;
  const int L = g->n_layers;
  if (L < 1 || L > CSA2_MAX_LAYERS) return CSA2_ERR_INVALID_ARG;
  if (g->B < 0 || g->Nq < 0 || g->cap < 0 || g->ratio < 1) return CSA2_ERR_INVALID_ARG;
  if (g->K < 1 || g->K > CSA2_MAX_ATTN_K || g->W < 0 || g->W > CSA2_MAX_W) return CSA2_ERR_INVALID_ARG;
  if (g->n_split < 0 || g->n_split > 32 || g->n_new < 0) return CSA2_ERR_INVALID_ARG;
  if (g->hierarchical && (g->n_blocks_keep < 1 || g->n_blocks_keep > CSA2_MAX_K)) return CSA2_ERR_INVALID_ARG;
  const int64_t rows = int64_t(g->B) * g->Nq;
  if (rows == 0) {
    *empty = true;
    return CSA2_OK;
  }
  if (rows > 65535) return CSA2_ERR_UNSUPPORTED;
  if (g->modes[0] != CSA2_MODE_FULL && g->modes[0] != CSA2_MODE_REINDEX) return CSA2_ERR_INVALID_ARG;
  if (!g->lens || !g->codes || !g->scales || !g->KI || !al16(g->codes) || !al16(g->scales) || !al16(g->KI))
    return CSA2_ERR_INVALID_ARG;
  if (g->hierarchical && (!g->block_keys || !g->pool || !g->pool_len || !al16(g->block_keys)))
    return CSA2_ERR_INVALID_ARG;
  if (g->W > 0 && !g->swa_len) return CSA2_ERR_INVALID_ARG;
  if (g->swa_format != CSA2_SWA_BF16 && g->swa_format != CSA2_SWA_E4M3) return CSA2_ERR_INVALID_ARG;
  bool any_full = false;
  for (int l = 0; l < L; ++l) {
    const int m = g->modes[l];
    if (m != CSA2_MODE_FULL && m != CSA2_MODE_REINDEX && m != CSA2_MODE_REUSE) return CSA2_ERR_INVALID_ARG;
    if (!g->q[l] || !g->out[l] || !al16(g->q[l]) || !al16(g->out[l])) return CSA2_ERR_INVALID_ARG;
    if (g->W > 0 && (!g->swa[l] || !al16(g->swa[l]))) return CSA2_ERR_INVALID_ARG;
    if (m != CSA2_MODE_REUSE) {
      if (!g->qI[l] || !g->w[l] || !g->idx[l] || !al16(g->qI[l])) return CSA2_ERR_INVALID_ARG;
      if (csa2::prefill_path(g->B, g->Nq, g->hierarchical, g->cap) && (!al16(g->w[l]) || !al16(g->idx[l])))
        return CSA2_ERR_INVALID_ARG;
      any_full |= (m == CSA2_MODE_FULL);
    }
  }
  if (g->n_new > 0 && (g->kv_new || g->ki_new)) {
    if (g->modes[0] != CSA2_MODE_FULL) return CSA2_ERR_INVALID_ARG;
    if ((g->kv_new && !al16(g->kv_new)) || (g->ki_new && !al16(g->ki_new))) return CSA2_ERR_INVALID_ARG;
  }
  (void)any_full;
  const csa2::GroupWs lay = csa2::group_ws_layout(g->B, g->Nq, g->cap, g->K, g->W, g->hierarchical,
                                                  g->n_blocks_keep, g->n_split);
  if (!ws || ws_bytes < lay.total || !al16(ws)) return CSA2_ERR_WORKSPACE;
  return CSA2_OK;
}
}  // namespace

extern "C" csa2_status csa2_group_step(const csa2_group_desc* g, void* ws, size_t ws_bytes,
                                       csa2_stream_t stream) {
  bool empty = false;
  const csa2_status chk = group_check(g, ws, ws_bytes, &empty);
  if (chk != CSA2_OK || empty) return chk;
  const int L = g->n_layers;
  const int64_t rows = int64_t(g->B) * g->Nq;
  const csa2::GroupWs lay = csa2::group_ws_layout(g->B, g->Nq, g->cap, g->K, g->W, g->hierarchical,
                                                  g->n_blocks_keep, g->n_split);

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* wsb = static_cast<char*>(ws);
  float* scores = reinterpret_cast<float*>(wsb + lay.scores_off);
  int32_t* nv = reinterpret_cast<int32_t*>(wsb + lay.nv_off);
  void* tws = wsb + lay.topk_off;
  float* attn_ws = reinterpret_cast<float*>(wsb + lay.attn_off);
  void* pf_ws = wsb + lay.pf_off;
  const bool pf = csa2::prefill_path(g->B, g->Nq, g->hierarchical, g->cap);
  const int64_t nb = g->cap / CSA2_BLOCK;
  const int64_t pool_w = int64_t(g->n_blocks_keep) * CSA2_BLOCK;
  const int64_t sld = lay.score_ld;
  const int Nq = g->Nq, K = g->K, SW = g->W - 1 + g->Nq;
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  auto rec = [&](csa2_event_t e, cudaStream_t s2) {
    return !e || cudaEventRecord(reinterpret_cast<cudaEvent_t>(e), s2) == cudaSuccess;
  };

  // Sequence chunks: the first indexer scan of chunk c runs on `stream` while the rest of chunk c-1
  // (selection, pool work, attention of every layer) runs on the side stream.
  int n_chunks = g->seq_chunks > 0 ? g->seq_chunks : 1;
  n_chunks = std::max(1, std::min({n_chunks, g->B, csa2::kMaxSeqChunks}));
  // A hierarchical group in one chunk whose Full layer 0 is followed by a Reindex layer l_rx: once
  // the pool is selected, l_rx's pool scan and selection run on a second side stream beside the
  // Full layer's pool scan, selection and attention (they share only the pool)
  int l_rx = -1;
  if (g->hierarchical && n_chunks == 1 && g->modes[0] == CSA2_MODE_FULL && nb > 0 && 2 * pool_w <= sld)
    for (int l = 1; l < g->n_layers; ++l)
      if (g->modes[l] != CSA2_MODE_REUSE) {
        if (g->modes[l] == CSA2_MODE_REINDEX) l_rx = l;
        break;
      }
  csa2::DeviceStreams* ds = nullptr;
  if (n_chunks > 1 || l_rx > 0) {
    ds = csa2::device_streams();
    if (!ds) return CSA2_ERR_CUDA;
  }
  std::unique_lock<std::mutex> lock;
  if (ds) lock = std::unique_lock<std::mutex>(ds->mu);
  cudaStream_t aux = ds && n_chunks > 1 ? ds->aux : st;

  // Top-K counters and attention tickets sit back to back in the workspace; every launch leaves them
  // zero, so clearing them once per step serves all layers of an unchunked step (by the append's
  // launch when the step has one)
  const bool zeroed = n_chunks == 1;
  const size_t zero_lo = csa2::topk_ws_bytes(int(rows), lay.score_ld) > 0
                             ? lay.topk_off + csa2::topk_counters_offset(int(rows))
                             : lay.attn_off;
  const size_t zero_hi = lay.attn_off + csa2::group_attn_ticket_bytes(rows, K, g->W, g->n_split);
  bool zero_done = false;

  // ---- append (Full layer of a decode step), before any scoring --------------------------------
  if (g->n_new > 0) {
    if (g->kv_new && g->ki_new) {
      // (the hierarchical step's completed block keys in the same launch)
      if (!ok(csa2::launch_append(g->kv_new, g->ki_new, g->B, g->n_new, g->codes, g->scales, g->KI, g->cap, g->lens,
                                  zeroed ? wsb + zero_lo : nullptr, zeroed ? zero_hi - zero_lo : 0,
                                  g->hierarchical ? g->block_keys : nullptr, st)))
        return CSA2_ERR_CUDA;
      zero_done = zeroed;
    } else if (g->kv_new &&
               !ok(csa2::launch_fp4_quantize(g->kv_new, g->B, g->n_new, g->codes, g->scales, g->cap, g->lens,
                                             -g->n_new, st))) {
      return CSA2_ERR_CUDA;
    }
    if (g->ki_new) {
      if (!g->kv_new &&
          !ok(csa2::launch_copy_rows_append(g->ki_new, g->B, g->n_new, CSA2_DI, g->KI, g->cap, g->lens, st)))
        return CSA2_ERR_CUDA;
      if (g->hierarchical && !g->kv_new &&
          !ok(csa2::launch_block_keys(g->KI, g->B, g->cap, g->lens, g->block_keys, 1, g->n_new, st)))
        return CSA2_ERR_CUDA;
    }
  }
  if (zeroed && !zero_done && !ok(csa2::launch_zero(wsb + zero_lo, zero_hi - zero_lo, st))) return CSA2_ERR_CUDA;
  if (!rec(g->ev_score_begin, st)) return CSA2_ERR_CUDA;
  bool attn_timed = false;  // the attention event pair brackets the step's first attention launch

  for (int c = 0; c < n_chunks; ++c) {
    const int b0 = int(int64_t(g->B) * c / n_chunks), b1 = int(int64_t(g->B) * (c + 1) / n_chunks);
    const int Bc = b1 - b0;
    const int64_t r0 = int64_t(b0) * Nq, rc = int64_t(Bc) * Nq;
    // chunk views
    const int32_t* lens = g->lens + b0;
    const int32_t* qpos = g->q_pos ? g->q_pos + r0 : nullptr;
    uint8_t* codes = g->codes + int64_t(b0) * g->cap * CSA2_CODE_BYTES;
    uint8_t* scl = g->scales + int64_t(b0) * g->cap * CSA2_SCALE_BYTES;
    const uint16_t* KI = g->KI + int64_t(b0) * g->cap * CSA2_DI;
    const uint16_t* bkeys = g->block_keys ? g->block_keys + int64_t(b0) * nb * CSA2_DI : nullptr;
    int32_t* pool = g->pool ? g->pool + r0 * pool_w : nullptr;
    int32_t* pool_len = g->pool_len ? g->pool_len + r0 : nullptr;
    float* sc = scores + r0 * sld;
    int32_t* nvc = nv + r0;
    const int32_t* swl = g->swa_len ? g->swa_len + b0 : nullptr;
    auto qI_of = [&](int l) { return g->qI[l] + r0 * (CSA2_HI * CSA2_DI); };
    auto w_of = [&](int l) { return g->w[l] + r0 * CSA2_HI; };
    auto idx_of = [&](int l) { return g->idx[l] + r0 * K; };
    // One attention launch for all the chunk's layers, each with its own selected rows (a Full or
    // Reindex layer's, which the Reuse layers after it share), after the last selection.  Its split:
    // the forced one, else the automatic one for all its queries (at most 4 when chunks overlap),
    // within the sized workspace.
    const size_t attn_cap = csa2::group_attn_ws_bytes(rows, K, g->W, g->n_split);
    csa2::AttnLayers run{};
    int run_n = 0;
    const int32_t* run_idx = nullptr;
    auto flush_run = [&]() -> bool {
      if (run_n == 0) return true;
      const bool timed = !attn_timed;
      attn_timed = true;
      if (timed && !rec(g->ev_attn_begin, aux)) return false;
      const int64_t inst = int64_t(run_n) * rc;
      int ns = csa2::attn_effective_split(
          K, g->W, g->n_split ? g->n_split : std::min(csa2::attn_auto_split(inst, K, g->W), n_chunks > 1 ? 4 : 32));
      while (ns > 1 && csa2::attn_ws_bytes(inst, ns) > attn_cap) --ns;
      const bool r = ok(csa2::launch_sparse_attn_layers(run, run_n, Bc, Nq, codes, scl, g->cap, run_idx, nullptr, K,
                                                         swl, g->W, g->softmax_scale, ns, attn_ws, aux, zeroed,
                                                         g->swa_format == CSA2_SWA_E4M3,
                                                         g->n_split == 0));
      if (timed && !rec(g->ev_attn_end, aux)) return false;
      run_n = 0;
      return r;
    };

    // stage 1 (stream): the first scan over this chunk's keys (layer 0 is Full or Reindex); prefill
    // chunks select on the tensor cores in stage 2 instead
    if (pf) {
    } else if (g->hierarchical && g->modes[0] == CSA2_MODE_FULL) {
      if (nb > 0 &&
          !ok(csa2::launch_index_score(qI_of(0), w_of(0), Bc, Nq, bkeys, nb, lens, g->cap, CSA2_BLOCK, nullptr,
                                       nullptr, 0, g->ratio, qpos, sc, nb, pool_len, st)))
        return CSA2_ERR_CUDA;
    } else if (!g->hierarchical) {
      if (!ok(csa2::launch_index_score(qI_of(0), w_of(0), Bc, Nq, KI, g->cap, lens, g->cap, 1, nullptr, nullptr, 0,
                                       g->ratio, qpos, sc, g->cap, nvc, st)))
        return CSA2_ERR_CUDA;
    }
    if (c == n_chunks - 1 && !rec(g->ev_score_end, st)) return CSA2_ERR_CUDA;
    if (ds && (!ok(cudaEventRecord(ds->fork[c], st)) || !ok(cudaStreamWaitEvent(aux, ds->fork[c], 0))))
      return CSA2_ERR_CUDA;

    // stage 2 (side stream): everything else of this chunk, layer by layer
    const int32_t* latest = nullptr;
    for (int l = 0; l < L; ++l) {
      const int mode = g->modes[l];
      if (mode != CSA2_MODE_REUSE) {
        if (l == l_rx) {
          // its selection ran on the second side stream
          if (!ok(cudaStreamWaitEvent(aux, ds->sel_done, 0))) return CSA2_ERR_CUDA;
        } else if (g->hierarchical) {
          if (mode == CSA2_MODE_FULL) {
            if (nb > 0 && l != 0 &&
                !ok(csa2::launch_index_score(qI_of(l), w_of(l), Bc, Nq, bkeys, nb, lens, g->cap, CSA2_BLOCK, nullptr,
                                             nullptr, 0, g->ratio, qpos, sc, nb, pool_len, aux)))
              return CSA2_ERR_CUDA;
            if (nb > 0) {
              if (!ok(csa2::launch_topk(sc, int(rc), nb, nb, pool_len, g->n_blocks_keep, nullptr, 0, pool, nullptr, 1,
                                        pool_len, tws, aux, zeroed)))
                return CSA2_ERR_CUDA;
              if (l == 0 && l_rx > 0) {
                // the Reindex layer's pool scores in the score buffer's second pool-sized region, its
                // own Top-K workspace and valid counts, on the second side stream
                float* sc2 = sc + rc * pool_w;
                int32_t* nv2 = reinterpret_cast<int32_t*>(wsb + lay.nv2_off) + r0;
                if (!ok(cudaEventRecord(ds->pool_ready, aux)) || !ok(cudaStreamWaitEvent(ds->aux2, ds->pool_ready, 0)) ||
                    !ok(csa2::launch_index_score(qI_of(l_rx), w_of(l_rx), Bc, Nq, KI, g->cap, lens, g->cap, 1, pool,
                                                 pool_len, pool_w, g->ratio, qpos, sc2, pool_w, nv2, ds->aux2)) ||
                    !ok(csa2::launch_topk(sc2, int(rc), pool_w, pool_w, nv2, K, pool, pool_w, idx_of(l_rx), nullptr, 0,
                                          nullptr, wsb + lay.topk2_off, ds->aux2, false)) ||
                    !ok(cudaEventRecord(ds->sel_done, ds->aux2)))
                  return CSA2_ERR_CUDA;
              }
            } else if (!ok(cudaMemsetAsync(pool_len, 0, size_t(rc) * sizeof(int32_t), aux))) {
              return CSA2_ERR_CUDA;
            }
          }
          if (!ok(csa2::launch_index_score(qI_of(l), w_of(l), Bc, Nq, KI, g->cap, lens, g->cap, 1, pool, pool_len,
                                           pool_w, g->ratio, qpos, sc, pool_w, nvc, aux)))
            return CSA2_ERR_CUDA;
          if (!ok(csa2::launch_topk(sc, int(rc), pool_w, pool_w, nvc, K, pool, pool_w, idx_of(l), nullptr, 0, nullptr,
                                    tws, aux, zeroed)))
            return CSA2_ERR_CUDA;
        } else if (pf) {
          if (!ok(csa2::launch_prefill_select(qI_of(l), w_of(l), Bc, Nq, KI, g->cap, lens, g->ratio, qpos, K,
                                              idx_of(l), nullptr, pf_ws, aux)))
            return CSA2_ERR_CUDA;
        } else {
          if (l != 0 &&
              !ok(csa2::launch_index_score(qI_of(l), w_of(l), Bc, Nq, KI, g->cap, lens, g->cap, 1, nullptr, nullptr, 0,
                                           g->ratio, qpos, sc, g->cap, nvc, aux)))
            return CSA2_ERR_CUDA;
          if (!ok(csa2::launch_topk(sc, int(rc), g->cap, g->cap, nvc, K, nullptr, 0, idx_of(l), nullptr, 0, nullptr,
                                    tws, aux, zeroed)))
            return CSA2_ERR_CUDA;
        }
        latest = idx_of(l);
      } else if (g->idx[l] && idx_of(l) != latest) {
        if (!ok(cudaMemcpyAsync(idx_of(l), latest, size_t(rc) * K * sizeof(int32_t), cudaMemcpyDeviceToDevice, aux)))
          return CSA2_ERR_CUDA;
      }
      run.q[run_n] = g->q[l] + r0 * (CSA2_H * CSA2_D);
      // window rows: 512 bf16 values, or 512 E4M3 bytes (the same pointer arithmetic in bytes)
      const int64_t win_off = int64_t(b0) * SW * CSA2_D;
      run.swa[run_n] = g->W <= 0 ? nullptr
                       : g->swa_format == CSA2_SWA_E4M3
                           ? reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(g->swa[l]) + win_off)
                           : g->swa[l] + win_off;
      run.out[run_n] = g->out[l] + r0 * (CSA2_H * CSA2_D);
      run.lse[run_n] = g->lse[l] ? g->lse[l] + r0 * CSA2_H : nullptr;
      run.idx[run_n] = latest;
      run_idx = latest;
      ++run_n;
    }
    if (!flush_run()) return CSA2_ERR_CUDA;
  }
  if (ds && (!ok(cudaEventRecord(ds->join, aux)) || !ok(cudaStreamWaitEvent(st, ds->join, 0))))
    return CSA2_ERR_CUDA;
  return CSA2_OK;
}

// A decoder stack's step: its layer groups in order over one cache.  Every group is checked before
// anything is launched.
extern "C" csa2_status csa2_stack_step(const csa2_group_desc* groups, int n_groups, void* ws, size_t ws_bytes,
                                       csa2_stream_t stream) {
  if (!groups || n_groups < 1) return CSA2_ERR_INVALID_ARG;
  const csa2_group_desc& g0 = groups[0];
  for (int i = 0; i < n_groups; ++i) {
    const csa2_group_desc* g = groups + i;
    bool empty = false;
    const csa2_status chk = group_check(g, ws, ws_bytes, &empty);
    if (chk != CSA2_OK) return chk;
    if (i == 0) continue;
    // one batch, one cache, one append (by the first group), one pool
    if (g->B != g0.B || g->Nq != g0.Nq || g->cap != g0.cap || g->lens != g0.lens || g->q_pos != g0.q_pos ||
        g->ratio != g0.ratio || g->codes != g0.codes || g->scales != g0.scales || g->KI != g0.KI ||
        g->hierarchical != g0.hierarchical)
      return CSA2_ERR_INVALID_ARG;
    if (g->n_new > 0 && (g->kv_new || g->ki_new)) return CSA2_ERR_INVALID_ARG;
    if (g->hierarchical && (g->block_keys != g0.block_keys || g->pool != g0.pool || g->pool_len != g0.pool_len))
      return CSA2_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n_groups; ++i) {
    const csa2_status st = csa2_group_step(groups + i, ws, ws_bytes, stream);
    if (st != CSA2_OK) return st;
  }
  return CSA2_OK;
}

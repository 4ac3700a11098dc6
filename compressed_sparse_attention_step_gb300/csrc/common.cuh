// Shared device helpers of the CSA2 library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/csa2.h"

namespace csa2 {

// Address of the current device's flag word (CSA2_FLAG_*), defined in group.cu; kernels that
// report data-dependent problems receive it as an argument.  NULL if the lookup failed.
unsigned int* device_flags_ptr();

// ---------------------------------------------------------------------------------------------
// bf16 bit helpers (values are carried as raw 16-bit patterns)
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16hi(uint32_t packed) { return __uint_as_float(packed & 0xFFFF0000u); }
__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// fp32 -> bf16 bits, round to nearest even (finite inputs).
__device__ __forceinline__ uint32_t f2bf_bits(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return u >> 16;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return f2bf_bits(lo) | (f2bf_bits(hi) << 16);
}

// Ordered 32-bit key of a score: larger key <=> larger score; -0 and +0 share one key.
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------------------------------------
// Memory helpers
// ---------------------------------------------------------------------------------------------
// Streaming 16-byte load: evict-first in L1 and L2 (data read once).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// cp.async of 16 bytes (or zero-fill when src_bytes == 0), cached in L2 only.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------------------------
// Warp-level tensor-core helpers (bf16 inputs, fp32 accumulate)
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                            uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D = A(16x16, row) * B(16x8, col) + D
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------------------------
// Block-wide exclusive scan of one uint32 per thread (blockDim.x multiple of 32, <= 1024).
// `tmp` is >= 32 words of shared memory.  Returns the exclusive prefix; *total gets the sum.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* tmp, uint32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    uint32_t s = (lane < nw) ? tmp[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    tmp[lane] = s;  // inclusive warp-sum prefix
  }
  __syncthreads();
  const uint32_t warp_base = (wid == 0) ? 0u : tmp[wid - 1];
  const uint32_t tot = tmp[nw - 1];
  __syncthreads();
  if (total) *total = tot;
  return warp_base + x - v;
}

// ---------------------------------------------------------------------------------------------
// Canonical indexer score s = sum_h w_h relu(qI_h . KI_t) in the fixed fp32 order: per head, eight
// fused-multiply-add chains over channels 16j..16j+15 from +0, then ((p0+p1)+(p2+p3))+((p4+p5)+
// (p6+p7)), relu, and (w0 r0 + w1 r1) + (w2 r2 + w3 r3) with every product and sum rounded.
// ---------------------------------------------------------------------------------------------
// Eight lanes per key: lane j = lane & 7 owns channels 16j..16j+15 (qf: its qI slice as fp32, k0/k1:
// its 32 key bytes) and head wh = w[2 (j & 1) + ((j >> 1) & 1)].  Every lane of the group of eight
// returns the same bits.  All 32 lanes of the warp must call it.
__device__ __forceinline__ float canon_score_lane8(const float (&qf)[4][16], float wh, uint4 k0, uint4 k1, int j) {
  const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
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
  const bool odd = (j & 1) != 0, second = (j & 2) != 0;
  const float s0 = odd ? P[0] : P[2], s1 = odd ? P[1] : P[3];
  const float k0v = odd ? P[2] : P[0], k1v = odd ? P[3] : P[1];
  const float A0 = __fadd_rn(k0v, __shfl_xor_sync(0xffffffffu, s0, 1));
  const float A1 = __fadd_rn(k1v, __shfl_xor_sync(0xffffffffu, s1, 1));
  const float sendB = second ? A0 : A1, keepB = second ? A1 : A0;
  const float Bv = __fadd_rn(keepB, __shfl_xor_sync(0xffffffffu, sendB, 2));
  const float dot = __fadd_rn(Bv, __shfl_xor_sync(0xffffffffu, Bv, 4));
  const float r = dot > 0.0f ? dot : 0.0f;
  const float m = __fmul_rn(wh, r);
  const float m2 = __fadd_rn(m, __shfl_xor_sync(0xffffffffu, m, 2));
  return __fadd_rn(m2, __shfl_xor_sync(0xffffffffu, m2, 1));
}

// ---------------------------------------------------------------------------------------------
// Programmatic dependent launch.  Every library kernel is launched with programmatic stream
// serialisation allowed: it may start while the kernel before it in the stream is still running,
// calls pdl_wait() before it touches anything an earlier kernel writes (or writes anything an
// earlier kernel reads), and calls pdl_trigger() only after that wait, so the next kernel can in
// turn rely on everything before this one having completed.  Without a preceding kernel both
// are no-ops.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace csa2

// Internal launchers shared across translation units (all return cudaGetLastError()).
namespace csa2 {
cudaError_t launch_fp4_quantize(const uint16_t* x, int B, int n_new, uint8_t* codes, uint8_t* scales,
                                int64_t cap, const int32_t* offsets, int offset_bias,
                                cudaStream_t st);
cudaError_t launch_copy_rows_append(const uint16_t* src, int B, int n_new, int row_elems,
                                    uint16_t* dst, int64_t cap, const int32_t* lens, cudaStream_t st);
// The decode append (new main-KV rows quantised to FP4, new indexer-K rows copied) in one launch;
// rows land at lens[b] - n_new + r.  The same launch clears zero_bytes at `zero` (nullable; both
// multiples of 16) and, when block_keys is not null, refreshes the keys of the blocks the append
// completes (as launch_block_keys with only_new).
cudaError_t launch_append(const uint16_t* kv_new, const uint16_t* ki_new, int B, int n_new, uint8_t* codes,
                          uint8_t* scales, uint16_t* KI, int64_t cap, const int32_t* lens, void* zero,
                          size_t zero_bytes, uint16_t* block_keys, cudaStream_t st);
// Clears `bytes` at p with a kernel launched like every other (a memset when p or bytes is not a
// multiple of 16).
cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t st);
cudaError_t launch_block_keys(const uint16_t* KI, int B, int64_t cap, const int32_t* lens,
                              uint16_t* block_keys, int only_new, int n_new, cudaStream_t st);
cudaError_t launch_index_score(const uint16_t* qI, const float* w, int B, int Nq, const uint16_t* KI,
                               int64_t key_stride_rows, const int32_t* lens, int64_t cap_entries,
                               int block_div, const int32_t* cand, const int32_t* cand_len,
                               int64_t n_cand, int ratio, const int32_t* q_pos, float* scores,
                               int64_t ld, int32_t* n_valid, cudaStream_t st);
// Exact Top-K of `rows` score rows.  Rows longer than one slice are spread over several CTAs and
// need workspace (topk_ws_bytes); ws may be NULL when topk_ws_bytes(...) == 0.
int sm_count();  // SMs of the current device
size_t topk_ws_bytes(int rows, int64_t n);
cudaError_t launch_topk(const float* scores, int rows, int64_t n, int64_t ld, const int32_t* n_valid,
                        int k, const int32_t* map, int64_t map_ld, int32_t* idx, int32_t* n_sel,
                        int expand8, int32_t* pool_len, void* ws, cudaStream_t st, bool counters_zeroed = false);
// Bytes from the start of a Top-K workspace for `rows` rows to its counters (which run to the end of
// topk_ws_bytes); a launch leaves them zero.
size_t topk_counters_offset(int rows);
size_t attn_ticket_bytes(int64_t instances);
// Per-layer operands of one attention launch over layers of one group: query, window buffer,
// output, lse, and the selected rows (null: the launch's shared `idx`, as for a Full or Reindex
// layer and the Reuse layers after it).
struct AttnLayers {
  const uint16_t* q[CSA2_MAX_LAYERS];
  const uint16_t* swa[CSA2_MAX_LAYERS];
  uint16_t* out[CSA2_MAX_LAYERS];
  float* lse[CSA2_MAX_LAYERS];
  const int32_t* idx[CSA2_MAX_LAYERS];
};
// n_layers layers of B*Nq queries each in one launch; the split workspace holds
// n_layers * B * Nq instances (attn_ws_bytes), tickets first.  win_fp8: the window buffers hold
// E4M3 bytes (rows of 512 B) instead of bf16.  allow_pairs: a run of layers that share their
// selected rows may take the pair path (attn_pair_path), which needs no workspace.
cudaError_t launch_sparse_attn_layers(const AttnLayers& layers, int n_layers, int B, int Nq, const uint8_t* codes,
                                      const uint8_t* scales, int64_t cap, const int32_t* idx,
                                      const int32_t* n_valid, int k, const int32_t* swa_len, int W,
                                      float softmax_scale, int n_split, float* ws, cudaStream_t st,
                                      bool tickets_zeroed, bool win_fp8, bool allow_pairs);
// The pair path of a run of n_layers layers that attend the same selected rows: two layers per CTA,
// one CTA per (query, pair), outputs written directly.  attn_pair_path: whether a run takes it.
bool attn_pair_path(int64_t per_layer, int n_layers);
cudaError_t launch_sparse_attn_pairs(const AttnLayers& layers, int n_layers, int per_layer, int Nq,
                                     const uint8_t* codes, const uint8_t* scales, int64_t cap, const int32_t* idx,
                                     const int32_t* n_valid, int k, const int32_t* swa_len, int W, float scale_log2,
                                     bool win_fp8, unsigned int* flags, cudaStream_t st);
// The warp-specialised attention kernel (attn_ws.cu), for launches of one CTA per SM: the split
// is effective, partials and tickets as in launch_sparse_attn_layers (tickets zero).
cudaError_t launch_sparse_attn_ws(const AttnLayers& layers, int n_layers, int per_layer, int Nq,
                                  const uint8_t* codes, const uint8_t* scales, int64_t cap, const int32_t* idx,
                                  const int32_t* n_valid, int k, const int32_t* swa_len, int W, float scale_log2,
                                  int n_split, float* partials, unsigned int* tickets, unsigned int* flags,
                                  bool win_fp8, cudaStream_t st);
// 8-bit window rows: n bf16 values -> E4M3 bytes (RNE, saturating to +-448).
cudaError_t launch_fp8_quantize(const uint16_t* x, int64_t n, uint8_t* out, cudaStream_t st);
cudaError_t launch_sparse_attn(const uint16_t* q, int B, int Nq, const uint8_t* codes,
                               const uint8_t* scales, int64_t cap, const int32_t* idx,
                               const int32_t* n_valid, int k, const uint16_t* swa,
                               const int32_t* swa_len, int W, float softmax_scale, uint16_t* out,
                               float* lse, int n_split, float* ws, cudaStream_t st, bool tickets_zeroed);
// Attention splits: at most one per 128-row tile; attn_ws_bytes with the effective split.
int attn_effective_split(int k, int W, int n_split);
size_t attn_ws_bytes(int64_t instances, int n_split);
// Prefill chunks: exact Top-k per query through the tensor-core filter (prefill.cu); the rescore
// and selection over the filter's bitmap (topk.cu).
size_t prefill_ws_bytes(int64_t rows, int64_t cap, int B);
int64_t prefill_max_groups();  // the longest cache (in groups of 32 entries) the filter handles
float prefill_delta_coef();
cudaError_t launch_prefill_select(const uint16_t* qI, const float* w, int B, int Nq, const uint16_t* KI,
                                  int64_t cap, const int32_t* lens, int ratio, const int32_t* q_pos, int k,
                                  int32_t* idx, int32_t* n_sel, void* ws, cudaStream_t st);
// The rows of the selection that several CTAs share: the first n_rows rows of the order take
// n_slices CTAs each; per (row, slice) up to k candidate keys and columns and their count, and one
// ticket per row (zero before the launch; the launch leaves it zero).
struct BmSlices {
  int n_rows, n_slices;
  uint32_t* key;
  int32_t* col;
  uint32_t* cnt;
  unsigned int* tickets;
};
// bitmap: [rows][n_words] marked keys; ubound: per row, the score key of an upper bound on every
// canonical score of the row (or null: no bound); order: the rows in processing order (or null:
// then no row is sliced).
cudaError_t launch_bitmap_select(const uint16_t* qI, const float* w, int B, int Nq, const uint16_t* KI,
                                 int64_t cap, const int32_t* lens, int ratio, const int32_t* q_pos, int k,
                                 const uint32_t* bitmap, int64_t n_words, const uint32_t* ubound,
                                 const int32_t* order, const BmSlices& sl, int32_t* idx, int32_t* n_sel,
                                 cudaStream_t st);
int bitmap_list_cap();  // marked keys that one list round of the selection rescores
// Context split: workspace of csa2_merge_topk_pairs for G shards' k pairs per row (shard.cu).
size_t merge_pairs_ws_bytes(int rows, int G, int k);
int attn_auto_split(int64_t instances, int k, int W);

// Library-owned side stream (highest priority) and events of the current device, created on first
// use; the group step overlaps sequence chunks with them.  `mu` serialises the enqueue of a step.
constexpr int kMaxSeqChunks = 16;
struct DeviceStreams {
  bool ready = false;
  cudaStream_t aux = nullptr;
  cudaEvent_t fork[kMaxSeqChunks] = {};
  cudaEvent_t join = nullptr;
  // a second side stream: a hierarchical group's Reindex selection beside its Full layer's
  cudaStream_t aux2 = nullptr;
  cudaEvent_t pool_ready = nullptr, sel_done = nullptr;
  std::mutex mu;
};
DeviceStreams* device_streams();
}  // namespace csa2

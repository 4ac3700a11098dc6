// Split-KV sparse attention whose scratch lives in a fixed array inside this library, for callers
// that cannot allocate device memory at the time they call: code running inside a device memory
// allocator's own callbacks (allocating there would re-enter the allocator), a service whose whole
// device memory budget is reserved up front (nothing is left to allocate from), and a plugin that is
// handed only its input and output buffers (it owns no allocator).  The computation is the same
// kernel as csa2_sparse_attn_decode; only where its split partials and per-query tickets live
// differs.  The tickets, which must start at zero, are cleared by an asynchronous memset on the
// caller's stream at the start of every call; the partials are written before they are read.
#include <mutex>

#include "attn_common.cuh"

namespace csa2 {
namespace {

// Scratch of the split partials (instances x splits x (16 x 512 + 32) floats) and one ticket per
// query.  Every GPU that loads the library reserves it until the process exits.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_attn_scratch[kStaticScratchBytes];

// Device address of g_attn_scratch for the current device (looked up once per device and kept for
// the life of the process, so a device reset or context teardown while the library is loaded is not
// supported), or NULL.
float* static_scratch() {
  static float* ptrs[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> guard(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<float*>(p);
  }
  return ptrs[dev];
}

}  // namespace
}  // namespace csa2

extern "C" size_t csa2_sparse_attn_static_scratch_bytes(void) { return csa2::kStaticScratchBytes; }

extern "C" csa2_status csa2_sparse_attn_decode_static(const uint16_t* q, int B, int Nq, const uint8_t* codes,
                                                      const uint8_t* scales, int64_t cap, const int32_t* idx,
                                                      const int32_t* n_valid, int k, const uint16_t* swa,
                                                      const int32_t* swa_len, int W, float softmax_scale,
                                                      uint16_t* out, float* lse, int n_split,
                                                      csa2_stream_t stream) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (B < 0 || Nq < 0 || cap < 0 || k < 0 || k > CSA2_MAX_ATTN_K || n_split < 0 || n_split > csa2::attn::kMaxSplit)
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
  if (csa2::attn_ws_bytes(instances, ns) > csa2::kStaticScratchBytes) return CSA2_ERR_TOO_LARGE;
  float* scratch = csa2::static_scratch();
  if (!scratch) return CSA2_ERR_CUDA;
  return csa2::launch_sparse_attn(q, B, Nq, codes, scales, cap, idx, n_valid, k, swa, swa_len, W, softmax_scale,
                                  out, lse, ns, scratch, reinterpret_cast<cudaStream_t>(stream), false) == cudaSuccess
             ? CSA2_OK
             : CSA2_ERR_CUDA;
}

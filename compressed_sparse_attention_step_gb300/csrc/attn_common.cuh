// Device helpers of the attention kernel (attn.cu): the 128-byte-swizzled operand layout, the FP4 /
// E4M3 hardware conversions, tcgen05 and mbarrier wrappers, tensor-memory loads and stores, and the
// warp reductions of the online softmax.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace csa2 {
namespace attn {

constexpr int kThreads = 256;
constexpr int kRows = 64;       // rows per tile = MMA M of S^T
constexpr int kMaxSplit = 32;   // split partials of one instance
constexpr float kLn2 = 0.6931471805599453f;

// byte offset of 16-byte chunk cc (0..63) of row r in a 128-byte-swizzled K-major operand whose
// 64-channel groups are `group` bytes apart
__device__ __forceinline__ uint32_t sw128(uint32_t group, int r, int cc) {
  return uint32_t(cc >> 3) * group + uint32_t(r) * 128u + uint32_t(((cc & 7) ^ (r & 7)) << 4);
}
// byte offset of 16-byte piece p (0..15) of staged FP4 row r (XOR-swizzled against bank conflicts)
__device__ __forceinline__ uint32_t raw_off(int r, int p) {
  return uint32_t(r) * CSA2_CODE_BYTES + uint32_t((p ^ (r & 7)) << 4);
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Four code bytes (eight E2M1 codes, the even channel in the low nibble of each byte) -> four f16x2
// (even channel in the low half), with the hardware conversion.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t& o0, uint32_t& o1, uint32_t& o2,
                                                  uint32_t& o3) {
  asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
      : "r"(w));
}
// Two E4M3 (FN) scale bytes (first in the low byte) -> f16x2 (first in the low half); exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t u) {
  return h2_bits(__floats2half2_rn(bf16lo(u), bf16hi(u)));
}

// 2^x with the hardware approximation (relative error about 2^-22; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- tcgen05 / mbarrier wrappers -----------------------------------------------------------------
// Shared-memory matrix descriptor: start address, leading / stride byte offsets, descriptor
// version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return uint64_t((addr >> 4) & 0x3FFFu) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}
// Instruction descriptor of kind::f16: fp32 accumulator, A/B f16 or bf16, A K-major or MN-major,
// B K-major, M = m, N = n (16 heads by default).
__device__ __forceinline__ uint32_t instr_desc(int m, bool bf16, bool a_mn_major, int n = CSA2_H) {
  return (1u << 4) | (bf16 ? (1u << 7) | (1u << 10) : 0u) | (a_mn_major ? (1u << 15) : 0u) |
         ((uint32_t(n) >> 3) << 17) | ((uint32_t(m) >> 4) << 24);
}
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(mbar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Waits for phase `parity` of the mbarrier, for at most about one second.  Each test suspends the
// thread until the phase completes or 20 us pass, so waiting warps take no issue slots from the
// working ones.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p; }\n"
        : "=r"(done)
        : "r"(mbar), "r"(parity), "n"(20000)
        : "memory");
    if (done) return true;
    if ((it & 63u) == 0u) {
      const uint64_t now = global_ns();
      if (it == 0u) t0 = now;
      else if (now - t0 > 1000000000ull) return false;
    }
  }
}

// Columns c, c + 16, c + 32, c + 48 (8 each) of this warp's 32 lanes, one wait for all four.
__device__ __forceinline__ void tmem_ld8x4(uint32_t taddr, float (&v)[4][8]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8, %9, %10, %11, %12, %13, %14, %15}, [%33];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16, %17, %18, %19, %20, %21, %22, %23}, [%34];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%24, %25, %26, %27, %28, %29, %30, %31}, [%35];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr), "r"(taddr + 16), "r"(taddr + 32), "r"(taddr + 48)
      : "memory");
#pragma unroll
  for (int g = 0; g < 4; ++g)
#pragma unroll
    for (int i = 0; i < 8; ++i) v[g][i] = __uint_as_float(r[8 * g + i]);
}
// Columns c .. c + 31 of this warp's 32 lanes as two groups of 16, one wait.
__device__ __forceinline__ void tmem_ld16x2(uint32_t taddr, float (&v)[2][16]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr), "r"(taddr + 16)
      : "memory");
#pragma unroll
  for (int g = 0; g < 2; ++g)
#pragma unroll
    for (int i = 0; i < 16; ++i) v[g][i] = __uint_as_float(r[16 * g + i]);
}
__device__ __forceinline__ void tmem_st16x2(uint32_t taddr, const float (&v)[2][16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17};\n\t"
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%1], {%18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33};\n\t"
      "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr), "r"(taddr + 16),
      "r"(__float_as_uint(v[0][0])), "r"(__float_as_uint(v[0][1])), "r"(__float_as_uint(v[0][2])), "r"(__float_as_uint(v[0][3])), "r"(__float_as_uint(v[0][4])), "r"(__float_as_uint(v[0][5])), "r"(__float_as_uint(v[0][6])), "r"(__float_as_uint(v[0][7])), "r"(__float_as_uint(v[0][8])), "r"(__float_as_uint(v[0][9])), "r"(__float_as_uint(v[0][10])), "r"(__float_as_uint(v[0][11])), "r"(__float_as_uint(v[0][12])), "r"(__float_as_uint(v[0][13])), "r"(__float_as_uint(v[0][14])), "r"(__float_as_uint(v[0][15])), "r"(__float_as_uint(v[1][0])), "r"(__float_as_uint(v[1][1])), "r"(__float_as_uint(v[1][2])), "r"(__float_as_uint(v[1][3])), "r"(__float_as_uint(v[1][4])), "r"(__float_as_uint(v[1][5])), "r"(__float_as_uint(v[1][6])), "r"(__float_as_uint(v[1][7])), "r"(__float_as_uint(v[1][8])), "r"(__float_as_uint(v[1][9])), "r"(__float_as_uint(v[1][10])), "r"(__float_as_uint(v[1][11])), "r"(__float_as_uint(v[1][12])), "r"(__float_as_uint(v[1][13])), "r"(__float_as_uint(v[1][14])), "r"(__float_as_uint(v[1][15]))
      : "memory");
}

// Eight values per lane (heads 0..7 of a row) -> lane l returns the combination over the warp's
// 32 lanes for head (l >> 2), in a fixed tree order.
template <bool kMax>
__device__ __forceinline__ float reduce_scatter8(const float (&v)[8], int lane) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4;
  float a[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = u16 ? v[i] : v[i + 4], keep = u16 ? v[i + 4] : v[i];
    a[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
  float b[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = u8 ? a[i] : a[i + 2], keep = u8 ? a[i + 2] : a[i];
    b[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
  float c;
  {
    const float send = u4 ? b[0] : b[1], keep = u4 ? b[1] : b[0];
    c = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  }
  c = op(c, __shfl_xor_sync(0xffffffffu, c, 2));
  c = op(c, __shfl_xor_sync(0xffffffffu, c, 1));
  return c;
}

}  // namespace attn
}  // namespace csa2

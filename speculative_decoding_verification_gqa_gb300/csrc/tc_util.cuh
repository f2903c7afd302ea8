// tc_util.cuh -- helpers of the tcgen05 attention kernels: mbarriers with bounded waits,
// TMA tile loads, tcgen05 shared-memory and instruction descriptors, MMA issue and commit,
// TMEM loads and stores, and the packing of scores into 16-bit operands. Each kernel file
// includes it into its own anonymous namespace.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.cuh"

namespace sv {

// [kv_rows, Hkv, hd] K or V cache -> a tensor map of boxes of 128 bytes x 1 head x box_rows
// rows with 128-byte swizzle (attn_tc.cu). False if the driver entry point is missing or
// the encoding fails.
bool kv_tensor_map(CUtensorMap* map, const void* base, int64_t kv_rows, int hkv, int hd,
                   bool fp8, int box_rows);

namespace {

constexpr long long TIMEOUT_CYCLES = 4000000000LL;  // ~2 s at 2 GHz
constexpr float RESCALE_THRESHOLD = 8.f;            // log2 units

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(b)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(saddr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// What a bounded wait needs: the CTA's abort flag (shared memory), the workspace flag word
// and the limit in clock cycles (a kernel parameter).
struct Waiter {
  volatile int* abort;
  uint32_t* flags;
  long long limit;
};

// Bounded wait for the phase with the given parity. Returns false (and raises the CTA's
// abort flag and the workspace timeout flag) if it gives up or another role already did.
__device__ __noinline__ bool mbar_wait_slow(uint64_t* b, uint32_t parity, const Waiter w) {
  const long long t0 = clock64();
  while (true) {
    if (mbar_try(b, parity)) return true;
    if (*w.abort) return false;
    if (clock64() - t0 > w.limit) {
      *w.abort = 1;
      atomicOr(w.flags, FLAG_TIMEOUT);
      return false;
    }
  }
}

// The common case (phase already complete) costs one try_wait and no call.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, const Waiter& w) {
  return mbar_try(b, parity) || mbar_wait_slow(b, parity, w);
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(c2), "r"(saddr(bar))
      : "memory");
}

// tcgen05 shared-memory matrix descriptor: start address, leading / stride byte offsets,
// descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A K-major,
// B K-major (b_mn = 0) or MN-major (b_mn = 1), M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_bf16(int n, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
// The same with f16 A and B (FP8 K/V decoded to f16).
__host__ __device__ constexpr uint32_t idesc_f16(int n, int b_mn) {
  return (1u << 4) | ((uint32_t)b_mn << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(128 >> 4) << 24);
}

// Instruction descriptor, kind::f8f6f4: fp32 accumulator, E4M3 A and B (format code 0),
// both K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_e4m3(int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
// The same on the 8-bit path: A (TMEM) and B (shared memory) both E4M3, 32 K-elements.
__device__ __forceinline__ void mma_ts_e4m3(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          saddr(bar))
      : "memory");
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

#define SV_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                 "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define SV_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                 "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// 32 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : SV_R8(0), SV_R8(8), SV_R8(16), SV_R8(24)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      SV_W8(0), SV_W8(8), SV_W8(16), SV_W8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      SV_W8(0), SV_W8(8)
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                   taddr),
               SV_W8(0)
               : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15}, [%16];"
      : SV_R8(0), SV_R8(8)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Ties registers written by tcgen05.ld to a point after tcgen05.wait::ld, so the compiler
// cannot move their first use above the wait.
__device__ __forceinline__ void reg_fence32(uint32_t* r) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
               "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
               "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
               "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
               "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
               "+r"(r[30]), "+r"(r[31]));
}
__device__ __forceinline__ void reg_fence16(uint32_t* r) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
               "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
               "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Named barrier 1 over the 256 softmax threads with an AND of `v`: the two warpgroups meet
// here once per tile (and once per unit epilogue), and a failed wait in either one makes
// both leave together, so neither can be left waiting at the barrier.
__device__ __forceinline__ bool softmax_pair_and(bool v) {
  __syncwarp();  // the reduction counts whole warps: arrive converged
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.red.and.pred q, 1, 256, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// (x0, x1) = (x0 * a + b, x1 * a + b), each rounded to nearest: one paired instruction
__device__ __forceinline__ void fma2(float& x0, float& x1, float a, float b) {
  asm("{\n .reg .b64 v, s, m;\n mov.b64 v, {%0, %1};\n mov.b64 s, {%2, %2};\n"
      " mov.b64 m, {%3, %3};\n fma.rn.f32x2 v, v, s, m;\n mov.b64 {%0, %1}, v;\n}"
      : "+f"(x0), "+f"(x1)
      : "f"(a), "f"(b));
}
// (s0, s1) += (a0, a1), each rounded to nearest: one paired instruction
__device__ __forceinline__ void add2(float& s0, float& s1, float a0, float a1) {
  asm("{\n .reg .b64 v, w;\n mov.b64 v, {%0, %1};\n mov.b64 w, {%2, %3};\n"
      " add.rn.f32x2 v, v, w;\n mov.b64 {%0, %1}, v;\n}"
      : "+f"(s0), "+f"(s1)
      : "f"(a0), "f"(a1));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
template <bool F16>
__device__ __forceinline__ uint32_t pack_p(float lo, float hi) {
  return F16 ? pack_f16(lo, hi) : pack_bf16(lo, hi);
}
// Four E4M3 codes (low byte first) -> two f16 pairs of the same values; exact, every E4M3
// value is an f16 value. The 32-bit word splits into its two 16-bit halves for free.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.rn.f16x2.e4m3x2 %0, a;\n"
      " cvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Two floats -> two E4M3 codes (the first in the low byte), nearest even, saturating.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// Two E4M3 codes (low byte first, in the low 16 bits) -> their values.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t c) {
  uint32_t h;
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %1;\n cvt.rn.f16x2.e4m3x2 %0, a;\n}\n"
      : "=r"(h)
      : "r"(c));
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

}  // namespace
}  // namespace sv

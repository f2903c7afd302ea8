// logits_vec.cuh -- 16-byte vectors of logits (8 bf16 or 4 fp32 values), shared by the
// acceptance and draft-signal scans.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace sv {

// Element `hi` (0 = low half) of a bf16 pair, widened exactly to fp32.
__device__ __forceinline__ float bf16_at(uint32_t w, int hi) {
  return __uint_as_float(hi ? (w & 0xffff0000u) : (w << 16));
}

__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t w) {
  return *reinterpret_cast<const __nv_bfloat162*>(&w);
}

// Largest of eight bf16 values (NaN ignored unless all are NaN), widened to fp32.
__device__ __forceinline__ float vmax_bf16x8(const uint4& w) {
  const __nv_bfloat162 m = __hmax2(__hmax2(as_bf2(w.x), as_bf2(w.y)), __hmax2(as_bf2(w.z), as_bf2(w.w)));
  const uint32_t u = *reinterpret_cast<const uint32_t*>(&m);
  return fmaxf(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

}  // namespace sv

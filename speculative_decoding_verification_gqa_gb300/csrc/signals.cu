// signals.cu -- draft signals for adaptive speculation length ("SpecKV: Adaptive
// Speculative Decoding with Compression-Aware Gamma Selection", summary, "technical core",
// item 1): per row of logits, the confidence (the largest probability of its softmax) and
// the entropy (nats) of that softmax, the two inputs of the speculation-length controller.
//
// One streaming pass. In log2 units t = x log2(e), each thread keeps for its part of a
// row a running maximum m, z = sum 2^(t - m) and s = sum (t - m) 2^(t - m); parts merge
// with the online-softmax rule ("GPU and LLM, chapter 5", "Online softmax": rescale by
// 2^(m_old - m_new)), extended to s: s' = 2^(m - m')(s + (m - m') z). For the whole row
// p_j = 2^(t_j - m) / z, so confidence = 1 / z and entropy = ln z - ln(2) s / z.
//
// Persistent CTAs scan equal contiguous ranges of the packed logits (as the acceptance
// kernel does), leave one (m, z, s) partial per (CTA, row) they touch, and the last CTA
// to finish (a completion ticket) merges each row's partials and writes the signals.
#include <cuda_bf16.h>

#include "internal.cuh"
#include "logits_vec.cuh"

namespace sv {
namespace {

#ifndef SV_SIG_THREADS
#define SV_SIG_THREADS 512
#endif
#ifndef SV_SIG_UNROLL
#define SV_SIG_UNROLL 4
#endif
#ifndef SV_SIG_CTAS_PER_SM
#define SV_SIG_CTAS_PER_SM 2
#endif
constexpr int SIG_THREADS = SV_SIG_THREADS;
constexpr int SIG_UNROLL = SV_SIG_UNROLL;  // 16-byte loads in flight per thread
constexpr int SIG_CTAS_PER_SM = SV_SIG_CTAS_PER_SM;  // all resident at once
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr float T_FLOOR = -150.f;  // 2^-150 is 0 in fp32: keeps (t - m) * 0 finite

struct Part {
  float m, z, s, pad;
};

struct SigArgs {
  const void* logits;
  float* confidence;
  float* entropy;
  uint32_t* ticket;  // CTAs of this call that have finished; reset by the last one
  Part* part;        // [nctas + rows]: slot c + r = CTA c's part of row r
  int64_t rows;
  int vocab, nctas;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Rescale factor 2^d for d <= 0: exactly 1 when the maximum did not move (the approximate
// exponential of 0 is not exactly 1, and the factor is applied once per vector and merge).
__device__ __forceinline__ float rescale_factor(float d) { return d == 0.f ? 1.f : ex2(d); }

// (m, z, s) <- (m, z, s) merged with (m2, z2, s2); an empty part has z = 0.
__device__ __forceinline__ void merge(float& m, float& z, float& s, float m2, float z2, float s2) {
  const float mn = fmaxf(m, m2);
  const float d1 = z > 0.f ? m - mn : 0.f, d2 = z2 > 0.f ? m2 - mn : 0.f;
  const float c1 = z > 0.f ? rescale_factor(d1) : 0.f, c2 = z2 > 0.f ? rescale_factor(d2) : 0.f;
  s = c1 * (s + d1 * z) + c2 * (s2 + d2 * z2);
  z = c1 * z + c2 * z2;
  m = z > 0.f ? mn : m;
}

// Adds element t (log2 units) to a thread's running (m, z, s) whose m already bounds it.
__device__ __forceinline__ void add(float t, float m, float& z, float& s) {
  const float d = fmaxf(t - m, T_FLOOR);
  const float e = ex2(d);
  z += e;
  s = fmaf(d, e, s);
}

// Raises the running max to at least mt (log2 units), rescaling z and s.
__device__ __forceinline__ void raise_max(float mt, float& m, float& z, float& s) {
  const float mn = fmaxf(m, mt);
  const float d = z > 0.f ? m - mn : 0.f;  // m may still be -inf while z is 0
  const float c = rescale_factor(d);
  s = c * (s + d * z);
  z = c * z;
  m = mn;
}

template <bool BF16>
__global__ void __launch_bounds__(SIG_THREADS, SIG_CTAS_PER_SM) signals_kernel(SigArgs a) {
  __shared__ Part sh[SIG_THREADS / 32];
  __shared__ int s_last;
  pdl_trigger();
  pdl_wait();
  constexpr int ES = BF16 ? 2 : 4;
  constexpr int VE = 16 / ES;  // elements per 16-byte vector
  const int64_t V = a.vocab, N = a.rows * V;
  const int64_t e0 = N * blockIdx.x / a.nctas, e1 = N * (blockIdx.x + 1) / a.nctas;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int64_t r = e0 / V; r * V < e1; ++r) {
    const int64_t c0 = max(e0, r * V) - r * V, c1 = min(e1, (r + 1) * V) - r * V;
    const uint8_t* row = (const uint8_t*)a.logits + r * V * ES;
    auto elem = [&](int e) -> float {
      if constexpr (BF16)
        return __uint_as_float((uint32_t)((const uint16_t*)row)[e] << 16);
      else
        return ((const float*)row)[e];
    };
    // scalar head up to a 16-byte boundary, 16-byte vectors, scalar tail (row-local
    // indices fit in 32 bits)
    const int h0 = (int)(((16 - ((uintptr_t)(row + c0 * ES) & 15)) & 15) / ES);
    const int vb = (int)c0 + (h0 < c1 - c0 ? h0 : (int)(c1 - c0));
    const int nvec = ((int)c1 - vb) / VE;
    const int tb = vb + nvec * VE;
    float m = -INFINITY, z = 0.f, s = 0.f;
    for (int e = (int)c0 + threadIdx.x; e < vb; e += blockDim.x) {
      const float t = elem(e) * LOG2E;
      raise_max(t, m, z, s);
      add(t, m, z, s);
    }
    const uint4* vec = reinterpret_cast<const uint4*>(row + vb * ES);
    for (int base = threadIdx.x; base < nvec; base += blockDim.x * SIG_UNROLL) {
      uint4 w[SIG_UNROLL];
#pragma unroll
      for (int k = 0; k < SIG_UNROLL; ++k) {
        const int vi = base + k * blockDim.x;
        w[k] = vi < nvec ? __ldcs(vec + vi) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < SIG_UNROLL; ++k) {
        if (base + k * blockDim.x >= nvec) break;
        const uint32_t ww[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
        float vm;
        if constexpr (BF16)
          vm = vmax_bf16x8(w[k]);
        else
          vm = fmaxf(fmaxf(__uint_as_float(ww[0]), __uint_as_float(ww[1])),
                     fmaxf(__uint_as_float(ww[2]), __uint_as_float(ww[3])));
        raise_max(vm * LOG2E, m, z, s);  // once per vector, without branches
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if constexpr (BF16) {
            add(bf16_at(ww[q], 0) * LOG2E, m, z, s);
            add(bf16_at(ww[q], 1) * LOG2E, m, z, s);
          } else {
            add(__uint_as_float(ww[q]) * LOG2E, m, z, s);
          }
        }
      }
    }
    for (int e = tb + threadIdx.x; e < c1; e += blockDim.x) {
      const float t = elem(e) * LOG2E;
      raise_max(t, m, z, s);
      add(t, m, z, s);
    }
    // merge the row segment across the CTA: warp shuffles, then the warps' parts
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float z2 = __shfl_xor_sync(0xffffffffu, z, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      merge(m, z, s, m2, z2, s2);
    }
    if (lane == 0) sh[wid] = Part{m, z, s, 0.f};
    __syncthreads();
    if (wid == 0) {
      const Part q = lane < (int)(blockDim.x >> 5) ? sh[lane] : Part{-INFINITY, 0.f, 0.f, 0.f};
      m = q.m;
      z = q.z;
      s = q.s;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float z2 = __shfl_xor_sync(0xffffffffu, z, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        merge(m, z, s, m2, z2, s2);
      }
      if (lane == 0) a.part[(size_t)blockIdx.x + r] = Part{m, z, s, 0.f};
    }
    __syncthreads();  // sh is reused by the next row
  }
  // completion ticket: the last CTA merges every row's parts
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(a.ticket, 1u) == (uint32_t)a.nctas - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x == 0) atomicExch(a.ticket, 0u);
  for (int64_t r = threadIdx.x; r < a.rows; r += blockDim.x) {
    const int c_lo = cta_of_tile(r * V, N, a.nctas), c_hi = cta_of_tile((r + 1) * V - 1, N, a.nctas);
    float m = -INFINITY, z = 0.f, s = 0.f;
    for (int c = c_lo; c <= c_hi; ++c) {
      if (!cta_has_tiles(c, N, a.nctas)) continue;
      const float4 q = __ldcg(reinterpret_cast<const float4*>(a.part + (size_t)c + r));
      merge(m, z, s, q.x, q.y, q.z);
    }
    a.confidence[r] = 1.f / z;
    a.entropy[r] = logf(z) - LN2 * s / z;
  }
}

}  // namespace

SigWs signals_ws_layout(int64_t rows, int vocab, int num_sms) {
  SigWs w;
  const int64_t n = rows * (int64_t)vocab;
  int64_t c = (int64_t)SIG_CTAS_PER_SM * num_sms;
  if (c > n / 8192) c = n / 8192;
  if (c < 1) c = 1;
  w.nctas = (int)c;
  w.ctrl = 0;  // ticket at +64
  w.part = 256;
  w.total = align_up(w.part + sizeof(Part) * (size_t)(rows + c), 256);
  return w;
}

cudaError_t launch_signals(int64_t rows, int vocab, int dtype, const void* logits,
                           float* confidence, float* entropy, void* ws, const SigWs& lay,
                           cudaStream_t s) {
  SigArgs a;
  a.logits = logits;
  a.confidence = confidence;
  a.entropy = entropy;
  a.ticket = (uint32_t*)((uint8_t*)ws + lay.ctrl + 64);
  a.part = (Part*)((uint8_t*)ws + lay.part);
  a.rows = rows;
  a.vocab = vocab;
  a.nctas = lay.nctas;
  return dtype == SV_BF16
             ? launch_pdl(signals_kernel<true>, dim3(a.nctas), dim3(SIG_THREADS), 0, s, a)
             : launch_pdl(signals_kernel<false>, dim3(a.nctas), dim3(SIG_THREADS), 0, s, a);
}

}  // namespace sv

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
// to finish (a completion ticket) merges each row's partials and writes the signals. When
// rows are whole 32-byte vectors and a range touches at most FLAT_ROWS rows, the range is
// one stream of 32-byte vectors across row boundaries: at a row's end each warp merges its
// lanes and leaves its part in shared memory, and the CTA merges its rows' warp parts once,
// at the end of its range (no CTA barrier per row). Otherwise the range is taken row by
// row, with the CTA's merge at each row's end.
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
constexpr int NW = SIG_THREADS / 32;
constexpr int FLAT_U = 4;       // continuous path: 32-byte vectors per thread per batch
constexpr int FLAT_ROWS = 16;   // continuous path: rows a CTA's range may touch
constexpr int64_t FLAT_BATCH_VECS = (int64_t)SIG_THREADS * FLAT_U;

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
  int64_t row_vecs;  // continuous path: 32-byte vectors per row
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

// Merges (m, z, s) across the 32 lanes of a warp (every lane ends with the warp's part).
__device__ __forceinline__ void warp_merge(float& m, float& z, float& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float z2 = __shfl_xor_sync(0xffffffffu, z, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    merge(m, z, s, m2, z2, s2);
  }
}

// 32 bytes (16 bf16 or 8 fp32 logits) in one load; read once, so not kept in L1.
__device__ __forceinline__ void load32(const uint8_t* p, uint32_t (&w)[8]) {
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::256B.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
        "=r"(w[7])
      : "l"(p));
}

// Adds a 32-byte vector of logits to a thread's running (m, z, s): the maximum raised once
// per vector, then every element.
template <bool BF16>
__device__ __forceinline__ void add_vec32(const uint32_t (&w)[8], float& m, float& z, float& s) {
  float vm;
  if constexpr (BF16) {
    vm = fmaxf(vmax_bf16x8(make_uint4(w[0], w[1], w[2], w[3])),
               vmax_bf16x8(make_uint4(w[4], w[5], w[6], w[7])));
  } else {
    vm = fmaxf(fmaxf(fmaxf(__uint_as_float(w[0]), __uint_as_float(w[1])),
                     fmaxf(__uint_as_float(w[2]), __uint_as_float(w[3]))),
               fmaxf(fmaxf(__uint_as_float(w[4]), __uint_as_float(w[5])),
                     fmaxf(__uint_as_float(w[6]), __uint_as_float(w[7]))));
  }
  raise_max(vm * LOG2E, m, z, s);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    if constexpr (BF16) {
      add(bf16_at(w[q], 0) * LOG2E, m, z, s);
      add(bf16_at(w[q], 1) * LOG2E, m, z, s);
    } else {
      add(__uint_as_float(w[q]) * LOG2E, m, z, s);
    }
  }
}

// Continuous path: CTA blockIdx.x's equal share of the rows * row_vecs vectors, one batch of
// FLAT_U vectors per thread at a time, taken in one pass per row it touches; at each row's
// end (uniform over the CTA) every warp merges its lanes into sp[row - first row][warp].
template <bool BF16>
__device__ void scan_flat(const SigArgs& a, int64_t v0, int64_t v1, Part (*sp)[NW]) {
  const int64_t rv = a.row_vecs, rfirst = v0 / rv;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const uint8_t* base = (const uint8_t*)a.logits;
  int64_t r = rfirst, row0 = r * rv, rb = row0 + rv;  // current row [row0, rb)
  float m = -INFINITY, z = 0.f, s = 0.f;
  auto flush = [&]() {
    warp_merge(m, z, s);
    if (lane == 0) sp[r - rfirst][wid] = Part{m, z, s, 0.f};
    m = -INFINITY;
    z = 0.f;
    s = 0.f;
  };
  for (int64_t b0 = v0; b0 < v1; b0 += FLAT_BATCH_VECS) {
    uint32_t w[FLAT_U][8];
#pragma unroll
    for (int k = 0; k < FLAT_U; ++k) {
      const int64_t vi = b0 + (int64_t)k * SIG_THREADS + threadIdx.x;
      if (vi < v1) load32(base + vi * 32, w[k]);
    }
    const int64_t se = min(b0 + FLAT_BATCH_VECS, v1);  // end of the batch's valid vectors
    while (true) {
      const int64_t cut = min(rb, se);
#pragma unroll
      for (int k = 0; k < FLAT_U; ++k) {
        const int64_t vi = b0 + (int64_t)k * SIG_THREADS + threadIdx.x;
        if (vi >= row0 && vi < cut) add_vec32<BF16>(w[k], m, z, s);
      }
      if (rb >= se) break;
      flush();  // row r is finished
      ++r;
      row0 = rb;
      rb += rv;
    }
  }
  flush();  // the range's last row
}

template <bool BF16, bool FLAT>
__global__ void __launch_bounds__(SIG_THREADS, SIG_CTAS_PER_SM) signals_kernel(SigArgs a) {
  __shared__ Part sh[SIG_THREADS / 32];
  __shared__ Part sp[FLAT ? FLAT_ROWS : 1][NW];
  __shared__ int s_last;
  pdl_trigger();
  pdl_wait();
  constexpr int ES = BF16 ? 2 : 4;
  constexpr int VE = 16 / ES;  // elements per 16-byte vector
  const int64_t V = a.vocab;
  // the line of positions split over the CTAs: elements, or 32-byte vectors (continuous)
  const int64_t N = FLAT ? a.rows * a.row_vecs : a.rows * V;
  const int64_t e0 = N * blockIdx.x / a.nctas, e1 = N * (blockIdx.x + 1) / a.nctas;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if constexpr (FLAT) {
    if (e0 < e1) {
      scan_flat<BF16>(a, e0, e1, sp);
      __syncthreads();
      // this CTA's part of each row it touched: one warp per row merges the warps' parts
      const int64_t rfirst = e0 / a.row_vecs;
      const int nloc = (int)((e1 - 1) / a.row_vecs - rfirst + 1);
      for (int lr = wid; lr < nloc; lr += NW) {
        const Part q = lane < NW ? sp[lr][lane] : Part{-INFINITY, 0.f, 0.f, 0.f};
        float m = q.m, z = q.z, s = q.s;
        warp_merge(m, z, s);
        if (lane == 0) a.part[(size_t)blockIdx.x + rfirst + lr] = Part{m, z, s, 0.f};
      }
    }
  }
  for (int64_t r = e0 / V; !FLAT && r * V < e1; ++r) {
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
  const int64_t RL = FLAT ? a.row_vecs : V;  // positions per row on the split line
  for (int64_t r = threadIdx.x; r < a.rows; r += blockDim.x) {
    const int c_lo = cta_of_tile(r * RL, N, a.nctas), c_hi = cta_of_tile((r + 1) * RL - 1, N, a.nctas);
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
  // continuous path: rows of whole, 32-byte aligned vectors, and every CTA's range within
  // FLAT_ROWS rows
  const int64_t row_bytes = (int64_t)vocab * (dtype == SV_BF16 ? 2 : 4);
  a.row_vecs = row_bytes / 32;
  bool flat = ((uintptr_t)logits & 31) == 0 && row_bytes % 32 == 0;
  if (flat) {
    const int64_t nv = rows * a.row_vecs;
    const int64_t per = (nv + a.nctas - 1) / a.nctas;  // vectors of the longest range
    flat = (per + a.row_vecs - 1) / a.row_vecs + 1 <= FLAT_ROWS;
  }
  const dim3 g(a.nctas), b(SIG_THREADS);
  if (dtype == SV_BF16)
    return flat ? launch_pdl(signals_kernel<true, true>, g, b, 0, s, a)
                : launch_pdl(signals_kernel<true, false>, g, b, 0, s, a);
  return flat ? launch_pdl(signals_kernel<false, true>, g, b, 0, s, a)
              : launch_pdl(signals_kernel<false, false>, g, b, 0, s, a);
}

}  // namespace sv

// accept.cu -- greedy acceptance ("Co-Designing AI Models Using Speculative Decoding",
// basic structure: keep the drafts up to the first mismatch; "GPU and LLM, chapter 5",
// "Speculative decoding (2)": the target's own token takes the place of the first
// rejected draft).
//
// Kernel 1 (argmax_partial): persistent CTAs, each scanning an equal contiguous range of
//   the packed logits with 16-byte streaming loads, a running (value, index) per thread, then
//   warp-shuffle and shared-memory reductions with the comparator "larger value wins, equal
//   values: smaller index wins", one candidate per row the range touches. Values are
//   compared exactly in fp32 (bf16 widens exactly).
// Kernel 2 (finalize): one CTA per sequence. Merges the candidates of its 1 + D_b rows,
//   then finds the first position whose draft differs from the target's token.
#include <cuda_bf16.h>

#include "internal.cuh"

namespace sv {
namespace {

constexpr int ARGMAX_THREADS = 512;
constexpr int UNROLL = 4;
constexpr int NONE = 0x7fffffff;  // "no candidate yet"

struct Cand {
  float v;
  int i;
};

__device__ __forceinline__ bool better(float v1, int i1, float v2, int i2) {
  if (i1 == NONE) return false;
  if (i2 == NONE) return true;
  return v1 > v2 || (v1 == v2 && i1 < i2);
}

__device__ __forceinline__ void take(float x, int idx, float& bv, int& bi) {
  // indices reach a thread in increasing order, so a strict '>' keeps the first maximum
  if (x > bv || (bi == NONE && x == x)) {
    bv = x;
    bi = idx;
  }
}

__device__ __forceinline__ float bf16_at(uint32_t w, int hi) {
  return __uint_as_float(hi ? (w & 0xffff0000u) : (w << 16));
}

__device__ __forceinline__ void block_argmax(float& bv, int& bi, Cand* sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(v2, i2, bv, bi)) {
      bv = v2;
      bi = i2;
    }
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane == 0) sh[wid] = Cand{bv, bi};
  __syncthreads();
  if (wid == 0) {
    const int nw = blockDim.x >> 5;
    bv = lane < nw ? sh[lane].v : 0.f;
    bi = lane < nw ? sh[lane].i : NONE;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      if (better(v2, i2, bv, bi)) {
        bv = v2;
        bi = i2;
      }
    }
  }
}

// Sum of (1 + D_b') and D_b' over b' < b; returns false if any D_b' is out of range.
__device__ bool prefix_offsets(const int32_t* draft_len, int b, int max_draft, int64_t* q_off,
                               int64_t* d_off) {
  __shared__ long long s_q, s_d;
  __shared__ int s_bad;
  if (threadIdx.x == 0) {
    s_q = 0;
    s_d = 0;
    s_bad = 0;
  }
  __syncthreads();
  long long q = 0, d = 0;
  int bad = 0;
  for (int bb = threadIdx.x; bb < b; bb += blockDim.x) {
    const int D = draft_len[bb];
    bad |= (D < 0 || D > max_draft);
    q += 1 + D;
    d += D;
  }
  if (q) atomicAdd((unsigned long long*)&s_q, (unsigned long long)q);
  if (d) atomicAdd((unsigned long long*)&s_d, (unsigned long long)d);
  if (bad) s_bad = 1;
  __syncthreads();
  *q_off = s_q;
  *d_off = s_d;
  const bool ok = !s_bad;
  __syncthreads();
  return ok;
}

struct AcceptArgs {
  const void* logits;
  const int32_t* draft_tokens;
  const int32_t* draft_len;
  int32_t* accept_len;
  int32_t* next_token;
  int32_t* target_tokens;
  uint32_t* flags;
  Cand* part;  // [nctas + B * (1 + max_draft)]: slot c + r = CTA c's part of row r
  int B, max_draft, vocab, nctas;
};

// Total window rows sum_b (1 + D_b); false if any D_b is out of range.
__device__ bool total_rows(const int32_t* draft_len, int B, int max_draft, int64_t* rows) {
  __shared__ long long s_rows;
  __shared__ int s_bad;
  if (threadIdx.x == 0) {
    s_rows = 0;
    s_bad = 0;
  }
  __syncthreads();
  long long q = 0;
  int bad = 0;
  for (int bb = threadIdx.x; bb < B; bb += blockDim.x) {
    const int D = draft_len[bb];
    bad |= (D < 0 || D > max_draft);
    q += 1 + D;
  }
  if (q) atomicAdd((unsigned long long*)&s_rows, (unsigned long long)q);
  if (bad) s_bad = 1;
  __syncthreads();
  *rows = s_rows;
  const bool ok = !s_bad;
  __syncthreads();
  return ok;
}

// The packed logits are one array of rows * V elements; CTA c scans the contiguous range
// [c*N/C, (c+1)*N/C), so every CTA reads the same number of bytes whatever the row count,
// and leaves one (value, index) candidate per row it touches (a range spans at most a few
// rows).
template <bool BF16>
__global__ void __launch_bounds__(ARGMAX_THREADS) argmax_partial_kernel(AcceptArgs a) {
  __shared__ Cand sh[32];
  pdl_trigger();
  pdl_wait();
  int64_t rows;
  if (!total_rows(a.draft_len, a.B, a.max_draft, &rows)) return;  // finalize raises the flag
  constexpr int ES = BF16 ? 2 : 4;
  constexpr int VE = 16 / ES;  // elements per 16-byte vector
  const int64_t V = a.vocab, N = rows * V;
  const int64_t e0 = N * blockIdx.x / a.nctas, e1 = N * (blockIdx.x + 1) / a.nctas;
  if (e0 >= e1) return;
  for (int64_t r = e0 / V; r * V < e1; ++r) {
    const int64_t c0 = max(e0, r * V) - r * V, c1 = min(e1, (r + 1) * V) - r * V;
    const uint8_t* row = (const uint8_t*)a.logits + r * V * ES;
    auto elem = [&](int64_t e) -> float {
      if constexpr (BF16)
        return __uint_as_float((uint32_t)((const uint16_t*)row)[e] << 16);
      else
        return ((const float*)row)[e];
    };
    // scalar head up to a 16-byte boundary, 16-byte vectors, scalar tail
    const int64_t h0 = (int64_t)(((16 - ((uintptr_t)(row + c0 * ES) & 15)) & 15) / ES);
    const int64_t vb = c0 + (h0 < c1 - c0 ? h0 : c1 - c0);
    const int64_t nvec = (c1 - vb) / VE;
    const int64_t tb = vb + nvec * VE;
    float bv = -INFINITY;
    int bi = NONE;
    for (int64_t e = c0 + threadIdx.x; e < vb; e += blockDim.x) take(elem(e), (int)e, bv, bi);
    const uint4* vec = reinterpret_cast<const uint4*>(row + vb * ES);
    for (int64_t base = threadIdx.x; base < nvec; base += (int64_t)blockDim.x * UNROLL) {
      uint4 w[UNROLL];
#pragma unroll
      for (int k = 0; k < UNROLL; ++k) {
        const int64_t vi = base + (int64_t)k * blockDim.x;
        w[k] = vi < nvec ? __ldcs(vec + vi) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < UNROLL; ++k) {
        const int64_t vi = base + (int64_t)k * blockDim.x;
        if (vi >= nvec) break;
        const int e = (int)(vb + vi * VE);
        const uint32_t ww[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if constexpr (BF16) {
            take(bf16_at(ww[q], 0), e + 2 * q, bv, bi);
            take(bf16_at(ww[q], 1), e + 2 * q + 1, bv, bi);
          } else {
            take(__uint_as_float(ww[q]), e + q, bv, bi);
          }
        }
      }
    }
    for (int64_t e = tb + threadIdx.x; e < c1; e += blockDim.x) take(elem(e), (int)e, bv, bi);
    block_argmax(bv, bi, sh);
    if (threadIdx.x == 0) a.part[(size_t)blockIdx.x + r] = Cand{bv, bi};
    __syncthreads();  // sh is reused by the next row
  }
}

__global__ void __launch_bounds__(256) accept_finalize_kernel(AcceptArgs a) {
  __shared__ int s_amax[256];
  __shared__ int s_first;
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  const int D = a.draft_len[b];
  if (D < 0 || D > a.max_draft) {
    if (threadIdx.x == 0) atomicOr(a.flags, FLAG_ACCEPT_SHAPE);
    return;
  }
  int64_t q_off, d_off, rows;
  if (!prefix_offsets(a.draft_len, b, a.max_draft, &q_off, &d_off)) return;
  if (!total_rows(a.draft_len, a.B, a.max_draft, &rows)) return;
  const int64_t V = a.vocab, N = rows * V;
  for (int i = threadIdx.x; i <= D; i += blockDim.x) {
    const int64_t r = q_off + i;
    const int c_lo = cta_of_tile(r * V, N, a.nctas), c_hi = cta_of_tile((r + 1) * V - 1, N, a.nctas);
    float bv = 0.f;
    int bi = NONE;
    for (int c = c_lo; c <= c_hi; ++c) {
      if (!cta_has_tiles(c, N, a.nctas)) continue;
      const Cand pc = a.part[(size_t)c + r];
      if (better(pc.v, pc.i, bv, bi)) {
        bv = pc.v;
        bi = pc.i;
      }
    }
    if (bi == NONE) bi = 0;  // a row made only of NaN: unspecified, report index 0
    s_amax[i] = bi;
    if (a.target_tokens) a.target_tokens[r] = bi;
  }
  if (threadIdx.x == 0) s_first = D;
  __syncthreads();
  for (int j = threadIdx.x; j < D; j += blockDim.x)
    if (a.draft_tokens[d_off + j] != s_amax[j]) atomicMin(&s_first, j);
  __syncthreads();
  if (threadIdx.x == 0) {
    const int n = s_first;
    a.accept_len[b] = n + 1;
    a.next_token[b] = s_amax[n];
  }
}

}  // namespace

AcceptWs accept_ws_layout(int B, int max_draft, int vocab, int num_sms) {
  AcceptWs w;
  const int64_t rows = (int64_t)B * (1 + max_draft);
  // persistent CTAs: 4 per SM, fewer for small inputs (at least ~8K elements each)
  const int64_t n_max = rows * (int64_t)vocab;
  int64_t c = 4LL * num_sms;
  if (c > n_max / 8192) c = n_max / 8192;
  if (c < 1) c = 1;
  w.nctas = (int)c;
  w.ctrl = 0;
  w.part = 256;
  w.total = align_up(256 + sizeof(Cand) * (size_t)(rows + c), 256);
  return w;
}

cudaError_t launch_accept(int B, int max_draft, int vocab, int dtype, const void* logits,
                          const int32_t* draft_tokens, const int32_t* draft_len,
                          int32_t* accept_len, int32_t* next_token, int32_t* target_tokens,
                          void* ws, const AcceptWs& lay, cudaStream_t s) {
  AcceptArgs a;
  a.logits = logits;
  a.draft_tokens = draft_tokens;
  a.draft_len = draft_len;
  a.accept_len = accept_len;
  a.next_token = next_token;
  a.target_tokens = target_tokens;
  a.flags = (uint32_t*)((uint8_t*)ws + lay.ctrl);
  a.part = (Cand*)((uint8_t*)ws + lay.part);
  a.B = B;
  a.max_draft = max_draft;
  a.vocab = vocab;
  a.nctas = lay.nctas;
  cudaError_t e = dtype == SV_BF16
                      ? launch_pdl(argmax_partial_kernel<true>, dim3(lay.nctas), dim3(ARGMAX_THREADS), 0, s, a)
                      : launch_pdl(argmax_partial_kernel<false>, dim3(lay.nctas), dim3(ARGMAX_THREADS), 0, s, a);
  if (e != cudaSuccess) return e;
  return launch_pdl(accept_finalize_kernel, dim3(B), dim3(256), 0, s, a);
}

}  // namespace sv

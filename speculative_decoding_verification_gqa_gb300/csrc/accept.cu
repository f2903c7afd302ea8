// accept.cu -- greedy acceptance ("Co-Designing AI Models Using Speculative Decoding",
// basic structure: keep the drafts up to the first mismatch; "GPU and LLM, chapter 5",
// "Speculative decoding (2)": the target's own token takes the place of the first
// rejected draft).
//
// Kernel 1 (argmax_partial): one CTA per (window row, vocab split). 16-byte vector loads
//   over the row, a running (value, index) per thread, then warp-shuffle and shared-memory
//   reductions with the comparator "larger value wins, equal values: smaller index wins".
//   Values are compared exactly in fp32 (bf16 widens exactly).
// Kernel 2 (finalize): one CTA per sequence. Merges the splits of its 1 + D_b rows, then
//   finds the first position whose draft differs from the target's token.
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
  Cand* part;  // [B * (1 + max_draft), splits]
  int B, max_draft, vocab, splits;
};

template <bool BF16>
__global__ void __launch_bounds__(ARGMAX_THREADS) argmax_partial_kernel(AcceptArgs a) {
  __shared__ Cand sh[32];
  const int W = 1 + a.max_draft;
  const int b = blockIdx.x / W, i = blockIdx.x % W, split = blockIdx.y;
  const int D = a.draft_len[b];
  if (D < 0 || D > a.max_draft || i > D) return;
  int64_t q_off, d_off;
  if (!prefix_offsets(a.draft_len, b, a.max_draft, &q_off, &d_off)) return;
  constexpr int ES = BF16 ? 2 : 4;
  constexpr int VE = 16 / ES;  // elements per 16-byte vector
  const int64_t V = a.vocab;
  const uint8_t* row = (const uint8_t*)a.logits + (q_off + i) * V * ES;
  const int64_t head0 = (int64_t)(((16 - ((uintptr_t)row & 15)) & 15) / ES);
  const int64_t head = head0 < V ? head0 : V;
  const int64_t nvec = (V - head) / VE;
  const int64_t tail0 = head + nvec * VE;
  const int64_t vb = nvec * split / a.splits, ve = nvec * (split + 1) / a.splits;
  float bv = -INFINITY;
  int bi = NONE;
  auto elem = [&](int64_t e) -> float {
    if constexpr (BF16)
      return __uint_as_float((uint32_t)((const uint16_t*)row)[e] << 16);
    else
      return ((const float*)row)[e];
  };
  if (split == 0)
    for (int64_t e = threadIdx.x; e < head; e += blockDim.x) take(elem(e), (int)e, bv, bi);
  const uint4* vec = reinterpret_cast<const uint4*>(row + head * ES);
  for (int64_t base = vb + threadIdx.x; base < ve; base += (int64_t)blockDim.x * UNROLL) {
    uint4 w[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int64_t vi = base + (int64_t)k * blockDim.x;
      w[k] = vi < ve ? __ldcs(vec + vi) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int64_t vi = base + (int64_t)k * blockDim.x;
      if (vi >= ve) break;
      const int e0 = (int)(head + vi * VE);
      const uint32_t ww[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if constexpr (BF16) {
          take(bf16_at(ww[q], 0), e0 + 2 * q, bv, bi);
          take(bf16_at(ww[q], 1), e0 + 2 * q + 1, bv, bi);
        } else {
          take(__uint_as_float(ww[q]), e0 + q, bv, bi);
        }
      }
    }
  }
  if (split == a.splits - 1)
    for (int64_t e = tail0 + threadIdx.x; e < V; e += blockDim.x) take(elem(e), (int)e, bv, bi);
  block_argmax(bv, bi, sh);
  if (threadIdx.x == 0) a.part[(size_t)blockIdx.x * a.splits + split] = Cand{bv, bi};
}

__global__ void __launch_bounds__(256) accept_finalize_kernel(AcceptArgs a) {
  __shared__ int s_amax[256];
  __shared__ int s_first;
  const int b = blockIdx.x;
  const int D = a.draft_len[b];
  if (D < 0 || D > a.max_draft) {
    if (threadIdx.x == 0) atomicOr(a.flags, FLAG_ACCEPT_SHAPE);
    return;
  }
  int64_t q_off, d_off;
  if (!prefix_offsets(a.draft_len, b, a.max_draft, &q_off, &d_off)) return;
  const int W = 1 + a.max_draft;
  for (int i = threadIdx.x; i <= D; i += blockDim.x) {
    const Cand* pc = a.part + ((size_t)b * W + i) * a.splits;
    float bv = pc[0].v;
    int bi = pc[0].i;
    for (int s = 1; s < a.splits; ++s)
      if (better(pc[s].v, pc[s].i, bv, bi)) {
        bv = pc[s].v;
        bi = pc[s].i;
      }
    if (bi == NONE) bi = 0;  // a row made only of NaN: unspecified, report index 0
    s_amax[i] = bi;
    if (a.target_tokens) a.target_tokens[q_off + i] = bi;
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
  int splits = 1;
  if (rows > 0) {
    const int64_t target = 4LL * num_sms;
    splits = (int)((target + rows - 1) / rows);
    const int cap = vocab / 8192 > 1 ? vocab / 8192 : 1;
    if (splits > cap) splits = cap;
    if (splits < 1) splits = 1;
  }
  w.splits = splits;
  w.ctrl = 0;
  w.part = 256;
  w.total = align_up(256 + sizeof(Cand) * (size_t)rows * splits, 256);
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
  a.splits = lay.splits;
  const dim3 grid((unsigned)(B * (1 + max_draft)), (unsigned)lay.splits);
  if (dtype == SV_BF16)
    argmax_partial_kernel<true><<<grid, ARGMAX_THREADS, 0, s>>>(a);
  else
    argmax_partial_kernel<false><<<grid, ARGMAX_THREADS, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  accept_finalize_kernel<<<B, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace sv

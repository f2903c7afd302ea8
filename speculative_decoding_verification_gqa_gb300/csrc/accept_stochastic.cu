// accept_stochastic.cu -- distribution-preserving acceptance ("GPU and LLM, chapter 5",
// "Speculative decoding (2)": the acceptance rule keeps the distribution of the output that
// of the large model alone). The rule with that property is the one of the paper that page
// cites (Leviathan, Kalman and Matias, "Fast Inference from Transformers via Speculative
// Decoding", 2023). With p the target's and q the drafter's softmax (logits divided by the
// temperature) at draft position j of a sequence, draft x_j is kept iff u_j q(x_j) <
// p(x_j), u_j uniform in [0, 1) (an input). At the first rejection the emitted token is
// drawn from the normalised max(0, p - q), or from p if every such weight is 0. With every
// draft kept, it is drawn from the target's row D_b. A token is drawn as the smallest index
// whose running sum of weights exceeds u_sample times their total.
//
// One CTA per sequence walks its draft positions in order. For each position, one pass
// over the target's and the drafter's rows gives both softmax normalisers (a running max
// and sum per thread, merged across the CTA); the decision needs p and q at x_j only, and
// every thread computes it alike. The draw reads its row once more: each thread sums the
// weights of a contiguous segment, a CTA-wide exclusive scan of the segment sums finds the
// first segment whose end passes u times the total, and that segment's thread walks it.
// Every loop is bounded by the row length; there are no waits.
#include <cuda_bf16.h>

#include "internal.cuh"

namespace sv {
namespace {

constexpr int ST_THREADS = 512;
constexpr int ST_WARPS = ST_THREADS / 32;

struct StArgs {
  const void* target;  // [sum_b (1 + D_b), V]
  const void* draft;   // [sum_b D_b, V]
  const int32_t* draft_tokens;
  const int32_t* draft_len;
  const float* u_accept;  // [sum_b D_b]
  const float* u_sample;  // [B]
  int32_t* accept_len;
  int32_t* next_token;
  uint32_t* flags;
  float inv_temp;
  int B, max_draft, vocab;
};

template <bool BF16>
__device__ __forceinline__ float logit(const void* base, int64_t row, int vocab, int k) {
  const int64_t i = row * vocab + k;
  if constexpr (BF16)
    return __uint_as_float((uint32_t)((const uint16_t*)base)[i] << 16);
  else
    return ((const float*)base)[i];
}

// Running max m and sum s of exp(x - m) (x = logit / temperature); -inf adds nothing.
struct MS {
  float m, s;
};
__device__ __forceinline__ void ms_add(MS& a, float x) {
  if (x == -INFINITY) return;
  if (x > a.m) {
    a.s = a.s * expf(a.m - x) + 1.f;  // a.m = -inf: a.s is 0 and stays 0 before the + 1
    a.m = x;
  } else {
    a.s += expf(x - a.m);
  }
}
__device__ __forceinline__ MS ms_merge(MS a, MS b) {
  if (b.m == -INFINITY) return a;
  if (a.m == -INFINITY) return b;
  const float m = fmaxf(a.m, b.m);
  return MS{m, a.s * expf(a.m - m) + b.s * expf(b.m - m)};
}
__device__ __forceinline__ MS ms_shfl(MS a, int o) {
  return MS{__shfl_xor_sync(0xffffffffu, a.m, o), __shfl_xor_sync(0xffffffffu, a.s, o)};
}

// Merges (a, c) over the CTA; every thread returns with the same two results (the warps'
// parts are folded in the same order by every thread).
__device__ void block_ms2(MS& a, MS& c, MS* sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = ms_merge(a, ms_shfl(a, o));
    c = ms_merge(c, ms_shfl(c, o));
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane == 0) {
    sh[wid] = a;
    sh[ST_WARPS + wid] = c;
  }
  __syncthreads();
  a = sh[0];
  c = sh[ST_WARPS];
  for (int w = 1; w < ST_WARPS; ++w) {
    a = ms_merge(a, sh[w]);
    c = ms_merge(c, sh[ST_WARPS + w]);
  }
  __syncthreads();  // sh is reused by the next call
}

// Sum of int64 values over the CTA (every thread gets it).
__device__ int64_t block_sum64(int64_t v, int64_t* sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
  __syncthreads();
  int64_t t = 0;
  for (int w = 0; w < ST_WARPS; ++w) t += sh[w];
  __syncthreads();
  return t;
}

// Draws from the weights weight(k) >= 0 of a row at u (see the file comment). Returns the
// token on every thread, or -1 if every weight is 0.
template <class Weight>
__device__ int draw(int vocab, float u, const Weight& weight, float* shf, int* shi) {
  const int seg = (vocab + ST_THREADS - 1) / ST_THREADS;
  const int k0 = min(vocab, (int)threadIdx.x * seg), k1 = min(vocab, k0 + seg);
  float sum = 0.f;
  int last = -1;  // last index of positive weight in the segment
  for (int k = k0; k < k1; ++k) {
    const float w = weight(k);
    sum += w;
    if (w > 0.f) last = k;
  }
  // exclusive scan of the segment sums in thread order
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  float incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) shf[wid] = incl;
  if (threadIdx.x == 0) {
    shi[0] = 0x7fffffff;  // first thread whose segment end passes the target
    shi[1] = -1;          // last index of positive weight in the row
    shi[2] = -1;          // the drawn token
  }
  __syncthreads();
  float before = 0.f, total = 0.f;
  for (int w = 0; w < ST_WARPS; ++w) {
    if (w < wid) before += shf[w];
    total += shf[w];
  }
  const float ex = before + incl - sum;
  const float target = u * total;
  if (sum > 0.f && target < ex + sum) atomicMin(&shi[0], (int)threadIdx.x);
  if (last >= 0) atomicMax(&shi[1], last);
  __syncthreads();
  if ((int)threadIdx.x == shi[0]) {
    float c = ex;
    int pick = last;
    for (int k = k0; k < k1; ++k) {
      const float w = weight(k);
      c += w;
      if (w > 0.f && c > target) {
        pick = k;
        break;
      }
    }
    shi[2] = pick;
  }
  __syncthreads();
  const int tok = shi[0] == 0x7fffffff ? shi[1] : shi[2];
  __syncthreads();  // shf and shi are reused by the next draw
  return tok;
}

template <bool BF16>
__global__ void __launch_bounds__(ST_THREADS) accept_stochastic_kernel(StArgs a) {
  __shared__ MS sh_ms[2 * ST_WARPS];
  __shared__ int64_t sh64[ST_WARPS];
  __shared__ float shf[ST_WARPS];
  __shared__ int shi[4];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, V = a.vocab;
  // this sequence's rows: q_off = sum over earlier sequences of (1 + D), d_off of D; every
  // length up to this one must be in range for the offsets to mean anything
  int64_t dsum = 0, nbad = 0;
  for (int bb = threadIdx.x; bb <= b; bb += ST_THREADS) {
    const int D = a.draft_len[bb];
    if (D < 0 || D > a.max_draft) ++nbad;
    if (bb < b) dsum += D;
  }
  nbad = block_sum64(nbad, sh64);
  const int64_t d_off = block_sum64(dsum, sh64);
  const int D = a.draft_len[b];
  if (nbad == 0) {
    for (int j = threadIdx.x; j < D; j += ST_THREADS) {
      const int x = a.draft_tokens[d_off + j];
      if (x < 0 || x >= V) ++nbad;
    }
    nbad = block_sum64(nbad, sh64);
  }
  if (nbad != 0) {  // leave this sequence's outputs untouched
    if (threadIdx.x == 0) atomicOr(a.flags, FLAG_ACCEPT_SHAPE);
    return;
  }
  const int64_t q_off = d_off + b;
  const float it = a.inv_temp;
  int n = D;  // drafts kept
  MS sp{-INFINITY, 0.f}, sq{-INFINITY, 0.f};
  for (int j = 0; j < D; ++j) {
    const int64_t tr = q_off + j, dr = d_off + j;
    sp = MS{-INFINITY, 0.f};
    sq = MS{-INFINITY, 0.f};
    for (int k = threadIdx.x; k < V; k += ST_THREADS) {
      ms_add(sp, logit<BF16>(a.target, tr, V, k) * it);
      ms_add(sq, logit<BF16>(a.draft, dr, V, k) * it);
    }
    block_ms2(sp, sq, sh_ms);
    const int x = a.draft_tokens[dr];
    const float px = expf(logit<BF16>(a.target, tr, V, x) * it - sp.m) / sp.s;
    const float qx = expf(logit<BF16>(a.draft, dr, V, x) * it - sq.m) / sq.s;
    if (!(a.u_accept[dr] * qx < px)) {  // the same decision on every thread
      n = j;
      break;
    }
  }
  const float us = a.u_sample[b];
  int tok = -1;
  if (n < D) {  // sp, sq hold row n's normalisers: draw from max(0, p - q)
    const int64_t tr = q_off + n, dr = d_off + n;
    const MS P = sp, Q = sq;
    auto resid = [&](int k) {
      const float pk = expf(logit<BF16>(a.target, tr, V, k) * it - P.m) / P.s;
      const float qk = expf(logit<BF16>(a.draft, dr, V, k) * it - Q.m) / Q.s;
      return fmaxf(pk - qk, 0.f);
    };
    tok = draw(V, us, resid, shf, shi);
  }
  if (tok < 0) {  // every draft kept (row D), or an all-zero residual (row n)
    const int64_t tr = q_off + (n < D ? n : D);
    if (n == D) {
      sp = MS{-INFINITY, 0.f};
      MS unused{-INFINITY, 0.f};
      for (int k = threadIdx.x; k < V; k += ST_THREADS) ms_add(sp, logit<BF16>(a.target, tr, V, k) * it);
      block_ms2(sp, unused, sh_ms);
    }
    const MS P = sp;
    auto prob = [&](int k) { return expf(logit<BF16>(a.target, tr, V, k) * it - P.m) / P.s; };
    tok = draw(V, us, prob, shf, shi);
  }
  if (threadIdx.x == 0) {
    a.accept_len[b] = n + 1;
    a.next_token[b] = tok;
  }
}

}  // namespace

cudaError_t launch_accept_stochastic(int B, int max_draft, int vocab, int dtype,
                                     const void* target, const void* draft,
                                     const int32_t* draft_tokens, const int32_t* draft_len,
                                     const float* u_accept, const float* u_sample,
                                     float inv_temp, int32_t* accept_len, int32_t* next_token,
                                     void* ws, cudaStream_t s) {
  StArgs a;
  a.target = target;
  a.draft = draft;
  a.draft_tokens = draft_tokens;
  a.draft_len = draft_len;
  a.u_accept = u_accept;
  a.u_sample = u_sample;
  a.accept_len = accept_len;
  a.next_token = next_token;
  a.flags = (uint32_t*)ws;
  a.inv_temp = inv_temp;
  a.B = B;
  a.max_draft = max_draft;
  a.vocab = vocab;
  return dtype == SV_BF16
             ? launch_pdl(accept_stochastic_kernel<true>, dim3(B), dim3(ST_THREADS), 0, s, a)
             : launch_pdl(accept_stochastic_kernel<false>, dim3(B), dim3(ST_THREADS), 0, s, a);
}

}  // namespace sv

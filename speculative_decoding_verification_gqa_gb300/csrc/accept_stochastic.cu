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
// One thread-block cluster of CL CTAs per sequence; CTA c of the cluster owns the vocabulary
// slice [c S, (c + 1) S). The cluster walks the sequence's draft positions in order:
//   * each CTA streams its slice of the target's and the drafter's row with 16-byte loads
//     (L2 prefetch of the next position's slices is issued at once) and reduces a running
//     max and sum of 2^t per row (t = logit / temperature in log2 units);
//   * the CTAs exchange their (max, sum) pairs through distributed shared memory at a
//     cluster barrier, and every CTA merges them in the same order, so every CTA holds the
//     same normalisers and takes the same keep / reject decision from p(x) and q(x);
//   * rows after the first rejection are never read.
// The draw: each thread sums the weights of a contiguous segment of its CTA's slice; the
// segment sums are scanned within the CTA and the CTA totals across the cluster; the CTA
// whose interval holds u times the total finds the thread, and that thread walks its
// segment. Every loop is bounded by the row length. There are no spin waits: the CTAs of a
// cluster meet only at hardware cluster barriers, which every CTA of the cluster reaches
// the same number of times because every branch between them is taken on values that all
// of them hold identically.
#include <cuda_bf16.h>

#include "internal.cuh"
#include "logits_vec.cuh"

namespace sv {
namespace {

constexpr int CL = 8;             // CTAs per cluster (one cluster per sequence)
constexpr int NT = 256;           // threads per CTA
constexpr int NW = NT / 32;
constexpr int UB = 8;             // 16-byte loads per row and thread in flight
constexpr float LOG2E = 1.4426950408889634f;

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
  float c2;    // log2(e) / temperature: logit -> t in log2 units
  int B, max_draft, vocab;
  int slice;   // vocabulary elements per CTA (a multiple of the vector width)
  int vec;     // 1: every row starts on a 16-byte boundary (vector loads)
};

template <bool BF16>
struct Vec {
  static constexpr int N = BF16 ? 8 : 4;  // elements per 16-byte vector
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// 2^(a - m) for a <= m, exactly 1 when a == m (the approximation of 2^0 is not exactly 1)
__device__ __forceinline__ float rescale(float a, float m) { return a == m ? 1.f : ex2(a - m); }

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster; writes to shared memory before it are visible
// to the other CTAs' distributed-shared-memory reads after it.
__device__ __forceinline__ void cluster_sync() {
  __syncwarp();  // the .aligned forms are executed by whole, converged warps
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
__device__ __forceinline__ float4 ld_remote(const float4* local, uint32_t rank) {
  uint32_t ra;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(saddr(local)), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(ra)
               : "memory");
  return v;
}

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

template <bool BF16>
__device__ __forceinline__ float logit(const void* base, int64_t row, int vocab, int k) {
  const int64_t i = row * vocab + k;
  if constexpr (BF16)
    return __uint_as_float((uint32_t)((const uint16_t*)base)[i] << 16);
  else
    return ((const float*)base)[i];
}
// Element e of a 16-byte vector.
template <bool BF16>
__device__ __forceinline__ float velem(const uint4& v, int e) {
  const uint32_t w = e / (BF16 ? 2 : 1) == 0 ? v.x
                     : e / (BF16 ? 2 : 1) == 1 ? v.y
                     : e / (BF16 ? 2 : 1) == 2 ? v.z : v.w;
  if constexpr (BF16) return bf16_at(w, e & 1);
  else return __uint_as_float(w);
}
template <bool BF16>
__device__ __forceinline__ float vmax(const uint4& v) {
  if constexpr (BF16) return vmax_bf16x8(v);
  else return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                    fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
}

// Running max m (log2 units) and sum s of 2^(t - m); empty: (-inf, 0).
struct MS {
  float m, s;
};
// The arithmetic of these reductions is spelled out with explicitly rounded operations, so
// no instance can be contracted into a fused multiply-add differently from another: merges
// are then exactly commutative (a + b == b + a in IEEE arithmetic), and two identical rows
// give bitwise identical normalisers wherever they are reduced.
__device__ __forceinline__ MS ms_merge(MS a, MS b) {
  const float m = fmaxf(a.m, b.m);
  const float fa = a.s > 0.f ? rescale(a.m, m) : 0.f;
  const float fb = b.s > 0.f ? rescale(b.m, m) : 0.f;
  return MS{m, __fadd_rn(__fmul_rn(a.s, fa), __fmul_rn(b.s, fb))};
}
__device__ __forceinline__ MS ms_shfl(MS a, int o) {
  return MS{__shfl_xor_sync(0xffffffffu, a.m, o), __shfl_xor_sync(0xffffffffu, a.s, o)};
}
// Adds values t_i (log2 units; -inf adds nothing) whose max is bm to (m, s).
__device__ __forceinline__ void ms_raise(MS& a, float bm) {
  if (bm > a.m) {
    a.s = a.s > 0.f ? __fmul_rn(a.s, ex2(__fsub_rn(a.m, bm))) : 0.f;
    a.m = bm;
  }
}

// This CTA's (max, sum) of one or two rows (target row tr; draft row dr when `two`) over
// the slice [k0, k1), reduced over the CTA; every thread returns the same values.
template <bool BF16>
__device__ __forceinline__ void slice_norms(const StArgs& a, int64_t tr, int64_t dr, bool two,
                                            int k0, int k1, MS& P, MS& Q, MS* sh) {
  constexpr int VN = Vec<BF16>::N;
  const int V = a.vocab, tid = threadIdx.x;
  const float c2 = a.c2;
  P = MS{-INFINITY, 0.f};
  Q = MS{-INFINITY, 0.f};
  if (a.vec) {
    const uint4* tp = reinterpret_cast<const uint4*>((const char*)a.target +
                                                     (tr * V + k0) * (BF16 ? 2 : 4));
    const uint4* dp = two ? reinterpret_cast<const uint4*>((const char*)a.draft +
                                                           (dr * V + k0) * (BF16 ? 2 : 4))
                          : tp;
    const int nv = (k1 - k0) / VN;
    for (int v0 = 0; v0 < nv; v0 += NT * UB) {
      uint4 tv[UB], dv[UB];
#pragma unroll
      for (int i = 0; i < UB; ++i) {
        const int v = v0 + i * NT + tid;
        if (v < nv) {
          tv[i] = ld_stream(tp + v);
          if (two) dv[i] = ld_stream(dp + v);
        }
      }
      float bt = -INFINITY, bd = -INFINITY;
#pragma unroll
      for (int i = 0; i < UB; ++i)
        if (v0 + i * NT + tid < nv) {
          bt = fmaxf(bt, vmax<BF16>(tv[i]));
          if (two) bd = fmaxf(bd, vmax<BF16>(dv[i]));
        }
      ms_raise(P, __fmul_rn(bt, c2));
      if (two) ms_raise(Q, __fmul_rn(bd, c2));
      const float nmp = P.m == -INFINITY ? 0.f : -P.m, nmq = Q.m == -INFINITY ? 0.f : -Q.m;
#pragma unroll
      for (int i = 0; i < UB; ++i)
        if (v0 + i * NT + tid < nv) {
#pragma unroll
          for (int e = 0; e < VN; ++e) {
            P.s = __fadd_rn(P.s, ex2(__fmaf_rn(velem<BF16>(tv[i], e), c2, nmp)));
            if (two) Q.s = __fadd_rn(Q.s, ex2(__fmaf_rn(velem<BF16>(dv[i], e), c2, nmq)));
          }
        }
    }
  } else {
    for (int k = k0 + tid; k < k1; k += NT) {
      const float t = __fmul_rn(logit<BF16>(a.target, tr, V, k), c2);
      ms_raise(P, t);
      if (P.m != -INFINITY) P.s = __fadd_rn(P.s, ex2(__fsub_rn(t, P.m)));
      if (two) {
        const float d = __fmul_rn(logit<BF16>(a.draft, dr, V, k), c2);
        ms_raise(Q, d);
        if (Q.m != -INFINITY) Q.s = __fadd_rn(Q.s, ex2(__fsub_rn(d, Q.m)));
      }
    }
  }
  // A row of -inf alone keeps (-inf, 0); a -inf element adds 2^-inf = 0.
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    P = ms_merge(P, ms_shfl(P, o));
    Q = ms_merge(Q, ms_shfl(Q, o));
  }
  const int lane = tid & 31, w = tid >> 5;
  if (lane == 0) {
    sh[w] = P;
    sh[NW + w] = Q;
  }
  __syncthreads();
  P = sh[0];
  Q = sh[NW];
  for (int i = 1; i < NW; ++i) {
    P = ms_merge(P, sh[i]);
    Q = ms_merge(Q, sh[NW + i]);
  }
  __syncthreads();  // sh is reused by the next call
}

// Exchange of one float4 per CTA through distributed shared memory: each CTA publishes
// `mine`, and every CTA returns all CL values in rank order (the same in every CTA).
// `slots` has two buffers of CL entries, used alternately (`round` parity), so a fast CTA
// never overwrites values a slower one has yet to read: it can only start round r + 2 after
// every CTA has reached the barrier of round r + 1, i.e. finished reading round r.
__device__ __forceinline__ void exchange(float4 mine, float4 (*slots)[CL], uint32_t& round, float4* all) {
  const uint32_t rank = cluster_rank();
  float4* buf = slots[round & 1];
  if (threadIdx.x == 0) buf[rank] = mine;
  cluster_sync();
#pragma unroll
  for (int c = 0; c < CL; ++c) all[c] = ld_remote(&buf[c], (uint32_t)c);  // CTA c's own slot
  ++round;
}

// The weight of token k: max(0, p_k - q_k) (residual) or p_k up to a constant factor.
template <bool BF16>
struct Weight {
  const void* target;
  const void* draft;
  int vocab;
  float c2;
  int64_t tr, dr;
  float pm, pinv, qm, qinv;
  bool residual;
  // from the two logits (p and q by the same explicitly rounded steps: identical rows give
  // p_k - q_k = 0)
  __device__ __forceinline__ float eval(float lt, float ld) const {
    const float p = __fmul_rn(ex2(__fmaf_rn(lt, c2, -pm)), pinv);
    if (!residual) return p;
    const float q = __fmul_rn(ex2(__fmaf_rn(ld, c2, -qm)), qinv);
    return fmaxf(__fsub_rn(p, q), 0.f);
  }
  __device__ __forceinline__ float operator()(int k) const {
    return eval(logit<BF16>(target, tr, vocab, k),
                residual ? logit<BF16>(draft, dr, vocab, k) : 0.f);
  }
};

constexpr int DV = 8;  // vectors per row loaded at once by a drawing thread

// Visits the weights of tokens [s0, s1) in token order: f(k, w) returns true to stop.
// With 16-byte rows (vec) s0 is a multiple of the vector width and the segment is read
// DV vectors per row at a time, every load of a chunk issued before the first is used.
template <bool BF16, class F>
__device__ __forceinline__ void visit(const Weight<BF16>& wt, bool vec, int s0, int s1, F&& f) {
  constexpr int VN = Vec<BF16>::N;
  if (vec) {
    const uint4* tp = reinterpret_cast<const uint4*>(
        (const char*)wt.target + (wt.tr * wt.vocab + s0) * (BF16 ? 2 : 4));
    const uint4* dp = reinterpret_cast<const uint4*>(
        (const char*)wt.draft + (wt.dr * wt.vocab + s0) * (BF16 ? 2 : 4));
    const int nv = (s1 - s0 + VN - 1) / VN;  // the last vector may end past s1 (not past V)
    for (int i0 = 0; i0 < nv; i0 += DV) {
      uint4 tv[DV], dv[DV];
#pragma unroll
      for (int i = 0; i < DV; ++i)
        if (i0 + i < nv) {
          tv[i] = tp[i0 + i];
          if (wt.residual) dv[i] = dp[i0 + i];
        }
#pragma unroll
      for (int i = 0; i < DV; ++i)
        if (i0 + i < nv) {
#pragma unroll
          for (int e = 0; e < VN; ++e) {
            const int k = s0 + (i0 + i) * VN + e;
            if (k < s1 && f(k, wt.eval(velem<BF16>(tv[i], e),
                                       wt.residual ? velem<BF16>(dv[i], e) : 0.f)))
              return;
          }
        }
    }
  } else {
#pragma unroll 8
    for (int k = s0; k < s1; ++k)
      if (f(k, wt(k))) return;
  }
}

// Draws from the weights over the whole row (all CTAs of the cluster take part). Returns
// -1 on every CTA if every weight is 0; otherwise the drawing CTA writes the token to
// *out and the function returns 0.
template <bool BF16>
__device__ __forceinline__ int cluster_draw(const Weight<BF16>& wt, bool vec, float u, int k0,
                                            int k1, float4 (*slots)[CL], uint32_t& round,
                                            float* shf, int* shi, int32_t* out) {
  constexpr int VN = Vec<BF16>::N;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int n = max(k1 - k0, 0);
  int seg = (n + NT - 1) / NT;
  if (vec) seg = (seg + VN - 1) / VN * VN;  // segments of whole vectors
  const int s0 = min(k0 + tid * seg, k1), s1 = min(s0 + seg, k1);
  float sum = 0.f;
  int last = -1;
  visit<BF16>(wt, vec, s0, s1, [&](int k, float w) {
    sum = __fadd_rn(sum, w);
    if (w > 0.f) last = k;
    return false;
  });
  // exclusive scan of the segment sums in thread order
  float incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int lmax = last;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lmax = max(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
  if (lane == 31) shf[wid] = incl;
  if (lane == 0) shi[wid] = lmax;
  __syncthreads();
  float before = 0.f, ctot = 0.f;
  int clast = -1;
  for (int w = 0; w < NW; ++w) {
    if (w < wid) before += shf[w];
    ctot += shf[w];
    clast = max(clast, shi[w]);
  }
  const float ex = before + incl - sum;
  __syncthreads();
  float4 all[CL];
  exchange(make_float4(ctot, __int_as_float(clast), 0.f, 0.f), slots, round, all);
  float pre = 0.f, total = 0.f;
  int glast = -1;
  for (int c = 0; c < CL; ++c) {
    total += all[c].x;
    glast = max(glast, __float_as_int(all[c].y));
  }
  if (!(total > 0.f)) return -1;  // the same on every CTA
  const float target = u * total;
  int cstar = -1;
  for (int c = 0; c < CL; ++c) {
    if (cstar < 0 && all[c].x > 0.f && target < pre + all[c].x) cstar = c;
    if (cstar < 0) pre += all[c].x;
  }
  const uint32_t rank = cluster_rank();
  if (cstar < 0) {  // rounding left the target at the end: the last token of positive weight
    if (rank == 0 && tid == 0) *out = glast;
    return 0;
  }
  if ((int)rank != cstar) return 0;
  const float tl = target - pre;
  if (tid == 0) shi[NW] = 0x7fffffff;
  __syncthreads();
  if (sum > 0.f && tl < ex + sum) atomicMin(&shi[NW], tid);
  __syncthreads();
  const int who = shi[NW];
  if (who == 0x7fffffff) {
    if (tid == 0) *out = clast;
  } else if (tid == who) {
    float c = ex;
    int pick = last;
    visit<BF16>(wt, vec, s0, s1, [&](int k, float w) {
      c = __fadd_rn(c, w);
      if (w > 0.f && c > tl) {
        pick = k;
        return true;
      }
      return false;
    });
    *out = pick;
  }
  return 0;
}

template <bool BF16>
__global__ void __launch_bounds__(NT) accept_stochastic_kernel(StArgs a) {
  __shared__ MS sh_ms[2 * NW];
  __shared__ float4 slots[2][CL];
  __shared__ float shf[NW];
  __shared__ int shi[NW + 1];
  __shared__ int64_t sh64[NW];
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x;
  const int b = blockIdx.x / CL;
  const uint32_t rank = cluster_rank();
  const int V = a.vocab;
  if (cluster_size() != CL || rank != blockIdx.x % CL) {  // launched without its cluster shape
    if (tid == 0) atomicOr(a.flags, FLAG_ACCEPT_SHAPE);
    return;  // (before any cluster barrier or remote access)
  }

  // this sequence's rows: d_off = sum of D over earlier sequences, q_off = d_off + b. Every
  // length up to this one must be in range for the offsets to mean anything. Every CTA of
  // the cluster computes the same sums, so all of them return here together or none does.
  auto block_sum = [&](int64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((tid & 31) == 0) sh64[tid >> 5] = v;
    __syncthreads();
    int64_t t = 0;
    for (int w = 0; w < NW; ++w) t += sh64[w];
    __syncthreads();
    return t;
  };
  int64_t dsum = 0, nbad = 0;
  for (int bb = tid; bb <= b; bb += NT) {
    const int D = a.draft_len[bb];
    if (D < 0 || D > a.max_draft) ++nbad;
    if (bb < b) dsum += D;
  }
  nbad = block_sum(nbad);
  const int64_t d_off = block_sum(dsum);
  const int D = a.draft_len[b];
  if (nbad == 0) {
    for (int j = tid; j < D; j += NT) {
      const int x = a.draft_tokens[d_off + j];
      if (x < 0 || x >= V) ++nbad;
    }
    nbad = block_sum(nbad);
  }
  if (nbad != 0) {  // leave this sequence's outputs untouched
    if (rank == 0 && tid == 0) atomicOr(a.flags, FLAG_ACCEPT_SHAPE);
    return;
  }
  const int64_t q_off = d_off + b;
  const int k0 = min((int)rank * a.slice, V), k1 = min(k0 + a.slice, V);
  const uint32_t esz = BF16 ? 2 : 4;
  auto prefetch_rows = [&](int64_t tr, int64_t dr, bool two) {
    if (a.vec && tid == 0 && k1 > k0) {
      const uint32_t bytes = (uint32_t)(k1 - k0) * esz;
      prefetch_l2((const char*)a.target + (tr * V + k0) * esz, bytes);
      if (two) prefetch_l2((const char*)a.draft + (dr * V + k0) * esz, bytes);
    }
  };
  uint32_t round = 0;
  float4 all[CL];
  auto cluster_norms = [&](MS& P, MS& Q) {  // merge every CTA's parts in rank order
    exchange(make_float4(P.m, P.s, Q.m, Q.s), slots, round, all);
    P = MS{all[0].x, all[0].y};
    Q = MS{all[0].z, all[0].w};
    for (int c = 1; c < CL; ++c) {
      P = ms_merge(P, MS{all[c].x, all[c].y});
      Q = ms_merge(Q, MS{all[c].z, all[c].w});
    }
  };

  int n = D;  // drafts kept
  MS P, Q;
  prefetch_rows(q_off, d_off, D > 0);
  for (int j = 0; j < D; ++j) {
    const int64_t tr = q_off + j, dr = d_off + j;
    // what the decision needs besides the normalisers, loaded before the rows stream
    const int x = a.draft_tokens[dr];
    const float lx = logit<BF16>(a.target, tr, V, x), dx = logit<BF16>(a.draft, dr, V, x);
    const float ua = a.u_accept[dr];
    slice_norms<BF16>(a, tr, dr, true, k0, k1, P, Q, sh_ms);
    prefetch_rows(tr + 1, dr + 1, j + 1 < D);  // the next position's rows (the bonus row last)
    cluster_norms(P, Q);
    const float px = __fdiv_rn(ex2(__fmaf_rn(lx, a.c2, -P.m)), P.s);
    const float qx = __fdiv_rn(ex2(__fmaf_rn(dx, a.c2, -Q.m)), Q.s);
    if (!(__fmul_rn(ua, qx) < px)) {  // the same decision on every thread of the cluster
      n = j;
      break;
    }
  }
  const float us = a.u_sample[b];
  int status = -1;
  if (n < D) {  // P, Q hold row n's normalisers: draw from max(0, p - q)
    const Weight<BF16> w{a.target, a.draft, V, a.c2, q_off + n, d_off + n,
                         P.m, __frcp_rn(P.s), Q.m, __frcp_rn(Q.s), true};
    status = cluster_draw<BF16>(w, a.vec, us, k0, k1, slots, round, shf, shi, a.next_token + b);
  }
  if (status < 0) {  // every draft kept (row D), or an all-zero residual (row n)
    const int64_t tr = q_off + n;
    if (n == D) {
      MS unused;
      slice_norms<BF16>(a, tr, 0, false, k0, k1, P, unused, sh_ms);
      cluster_norms(P, unused);
    }
    const Weight<BF16> w{a.target, a.draft, V, a.c2, tr, 0, P.m, 1.f, 0.f, 0.f, false};
    cluster_draw<BF16>(w, a.vec, us, k0, k1, slots, round, shf, shi, a.next_token + b);
  }
  if (rank == 0 && tid == 0) a.accept_len[b] = n + 1;
  cluster_sync();  // no CTA leaves while another may still read its shared memory
}

template <bool BF16>
cudaError_t launch_st(const StArgs& a, cudaStream_t s) {
  if (take_injected_launch_failure()) return cudaErrorLaunchFailure;  // nothing launched
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.B * CL);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CL;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, accept_stochastic_kernel<BF16>, a);
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
  a.c2 = inv_temp * LOG2E;
  a.B = B;
  a.max_draft = max_draft;
  a.vocab = vocab;
  const bool bf16 = dtype == SV_BF16;
  const int vn = bf16 ? 8 : 4;
  const uintptr_t al = 16;
  a.vec = vocab % vn == 0 && ((uintptr_t)target % al) == 0 &&
          (draft == nullptr || ((uintptr_t)draft % al) == 0);
  // slices of whole vectors: every slice of an aligned row starts on a 16-byte boundary
  a.slice = ((vocab + CL - 1) / CL + vn - 1) / vn * vn;
  return bf16 ? launch_st<true>(a, s) : launch_st<false>(a, s);
}

}  // namespace sv

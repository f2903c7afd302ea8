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
// slice [c S, (c + 1) S). The cluster walks the sequence's draft positions in rounds of R:
//   * each CTA streams its slice of the target's and the drafter's rows of the round's
//     positions with 16-byte loads, all rows' loads in flight together (the slices of the
//     positions ahead are prefetched into L2), and reduces a running max and sum of 2^t
//     per row (t = logit / temperature in log2 units);
//   * each CTA stores its (max, sum) pairs into every CTA's shared memory (distributed
//     shared memory) before one cluster barrier per round, after which every CTA merges
//     them from its own shared memory in the same order, so every CTA
//     holds the same normalisers and takes the same keep / reject decisions from p(x) and
//     q(x), in order, up to the first rejection;
//   * rows of positions after the first rejection are read at most by the round that
//     holds it and the prefetch window.
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
constexpr int R = 1;              // draft positions reduced per round
constexpr int UBR = 8;            // 16-byte loads per row and thread in flight (2 R rows)
constexpr int PF = 4;             // draft positions whose rows are prefetched ahead
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
// Every thread of every CTA of the cluster; writes to the cluster's shared memory before it
// (a CTA's own or, through distributed shared memory, another's) are visible to every
// thread of the cluster after it.
// Only thread 0 of a CTA writes what other CTAs read (the exchange slots), so only warp 0
// arrives with release semantics.
__device__ __forceinline__ void cluster_sync() {
  __syncwarp();  // the .aligned forms are executed by whole, converged warps
  if ((threadIdx.x >> 5) == 0)
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  else
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Stores v at the address of `local` in the shared memory of CTA `rank` of the cluster.
__device__ __forceinline__ void st_remote(float4* local, uint32_t rank, const float4& v) {
  uint32_t ra;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(saddr(local)), "r"(rank));
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(ra), "f"(v.x),
               "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
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

template <int N>
__device__ __forceinline__ void cta_merge(MS (&acc)[N], MS* sh);

// This CTA's (max, sum) over the slice [k0, k1) of NR = 2 R rows at once (the target's and
// the drafter's row of R draft positions; row r is read only where use[r]), reduced over
// the CTA; every thread returns the same values. The rows' loads are issued together, UBR
// vectors per row and thread, so their latencies overlap.
template <bool BF16>
__device__ __forceinline__ void round_norms(const StArgs& a, const int64_t (&row)[2 * R],
                                            const bool (&use)[2 * R], int k0, int k1,
                                            MS (&acc)[2 * R], MS* sh) {
  constexpr int VN = Vec<BF16>::N, NR = 2 * R;
  const int V = a.vocab, tid = threadIdx.x;
  const float c2 = a.c2;
#pragma unroll
  for (int r = 0; r < NR; ++r) acc[r] = MS{-INFINITY, 0.f};
  if (a.vec) {
    const uint4* base[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r)
      base[r] = reinterpret_cast<const uint4*>((const char*)((r & 1) ? a.draft : a.target) +
                                               (row[r] * V + k0) * (BF16 ? 2 : 4));
    const int nv = (k1 - k0) / VN;
    for (int v0 = 0; v0 < nv; v0 += NT * UBR) {
      uint4 w[NR][UBR];
#pragma unroll
      for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int i = 0; i < UBR; ++i) {
          const int v = v0 + i * NT + tid;
          if (use[r] && v < nv) w[r][i] = ld_stream(base[r] + v);
        }
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        if (!use[r]) continue;
        float bm = -INFINITY;
#pragma unroll
        for (int i = 0; i < UBR; ++i)
          if (v0 + i * NT + tid < nv) bm = fmaxf(bm, vmax<BF16>(w[r][i]));
        ms_raise(acc[r], __fmul_rn(bm, c2));
        const float nm = acc[r].m == -INFINITY ? 0.f : -acc[r].m;
#pragma unroll
        for (int i = 0; i < UBR; ++i)
          if (v0 + i * NT + tid < nv) {  // a vector's terms summed as a tree (depth 3)
            float t[VN];
#pragma unroll
            for (int e = 0; e < VN; ++e) t[e] = ex2(__fmaf_rn(velem<BF16>(w[r][i], e), c2, nm));
#pragma unroll
            for (int h = VN / 2; h > 0; h >>= 1)
#pragma unroll
              for (int e = 0; e < h; ++e) t[e] = __fadd_rn(t[e], t[e + h]);
            acc[r].s = __fadd_rn(acc[r].s, t[0]);
          }
      }
    }
  } else {
    for (int k = k0 + tid; k < k1; k += NT) {
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        if (!use[r]) continue;
        const float t = __fmul_rn(logit<BF16>((r & 1) ? a.draft : a.target, row[r], V, k), c2);
        ms_raise(acc[r], t);
        if (acc[r].m != -INFINITY) acc[r].s = __fadd_rn(acc[r].s, ex2(__fsub_rn(t, acc[r].m)));
      }
    }
  }
  cta_merge<NR>(acc, sh);
}

// Threads' parts (acc, the same count N on every thread) merged over the CTA; every thread
// returns the same values.
template <int N>
__device__ __forceinline__ void cta_merge(MS (&acc)[N], MS* sh) {
  const int tid = threadIdx.x;
  // A row of -inf alone keeps (-inf, 0); a -inf element adds 2^-inf = 0.
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int r = 0; r < N; ++r) acc[r] = ms_merge(acc[r], ms_shfl(acc[r], o));
  const int lane = tid & 31, wid = tid >> 5;
  if (lane == 0)
#pragma unroll
    for (int r = 0; r < N; ++r) sh[r * NW + wid] = acc[r];
  __syncthreads();
  // the NW warp parts merged as a tree over lanes 0 .. NW - 1 of every warp: the same
  // operations in the same order in every warp, so every thread holds the same result
#pragma unroll
  for (int r = 0; r < N; ++r) {
    MS v = lane < NW ? sh[r * NW + lane] : MS{-INFINITY, 0.f};
#pragma unroll
    for (int o = NW / 2; o > 0; o >>= 1) v = ms_merge(v, ms_shfl(v, o));
    acc[r] = MS{__shfl_sync(0xffffffffu, v.m, 0), __shfl_sync(0xffffffffu, v.s, 0)};
  }
  __syncthreads();  // sh is reused by the next call
}

// One position's row slices, one batch (every vector of the thread at once): the loads of
// the target's row tr and, when `two`, the drafter's row dr.
template <bool BF16>
__device__ __forceinline__ void issue_rows(const StArgs& a, int64_t tr, int64_t dr, bool two,
                                           int k0, int nv, uint4 (&tv)[UBR], uint4 (&dv)[UBR]) {
  const int V = a.vocab, tid = threadIdx.x;
  const uint4* tp = reinterpret_cast<const uint4*>((const char*)a.target + (tr * V + k0) * (BF16 ? 2 : 4));
  const uint4* dp = reinterpret_cast<const uint4*>((const char*)a.draft + (dr * V + k0) * (BF16 ? 2 : 4));
#pragma unroll
  for (int i = 0; i < UBR; ++i) {
    const int v = i * NT + tid;
    if (v < nv) {
      tv[i] = ld_stream(tp + v);
      if (two) dv[i] = ld_stream(dp + v);
    }
  }
}

// The thread's (max, sum) parts of the vectors loaded by issue_rows.
template <bool BF16>
__device__ __forceinline__ void thread_parts(const uint4 (&tv)[UBR], const uint4 (&dv)[UBR],
                                             bool two, int nv, float c2, MS (&acc)[2]) {
  constexpr int VN = Vec<BF16>::N;
  const int tid = threadIdx.x;
  acc[0] = MS{-INFINITY, 0.f};
  acc[1] = MS{-INFINITY, 0.f};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (r == 1 && !two) continue;
    const uint4(&w)[UBR] = r ? dv : tv;
    float bm = -INFINITY;
#pragma unroll
    for (int i = 0; i < UBR; ++i)
      if (i * NT + tid < nv) bm = fmaxf(bm, vmax<BF16>(w[i]));
    ms_raise(acc[r], __fmul_rn(bm, c2));
    const float nm = acc[r].m == -INFINITY ? 0.f : -acc[r].m;
#pragma unroll
    for (int i = 0; i < UBR; ++i)
      if (i * NT + tid < nv) {  // a vector's terms summed as a tree (depth 3)
        float t[VN];
#pragma unroll
        for (int e = 0; e < VN; ++e) t[e] = ex2(__fmaf_rn(velem<BF16>(w[i], e), c2, nm));
#pragma unroll
        for (int h = VN / 2; h > 0; h >>= 1)
#pragma unroll
          for (int e = 0; e < h; ++e) t[e] = __fadd_rn(t[e], t[e + h]);
        acc[r].s = __fadd_rn(acc[r].s, t[0]);
      }
  }
}

// Exchange of N float4 per CTA through distributed shared memory: each CTA stores `mine`
// into its slot of every CTA's buffer (its own included) before the cluster barrier, and
// after it every CTA reads all CL x N values from its own shared memory, in rank order
// (the same in every CTA). `slots` has two buffers, used alternately (`round` parity), so
// a fast CTA never overwrites values a slower one has yet to read: it can only start round
// r + 2 after every CTA has reached the barrier of round r + 1, i.e. finished reading
// round r.
template <int N>
__device__ __forceinline__ void exchange(const float4 (&mine)[N], float4 (*slots)[CL][R],
                                         uint32_t& round, float4 (&all)[CL][N]) {
  const uint32_t rank = cluster_rank();
  float4 (*buf)[R] = slots[round & 1];
  if (threadIdx.x == 0)
#pragma unroll
    for (int c = 0; c < CL; ++c)
#pragma unroll
      for (int n = 0; n < N; ++n) st_remote(&buf[rank][n], (uint32_t)c, mine[n]);
  cluster_sync();
#pragma unroll
  for (int c = 0; c < CL; ++c)
#pragma unroll
    for (int n = 0; n < N; ++n) all[c][n] = buf[c][n];  // CTA c's slot, stored here by CTA c
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
                                            int k1, float4 (*slots)[CL][R], uint32_t& round,
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
  float4 all[CL][1];
  const float4 mine[1] = {make_float4(ctot, __int_as_float(clast), 0.f, 0.f)};
  exchange<1>(mine, slots, round, all);
  float pre = 0.f, total = 0.f;
  int glast = -1;
  for (int c = 0; c < CL; ++c) {
    total += all[c][0].x;
    glast = max(glast, __float_as_int(all[c][0].y));
  }
  if (!(total > 0.f)) return -1;  // the same on every CTA
  const float target = u * total;
  int cstar = -1;
  for (int c = 0; c < CL; ++c) {
    if (cstar < 0 && all[c][0].x > 0.f && target < pre + all[c][0].x) cstar = c;
    if (cstar < 0) pre += all[c][0].x;
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

// Two CTAs per SM (at most 128 registers a thread), so that the clusters of a batch of up to
// 2 x SMs / CL sequences are resident at once.
// PIPE: rows start on 16-byte boundaries and a CTA's slice of a row is one batch per thread
// (the next position's loads are issued during this one's reductions).
template <bool BF16, bool PIPE>
__global__ void __launch_bounds__(NT, 2) accept_stochastic_kernel(StArgs a) {
  __shared__ MS sh_ms[2 * R * NW];
  __shared__ float4 slots[2][CL][R];
  __shared__ float s_lx[256], s_dx[256], s_ua[256];  // per draft position (D <= 255)
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
  // L2 prefetch of position j's rows (the target's bonus row for j = D); rows of positions
  // after the first rejection may be fetched for nothing (at most the window's)
  auto prefetch_pos = [&](int j) {
    if (j <= D) prefetch_rows(q_off + j, d_off + j, j < D);
  };
  for (int j = 0; j < PF; ++j) prefetch_pos(j);

  // What each decision needs besides the normalisers (the drafted token's two logits and
  // its uniform), loaded for every position at once.
  for (int j = tid; j < D; j += NT) {
    const int x = a.draft_tokens[d_off + j];
    s_lx[j] = logit<BF16>(a.target, q_off + j, V, x);
    s_dx[j] = logit<BF16>(a.draft, d_off + j, V, x);
    s_ua[j] = a.u_accept[d_off + j];
  }
  // Positions in order, each: every CTA reduces its slice of the position's rows (the
  // target's and the drafter's row of a draft position, the target's row alone for the
  // bonus position D), the CTAs exchange and merge their parts in rank order, and the
  // draft is decided. With 16-byte rows whose slice is one batch per thread, the next
  // position's loads are issued as soon as this position's vectors are consumed, so they
  // are in flight during its reductions and exchange.
  const int nv = PIPE ? (k1 - k0) / Vec<BF16>::N : 0;
  uint4 tv[PIPE ? UBR : 1], dv[PIPE ? UBR : 1];
  if constexpr (PIPE) issue_rows<BF16>(a, q_off, d_off, D > 0, k0, nv, tv, dv);
  // every CTA of the cluster is running before the first exchange stores into its shared
  // memory (all of them get here: the checks above return in all of them or in none)
  cluster_sync();
  int n = D;  // drafts kept
  MS P, Q;    // normalisers of row n (the draw's row)
  for (int j = 0; j <= D; ++j) {
    prefetch_pos(j + PF);
    MS acc[2];
    if constexpr (PIPE) {
      thread_parts<BF16>(tv, dv, j < D, nv, a.c2, acc);
      if (j + 1 <= D) issue_rows<BF16>(a, q_off + j + 1, d_off + j + 1, j + 1 < D, k0, nv, tv, dv);
      cta_merge<2>(acc, sh_ms);
    } else {
      const int64_t row[2] = {q_off + j, d_off + j};
      const bool use[2] = {true, j < D};
      round_norms<BF16>(a, row, use, k0, k1, acc, sh_ms);
    }
    float4 mine[1], all[CL][1];
    mine[0] = make_float4(acc[0].m, acc[0].s, acc[1].m, acc[1].s);
    exchange<1>(mine, slots, round, all);
    // every CTA's part, merged as a tree over lanes 0 .. CL - 1 (the same in every warp of
    // every CTA)
    const int lane = tid & 31;
    float4 mc = all[0][0];
#pragma unroll
    for (int c = 1; c < CL; ++c)
      if (lane == c) mc = all[c][0];
    P = lane < CL ? MS{mc.x, mc.y} : MS{-INFINITY, 0.f};
    Q = lane < CL ? MS{mc.z, mc.w} : MS{-INFINITY, 0.f};
#pragma unroll
    for (int o = CL / 2; o > 0; o >>= 1) {
      P = ms_merge(P, ms_shfl(P, o));
      Q = ms_merge(Q, ms_shfl(Q, o));
    }
    P = MS{__shfl_sync(0xffffffffu, P.m, 0), __shfl_sync(0xffffffffu, P.s, 0)};
    Q = MS{__shfl_sync(0xffffffffu, Q.m, 0), __shfl_sync(0xffffffffu, Q.s, 0)};
    if (j == D) break;  // every draft kept: P is the bonus row's normaliser
    const float px = __fdiv_rn(ex2(__fmaf_rn(s_lx[j], a.c2, -P.m)), P.s);
    const float qx = __fdiv_rn(ex2(__fmaf_rn(s_dx[j], a.c2, -Q.m)), Q.s);
    if (!(__fmul_rn(s_ua[j], qx) < px)) {  // the same decision on every thread of the cluster
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
  if (status < 0) {  // every draft kept (row D: P already holds it), or an all-zero residual
    const Weight<BF16> w{a.target, a.draft, V, a.c2, q_off + n, 0, P.m, 1.f, 0.f, 0.f, false};
    cluster_draw<BF16>(w, a.vec, us, k0, k1, slots, round, shf, shi, a.next_token + b);
  }
  if (rank == 0 && tid == 0) a.accept_len[b] = n + 1;
  cluster_sync();  // no CTA leaves while another may still read its shared memory
}

template <bool BF16, bool PIPE>
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
  return cudaLaunchKernelEx(&cfg, accept_stochastic_kernel<BF16, PIPE>, a);
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
  const bool pipe = a.vec && a.slice / vn <= NT * UBR;
  if (bf16) return pipe ? launch_st<true, true>(a, s) : launch_st<true, false>(a, s);
  return pipe ? launch_st<false, true>(a, s) : launch_st<false, false>(a, s);
}

}  // namespace sv

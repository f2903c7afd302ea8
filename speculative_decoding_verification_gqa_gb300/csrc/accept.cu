// accept.cu -- greedy acceptance ("Co-Designing AI Models Using Speculative Decoding",
// basic structure: keep the drafts up to the first mismatch; "GPU and LLM, chapter 5",
// "Speculative decoding (2)": the target's own token takes the place of the first
// rejected draft).
//
// One kernel of persistent CTAs, each scanning an equal contiguous range of the packed
// logits. When rows are whole 32-byte vectors (and the logits 32-byte aligned) the range is
// one stream of 32-byte vectors that runs across row boundaries, so a CTA's loads do not
// drain at every row end: a batch is taken in one pass per row it touches, and a row that
// ends inside it is reduced before the next row's pass. Otherwise the range is scanned row
// by row with 16-byte loads and scalar heads and tails. Either way only each vector's
// maximum (packed max instructions) is compared, without branches, the best vector and its
// words are kept, and the element index inside it is resolved once per row. Warp-shuffle
// reductions with the comparator "larger value wins, equal values: smaller index wins"
// give one candidate per warp and row, folded into the row's 64-bit key (order-preserving
// value bits above the inverted index) with one atomicMax. Values are compared exactly in
// fp32 (bf16 widens exactly). Every CTA stages the drafts in shared memory while it scans;
// the last CTA to finish (a completion ticket in the workspace) reads and clears every
// row's key, which is the target's token, and, per sequence, finds the first position
// whose draft differs from it.
#include <cuda_bf16.h>

#include "internal.cuh"
#include "logits_vec.cuh"

namespace sv {
namespace {

constexpr int ARGMAX_THREADS = 512;
// Two CTAs of 512 threads per SM, each thread with eight 16-byte loads in flight (64
// registers): measured faster than four CTAs with four loads each (32 registers).
constexpr int ARGMAX_CTAS_PER_SM = 2;
constexpr int UNROLL = 8;
constexpr int NONE = 0x7fffffff;  // "no candidate yet"
// Continuous scan: FLAT_U 32-byte vectors per thread per batch (ARGMAX_THREADS * FLAT_U
// vectors, 64 KB per CTA); measured faster than 16-byte vectors eight at a time, and than
// issuing the next batch before processing the current one.
constexpr int FLAT_U = 4;
constexpr int VW = 8;       // 32-bit words per vector
constexpr int VB = VW * 4;  // bytes per vector
constexpr int64_t FLAT_BATCH_VECS = (int64_t)ARGMAX_THREADS * FLAT_U;

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

__device__ __forceinline__ void warp_argmax(float& bv, int& bi) {
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


// Row key: the value's bits mapped to an unsigned integer of the same order (-0 taken as
// +0, so the two tie) above 0xffffffff - index, so a larger key is a larger value or the
// same value at a smaller index. 0 means "no candidate" (below every value's key).
__device__ __forceinline__ unsigned long long row_key(float v, int i) {
  uint32_t u = v == 0.f ? 0u : __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (0xffffffffu - (uint32_t)i);
}
__device__ __forceinline__ int key_index(unsigned long long k) {
  return (int)(0xffffffffu - (uint32_t)k);
}

struct AcceptArgs {
  const void* logits;
  const int32_t* draft_tokens;
  const int32_t* draft_len;
  int32_t* accept_len;
  int32_t* next_token;
  int32_t* target_tokens;
  uint32_t* flags;
  uint32_t* ticket;         // CTAs of this call that have finished; reset by the last one
  unsigned long long* key;  // [B * (1 + max_draft)]: best (value, index) of every row so
                            // far; read and reset to 0 by the last CTA
  int32_t* amax;            // [B * (1 + max_draft)]: the target's token of every row
  int B, max_draft, vocab, nctas;
  int64_t row_vecs;  // vectors per row (continuous scan only)
};

constexpr int FIN_B = 1024;   // sequences whose D_b stay in shared memory
constexpr int FIN_CAP = 4096;  // rows / drafts the last CTA finalizes in shared memory

// Total window rows sum_b (1 + D_b); false if any D_b is out of range. D_b of the first
// FIN_B sequences are left in s_D.
__device__ bool total_rows(const int32_t* draft_len, int B, int max_draft, int64_t* rows,
                           int* s_D) {
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
    if (bb < FIN_B) s_D[bb] = D;
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
__device__ void scan_range(const AcceptArgs& a, int64_t rows) {
  constexpr int ES = BF16 ? 2 : 4;
  constexpr int VE = 16 / ES;  // elements per 16-byte vector
  const int64_t V = a.vocab, N = rows * V;
  const int64_t e0 = N * blockIdx.x / a.nctas, e1 = N * (blockIdx.x + 1) / a.nctas;
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
    // (row-local indices fit in 32 bits: V < 2^31)
    const int h0 = (int)(((16 - ((uintptr_t)(row + c0 * ES) & 15)) & 15) / ES);
    const int vb = (int)c0 + (h0 < c1 - c0 ? h0 : (int)(c1 - c0));
    const int nvec = ((int)c1 - vb) / VE;
    const int tb = vb + nvec * VE;
    float bv = -INFINITY;
    int bi = NONE;
    for (int e = (int)c0 + threadIdx.x; e < vb; e += blockDim.x) take(elem(e), e, bv, bi);
    // Vectors: only the maximum of each is compared, without branches; the best vector so
    // far (strictly larger maximum, so the earliest of equal ones) and its words are kept,
    // and the element index inside it is resolved once at the end.
    const uint4* vec = reinterpret_cast<const uint4*>(row + vb * ES);
    int bvec = -1;
    uint4 bw = make_uint4(0, 0, 0, 0);
    for (int base = threadIdx.x; base < nvec; base += blockDim.x * UNROLL) {
      uint4 w[UNROLL];
#pragma unroll
      for (int k = 0; k < UNROLL; ++k) {
        const int vi = base + k * blockDim.x;
        w[k] = vi < nvec ? __ldcs(vec + vi) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < UNROLL; ++k) {
        const int vi = base + k * blockDim.x;
        float vm;
        if constexpr (BF16)
          vm = vmax_bf16x8(w[k]);
        else
          vm = fmaxf(fmaxf(__uint_as_float(w[k].x), __uint_as_float(w[k].y)),
                     fmaxf(__uint_as_float(w[k].z), __uint_as_float(w[k].w)));
        const bool win = vi < nvec && (vm > bv || (bi == NONE && bvec < 0 && vm == vm));
        bv = win ? vm : bv;
        bvec = win ? vi : bvec;
        bw.x = win ? w[k].x : bw.x;
        bw.y = win ? w[k].y : bw.y;
        bw.z = win ? w[k].z : bw.z;
        bw.w = win ? w[k].w : bw.w;
      }
    }
    if (bvec >= 0) {  // the first element of the best vector that equals its maximum
      const int e = vb + bvec * VE;
      const uint32_t ww[4] = {bw.x, bw.y, bw.z, bw.w};
      int q = VE - 1;
#pragma unroll
      for (int t = VE - 1; t >= 0; --t) {
        const float x = BF16 ? bf16_at(ww[t / 2], t & 1) : __uint_as_float(ww[t]);
        if (x == bv) q = t;
      }
      bi = e + q;
    }
    for (int e = tb + threadIdx.x; e < c1; e += blockDim.x) take(elem(e), e, bv, bi);
    warp_argmax(bv, bi);  // one key update per warp and row: no CTA-wide barrier
    if ((threadIdx.x & 31) == 0 && bi != NONE) atomicMax(a.key + r, row_key(bv, bi));
  }
}

// One vector of logits in one load; read once, so not kept in L1.
__device__ __forceinline__ void load_vec(const uint8_t* p, uint32_t (&w)[VW]) {
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::256B.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
        "=r"(w[7])
      : "l"(p));
}

template <bool BF16>
__device__ __forceinline__ float elem_of(const uint32_t (&w)[VW], int t) {
  if constexpr (BF16)
    return bf16_at(w[t >> 1], t & 1);
  else
    return __uint_as_float(w[t]);
}

// Largest value of a vector (NaN ignored unless all are NaN).
template <bool BF16>
__device__ __forceinline__ float vmax_vec(const uint32_t (&w)[VW]) {
  if constexpr (BF16) {
    return fmaxf(vmax_bf16x8(make_uint4(w[0], w[1], w[2], w[3])),
                 vmax_bf16x8(make_uint4(w[4], w[5], w[6], w[7])));
  } else {
    const float m0 = fmaxf(__uint_as_float(w[0]), __uint_as_float(w[1]));
    const float m1 = fmaxf(__uint_as_float(w[2]), __uint_as_float(w[3]));
    const float m2 = fmaxf(__uint_as_float(w[4]), __uint_as_float(w[5]));
    const float m3 = fmaxf(__uint_as_float(w[6]), __uint_as_float(w[7]));
    return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
  }
}

// A thread's best vector of its current row: its maximum bv, its row-local index bvec
// (-1: none yet) and its words, kept without branches; only a strictly larger maximum
// replaces it (vectors reach a thread in increasing order, so the earliest of equal maxima
// stays). The element index inside it is resolved once, when the row is flushed.
struct Best {
  float bv;
  int bvec;
  uint32_t bw[VW];
};

template <bool BF16>
__device__ __forceinline__ void consider(const uint32_t (&w)[VW], int vrow, bool valid,
                                         Best& b) {
  const float vm = vmax_vec<BF16>(w);
  const bool win = valid && (vm > b.bv || (b.bvec < 0 && vm == vm));
  b.bv = win ? vm : b.bv;
  b.bvec = win ? vrow : b.bvec;
#pragma unroll
  for (int t = 0; t < VW; ++t) b.bw[t] = win ? w[t] : b.bw[t];
}

// Row r's candidate: each thread's first element equal to its best vector's maximum, then
// one key update per warp (the whole warp calls it); the thread's best is reset.
template <bool BF16>
__device__ __forceinline__ void flush_row(const AcceptArgs& a, int64_t r, Best& b) {
  constexpr int VE = VB / (BF16 ? 2 : 4);  // elements per vector
  float bv = b.bv;
  int bi = NONE;
  if (b.bvec >= 0) {
    int q = VE - 1;
#pragma unroll
    for (int t = VE - 1; t >= 0; --t)
      if (elem_of<BF16>(b.bw, t) == bv) q = t;
    bi = b.bvec * VE + q;
  }
  warp_argmax(bv, bi);
  if ((threadIdx.x & 31) == 0 && bi != NONE) atomicMax(a.key + r, row_key(bv, bi));
  b.bv = -INFINITY;
  b.bvec = -1;
}

// Continuous scan of CTA blockIdx.x's equal share of the rows * row_vecs vectors.
// Thread t's batch at s holds vectors s + k * ARGMAX_THREADS + t (k < FLAT_U). A batch is
// taken in one pass per row it touches: the vectors of the current row, then, while the
// row ends inside the batch, the flush of the finished row (uniform over the CTA, so whole
// warps reduce it) and a pass over the next row's vectors.
template <bool BF16>
__device__ void scan_flat(const AcceptArgs& a, int64_t rows) {
  const int64_t rv = a.row_vecs, nv = rows * rv;
  const int64_t v0 = nv * blockIdx.x / a.nctas, v1 = nv * (blockIdx.x + 1) / a.nctas;
  const uint8_t* base = (const uint8_t*)a.logits;
  int64_t r = v0 / rv, row0 = r * rv, rb = row0 + rv;  // current row [row0, rb)
  Best b;
  b.bv = -INFINITY;
  b.bvec = -1;
  auto issue = [&](uint32_t (&w)[FLAT_U][VW], int64_t s) {
#pragma unroll
    for (int k = 0; k < FLAT_U; ++k) {
      const int64_t vi = s + (int64_t)k * ARGMAX_THREADS + threadIdx.x;
      if (vi < v1) load_vec(base + vi * VB, w[k]);
    }
  };
  auto process = [&](const uint32_t (&w)[FLAT_U][VW], int64_t s) {
    const int64_t se = min(s + FLAT_BATCH_VECS, v1);  // end of the batch's valid vectors
    while (true) {
      const int64_t cut = min(rb, se);
#pragma unroll
      for (int k = 0; k < FLAT_U; ++k) {
        const int64_t vi = s + (int64_t)k * ARGMAX_THREADS + threadIdx.x;
        consider<BF16>(w[k], (int)(vi - row0), vi >= row0 && vi < cut, b);
      }
      if (rb >= se) break;
      flush_row<BF16>(a, r, b);  // row r is finished
      ++r;
      row0 = rb;
      rb += rv;
    }
  };
  for (int64_t s = v0; s < v1; s += FLAT_BATCH_VECS) {
    uint32_t w[FLAT_U][VW];
    issue(w, s);
    process(w, s);
  }
  flush_row<BF16>(a, r, b);  // the range's last row (no key update if it has no candidate)
}

// Exclusive scan over the CTA of (1 + D, D); returns the running totals through `carry`.
__device__ __forceinline__ void block_scan2(long long& x, long long& y, long long* sh2,
                                            long long& cx, long long& cy) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  long long ix = x, iy = y;  // inclusive within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long ux = __shfl_up_sync(0xffffffffu, ix, o);
    const long long uy = __shfl_up_sync(0xffffffffu, iy, o);
    if (lane >= o) {
      ix += ux;
      iy += uy;
    }
  }
  if (lane == 31) {
    sh2[2 * wid] = ix;
    sh2[2 * wid + 1] = iy;
  }
  __syncthreads();
  long long wx = 0, wy = 0, tx = 0, ty = 0;
  for (int w = 0; w < nw; ++w) {
    if (w < wid) {
      wx += sh2[2 * w];
      wy += sh2[2 * w + 1];
    }
    tx += sh2[2 * w];
    ty += sh2[2 * w + 1];
  }
  x = cx + wx + ix - x;
  y = cy + wy + iy - y;
  cx += tx;
  cy += ty;
  __syncthreads();  // sh2 is reused by the next chunk
}

__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(smem_dst)),
               "l"(gmem_src)
               : "memory");
}

// Run by the last CTA: every row's target token, then per sequence (one warp each) the
// accepted length. For up to FIN_CAP rows and drafts everything stays in shared memory,
// where every CTA staged the drafts during its scan, so the only global round trip left
// is the read of the candidates.
__device__ __forceinline__ void finalize_all(const AcceptArgs& a, int64_t rows, const int* s_D,
                                             const int* s_draft, bool in_smem) {
  __shared__ long long sh2[2 * (ARGMAX_THREADS / 32)];
  __shared__ long long s_q[ARGMAX_THREADS], s_d[ARGMAX_THREADS];
  __shared__ int s_n[ARGMAX_THREADS];
  __shared__ int s_amax[FIN_CAP];
  int* amax = in_smem ? s_amax : a.amax;
  const int* draft = in_smem ? s_draft : a.draft_tokens;
  for (int64_t r = threadIdx.x; r < rows; r += blockDim.x) {
    const unsigned long long k = __ldcg(a.key + r);
    a.key[r] = 0ull;  // clean for the next call
    // a row made only of NaN has no candidate: unspecified, report index 0
    const int bi = k == 0ull ? 0 : key_index(k);
    amax[r] = bi;
    if (a.target_tokens) a.target_tokens[r] = bi;
  }
  __syncthreads();  // amax is visible to the whole CTA
  long long cq = 0, cd = 0;
  for (int b0 = 0; b0 < a.B; b0 += blockDim.x) {
    const int b = b0 + threadIdx.x;
    const int D = b >= a.B ? 0 : (b < FIN_B ? s_D[b] : a.draft_len[b]);
    long long q_off = b < a.B ? 1 + D : 0, d_off = D;
    block_scan2(q_off, d_off, sh2, cq, cd);
    s_q[threadIdx.x] = q_off;
    s_d[threadIdx.x] = d_off;
    s_n[threadIdx.x] = D;
    __syncthreads();
    const int lane = threadIdx.x & 31, nb = min((int)blockDim.x, a.B - b0);
    for (int bb = threadIdx.x >> 5; bb < nb; bb += blockDim.x >> 5) {
      const int Db = s_n[bb];
      const long long qb = s_q[bb], db = s_d[bb];
      int n = Db;  // first draft position that differs from the target's token
      for (int j0 = 0; j0 < Db; j0 += 32) {
        const int j = j0 + lane;
        const bool differs = j < Db && draft[db + j] != amax[qb + j];
        const uint32_t m = __ballot_sync(0xffffffffu, differs);
        if (m) {
          n = j0 + __ffs(m) - 1;
          break;
        }
      }
      if (lane == 0) {
        a.accept_len[b0 + bb] = n + 1;
        a.next_token[b0 + bb] = amax[qb + n];
      }
    }
    __syncthreads();  // s_q / s_d / s_n are reused by the next chunk
  }
  if (!in_smem)  // leave the workspace as it was found (zero) for the next call
    for (int64_t r = threadIdx.x; r < rows; r += blockDim.x) amax[r] = 0;
}

template <bool BF16, bool FLAT>
__global__ void __launch_bounds__(ARGMAX_THREADS, ARGMAX_CTAS_PER_SM) accept_kernel(AcceptArgs a) {
  __shared__ int s_last;
  __shared__ int s_D[FIN_B];
  __shared__ int s_draft[FIN_CAP];
  pdl_trigger();
  pdl_wait();
  int64_t rows;
  const bool ok = total_rows(a.draft_len, a.B, a.max_draft, &rows, s_D);
  const bool in_smem = ok && rows <= FIN_CAP && a.B <= FIN_B;
  if (in_smem) {  // the drafts, for whichever CTA finishes last; they arrive during the scan
    for (int j = threadIdx.x; j < rows - a.B; j += blockDim.x)
      cp_async4(s_draft + j, a.draft_tokens + j);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  if (ok) {
    if constexpr (FLAT)
      scan_flat<BF16>(a, rows);
    else
      scan_range<BF16>(a, rows);
  }
  if (in_smem) asm volatile("cp.async.wait_all;" ::: "memory");
  // completion ticket: every CTA takes one after its candidates are written; the fences
  // order this CTA's key updates before its ticket and, in the last CTA, every other CTA's
  // key updates before its reads
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const bool last = atomicAdd(a.ticket, 1u) == (uint32_t)a.nctas - 1;
    if (last) {
      __threadfence();
      *a.ticket = 0u;  // no CTA of this call touches it again
    }
    s_last = last;
  }
  __syncthreads();
  if (!s_last) return;
  if (!ok) {
    if (threadIdx.x == 0) atomicOr(a.flags, FLAG_ACCEPT_SHAPE);
    return;
  }
  finalize_all(a, rows, s_D, s_draft, in_smem);
}

}  // namespace

AcceptWs accept_ws_layout(int B, int max_draft, int vocab, int num_sms) {
  AcceptWs w;
  const int64_t rows = (int64_t)B * (1 + max_draft);
  // persistent CTAs: all resident at once (4 per SM), fewer for small inputs (at least
  // ~8K elements each)
  const int64_t n_max = rows * (int64_t)vocab;
  int64_t c = (int64_t)ARGMAX_CTAS_PER_SM * num_sms;
  if (c > n_max / 8192) c = n_max / 8192;
  if (c < 1) c = 1;
  w.nctas = (int)c;
  w.ctrl = 0;  // flags word at +0, completion ticket at +64
  w.key = 256;
  w.amax = align_up(w.key + sizeof(unsigned long long) * (size_t)rows, 256);
  w.total = align_up(w.amax + sizeof(int32_t) * (size_t)rows, 256);
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
  a.ticket = (uint32_t*)((uint8_t*)ws + lay.ctrl + 64);
  a.key = (unsigned long long*)((uint8_t*)ws + lay.key);
  a.amax = (int32_t*)((uint8_t*)ws + lay.amax);
  a.B = B;
  a.max_draft = max_draft;
  a.vocab = vocab;
  a.nctas = lay.nctas;
  // continuous scan: rows of whole, aligned vectors
  const int64_t row_bytes = (int64_t)vocab * (dtype == SV_BF16 ? 2 : 4);
  const bool flat = ((uintptr_t)logits % VB) == 0 && row_bytes % VB == 0;
  a.row_vecs = row_bytes / VB;
  const dim3 g(lay.nctas), b(ARGMAX_THREADS);
  if (dtype == SV_BF16)
    return flat ? launch_pdl(accept_kernel<true, true>, g, b, 0, s, a)
                : launch_pdl(accept_kernel<true, false>, g, b, 0, s, a);
  return flat ? launch_pdl(accept_kernel<false, true>, g, b, 0, s, a)
              : launch_pdl(accept_kernel<false, false>, g, b, 0, s, a);
}

}  // namespace sv

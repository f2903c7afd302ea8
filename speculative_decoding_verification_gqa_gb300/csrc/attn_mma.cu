// attn_mma.cu -- verify attention on warp-level tensor-core MMA (mma.sync m16n8k16).
//
// One persistent CTA per SM walks its contiguous range of the global tile line (see
// internal.cuh). For each unit it holds the unit's query-row tile (up to 128 rows =
// G heads x window positions of one KV head) in shared memory and streams 64-key K/V
// tiles through a 3-stage cp.async ring. Eight warps own 16 query rows each:
//   S = Q K^T (fp32 accumulate) -> scale, window-causal mask -> online softmax
//   (running max m and sum l per row, "GPU and LLM, chapter 5", "Online softmax") ->
//   P rounded to 16 bits -> O = O * 2^(m_old - m_new) + P V.
// Nothing but the final O (or a split-KV partial) is written to global memory.
//
// FP8 E4M3 K/V: the raw 8-bit tile is staged by cp.async, then converted in shared memory
// to f16 (every E4M3 value is exact in f16); Q is converted bf16 -> f16 on load and the
// MMAs run in f16 with fp32 accumulation. The per-head K scale is folded into the score
// scale and the V scale into the final normalisation.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "internal.cuh"

namespace sv {
namespace {

constexpr int KT = 64;       // keys per tile
constexpr int NSTAGE = 3;    // cp.async ring depth
constexpr int NTHREADS = 256;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // n = 0: fill the 16 bytes with zeros, read nothing
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                        uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <bool F16>
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0,
                                         uint32_t b1) {
  if constexpr (F16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
        "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
        "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (F16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// bf16 x8 -> f16 x8 (exact for |x| in f16's normal range; tiny values round to f16).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w[e]));
    __half2 h = __float22half2_rn(f);
    w[e] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// e4m3 x2 (low byte = first element) -> f16 x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t x) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)x, __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

template <int HD>
struct Layout {
  static constexpr int ROWB = HD * 2;    // bytes of one 16-bit row
  static constexpr int CH = HD / 8;      // 16-byte chunks per 16-bit row
  static constexpr int Q_BYTES = MT * ROWB;
  static constexpr int T16_BYTES = KT * ROWB;   // one 16-bit K or V tile
  static constexpr int T8_BYTES = KT * HD;      // one raw fp8 K or V tile
  // byte offset of 16-byte chunk c of row r, XOR-swizzled so ldmatrix is conflict-free
  __device__ static __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)(r * ROWB + ((c ^ (r & 7)) << 4));
  }
  static constexpr size_t smem_bytes(bool fp8) {
    return fp8 ? (size_t)Q_BYTES + 2 * NSTAGE * T8_BYTES + 2 * T16_BYTES
               : (size_t)Q_BYTES + 2 * NSTAGE * T16_BYTES;
  }
};

template <int HD, bool FP8>
__global__ void __launch_bounds__(NTHREADS, 1) attn_mma_kernel(const AttnParams p) {
  using L = Layout<HD>;
  constexpr int KS = HD / 16;   // k-steps of S = Q K^T
  constexpr int NS = KT / 8;    // n8 tiles of S
  constexpr int NO = HD / 8;    // n8 tiles of O
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + L::Q_BYTES;  // ring: [stage][K|V]
  const int STAGE_BYTES = FP8 ? 2 * L::T8_BYTES : 2 * L::T16_BYTES;
  uint8_t* sConv = sKV + NSTAGE * STAGE_BYTES;  // fp8 only: converted K | V (f16)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_trigger();
  pdl_wait();  // the plan of this call is complete
  const int2 rb = p.cta_tab[blockIdx.x], re = p.cta_tab[blockIdx.x + 1];
  const int64_t t_begin = rb.x, t_end = re.x;  // this CTA's tiles (see the plan kernel)
  if (t_begin >= t_end) return;
  int u = rb.y;
  const size_t elem = FP8 ? 1 : 2;

  for (int64_t t = t_begin; t < t_end; ++u) {
    if (u >= p.hdr->num_units) break;  // cannot happen for a valid plan
    const int4 info = p.units[u];
    const int b = info.x, g = info.y, mt = info.z;
    const int64_t ub = p.ubeg[u];
    const int nt = p.ubeg[u + 1] - (int)ub;
    const int l0 = (int)(t - ub);
    const int l1 = (int)(min(t_end, ub + nt) - ub);
    if (l1 <= l0) break;  // cannot happen for a valid plan
    t = ub + l1;
    const int T = p.seq_lens[b];
    const int D = p.draft_len[b];
    // key tiles [j0, j1) of the sequence (tile j holds positions j*KT ..), out of the
    // unit's tiles [kb, kb + nt)
    const int kb = info.w / KT;
    const int j0 = kb + l0, j1 = kb + l1;
    const int rows_total = p.G * (D + 1);
    const int rows = min(MT, rows_total - mt * MT);
    const int nkeys = T + D + 1;
    const int kvis = first_visible_key(T, p.window);  // earlier rows left the window
    const int64_t qo = p.q_off[b], ko = p.kv_off[b];
    const float ks = FP8 ? p.kv_scale[g] : 1.f;
    const float sc = p.scale_log2 * ks;

    __syncthreads();  // the previous segment is done with shared memory
    // ---- query-row tile: row r = (window position i, head in group hl)
    for (int idx = tid; idx < MT * L::CH; idx += NTHREADS) {
      const int r = idx / L::CH, c = idx % L::CH;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (r < rows) {
        const int rg = mt * MT + r;
        const int i = rg / p.G, hl = rg % p.G;
        const uint4* src = reinterpret_cast<const uint4*>(
                               (const uint16_t*)p.q + ((qo + i) * p.Hq + (int64_t)g * p.G + hl) * HD) + c;
        val = __ldg(src);
        if (FP8) val = bf16x8_to_f16x8(val);
      }
      *reinterpret_cast<uint4*>(sQ + L::swz(r, c)) = val;
    }

    // ---- K/V tile loader (cp.async; zero fill beyond the sequence's last key and, under a
    // sliding window, before its first visible key: P = 0 there must not meet NaN). The
    // cache row of position `key`: packed, ko + key; paged, row key % block_size of the
    // block the block table names (an entry outside the pool sets the shape flag and
    // reads as zeros).
    const int32_t* tab = p.block_table + (size_t)b * p.bt_stride;
    auto cache_row = [&](int key, bool& ok) -> int64_t {
      if (p.block_size == 0) return ko + key;
      if (!ok) return 0;
      const int blk = __ldg(tab + (key >> p.bs_log2));
      if (blk < 0 || blk >= p.num_blocks) {
        atomicOr(p.flags, FLAG_ATTN_SHAPE);
        ok = false;
        return 0;
      }
      return (int64_t)blk * p.block_size + (key & (p.block_size - 1));
    };
    auto load_tile = [&](int j, int stage) {
      uint8_t* dK = sKV + stage * STAGE_BYTES;
      uint8_t* dV = dK + STAGE_BYTES / 2;
      const int key0 = j * KT;
      if constexpr (FP8) {
        constexpr int CH8 = HD / 16;
        for (int idx = tid; idx < KT * CH8; idx += NTHREADS) {
          const int r = idx / CH8, c = idx % CH8;
          const int key = key0 + r;
          bool ok = key >= kvis && key < nkeys;
          const int64_t row = cache_row(key, ok);
          const size_t off = ok ? ((row * p.Hkv + g) * (size_t)HD + c * 16) : 0;
          cp_async16(smem_u32(dK + r * HD + c * 16), (const uint8_t*)p.k + off, ok);
          cp_async16(smem_u32(dV + r * HD + c * 16), (const uint8_t*)p.v + off, ok);
        }
      } else {
        for (int idx = tid; idx < KT * L::CH; idx += NTHREADS) {
          const int r = idx / L::CH, c = idx % L::CH;
          const int key = key0 + r;
          bool ok = key >= kvis && key < nkeys;
          const int64_t row = cache_row(key, ok);
          const size_t off = ok ? ((row * p.Hkv + g) * (size_t)HD + c * 8) * elem : 0;
          cp_async16(smem_u32(dK + L::swz(r, c)), (const uint8_t*)p.k + off, ok);
          cp_async16(smem_u32(dV + L::swz(r, c)), (const uint8_t*)p.v + off, ok);
        }
      }
    };

#pragma unroll
    for (int s = 0; s < NSTAGE - 1; ++s) {
      if (j0 + s < j1) load_tile(j0 + s, s);
      cp_async_commit();
    }
    __syncthreads();  // query tile visible

    const bool active = warp * 16 < rows;
    uint32_t qf[KS][4];
    if (active) {
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = 2 * kk + (lane >> 4);
        ldsm_x4(smem_u32(sQ) + L::swz(r, c), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }
    // rows owned by this thread: rA = warp*16 + lane/4, rB = rA + 8
    const int rA = warp * 16 + (lane >> 2), rB = rA + 8;
    const int rgA = mt * MT + rA, rgB = mt * MT + rB;
    const int iA = rgA < rows_total ? rgA / p.G : D;  // padding rows see every key
    const int iB = rgB < rows_total ? rgB / p.G : D;
    // sliding window: first visible key of each row, and the largest over the unit
    const int loA = p.window > 0 ? max(T + iA + 1 - p.window, 0) : 0;
    const int loB = p.window > 0 ? max(T + iB + 1 - p.window, 0) : 0;
    const int lo_max = p.window > 0 ? max(T + D + 1 - p.window, 0) : 0;
    float o[NO][4];
#pragma unroll
    for (int n = 0; n < NO; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

    for (int j = j0; j < j1; ++j) {
      cp_async_wait<NSTAGE - 2>();
      __syncthreads();
      {
        const int jn = j + NSTAGE - 1;
        if (jn < j1) load_tile(jn, (jn - j0) % NSTAGE);
        cp_async_commit();
      }
      const int stage = (j - j0) % NSTAGE;
      uint8_t* tK;
      uint8_t* tV;
      if constexpr (FP8) {
        const uint8_t* rK = sKV + stage * STAGE_BYTES;
        const uint8_t* rV = rK + STAGE_BYTES / 2;
        tK = sConv;
        tV = sConv + L::T16_BYTES;
        constexpr int CH8 = HD / 16;
        for (int idx = tid; idx < 2 * KT * CH8; idx += NTHREADS) {
          const int which = idx / (KT * CH8);
          const int rem = idx % (KT * CH8);
          const int r = rem / CH8, c = rem % CH8;
          const uint4 raw = *reinterpret_cast<const uint4*>((which ? rV : rK) + r * HD + c * 16);
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t h[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            h[2 * e] = e4m3x2_to_f16x2((uint16_t)(w[e] & 0xffff));
            h[2 * e + 1] = e4m3x2_to_f16x2((uint16_t)(w[e] >> 16));
          }
          uint8_t* dst = which ? tV : tK;
          *reinterpret_cast<uint4*>(dst + L::swz(r, 2 * c)) = make_uint4(h[0], h[1], h[2], h[3]);
          *reinterpret_cast<uint4*>(dst + L::swz(r, 2 * c + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
        __syncthreads();
      } else {
        tK = sKV + stage * STAGE_BYTES;
        tV = tK + STAGE_BYTES / 2;
      }
      if (!active) continue;

      // ---- S = Q K^T
      float s[NS][4];
#pragma unroll
      for (int n = 0; n < NS; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
        for (int np = 0; np < NS / 2; ++np) {
          const int mi = lane >> 3;
          const int r = np * 16 + (lane & 7) + (mi >> 1) * 8;
          const int c = 2 * kk + (mi & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(smem_u32(tK) + L::swz(r, c), b0, b1, b2, b3);
          mma16816<FP8>(s[2 * np], qf[kk], b0, b1);
          mma16816<FP8>(s[2 * np + 1], qf[kk], b2, b3);
        }
      }
      // ---- scale (log2 units) and window-causal mask: key j visible to row i iff j <= T+i
      // (and, under a sliding window, j >= T+i-window+1)
      const int key0 = j * KT;
      const bool edge = key0 + KT > T || key0 < lo_max;
#pragma unroll
      for (int n = 0; n < NS; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float x = s[n][e] * sc;
          if (edge) {
            const int key = key0 + n * 8 + 2 * (lane & 3) + (e & 1);
            const int lim = T + (e < 2 ? iA : iB);
            if (key > lim || key < (e < 2 ? loA : loB)) x = -INFINITY;
          }
          s[n][e] = x;
        }
      }
      // ---- online softmax update
      float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
      for (int n = 0; n < NS; ++n) {
        mxA = fmaxf(mxA, fmaxf(s[n][0], s[n][1]));
        mxB = fmaxf(mxB, fmaxf(s[n][2], s[n][3]));
      }
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
      mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
      mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
      const float mnA = fmaxf(mA, mxA), mnB = fmaxf(mB, mxB);
      const float muA = mnA == -INFINITY ? 0.f : mnA;
      const float muB = mnB == -INFINITY ? 0.f : mnB;
      const float aA = ex2(mA - muA), aB = ex2(mB - muB);
      mA = mnA;
      mB = mnB;
      float sumA = 0.f, sumB = 0.f;
#pragma unroll
      for (int n = 0; n < NS; ++n) {
        s[n][0] = ex2(s[n][0] - muA);
        s[n][1] = ex2(s[n][1] - muA);
        s[n][2] = ex2(s[n][2] - muB);
        s[n][3] = ex2(s[n][3] - muB);
        sumA += s[n][0] + s[n][1];
        sumB += s[n][2] + s[n][3];
      }
      lA = lA * aA + sumA;
      lB = lB * aB + sumB;
#pragma unroll
      for (int n = 0; n < NO; ++n) {
        o[n][0] *= aA;
        o[n][1] *= aA;
        o[n][2] *= aB;
        o[n][3] *= aB;
      }
      // ---- O += P V
#pragma unroll
      for (int kk = 0; kk < KT / 16; ++kk) {
        uint32_t a[4];
        a[0] = pack2<FP8>(s[2 * kk][0], s[2 * kk][1]);
        a[1] = pack2<FP8>(s[2 * kk][2], s[2 * kk][3]);
        a[2] = pack2<FP8>(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        a[3] = pack2<FP8>(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
        for (int dp = 0; dp < HD / 16; ++dp) {
          const int mi = lane >> 3;
          const int r = kk * 16 + (lane & 7) + (mi & 1) * 8;
          const int c = 2 * dp + (mi >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(smem_u32(tV) + L::swz(r, c), b0, b1, b2, b3);
          mma16816<FP8>(o[2 * dp], a, b0, b1);
          mma16816<FP8>(o[2 * dp + 1], a, b2, b3);
        }
      }
    }
    cp_async_wait<0>();

    // ---- epilogue
    if (active) {
      lA += __shfl_xor_sync(0xffffffffu, lA, 1);
      lA += __shfl_xor_sync(0xffffffffu, lA, 2);
      lB += __shfl_xor_sync(0xffffffffu, lB, 1);
      lB += __shfl_xor_sync(0xffffffffu, lB, 2);
      const int col = 2 * (lane & 3);
      if (j0 == kb && j1 == kb + nt) {
        // this CTA saw every key of the unit: normalise and store bf16
        const float vs = FP8 ? p.kv_scale[p.Hkv + g] : 1.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int r = half ? rB : rA;
          if (r >= rows) continue;
          const int rg = mt * MT + r;
          const int i = rg / p.G, hl = rg % p.G;
          const float inv = vs / (half ? lB : lA);
          __nv_bfloat16* dst = (__nv_bfloat16*)p.out +
                               ((qo + i) * p.Hq + (int64_t)g * p.G + hl) * HD + col;
#pragma unroll
          for (int n = 0; n < NO; ++n)
            *reinterpret_cast<__nv_bfloat162*>(dst + n * 8) = __floats2bfloat162_rn(
                o[n][half * 2] * inv, o[n][half * 2 + 1] * inv);
        }
      } else {
        const size_t slot = (size_t)blockIdx.x + u;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int r = half ? rB : rA;
          float* dst = p.part_o + (slot * MT + r) * HD + col;
#pragma unroll
          for (int n = 0; n < NO; ++n)
            *reinterpret_cast<float2*>(dst + n * 8) = make_float2(o[n][half * 2], o[n][half * 2 + 1]);
          if ((lane & 3) == 0)
            p.part_ml[slot * MT + r] = make_float2(half ? mB : mA, half ? lB : lA);
        }
      }
    }
  }
}

template <int HD, bool FP8>
cudaError_t launch_one(const AttnParams& p, cudaStream_t s) {
  const size_t smem = Layout<HD>::smem_bytes(FP8);
  cudaError_t e = cudaFuncSetAttribute(attn_mma_kernel<HD, FP8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_mma_kernel<HD, FP8>, dim3(p.n_ctas), dim3(NTHREADS), smem, s, p);
}

}  // namespace

int attn_mma_kt() { return KT; }

cudaError_t launch_attn_mma(const AttnParams& p, bool fp8, cudaStream_t s) {
  if (p.d == 128) return fp8 ? launch_one<128, true>(p, s) : launch_one<128, false>(p, s);
  return fp8 ? launch_one<64, true>(p, s) : launch_one<64, false>(p, s);
}

}  // namespace sv

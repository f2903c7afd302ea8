// plan_combine.cu -- the two small kernels around verify attention.
//
// plan:    per-sequence offsets of the packed layout, the unit list, each unit's first
//          tile on the global tile line and each CTA's range of it; device-side length
//          checks.
// combine: merges the split-KV partials of one unit. For partials s with running max m_s,
//          sum l_s and unnormalised output O_s: m* = max m_s, l* = sum l_s 2^(m_s - m*),
//          O* = sum O_s 2^(m_s - m*) / l*. This is the online-softmax update of
//          "GPU and LLM, chapter 5", "Online softmax", applied across key ranges instead
//          of across tiles (log2 units: the scores were pre-multiplied by log2(e)).
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.cuh"

namespace sv {

constexpr int PLAN_THREADS = 256;

// Exclusive scans over the block of N int64 values per thread at once (one pair of
// barriers for all of them); total[k] receives the block's sum of v[k].
template <int N>
__device__ void block_excl_scan(const int64_t (&v)[N], int64_t (&ex)[N], int64_t (&total)[N],
                                int64_t (*s_warp)[N]) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  int64_t x[N];
#pragma unroll
  for (int k = 0; k < N; ++k) x[k] = v[k];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x[k], o);
      if (lane >= o) x[k] += y;
    }
  }
  if (lane == 31)
#pragma unroll
    for (int k = 0; k < N; ++k) s_warp[wid][k] = x[k];
  __syncthreads();
#pragma unroll
  for (int k = 0; k < N; ++k) {
    int64_t before = 0, all = 0;
    for (int w2 = 0; w2 < nw; ++w2) {
      before += w2 < wid ? s_warp[w2][k] : 0;
      all += s_warp[w2][k];
    }
    ex[k] = x[k] - v[k] + before;
    total[k] = all;
  }
  __syncthreads();  // s_warp is reused by the next scan
}

constexpr int PLAN_SMEM_UNITS = 4096;  // unit starts also kept in shared memory

__global__ void __launch_bounds__(PLAN_THREADS) plan_kernel(AttnParams p, int kt) {
  __shared__ int64_t s_warp[PLAN_THREADS / 32][4];
  __shared__ int32_t s_ubeg[PLAN_SMEM_UNITS + 1];
  __shared__ int64_t carry[4];
  __shared__ int bad, s_maxt, s_nmt_lo, s_nmt_hi;
  const int tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();
  if (tid == 0) {
    carry[0] = carry[1] = carry[2] = carry[3] = 0;
    bad = 0;
    s_maxt = 0;
    s_nmt_lo = 0x7fffffff;
    s_nmt_hi = 0;
  }
  __syncthreads();
  for (int base = 0; base < p.B; base += blockDim.x) {
    const int b = base + tid;
    int64_t w = 0, kvn = 0, nunits = 0, ntiles = 0, per_g = 0;
    int nmt = 0, nt = 0, T = 0;
    if (b < p.B) {
      T = p.seq_lens[b];
      const int D = p.draft_len[b];
      if (T < 0 || T > p.max_seq || D < 0 || D > p.max_draft ||
          (p.block_size > 0 &&
           (((int64_t)T + D + p.block_size) >> p.bs_log2) > p.bt_stride)) {
        bad = 1;  // a length out of range, or more blocks than the block table's row holds
      } else {
        w = 1 + D;
        kvn = T + w;
        nmt = (int)((p.G * w + MT - 1) / MT);
        nt = (int)((kvn + kt - 1) / kt);  // tiles up to the one holding T + D
        for (int mt = 0; mt < nmt; ++mt) per_g += nt - unit_first_tile(T, mt, p.G, p.window, kt);
        atomicMax(&s_maxt, nt - unit_first_tile(T, 0, p.G, p.window, kt));  // longest unit
        atomicMin(&s_nmt_lo, nmt);
        atomicMax(&s_nmt_hi, nmt);
        nunits = (int64_t)p.Hkv * nmt;
        ntiles = (int64_t)p.Hkv * per_g;
      }
    }
    const int64_t vals[4] = {w, kvn, nunits, ntiles};
    int64_t ex[4], tot[4];
    block_excl_scan<4>(vals, ex, tot, s_warp);
    const int64_t eq = ex[0], ekv = ex[1], eu = ex[2], et = ex[3];
    const int64_t tq = tot[0], tkv = tot[1], tu = tot[2], tt = tot[3];
    if (b < p.B) {
      p.q_off[b] = carry[0] + eq;
      p.kv_off[b] = carry[1] + ekv;
      const int64_t ub = carry[2] + eu, tb = carry[3] + et;
      for (int g = 0; g < p.Hkv; ++g) {
        int64_t t0 = tb + (int64_t)g * per_g;
        for (int mt = 0; mt < nmt; ++mt) {
          const int64_t u = ub + (int64_t)g * nmt + mt;
          const int kb = unit_first_tile(T, mt, p.G, p.window, kt);
          const int ntu = nt - kb;
          if (u < p.max_units) {
            p.units[u] = make_int4(b, g, mt, kb * kt);
            p.ubeg[u] = (int32_t)t0;
            if (u < PLAN_SMEM_UNITS) s_ubeg[u] = (int32_t)t0;
          }
          t0 += ntu;
        }
      }
    }
    __syncthreads();
    if (tid == 0) {
      carry[0] += tq;
      carry[1] += tkv;
      carry[2] += tu;
      carry[3] += tt;
    }
    __syncthreads();
  }
  if (tid == 0) {
    const bool err = bad || carry[0] > p.q_rows || (p.block_size == 0 && carry[1] > p.kv_rows) ||
                     carry[2] > p.max_units || carry[3] >= (int64_t)0x7fffffff;
    p.q_off[p.B] = carry[0];
    p.kv_off[p.B] = carry[1];
    p.hdr->sum_w = carry[0];
    p.hdr->sum_kv = carry[1];
    p.hdr->kt = kt;
    if (err) {
      atomicOr(p.flags, FLAG_ATTN_SHAPE);
      p.hdr->num_units = 0;
      p.hdr->total_tiles = 0;
    } else {
      p.hdr->num_units = (int32_t)carry[2];
      p.hdr->total_tiles = (int32_t)carry[3];
      p.ubeg[carry[2]] = (int32_t)carry[3];
      if (carry[2] <= PLAN_SMEM_UNITS) s_ubeg[carry[2]] = (int32_t)carry[3];  // the end too
    }
  }
  __syncthreads();  // the header is visible to the whole block
  // Every sequence with the same number nm > 1 of row tiles per KV head: reorder the units
  // row-tile-major (all row tiles 0, then all row tiles 1, ...). The row tiles of one
  // (sequence, KV head) read the same K/V; on the split tile line the CTAs of slice mt
  // then walk the same key tiles at the same time as those of slice 0, so the K/V of all
  // but one of them comes from L2 instead of HBM.
  const int nm = s_nmt_hi;
  if (p.hdr->num_units > 0 && nm > 1 && s_nmt_lo == nm) {
    if (tid == 0) carry[3] = 0;
    __syncthreads();
    for (int mt = 0; mt < nm; ++mt) {
      for (int base = 0; base < p.B; base += blockDim.x) {
        const int b = base + tid;
        int T = 0, nt = 0, kb = 0;
        if (b < p.B) {
          T = p.seq_lens[b];
          nt = (int)(((int64_t)T + p.draft_len[b] + kt) / kt);  // tiles up to T + D
          kb = unit_first_tile(T, mt, p.G, p.window, kt);
        }
        const int64_t v1[1] = {b < p.B ? (int64_t)p.Hkv * (nt - kb) : 0};
        int64_t e1[1], t1[1];
        block_excl_scan<1>(v1, e1, t1, reinterpret_cast<int64_t (*)[1]>(&s_warp[0][0]));
        const int64_t et = e1[0], tt = t1[0];
        if (b < p.B) {
          for (int g = 0; g < p.Hkv; ++g) {
            const int64_t u = ((int64_t)mt * p.B + b) * p.Hkv + g;
            const int32_t t0 = (int32_t)(carry[3] + et + (int64_t)g * (nt - kb));
            p.units[u] = make_int4(b, g, mt, kb * kt);
            p.ubeg[u] = t0;
            if (u < PLAN_SMEM_UNITS) s_ubeg[u] = t0;
          }
        }
        __syncthreads();
        if (tid == 0) carry[3] += tt;
        __syncthreads();
      }
    }
  }
  if (tid == 0) {
    // k CTAs per unit, or the split tile line (cost model in internal.cuh)
    const int64_t U = p.hdr->num_units, TT = p.hdr->total_tiles, C = p.n_ctas;
    int k = 0;
    if (U > 0 && U <= C) {
      if (p.unit_ctas_mode > 0) {  // forced by the caller
        k = (int)min((int64_t)p.unit_ctas_mode, C / U);
      } else if (p.unit_ctas_mode < 0 && p.tile_floor > 0) {  // the model, where it applies
        const double f = p.tile_floor;
        double best = (double)(TT + U * p.switch_tiles) / C * fmax(f, (double)C);
        for (int kk = 1; kk <= C / U; ++kk) {
          const double t = (double)((s_maxt + kk - 1) / kk) * fmax(f, (double)(U * kk));
          if (t < best) {
            best = t;
            k = kk;
          }
        }
      }
    }
    p.hdr->unit_ctas = k;
  }
  __syncthreads();  // ubeg and the header are visible to the whole block
  const int U = p.hdr->num_units;
  const int64_t TT = p.hdr->total_tiles, X = p.switch_tiles;
  const int32_t* ubeg = U <= PLAN_SMEM_UNITS ? s_ubeg : p.ubeg;
  if (p.hdr->unit_ctas > 0) {
    // CTA c = u * k + i takes the i-th of k equal parts of unit u's tiles
    const int k = p.hdr->unit_ctas;
    for (int c = tid; c <= p.n_ctas; c += blockDim.x) {
      int2 e = make_int2((int32_t)TT, U);
      if (c < U * k) {
        const int u = c / k, i = c % k;
        const int32_t n = ubeg[u + 1] - ubeg[u];
        e = make_int2(ubeg[u] + (int32_t)((int64_t)n * i / k), u);
      }
      p.cta_tab[c] = e;
    }
    return;
  }
  // CTA c starts at the first real tile at or after virtual position c*VT/C
  const int64_t VT = TT + (int64_t)U * X;
  for (int c = tid; c <= p.n_ctas; c += blockDim.x) {
    int2 e = make_int2((int32_t)TT, U);
    if (c < p.n_ctas && TT > 0) {
      const int64_t v0 = (int64_t)c * VT / p.n_ctas;
      int lo = 0, hi = U - 1;  // last unit whose virtual start ubeg[u] + u*X is <= v0
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ubeg[mid] + (int64_t)mid * X <= v0) lo = mid; else hi = mid - 1;
      }
      const int64_t into = v0 - (ubeg[lo] + (int64_t)lo * X) - X;  // < 0: before its tiles
      e = make_int2((int32_t)(ubeg[lo] + (into > 0 ? into : 0)), lo);
    }
    p.cta_tab[c] = e;
  }
}

sv_status host_plan(const AttnParams& p, int kt, const int32_t* Tv, const int32_t* Dv,
                    HostPlan* hp) {
  // the steps of plan_kernel, one sequence after another
  if (p.B > HP_MAX_B || p.n_ctas > HP_MAX_C) return SV_ERR_WORKSPACE;
  int64_t sum_w = 0, sum_kv = 0, U = 0, TT = 0;
  int maxt = 0, nmt_lo = 0x7fffffff, nmt_hi = 0;
  for (int b = 0; b < p.B; ++b) {
    const int T = Tv[b], D = Dv[b];
    if (T < 0 || T > p.max_seq || D < 0 || D > p.max_draft) return SV_ERR_SHAPE;
    const int w = 1 + D;
    const int nmt = (p.G * w + MT - 1) / MT;
    const int nt = (int)(((int64_t)T + w + kt - 1) / kt);
    hp->T[b] = T;
    hp->D[b] = D;
    hp->q_off[b] = sum_w;
    hp->kv_off[b] = sum_kv;
    sum_w += w;
    sum_kv += (int64_t)T + w;
    U += (int64_t)p.Hkv * nmt;
    maxt = std::max(maxt, nt - unit_first_tile(T, 0, p.G, p.window, kt));
    nmt_lo = std::min(nmt_lo, nmt);
    nmt_hi = std::max(nmt_hi, nmt);
  }
  hp->q_off[p.B] = sum_w;
  hp->kv_off[p.B] = sum_kv;
  if (sum_w > p.q_rows || (p.block_size == 0 && sum_kv > p.kv_rows) || U > p.max_units)
    return SV_ERR_SHAPE;
  if (U > HP_MAX_U) return SV_ERR_WORKSPACE;
  // units and their starts on the tile line: by sequence, KV head, row tile; row-tile-major
  // when every sequence has the same number (> 1) of row tiles
  const bool by_slice = p.B > 0 && nmt_hi > 1 && nmt_lo == nmt_hi;
  int64_t u = 0;
  auto add_unit = [&](int b, int g, int mt) {
    const int T = hp->T[b];
    const int nt = (int)(((int64_t)T + hp->D[b] + kt) / kt);
    const int kb = unit_first_tile(T, mt, p.G, p.window, kt);
    hp->units[u] = make_int4(b, g, mt, kb * kt);
    hp->ubeg[u] = (int32_t)TT;
    TT += nt - kb;
    ++u;
  };
  if (by_slice) {
    for (int mt = 0; mt < nmt_hi; ++mt)
      for (int b = 0; b < p.B; ++b)
        for (int g = 0; g < p.Hkv; ++g) add_unit(b, g, mt);
  } else {
    for (int b = 0; b < p.B; ++b) {
      const int nmt = (p.G * (1 + hp->D[b]) + MT - 1) / MT;
      for (int g = 0; g < p.Hkv; ++g)
        for (int mt = 0; mt < nmt; ++mt) add_unit(b, g, mt);
    }
  }
  if (TT >= (int64_t)0x7fffffff) return SV_ERR_SHAPE;
  hp->ubeg[U] = (int32_t)TT;
  hp->num_units = (int32_t)U;
  hp->total_tiles = (int32_t)TT;
  // the unit-to-CTA policy (the same model and arithmetic as plan_kernel)
  const int64_t C = p.n_ctas;
  int k = 0;
  if (U > 0 && U <= C) {
    if (p.unit_ctas_mode > 0) {
      k = (int)std::min((int64_t)p.unit_ctas_mode, C / U);
    } else if (p.unit_ctas_mode < 0 && p.tile_floor > 0) {
      const double f = p.tile_floor;
      double best = (double)(TT + U * p.switch_tiles) / C * fmax(f, (double)C);
      for (int kk = 1; kk <= C / U; ++kk) {
        const double t = (double)((maxt + kk - 1) / kk) * fmax(f, (double)(U * kk));
        if (t < best) {
          best = t;
          k = kk;
        }
      }
    }
  }
  hp->unit_ctas = k;
  for (int c = 0; c <= C; ++c) {
    int2 e = make_int2((int32_t)TT, (int32_t)U);
    if (k > 0) {
      if (c < U * k) {
        const int uu = c / k, i = c % k;
        const int32_t n = hp->ubeg[uu + 1] - hp->ubeg[uu];
        e = make_int2(hp->ubeg[uu] + (int32_t)((int64_t)n * i / k), uu);
      }
    } else if (c < C && TT > 0) {
      const int64_t X = p.switch_tiles, VT = TT + U * X;
      const int64_t v0 = (int64_t)c * VT / C;
      int lo = 0, hi = (int)U - 1;  // last unit whose virtual start ubeg[u] + u*X is <= v0
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (hp->ubeg[mid] + (int64_t)mid * X <= v0) lo = mid; else hi = mid - 1;
      }
      const int64_t into = v0 - (hp->ubeg[lo] + (int64_t)lo * X) - X;
      e = make_int2((int32_t)(hp->ubeg[lo] + (into > 0 ? into : 0)), lo);
    }
    hp->cta_tab[c] = e;
  }
  return SV_OK;
}

cudaError_t launch_plan(const AttnParams& p, int kt, cudaStream_t s) {
  return launch_pdl(plan_kernel, dim3(1), dim3(PLAN_THREADS), 0, s, p, kt);
}

// Work item = eight query rows of one unit: one warp per row, each lane d/32 consecutive
// columns; the rows of units that a single attention CTA covered are skipped at once.
constexpr int COMBINE_ROWS = 8;

template <int HD>
__device__ __forceinline__ void combine_row(const AttnParams& p, int u, int r, int lane, int kc) {
  constexpr int PER = HD / 32;
  constexpr int MAXP = 4;  // partials loaded in one batch
  const int64_t VT = p.hdr->total_tiles + (int64_t)p.hdr->num_units * p.switch_tiles;
  const int64_t ub = p.ubeg[u], ue = p.ubeg[u + 1];
  // the CTAs that covered the unit: u*k .. u*k + k - 1 (k CTAs per unit), or those whose
  // ranges of the split tile line hold its tiles
  const int c_lo = kc > 0 ? u * kc : cta_of_tile(vpos_of_tile(ub, u, p.switch_tiles), VT, p.n_ctas);
  const int c_hi = kc > 0 ? u * kc + kc - 1
                          : cta_of_tile(vpos_of_tile(ue - 1, u, p.switch_tiles), VT, p.n_ctas);
  // one CTA covered the unit and wrote the output itself
  if (c_lo == c_hi || (kc > 0 && ue - ub == 1)) return;
  const int4 info = p.units[u];
  const int b = info.x, g = info.y, mt = info.z;
  const int rows_total = p.G * (1 + p.draft_len[b]);
  if (r >= min(MT, rows_total - mt * MT)) return;
  float mx = -INFINITY, L = 0.f, acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  for (int c0 = c_lo; c0 <= c_hi; c0 += MAXP) {
    // issue every load of the batch before using any (one L2 round trip per batch)
    float2 ml[MAXP];
    float ov[MAXP][PER];
#pragma unroll
    for (int k = 0; k < MAXP; ++k) {
      const int c = c0 + k;
      const bool use = c <= c_hi && (kc > 0 ? (ue - ub) * (c - c_lo + 1) / kc > (ue - ub) * (c - c_lo) / kc
                                            : cta_has_tiles(c, VT, p.n_ctas));
      const size_t slot = (size_t)(c + u);
      ml[k] = use ? p.part_ml[slot * MT + r] : make_float2(-INFINITY, 0.f);
      const float* src = p.part_o + (slot * MT + r) * HD + lane * PER;
      if constexpr (PER == 4) {
        const float4 v = use ? __ldcs(reinterpret_cast<const float4*>(src)) : make_float4(0, 0, 0, 0);
        ov[k][0] = v.x;
        ov[k][1] = v.y;
        ov[k][2] = v.z;
        ov[k][3] = v.w;
      } else {
        const float2 v = use ? __ldcs(reinterpret_cast<const float2*>(src)) : make_float2(0, 0);
        ov[k][0] = v.x;
        ov[k][1] = v.y;
      }
    }
    float bm = mx;
#pragma unroll
    for (int k = 0; k < MAXP; ++k) bm = fmaxf(bm, ml[k].x);
    const float muse = bm == -INFINITY ? 0.f : bm;
    const float rs = exp2f(mx - muse);  // rescale what earlier batches accumulated
    L *= rs;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] *= rs;
#pragma unroll
    for (int k = 0; k < MAXP; ++k) {
      const float wgt = exp2f(ml[k].x - muse);  // 0 for unused slots (m = -inf)
      L += ml[k].y * wgt;
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] += wgt * ov[k][e];
    }
    mx = bm;
  }
  const float vs = p.kv_scale ? p.kv_scale[p.Hkv + g] : 1.f;
  const float inv = vs / L;
  const int rg = mt * MT + r;
  const int i = rg / p.G, hl = rg % p.G;
  __nv_bfloat16* dst = (__nv_bfloat16*)p.out +
                       ((p.q_off[b] + i) * p.Hq + (int64_t)g * p.G + hl) * HD + lane * PER;
  if constexpr (PER == 4) {
    __nv_bfloat162 a = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
    __nv_bfloat162 c = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
    uint2 w;
    w.x = *reinterpret_cast<uint32_t*>(&a);
    w.y = *reinterpret_cast<uint32_t*>(&c);
    *reinterpret_cast<uint2*>(dst) = w;
  } else {
    *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
  }
}

// Work items (unit, block of COMBINE_ROWS rows) in a grid-stride loop over a grid that is
// resident at once, so that a call with nothing to combine (one CTA per unit) ends at once.
template <int HD>
__global__ void __launch_bounds__(256) combine_kernel(AttnParams p) {
  pdl_trigger();
  pdl_wait();
  const int kc = p.hdr->unit_ctas;  // CTAs per unit (0: the split tile line)
  if (kc == 1) return;              // one CTA per unit: every unit is whole
  const int items = p.hdr->num_units * (MT / COMBINE_ROWS);
  for (int it = blockIdx.x; it < items; it += gridDim.x)
    combine_row<HD>(p, it / (MT / COMBINE_ROWS),
                    (it % (MT / COMBINE_ROWS)) * COMBINE_ROWS + (threadIdx.x >> 5),
                    threadIdx.x & 31, kc);
}

cudaError_t launch_combine(const AttnParams& p, cudaStream_t s) {
  if (p.max_units <= 0) return cudaSuccess;
  // at most 8 CTAs of 256 threads per CTA of the attention grid (about one SM each)
  const unsigned items = (unsigned)p.max_units * (MT / COMBINE_ROWS);
  const unsigned grid = min(items, 8u * (unsigned)(p.n_ctas > 0 ? p.n_ctas : 1));
  return p.d == 128 ? launch_pdl(combine_kernel<128>, dim3(grid), dim3(256), 0, s, p)
                    : launch_pdl(combine_kernel<64>, dim3(grid), dim3(256), 0, s, p);
}

}  // namespace sv

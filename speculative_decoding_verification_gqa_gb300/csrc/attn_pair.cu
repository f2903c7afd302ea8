// attn_pair.cu -- verify attention when a KV head serves more than one tensor-core tile of
// query rows: 128 < G (1 + D) <= 256 ("Co-Designing AI Models Using Speculative Decoding",
// summary, guideline 3: the runtime steps up when G (1 + D) crosses a multiple of 128,
// because the query tile no longer fits one M = 128 tile).
//
// One CTA per (sequence b, KV head g) holds both 128-row tiles of its G (1 + D_b) query
// rows and streams each 128-key K/V tile of the head once for both, so the second row tile
// costs tensor-core and softmax time but no second pass over the cache. Row tile r has its
// own softmax warpgroup, score buffer S_r and accumulator O_r in TMEM (4 x 128 columns, the
// whole of it); P_r is written over the first 64 columns of S_r once the scores are in
// registers, and Q_r sits in shared memory (A operand of the score MMA from shared memory).
//
//   warp 0      TMA producer: K and V tiles (128 keys x 128, bf16, 128-byte swizzle) into
//               a 2-stage ring; a stage is released when both P V MMAs have read it.
//   warp 1      S issuer: S_r = Q_r K^T for r = 0, 1 per key tile, each once P_r of the
//               previous tile has been consumed (the P V that reads it has completed).
//   warp 3      P V issuer: O_r += P_r V once warpgroup r has written P_r.
//   warps 4-7   row tile 0; warps 8-11 row tile 1. A thread owns one query row: it writes
//               Q into shared memory once, then per key tile reads its 128 scores, applies
//               the window-causal mask and the online-softmax update ("GPU and LLM, chapter
//               5", "Online softmax": running max, running sum, rescale by 2^(m_old -
//               m_new), lazily as in attn_tc.cu: only when the max grows by more than 2^8),
//               writes P = 2^(s - m) as bf16 and, at the end, O / l.
// The CTA works out its sequence's offsets in the packed layout from the lengths itself
// (every CTA checks every length), so no planning or combining kernel runs. Every
// mbarrier wait is bounded as in attn_tc.cu.
#include "tc_util.cuh"

namespace sv {
namespace {

constexpr int PKT = 128;   // keys per tile
constexpr int PHD = 128;   // head dimension
constexpr int PNS = 2;     // ring stages (K and V tile each)
constexpr int PTHREADS = 384;
constexpr int PWG0 = 4;    // warps 4..7: row tile 0, 8..11: row tile 1
constexpr uint32_t P_TMEM_COLS = 512;
constexpr uint32_t PCOL_O = 0;    // O_r: columns [128 r, 128 r + 128)
constexpr uint32_t PCOL_S = 256;  // S_r: [256 + 128 r, + 128); P_r: its first 64 columns

struct __align__(8) PairBars {
  uint64_t k_full[PNS], v_full[PNS], kv_empty[PNS];
  uint64_t q_full[2], s_full[2], p_full[2], o_done[2];
  uint64_t s_final[2];  // the two issuers' last MMAs
  uint32_t tmem_base;
  int abort;
  unsigned long long q_off, kv_off, q_tot, kv_tot;  // this sequence's offsets; batch totals
  int bad;
};

struct PairLayout {
  static constexpr int BLK = PKT * 128;        // one 128-byte-wide column block of a tile
  static constexpr int TILE = PKT * PHD * 2;   // one bf16 tile (Q rows, K or V)
  static constexpr int Q0 = 0;                 // Q_0, then Q_1
  static constexpr int RING = 2 * TILE;        // stage s: K at RING + s STAGE, V after it
  static constexpr int STAGE = 2 * TILE;
  static constexpr int BARS = RING + PNS * STAGE;
  static constexpr size_t SMEM = (size_t)BARS + sizeof(PairBars);
  static_assert(SMEM <= 227 * 1024, "dynamic shared memory above the per-CTA limit");
};

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

__global__ void __launch_bounds__(PTHREADS, 1)
    attn_pair_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
  using L = PairLayout;
  extern __shared__ __align__(1024) uint8_t smem[];  // 128-byte swizzled tiles: 1 KiB aligned
  PairBars* bars = (PairBars*)(smem + L::BARS);
  volatile int* abort = &bars->abort;
  const Waiter wt{abort, p.flags, p.wait_limit > 0 ? p.wait_limit : TIMEOUT_CYCLES};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_trigger();
  pdl_wait();  // the previous call on the stream is complete
  if (saddr(smem) & 1023) {  // the swizzle phases below assume a 1 KiB-aligned base
    if (tid == 0) atomicOr(p.flags, FLAG_ATTN_SHAPE);
    return;
  }
  const int b = blockIdx.x / p.Hkv, g = blockIdx.x % p.Hkv;

  if (tid == 0) {
    bars->q_off = bars->kv_off = bars->q_tot = bars->kv_tot = 0;
    bars->bad = 0;
    bars->abort = 0;
  }
  __syncthreads();
  // every length in range, and this sequence's offsets (every CTA scans every length, so
  // all of them skip the call together when one is out of range)
  {
    unsigned long long q = 0, kv = 0, qt = 0, kvt = 0;
    int bad = 0;
    for (int bb = tid; bb < p.B; bb += PTHREADS) {
      const int T = p.seq_lens[bb], D = p.draft_len[bb];
      if (T < 0 || T > p.max_seq || D < 0 || D > p.max_draft) {
        bad = 1;
        continue;
      }
      qt += 1 + D;
      kvt += (unsigned long long)T + 1 + D;
      if (bb < b) {
        q += 1 + D;
        kv += (unsigned long long)T + 1 + D;
      }
    }
    if (bad) atomicOr(&bars->bad, 1);
    if (q) atomicAdd(&bars->q_off, q);
    if (kv) atomicAdd(&bars->kv_off, kv);
    if (qt) atomicAdd(&bars->q_tot, qt);
    if (kvt) atomicAdd(&bars->kv_tot, kvt);
  }
  __syncthreads();
  if (bars->bad || bars->q_tot > (unsigned long long)p.q_rows ||
      bars->kv_tot > (unsigned long long)p.kv_rows) {
    if (blockIdx.x == 0 && tid == 0) atomicOr(p.flags, FLAG_ATTN_SHAPE);
    return;  // uniform: every CTA sees the same totals
  }
  const int64_t q_off = (int64_t)bars->q_off, kv_off = (int64_t)bars->kv_off;
  const int T = p.seq_lens[b], D = p.draft_len[b];
  const int rows_total = p.G * (D + 1);
  const int nr = rows_total > MT ? 2 : 1;  // row tiles with live rows
  const int nkeys = T + D + 1;
  const int nt = (nkeys + PKT - 1) / PKT;   // key tiles

  if (tid == 0) {
    for (int s = 0; s < PNS; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);  // the commit after the stage's last P V
    }
    for (int r = 0; r < 2; ++r) {
      mbar_init(&bars->q_full[r], 128);
      mbar_init(&bars->s_full[r], 1);
      mbar_init(&bars->p_full[r], 128);
      mbar_init(&bars->o_done[r], 1);
    }
    mbar_init(&bars->s_final[0], 1);
    mbar_init(&bars->s_final[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     saddr(&bars->tmem_base)),
                 "r"(P_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = bars->tmem_base;
  if (warp < PWG0) {  // warps 0-3: producer and MMA issuers
    if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmk) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmv) : "memory");
      // test hook: the first tile is never loaded, so the waits for it run out; stage 0
      // then holds no copy to wait for
      const bool withhold = p.stall_first_tile != 0;
      uint32_t it = 0;
      for (; it < (uint32_t)nt; ++it) {
        const uint32_t st = it % PNS;
        if (it >= PNS && !mbar_wait(&bars->kv_empty[st], ((it / PNS) - 1) & 1, wt)) break;
        if (withhold && it == 0) continue;
        const int row = (int)kv_off + (int)it * PKT;
        uint8_t* kst = smem + L::RING + st * L::STAGE;
        mbar_expect_tx(&bars->k_full[st], L::TILE);
        for (int c = 0; c < PHD / 64; ++c)
          tma_load_3d(saddr(kst + c * L::BLK), &tmk, &bars->k_full[st], c * 64, g, row);
        mbar_expect_tx(&bars->v_full[st], L::TILE);
        for (int c = 0; c < PHD / 64; ++c)
          tma_load_3d(saddr(kst + L::TILE + c * L::BLK), &tmv, &bars->v_full[st], c * 64, g,
                      row);
      }
      // leave no copy in flight: the last fill of every stage must have landed (normally
      // its readers waited for it; after another role gave up they may not have)
      for (uint32_t st = withhold ? 1 : 0; st < PNS && st < it; ++st) {
        const uint32_t fills = (it - 1 - st) / PNS + 1;
        const uint32_t par = (fills - 1) & 1;
        const long long t0 = clock64();
        while (!(mbar_try(&bars->k_full[st], par) && mbar_try(&bars->v_full[st], par)) &&
               clock64() - t0 < TIMEOUT_CYCLES) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S_r = Q_r K^T issuer
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_bf16(PKT, 0);
      // K and Q tiles: K-major, 128-byte rows, 8-row groups 1024 B apart; 16 elements (32
      // bytes) per K step, two 64-column blocks
      const uint64_t kdesc0 = smem_desc(saddr(smem + L::RING), 16, 1024);
      const uint64_t qdesc0 = smem_desc(saddr(smem + L::Q0), 16, 1024);
      bool ok = mbar_wait(&bars->q_full[0], 0, wt) && (nr < 2 || mbar_wait(&bars->q_full[1], 0, wt));
      for (int j = 0; ok && j < nt; ++j) {
        const uint32_t st = j % PNS;
        if (!mbar_wait(&bars->k_full[st], (j / PNS) & 1, wt)) break;
        fence_after();
        const uint64_t kd = kdesc0 + ((st * L::STAGE) >> 4);
        for (int r = 0; r < nr; ++r) {
          // S_r and P_r share columns: P_r of the previous tile must have been consumed
          if (j >= 1 && !mbar_wait(&bars->o_done[r], (j - 1) & 1, wt)) {
            ok = false;
            break;
          }
          fence_after();
          const uint64_t qd = qdesc0 + ((r * L::TILE) >> 4);
#pragma unroll
          for (int kk = 0; kk < PHD / 16; ++kk) {
            const uint32_t off = (((kk >> 2) * L::BLK) + (kk & 3) * 32) >> 4;
            mma_ss(tmem + PCOL_S + r * 128, qd + off, kd + off, ID_S, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars->s_full[r]);
        }
      }
      mma_commit(&bars->s_final[0]);
      const long long t0 = clock64();
      while (!mbar_try(&bars->s_final[0], 0) && clock64() - t0 < TIMEOUT_CYCLES) {
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ O_r += P_r V issuer
    // P V of row tile 1 is issued after that of row tile 0, so it also comes after row tile
    // 0's warpgroup has cleared the last tile's V rows past the sequence's end.
    if (lane == 0) {
      constexpr uint32_t ID_PV = idesc_bf16(PHD, 1);
      // V: MN-major, 64-column blocks L::BLK apart (LBO), 8-key groups 1024 B apart (SBO)
      const uint64_t vdesc0 = smem_desc(saddr(smem + L::RING + L::TILE), L::BLK, 1024);
      bool ok = true;
      for (int j = 0; ok && j < nt; ++j) {
        const uint32_t st = j % PNS;
        if (!mbar_wait(&bars->v_full[st], (j / PNS) & 1, wt)) break;
        const uint64_t vd = vdesc0 + ((st * L::STAGE) >> 4);
        for (int r = 0; r < nr; ++r) {
          if (!mbar_wait(&bars->p_full[r], j & 1, wt)) {
            ok = false;
            break;
          }
          fence_after();
          // keys [16 kk, 16 kk + 16): P_r columns [8 kk, 8 kk + 8), V rows 16 kk ..
#pragma unroll
          for (int kk = 0; kk < PKT / 16; ++kk)
            mma_ts(tmem + PCOL_O + r * 128, tmem + PCOL_S + r * 128 + kk * 8,
                   vd + ((kk * 16 * 128) >> 4), ID_PV, (j == 0 && kk == 0) ? 0u : 1u);
          mma_commit(&bars->o_done[r]);
        }
        if (!ok) break;
        mma_commit(&bars->kv_empty[st]);
      }
      mma_commit(&bars->s_final[1]);
      const long long t0 = clock64();
      while (!mbar_try(&bars->s_final[1], 0) && clock64() - t0 < TIMEOUT_CYCLES) {
      }
    }
  }
  } else {  // warps 4-11: softmax
  if ((warp - PWG0) / 4 < nr) {
    // ------------------------------------------------------------ softmax, row tile r
    const int r = (warp - PWG0) >> 2;
    const int rr = (warp & 3) * 32 + lane;  // the thread's row in its tile = TMEM lane
    const uint32_t tq = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int rg = r * MT + rr;
    const bool live = rg < rows_total;
    const int i_row = live ? rg / p.G : D;
    const int hl = live ? rg % p.G : 0;
    const int hi_row = T + i_row;  // the row's last visible key
    const float sc = p.scale_log2;
    auto wwait = [&](uint64_t* bar, uint32_t par) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, par, wt));
    };
    // Q row -> this row tile's shared-memory Q tile: 16-byte chunk k of column block c
    // goes to chunk k ^ (row & 7) of the row (the 128-byte swizzle the MMA reads)
    {
      const uint4* qsrc = reinterpret_cast<const uint4*>(
          (const __nv_bfloat16*)p.q + ((q_off + i_row) * p.Hq + (int64_t)g * p.G + hl) * PHD);
      uint8_t* qt = smem + L::Q0 + r * L::TILE + rr * 128;
#pragma unroll
      for (int c = 0; c < PHD / 64; ++c)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 v = live ? __ldg(qsrc + c * 8 + k) : make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(qt + c * L::BLK + ((k ^ (rr & 7)) << 4)) = v;
        }
      fence_proxy_async();
      mbar_arrive(&bars->q_full[r]);
    }
    float m_ref = -INFINITY, lh = 0.f;
    bool good = true;
    for (int j = 0; j < nt && good; ++j) {
      if (!(good = wwait(&bars->s_full[r], j & 1))) break;
      fence_after();
      float sv[PKT];
      {
        uint32_t* raw = reinterpret_cast<uint32_t*>(sv);
#pragma unroll
        for (int c = 0; c < PKT / 32; ++c) tmem_ld32(tq + PCOL_S + r * 128 + c * 32, raw + c * 32);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < PKT / 32; ++c) reg_fence32(raw + c * 32);
      }
      const int key0 = j * PKT;
      if (key0 + PKT - 1 > hi_row) {  // the window-causal mask reaches into this tile
        const int lim = hi_row - key0;
#pragma unroll
        for (int c = 0; c < PKT; ++c)
          if (c > lim) sv[c] = -INFINITY;
      }
      float m8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) m8[e] = sv[e];
#pragma unroll
      for (int c = 8; c < PKT; ++c) m8[c & 7] = fmaxf(m8[c & 7], sv[c]);
      const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                             fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      const float mt = mx * sc;  // tile max in log2 units (sc > 0)
      // Lazy rescale. O_r is not being written here: S_r of this tile was issued after the
      // P V of the previous one had completed. TMEM loads and stores are warp-collective,
      // so the whole warp rescales when any of its rows needs it (alpha = 1 for the rest).
      float alpha = 1.f;
      const bool grow = m_ref != -INFINITY && mt > m_ref + RESCALE_THRESHOLD;
      if (m_ref == -INFINITY) {
        m_ref = mt;
      } else if (grow) {
        alpha = ex2(m_ref - mt);
        lh *= alpha;
        m_ref = mt;
      }
      if (__any_sync(0xffffffffu, grow)) {
#pragma unroll 1
        for (int c = 0; c < PHD / 16; ++c) {
          uint32_t ro[16];
          tmem_ld16(tq + PCOL_O + r * 128 + c * 16, ro);
          tmem_wait_ld();
          reg_fence16(ro);
#pragma unroll
          for (int e = 0; e < 16; ++e) ro[e] = __float_as_uint(__uint_as_float(ro[e]) * alpha);
          tmem_st16(tq + PCOL_O + r * 128 + c * 16, ro);
        }
      }
      const float nmu = m_ref == -INFINITY ? 0.f : -m_ref;
      float s8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) s8[e] = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // 64 keys (32 columns of bf16 pairs) at a time
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float a0 = ex2(fmaf(sv[64 * h + 2 * e], sc, nmu));
          const float a1 = ex2(fmaf(sv[64 * h + 2 * e + 1], sc, nmu));
          s8[e & 7] += a0 + a1;
          pk[e] = pack_bf16(a0, a1);
        }
        tmem_st32(tq + PCOL_S + r * 128 + 32 * h, pk);
      }
      lh += ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
      tmem_wait_st();
      if (r == 0 && key0 + PKT > nkeys) {
        // the V rows past the sequence's end (the next sequence's rows, or memory past the
        // cache) are cleared so that P = 0 never meets non-finite data; both row tiles'
        // P V read this tile, and P V of row tile 1 is issued after that of row tile 0
        const uint32_t st = j % PNS;
        if (!(good = wwait(&bars->v_full[st], (j / PNS) & 1))) break;
        uint8_t* vt = smem + L::RING + st * L::STAGE + L::TILE;
        const int first = nkeys - key0;
        const int chunks = (PKT - first) * 8;  // 16-byte chunks per column block
        for (int q = rr; q < chunks * (PHD / 64); q += 128) {
          const int blk = q / chunks, rem = q % chunks;
          *reinterpret_cast<uint4*>(vt + blk * L::BLK + (first + rem / 8) * 128 + (rem % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();
      }
      fence_before();
      mbar_arrive(&bars->p_full[r]);
    }
    // the last P V of the row tile is complete: O_r / l_r to the output
    if (good && nt > 0) {
      good = wwait(&bars->o_done[r], (nt - 1) & 1);
      if (good) fence_after();
    }
    if (good) {
      const float inv = 1.f / lh;
#pragma unroll 1
      for (int c = 0; c < PHD / 16; ++c) {
        uint32_t ro[16];
        tmem_ld16(tq + PCOL_O + r * 128 + c * 16, ro);
        tmem_wait_ld();
        reg_fence16(ro);
        if (live) {
          __nv_bfloat16* dst = (__nv_bfloat16*)p.out +
                               ((q_off + i_row) * p.Hq + (int64_t)g * p.G + hl) * PHD + c * 16;
          uint32_t pw[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            pw[e] = pack_bf16(__uint_as_float(ro[2 * e]) * inv, __uint_as_float(ro[2 * e + 1]) * inv);
          uint4* d4 = reinterpret_cast<uint4*>(dst);
          d4[0] = make_uint4(pw[0], pw[1], pw[2], pw[3]);
          d4[1] = make_uint4(pw[4], pw[5], pw[6], pw[7]);
        }
      }
    }
  }

  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(P_TMEM_COLS)
                 : "memory");
  }
}

}  // namespace

bool attn_pair_applies(const AttnParams& p, bool fp8, int sms) {
  const int rows = p.G * (1 + p.max_draft);
  return !fp8 && p.d == PHD && p.block_size == 0 && p.window == 0 && rows > MT &&
         rows <= 2 * MT && p.B > 0 && (int64_t)p.B * p.Hkv <= sms && p.kv_rows > 0 &&
         p.kv_rows <= 0x7fffffffLL - PKT;
}

cudaError_t launch_attn_pair(const AttnParams& p, cudaStream_t s) {
  CUtensorMap mk, mv;
  if (!kv_tensor_map(&mk, p.k, p.kv_rows, p.Hkv, PHD, false, PKT) ||
      !kv_tensor_map(&mv, p.v, p.kv_rows, p.Hkv, PHD, false, PKT))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)PairLayout::SMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_pair_kernel, dim3(p.B * p.Hkv), dim3(PTHREADS), PairLayout::SMEM, s, p,
                    mk, mv);
}

}  // namespace sv

// attn_tc.cu -- verify attention on the fifth-generation tensor cores (tcgen05, TMEM, TMA).
//
// Persistent CTAs walk contiguous ranges of the global tile line (see internal.cuh) in
// 128-key tiles. The two softmax warpgroups split every tile by keys: warpgroup w owns
// keys [64w, 64w + 64) of each tile, each of its threads a whole query row of them, with
// its own running max m_w, running sum l_w, TMEM accumulator O_w and P buffer. So the
// warpgroups never exchange maxima per tile, and each half's P V starts as soon as that
// half's P is written. The two partial results of a unit merge once, at its end, with the
// online-softmax rule ("GPU and LLM, chapter 5", "Online softmax").
//
//   warp 0      TMA producer: K and V tiles of one KV head (128 keys x d, 128-byte swizzle)
//               into shared memory; a stage is released once every reader of it has
//               finished. E4M3: 4 stages of a K and a V tile. bf16: 3 such stages, or
//               (split rings, chosen per call) 4 stages of K tiles, each released by its
//               S MMA, while warp 2 fills 3 stages of V tiles, released by their P V, so
//               the K loads run further ahead. A paged cache's tile is one box per
//               block, each loaded by its own lane, the block-table entries read a
//               group of tiles ahead.
//   warp 1      S issuer (one thread): S = Q K^T (N = 128) into the score buffer, which is
//               free again as soon as both warpgroups have read their halves. bf16:
//               kind::f16 with Q (A) read from TMEM and K (B, K-major) from shared memory.
//               FP8: kind::f8f6f4 on the raw E4M3 K tile, with Q held exactly as the sum of
//               two E4M3 terms (see split_q_e4m3): two 8-bit MMAs per 32-element step.
//   warp 3      P V issuer (one thread): O_w += P_w V[64w .. 64w + 64) for each half, with
//               P_w (A) read from TMEM and V (B, MN-major) from shared memory.
//   warps 4..11 softmax, warpgroups 0 (warps 4-7) and 1 (8-11). Per unit they write Q into
//               TMEM (half of d each). Per tile a thread reads its row's 64 scores of its
//               half, releases the score buffer, applies the scale and the window-causal
//               mask (and a sliding window's lower edge), updates m_w and l_w, computes
//               P_w = 2^(s - m_w) into registers, and stores it into its P buffer once
//               its previous P V has consumed the last one. At the end of a unit
//               they merge (O_0, m_0, l_0) with (O_1, m_1, l_1) and store the output, or a
//               split partial.
//   warps 12-15 (FP8 K/V only) decode E4M3 V tiles to f16 tiles for P V (MMAs in f16, P
//               in f16). The K scale folds into the score scale, the V scale into the
//               normalisation.
//
// The online-softmax rescale O_w *= 2^(m_old - m_new) is applied lazily: a reference max
// only moves when a tile's max exceeds it by more than 2^8, so P stays below 256 and the
// exact result is unchanged (numerator and denominator use the same reference).
//
// Every mbarrier wait is bounded: on timeout the kernel sets a flag in the workspace,
// every role leaves its loop, the producers wait (bounded) for their copies in flight, and
// TMEM is freed before the kernel returns. The next kernel on the stream may launch once
// every CTA has finished its work (not at the CTAs' start).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.cuh"
#include "tc_util.cuh"

namespace sv {
namespace {

constexpr int KT = 128;           // keys per tile
constexpr int HK = KT / 2;        // keys per warpgroup per tile
constexpr int NS = 3;             // bf16, paired stages: ring depth (K and V tile each)
constexpr int NSK = 4;            // bf16, split rings: K stages (free after their S MMA)
constexpr int NSV = 3;            // bf16, split rings: V stages (free after their P V)
constexpr int NS8 = 4;            // shared-memory ring depth, E4M3 K/V
constexpr int NSMAX = 4;
constexpr int NCV = 2;            // FP8: decoded V stages
constexpr int NTHREADS = 384;
constexpr int SOFTMAX_WARP0 = 4;  // warps 4..7: warpgroup 0, 8..11: warpgroup 1
constexpr int NSOFT = 256;        // softmax threads (two warpgroups)
constexpr int CONV_WARP0 = 12;    // FP8 only: warps 12-15 decode V tiles
constexpr int NCONV = 128;        // decoding threads
constexpr uint32_t TMEM_COLS = 512;
// TMEM columns: O_0 and O_1 (128 each), the score tile (128), Q (64: bf16 pairs, or the
// E4M3 hi and lo terms), the warpgroups' P buffers (32 each: 64 keys of 16-bit pairs)
constexpr uint32_t COL_O = 0, COL_S = 256, COL_Q = 384, COL_P = 448;

struct __align__(8) Bars {
  uint64_t k_full[NSMAX], v_full[NSMAX];
  uint64_t kv_empty[NSMAX];  // a K + V stage is free (split bf16 rings: a K stage)
  uint64_t v_empty[NSMAX];   // split bf16 rings: a V stage is free
  uint64_t vc_full[NCV], vc_empty[NCV];  // FP8: decoded f16 V tiles
  uint64_t s_full, s_free;               // the score tile: written / read by both halves
  uint64_t p_full[2], o_done[2];         // per warpgroup: P published / its P V complete
  uint64_t q_full, s_final, pv_final;
  uint32_t tmem_base;
  int abort;
  float xm[2][128], xl[2][128];  // end of a unit: each warpgroup's (m, l) per row
};

// Four scaled Q elements x (|x| < 256, at most 8 significant bits each) as hi + lo, both
// E4M3 (the first element in the low byte): hi = x rounded to E4M3, lo = x - hi rounded
// to E4M3. hi keeps the top 4 significant bits and the remainder x - hi is k * ulp(x) with
// |k| <= 8, so lo is exact whenever ulp(x) >= 2^-9 (E4M3's finest step), i.e. |x| >= 1/4;
// below that, |x - hi - lo| <= 2^-10.
__device__ __forceinline__ void split_q_e4m3(const float* x, uint32_t& whi, uint32_t& wlo) {
  const uint32_t h01 = f32x2_to_e4m3x2(x[0], x[1]), h23 = f32x2_to_e4m3x2(x[2], x[3]);
  const float2 d01 = e4m3x2_to_f32x2(h01), d23 = e4m3x2_to_f32x2(h23);
  const uint32_t l01 = f32x2_to_e4m3x2(x[0] - d01.x, x[1] - d01.y);
  const uint32_t l23 = f32x2_to_e4m3x2(x[2] - d23.x, x[3] - d23.y);
  whi = h01 | (h23 << 16);
  wlo = l01 | (l23 << 16);
}

// Where a CTA reads the work plan: the workspace, written by the planning kernel, or a
// HostPlan passed with the launch (kernel parameter space, read through the constant
// cache; every read below is uniform across the threads that make it).
struct WsPlan {
  const AttnParams& p;
  __device__ int num_units() const { return p.hdr->num_units; }
  __device__ int2 cta(int c) const { return p.cta_tab[c]; }
  __device__ int4 unit(int u) const { return p.units[u]; }
  __device__ int32_t ubeg(int u) const { return p.ubeg[u]; }
  __device__ int64_t q_off(int b) const { return p.q_off[b]; }
  __device__ int64_t kv_off(int b) const { return p.kv_off[b]; }
  __device__ int T(int b) const { return p.seq_lens[b]; }
  __device__ int D(int b) const { return p.draft_len[b]; }
};
struct ParamPlan {
  const HostPlan& h;
  __device__ int num_units() const { return h.num_units; }
  __device__ int2 cta(int c) const { return h.cta_tab[c]; }
  __device__ int4 unit(int u) const { return h.units[u]; }
  __device__ int32_t ubeg(int u) const { return h.ubeg[u]; }
  __device__ int64_t q_off(int b) const { return h.q_off[b]; }
  __device__ int64_t kv_off(int b) const { return h.kv_off[b]; }
  __device__ int T(int b) const { return h.T[b]; }
  __device__ int D(int b) const { return h.D[b]; }
};

// One unit's share of a CTA's range: the unit's tiles [j0, j1), tile j holding cache
// positions kbase + j*KT .. (kbase: the first position of the unit's first tile, 0 without
// a sliding window); whole when they are all of the unit's tiles.
struct Seg {
  int u, b, g, mt, j0, j1, kbase;
  bool whole;
};

// Next (unit, tile range) of this CTA's contiguous range of the global tile line.
template <bool WIN, class Plan>
__device__ __forceinline__ bool seg_next(const Plan& pl, int num_units, int64_t& t,
                                         int64_t t_end, int& u, Seg& s) {
  if (t >= t_end || u >= num_units) return false;
  const int4 info = pl.unit(u);
  const int64_t ub = pl.ubeg(u);
  s.u = u;
  s.b = info.x;
  s.g = info.y;
  s.mt = info.z;
  s.kbase = WIN ? info.w : 0;
  const int nt = pl.ubeg(u + 1) - (int)ub;
  s.j0 = (int)(t - ub);
  s.j1 = (int)(min(t_end, ub + nt) - ub);
  if (s.j1 <= s.j0) return false;
  s.whole = s.j0 == 0 && s.j1 == nt;
  t = ub + s.j1;
  ++u;
  return true;
}

// Shared memory. bf16 K/V, paired stages (SPLIT = false): NS stages of (K tile, V tile),
// filled by one TMA producer and freed by the tile's P V. bf16 K/V, split rings (SPLIT):
// NSK K tiles and NSV V tiles, filled by two producers; a K tile is free once its S MMA is
// complete, a V tile once its P V is, so K loads run further ahead of the score MMAs.
// FP8 K/V: an NS8-stage ring of raw E4M3 K and V tiles filled by TMA (K read by the S MMAs
// as it is), and an NCV-stage ring of V tiles decoded to f16 for the P V MMAs.
template <int HD, bool F8, bool SPLIT>
struct TcLayout {
  static_assert(!F8 || HD == 128, "E4M3 rows of one head are one 128-byte swizzle row");
  static_assert(!(F8 && SPLIT), "split rings are a bf16 layout");
  static constexpr int NR = NS8;                               // FP8: raw ring stages
  static constexpr int NRK = F8 ? NS8 : (SPLIT ? NSK : NS);    // stages holding K tiles
  static constexpr int NRV = F8 ? NS8 : (SPLIT ? NSV : NS);    // stages holding V tiles
  static constexpr int BLK = KT * 128;            // one 128-byte-wide column block of a tile
  static constexpr int NBLK = HD / 64;            // 16-bit column blocks per tile
  static constexpr int TILE = KT * HD * 2;        // one 16-bit K or V tile
  // bf16: stage st of the K tiles at KRING + st * KSTEP, of the V tiles at VRING + st * VSTEP
  static constexpr int KRING = 0;
  static constexpr int KSTEP = SPLIT ? TILE : 2 * TILE;
  static constexpr int VRING = SPLIT ? NSK * TILE : TILE;
  static constexpr int VSTEP = SPLIT ? TILE : 2 * TILE;
  static constexpr int RAW = KT * HD;             // one E4M3 tile
  static constexpr int CV = 0;                    // FP8 offsets
  static constexpr int RK = CV + NCV * TILE;
  static constexpr int RV = RK + NR * RAW;
  static constexpr int BARS =
      F8 ? RV + NR * RAW : (SPLIT ? NSK * TILE + NSV * TILE : NS * 2 * TILE);  // barriers
  static constexpr size_t SMEM = (size_t)BARS + sizeof(Bars);
  static_assert(SMEM <= 227 * 1024, "dynamic shared memory above the per-CTA limit");
  static constexpr int THREADS = F8 ? NTHREADS + 4 * 32 : NTHREADS;
};

// WIN: a sliding window is in force (p.window > 0); without it the window's lower mask
// edge, the per-unit key base and the clearing of V rows before the window compile away.
template <int HD, bool F8, bool WIN, bool SPLIT, class Plan>
__device__ __forceinline__ void attn_tc_body(const AttnParams& p, const CUtensorMap& tmk,
                                             const CUtensorMap& tmv, const Plan& pl) {
  using L = TcLayout<HD, F8, SPLIT>;
  const int window = WIN ? p.window : 0;
  extern __shared__ __align__(1024) uint8_t smem[];  // 128-byte swizzled tiles: 1 KiB aligned
  Bars* bars = (Bars*)(smem + L::BARS);
  volatile int* abort = &bars->abort;
  const Waiter wt{abort, p.flags, p.wait_limit > 0 ? p.wait_limit : TIMEOUT_CYCLES};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();  // the plan of this call is complete

  const int num_units = pl.num_units();
  const int2 rb = pl.cta(blockIdx.x), re = pl.cta(blockIdx.x + 1);
  const int64_t t_begin = rb.x, t_end = re.x;  // this CTA's tiles (see the plan kernel)
  if (t_begin >= t_end) return;                // uniform across the CTA
  if (saddr(smem) & 1023) {  // the swizzle phases below assume a 1 KiB-aligned base
    if (tid == 0) atomicOr(p.flags, FLAG_ATTN_SHAPE);
    return;
  }

  if (tid == 0) {
    for (int s = 0; s < NSMAX; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      // FP8: freed by the S commit and the V decoders; bf16 paired stages: by the P V
      // commit; split rings: by the S commit
      mbar_init(&bars->kv_empty[s], F8 ? NCONV + 1 : 1);
      mbar_init(&bars->v_empty[s], 1);  // split rings: freed by the P V commit
    }
    for (int s = 0; s < NCV; ++s) {
      mbar_init(&bars->vc_full[s], NCONV);
      mbar_init(&bars->vc_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, NSOFT);
    for (int w = 0; w < 2; ++w) {
      mbar_init(&bars->p_full[w], NSOFT / 2);
      mbar_init(&bars->o_done[w], 1);
    }
    mbar_init(&bars->q_full, NSOFT);
    mbar_init(&bars->s_final, 1);
    mbar_init(&bars->pv_final, 1);
    bars->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     saddr(&bars->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = bars->tmem_base;
  const int u_first = rb.y;

  if (warp == 0 || (SPLIT && warp == 2)) {
    // ------------------------------------------------------------ TMA producers
    // FP8 and paired bf16 stages: warp 0 loads K and V. Split bf16 rings: warp 0 fills the
    // K ring and warp 2 the V ring, each waiting only for its own ring's stages.
    // Packed cache: lane 0 loads one box of KT rows per tile and tensor. Paged cache: a
    // tile is KT / box boxes of box = min(block_size, KT) rows, each from the physical
    // block the block table names, spread over the lanes (lane n loads box n). The table
    // entries are requested a group of tiles ahead (one entry per lane), so a lookup never
    // waits at its tile behind the copies in flight; a box holding no position a row of
    // the unit can see (past the sequence's end, or wholly before its sliding window) is
    // not looked up and loads from a negative row, which fills it with zeros. Lane 0 waits
    // for the stage and arms its barriers.
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmk) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmv) : "memory");
    }
    const bool do_k = !SPLIT || warp == 0, do_v = !SPLIT || warp == 2;
    const uint32_t nr = do_k ? L::NRK : L::NRV;  // this producer's ring depth
    uint64_t* empty = do_k ? bars->kv_empty : bars->v_empty;
    int64_t t = t_begin;
    int u = u_first;
    Seg s;
    uint32_t it = 0;
    bool ok = true;
    const int box = p.block_size > 0 ? min(p.block_size, KT) : KT;
    const int nbox = KT / box;  // boxes per tile, one per lane
    // test hook: the first tile of the CTA's range is never loaded (its barriers are never
    // armed), so every wait for it runs out; stage 0 then holds no copy to wait for
    const bool withhold = p.stall_first_tile != 0;
    auto load_k = [&](uint32_t st, int n, int g, int grow) {
      const uint32_t roff = (uint32_t)(n * box * 128);
      if constexpr (F8) {
        tma_load_3d(saddr(smem + L::RK + st * L::RAW) + roff, &tmk, &bars->k_full[st], 0, g,
                    grow);
      } else {
#pragma unroll
        for (int c = 0; c < L::NBLK; ++c)
          tma_load_3d(saddr(smem + L::KRING + st * L::KSTEP) + c * L::BLK + roff, &tmk,
                      &bars->k_full[st], c * 64, g, grow);
      }
    };
    auto load_v = [&](uint32_t st, int n, int g, int grow) {
      const uint32_t roff = (uint32_t)(n * box * 128);
      if constexpr (F8) {
        tma_load_3d(saddr(smem + L::RV + st * L::RAW) + roff, &tmv, &bars->v_full[st], 0, g,
                    grow);
      } else {
#pragma unroll
        for (int c = 0; c < L::NBLK; ++c)
          tma_load_3d(saddr(smem + L::VRING + st * L::VSTEP) + c * L::BLK + roff, &tmv,
                      &bars->v_full[st], c * 64, g, grow);
      }
    };
    while (ok && seg_next<WIN>(pl, num_units, t, t_end, u, s)) {
      const int row0 = (int)pl.kv_off(s.b) + s.kbase;
      const int T = pl.T(s.b);
      const int nkeys = T + pl.D(s.b) + 1;
      const int kvis = first_visible_key(T, window);
      const int32_t* tab = p.block_table + (size_t)s.b * p.bt_stride;
      // Paged: the block-table entries of a group of tg = 32 / nbox tiles are loaded one
      // per lane (lane l: tile l / nbox of the group, box l % nbox) a whole group ahead of
      // their use, so that no lookup waits behind this SM's copies in flight; at its tile
      // each box's lane takes its entry from the group's lanes.
      const int tg = 32 / nbox;
      auto box_pos = [&](int j, int n) { return s.kbase + j * KT + n * box; };
      auto visible = [&](int pos) { return pos < nkeys && pos + box > kvis; };
      auto fetch = [&](int jg) -> int {  // this lane's entry of the group starting at tile jg
        int e = 0;
        const int j = jg + lane / nbox, pos = box_pos(j, lane % nbox);
        if (p.block_size > 0 && j < s.j1 && visible(pos)) e = __ldg(tab + (pos >> p.bs_log2));
        return e;
      };
      int ent_cur = fetch(s.j0), ent_nxt = fetch(s.j0 + tg);
      // first cache row of box n of tile j (paged), from its table entry blk
      auto paged_row = [&](int j, int n, int blk) -> int {
        const int pos = box_pos(j, n);
        if (!visible(pos)) return -box;
        if (blk < 0 || blk >= p.num_blocks) {  // a table entry outside the pool
          atomicOr(p.flags, FLAG_ATTN_SHAPE);
          return -box;
        }
        return blk * p.block_size + (pos & (p.block_size - 1));
      };
      for (int j = s.j0; j < s.j1; ++j, ++it) {
        const uint32_t st = it % nr;
        const bool mine = p.block_size == 0 ? lane == 0 : lane < nbox;
        int grow = row0 + j * KT;
        if (p.block_size > 0) {
          const int q = (j - s.j0) % tg;
          if (q == 0 && j > s.j0) {  // the next group: its entries were requested tg tiles ago
            ent_cur = ent_nxt;
            ent_nxt = fetch(j + tg);
          }
          const int blk = __shfl_sync(0xffffffffu, ent_cur, q * nbox + lane % nbox);
          grow = mine ? paged_row(j, lane, blk) : 0;
        }
        bool w = true;
        if (it >= nr && lane == 0) w = mbar_wait(&empty[st], ((it / nr) - 1) & 1, wt);
        if (!__shfl_sync(0xffffffffu, w, 0)) {
          ok = false;
          break;
        }
        if (withhold && it == 0) continue;
        // the boxes of a tile add up to one full tile per tensor
        if (do_k) {
          if (lane == 0) mbar_expect_tx(&bars->k_full[st], F8 ? L::RAW : L::TILE);
          __syncwarp();
          if (mine) load_k(st, lane, s.g, grow);
        }
        if (do_v) {
          if (lane == 0) mbar_expect_tx(&bars->v_full[st], F8 ? L::RAW : L::TILE);
          __syncwarp();
          if (mine) load_v(st, lane, s.g, grow);
        }
      }
    }
    if (lane == 0) {
      // leave no copy in flight: wait (bounded) for the last fill of every stage. Normally
      // its readers have waited for it too; after another role gave up they may not have,
      // and the copy must land before the CTA's shared memory is released.
      for (uint32_t st = withhold ? 1 : 0; st < nr && st < it; ++st) {
        const uint32_t fills = (it - 1 - st) / nr + 1;
        const uint32_t par = (fills - 1) & 1;
        const long long t0 = clock64();
        while (!((!do_k || mbar_try(&bars->k_full[st], par)) &&
                 (!do_v || mbar_try(&bars->v_full[st], par))) &&
               clock64() - t0 < TIMEOUT_CYCLES) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S = Q K^T issuer
    if (lane == 0) {
      constexpr uint32_t ID_S = F8 ? idesc_e4m3(KT) : idesc_bf16(KT, 0);
      // K: K-major, 128-byte rows, 8-row groups 1024 B apart; 32 B per K step (16 bf16 or
      // 32 E4M3 elements)
      const uint64_t kdesc0 = smem_desc(saddr(smem + (F8 ? L::RK : L::KRING)), 16, 1024);
      int64_t t = t_begin;
      int u = u_first;
      Seg s;
      uint32_t it = 0, seg_i = 0;
      bool ok = true;
      while (ok && seg_next<WIN>(pl, num_units, t, t_end, u, s)) {
        if (!mbar_wait(&bars->q_full, seg_i & 1, wt)) break;
        fence_after();
        for (int j = s.j0; j < s.j1; ++j, ++it) {
          const uint32_t st = it % L::NRK;
          if (!mbar_wait(&bars->k_full[st], (it / L::NRK) & 1, wt) ||
              (it >= 1 && !mbar_wait(&bars->s_free, (it - 1) & 1, wt))) {
            ok = false;
            break;
          }
          fence_after();
          const uint64_t kd = kdesc0 + ((st * (F8 ? L::RAW : L::KSTEP)) >> 4);
          const uint32_t dcol = tmem + COL_S;
          if constexpr (F8) {
            // S = Q_hi K^T + Q_lo K^T: Q_hi in TMEM columns [COL_Q, +32), Q_lo in [+32, +64)
#pragma unroll
            for (int kk = 0; kk < HD / 32; ++kk) {
              mma_ts_e4m3(dcol, tmem + COL_Q + kk * 8, kd + ((kk * 32) >> 4), ID_S,
                          kk > 0 ? 1u : 0u);
              mma_ts_e4m3(dcol, tmem + COL_Q + 32 + kk * 8, kd + ((kk * 32) >> 4), ID_S, 1u);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk)
              mma_ts(dcol, tmem + COL_Q + kk * 8,
                     kd + ((((kk >> 2) * L::BLK) + (kk & 3) * 32) >> 4), ID_S, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars->s_full);
          // the K tile is read: an FP8 raw stage's K half, or a split ring's K stage
          if constexpr (F8 || SPLIT) mma_commit(&bars->kv_empty[st]);
        }
        ++seg_i;
      }
      mma_commit(&bars->s_final);
      const long long t0 = clock64();
      while (!mbar_try(&bars->s_final, 0) && clock64() - t0 < TIMEOUT_CYCLES) {
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ O_w += P V issuer
    if (lane == 0) {
      constexpr uint32_t ID_PV = F8 ? idesc_f16(HD, 1) : idesc_bf16(HD, 1);
      // V: MN-major, 64-column blocks L::BLK apart (LBO), 8-key groups 1024 B apart (SBO)
      const uint64_t vdesc0 = smem_desc(saddr(smem + (F8 ? L::CV : L::VRING)), L::BLK, 1024);
      int64_t t = t_begin;
      int u = u_first;
      Seg s;
      uint32_t it = 0;
      bool ok = true;
      while (ok && seg_next<WIN>(pl, num_units, t, t_end, u, s)) {
        bool first[2] = {true, true};  // each accumulator starts afresh in every unit
        for (int j = s.j0; j < s.j1; ++j, ++it) {
          const uint32_t st = F8 ? it % NCV : it % L::NRV;
          uint64_t* vready = F8 ? &bars->vc_full[st] : &bars->v_full[st];
          const uint32_t vpar = F8 ? (it / NCV) & 1 : (it / L::NRV) & 1;
          if (!mbar_wait(vready, vpar, wt)) {
            ok = false;
            break;
          }
          const uint64_t vd = vdesc0 + ((st * (F8 ? L::TILE : L::VSTEP)) >> 4);
          for (int w = 0; w < 2 && ok; ++w) {
            if (!mbar_wait(&bars->p_full[w], it & 1, wt)) {
              ok = false;
              break;
            }
            fence_after();
            // keys [64w + 16kk, +16): rows 64w + 16kk of the V tile (128 bytes each)
#pragma unroll
            for (int kk = 0; kk < HK / 16; ++kk)
              mma_ts(tmem + COL_O + w * 128, tmem + COL_P + w * (HK / 2) + kk * 8,
                     vd + (((w * HK + kk * 16) * 128) >> 4), ID_PV,
                     (first[w] && kk == 0) ? 0u : 1u);
            first[w] = false;
            mma_commit(&bars->o_done[w]);
          }
          if (!ok) break;
          mma_commit(F8 ? &bars->vc_empty[st] : SPLIT ? &bars->v_empty[st] : &bars->kv_empty[st]);
        }
      }
      mma_commit(&bars->pv_final);
      const long long t0 = clock64();
      while (!mbar_try(&bars->pv_final, 0) && clock64() - t0 < TIMEOUT_CYCLES) {
      }
    }
  } else if (warp >= SOFTMAX_WARP0 && warp < SOFTMAX_WARP0 + NSOFT / 32) {
    // ------------------------------------------------------------ softmax / epilogue
    const int wg = (warp - SOFTMAX_WARP0) >> 2;
    const int r = (warp & 3) * 32 + lane;  // query row = TMEM lane
    const uint32_t tq = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t colS = COL_S + wg * HK;
    constexpr int OC = HD / 2;             // output columns per warpgroup in the epilogue
    auto wwait = [&](uint64_t* bar, uint32_t par) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, par, wt));
    };
    int64_t t = t_begin;
    int u = u_first;
    Seg s;
    uint32_t it = 0;
    bool ok = true;
    while (ok && seg_next<WIN>(pl, num_units, t, t_end, u, s)) {
      // cache positions below are relative to the unit's first tile (kbase)
      const int T = pl.T(s.b) - s.kbase;
      const int D = pl.D(s.b);
      const int rows_total = p.G * (D + 1);
      const int rows = min(MT, rows_total - s.mt * MT);
      const int nkeys = T + D + 1;
      const int rg = s.mt * MT + r;
      const bool live = r < rows;
      const int i_row = live ? rg / p.G : D;
      const int hi_row = T + i_row;  // the row's last visible key
      const int hl = live ? rg % p.G : 0;
      const int64_t qrow = pl.q_off(s.b) + i_row;
      float sc = p.scale_log2;  // score scale in log2 units
      const float vs = F8 ? p.kv_scale[p.Hkv + s.g] : 1.f;
      const uint4* qsrc = reinterpret_cast<const uint4*>(
          (const __nv_bfloat16*)p.q + (qrow * p.Hq + (int64_t)s.g * p.G + hl) * HD);

      if constexpr (F8) {
        // Q row x 2^e -> E4M3 hi + lo terms in TMEM columns [COL_Q, +32) and [+32, +64),
        // this warpgroup's half of d in each. e puts the row's largest |q| in [128, 256),
        // so the pair holds every element to within 2^-17 of that maximum (exactly, for
        // elements within 2^-9 of it); 2^-e joins the K scale in the score scale.
        uint32_t rq[HD / 4];  // this warpgroup's half of the row
        uint32_t amax = 0;    // largest bf16 magnitude of the row (integer order = magnitude)
#pragma unroll
        for (int e = 0; e < HD / 16; ++e) {
          const uint4 v = live ? __ldg(qsrc + wg * (HD / 16) + e) : make_uint4(0, 0, 0, 0);
          const uint4 o = live ? __ldg(qsrc + (wg ^ 1) * (HD / 16) + e) : make_uint4(0, 0, 0, 0);
          rq[4 * e] = v.x;
          rq[4 * e + 1] = v.y;
          rq[4 * e + 2] = v.z;
          rq[4 * e + 3] = v.w;
          const uint32_t both[8] = {v.x, v.y, v.z, v.w, o.x, o.y, o.z, o.w};
#pragma unroll
          for (int k = 0; k < 8; ++k)
            amax = max(amax, max(both[k] & 0x7fffu, (both[k] >> 16) & 0x7fffu));
        }
        // amax in [2^(eb-127), 2^(eb-126)): e = 8 - (eb - 126), clamped to keep 2^+-e normal
        const int eb = max((int)(amax >> 7), 1);
        const int e2 = amax == 0 ? 0 : min(max(134 - eb, -120), 120);
        const float f = __int_as_float((e2 + 127) << 23);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {  // 8 columns (32 elements) at a time
          uint32_t hi[8], lo[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t a = rq[16 * hh + 2 * c], b = rq[16 * hh + 2 * c + 1];
            const float x[4] = {__uint_as_float(a << 16) * f, __uint_as_float(a & 0xffff0000u) * f,
                                __uint_as_float(b << 16) * f, __uint_as_float(b & 0xffff0000u) * f};
            split_q_e4m3(x, hi[c], lo[c]);
          }
          tmem_st8(tq + COL_Q + wg * 16 + 8 * hh, hi);
          tmem_st8(tq + COL_Q + 32 + wg * 16 + 8 * hh, lo);
        }
        tmem_wait_st();
        sc = p.scale_log2 * p.kv_scale[s.g] * __int_as_float((127 - e2) << 23);
      } else if (wg < HD / 64) {
        // Q row -> TMEM columns [COL_Q, COL_Q + HD/2) as packed bf16 pairs, 32 columns per
        // store (both warpgroups for d = 128, the first one for d = 64)
        uint32_t rq[32];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint4 v = live ? __ldg(qsrc + wg * 8 + e) : make_uint4(0, 0, 0, 0);
          rq[4 * e] = v.x;
          rq[4 * e + 1] = v.y;
          rq[4 * e + 2] = v.z;
          rq[4 * e + 3] = v.w;
        }
        tmem_st32(tq + COL_Q + wg * 32, rq);
        tmem_wait_st();
      }
      fence_before();
      mbar_arrive(&bars->q_full);

      // this warpgroup's half of every tile of the unit
      float m_ref = -INFINITY, lh = 0.f;
      uint32_t it_last = 0;
      bool good = true;
      for (int j = s.j0; j < s.j1; ++j, ++it) {
        if (!good) continue;
        it_last = it;
        if (!(good = wwait(&bars->s_full, it & 1))) continue;
        fence_after();
        float sv[HK];
        {
          uint32_t* raw = reinterpret_cast<uint32_t*>(sv);
#pragma unroll
          for (int c = 0; c < HK / 32; ++c) tmem_ld32(tq + colS + c * 32, raw + c * 32);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < HK / 32; ++c) reg_fence32(raw + c * 32);
        }
        fence_before();
        mbar_arrive(&bars->s_free);  // the scores are in registers: the next S may start
        const int key0 = j * KT + wg * HK;
        // the window-causal mask (key <= T + i) or the sliding window's lower edge
        // (key >= T + i - window + 1) reaches into this half tile for this row
        const int lo_row = hi_row + 1 - window;  // (used only under a sliding window)
        if (key0 + HK - 1 > hi_row) {
          const int lim = hi_row - key0;
#pragma unroll
          for (int c = 0; c < HK; ++c)
            if (c > lim) sv[c] = -INFINITY;
        }
        if (WIN && key0 < lo_row) {
          const int low = lo_row - key0;
#pragma unroll
          for (int c = 0; c < HK; ++c)
            if (c < low) sv[c] = -INFINITY;
        }
        // The E4M3 tile, whose softmax bounds the tile period, takes the maximum in chains
        // of three-operand maxima and the exponent arguments and row sums two at a time
        // (paired f32 instructions, each half rounded as alone): c3 122.9 -> 119.8 us. The
        // bf16 tiles keep single instructions (c2 and c4 D = 15, which stream at the HBM
        // rate, measured 0.5-0.9% slower with the paired forms).
        static_assert(HK == 64, "eight chains of eight scores");
        float m8[8];
        if constexpr (F8) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            m8[e] = max3f(sv[e], sv[e + 8], sv[e + 16]);
            m8[e] = max3f(m8[e], sv[e + 24], sv[e + 32]);
            m8[e] = max3f(m8[e], sv[e + 40], sv[e + 48]);
            m8[e] = fmaxf(m8[e], sv[e + 56]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) m8[e] = sv[e];
#pragma unroll
          for (int c = 8; c < HK; ++c) m8[c & 7] = fmaxf(m8[c & 7], sv[c]);
        }
        const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        const float mt = mx * sc;  // tile max in log2 units (sc > 0)
        // The decision is per row, but TMEM loads and stores are warp-collective: the whole
        // warp rescales when any of its rows needs it, with alpha = 1 for the others.
        float alpha = 1.f;
        const bool grow = m_ref != -INFINITY && mt > m_ref + RESCALE_THRESHOLD;
        if (m_ref == -INFINITY) {
          m_ref = mt;  // O_w holds nothing yet for this row (zeros or about to be overwritten)
        } else if (grow) {
          alpha = ex2(m_ref - mt);
          lh *= alpha;
          m_ref = mt;
        }
        // P = 2^(s - m_ref) in registers, packed, while this warpgroup's previous P V may
        // still be running
        const float nmu = m_ref == -INFINITY ? 0.f : -m_ref;
        float s8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) s8[e] = 0.f;
        if constexpr (F8) {
#pragma unroll
          for (int e = 0; e < HK / 2; ++e) {
            fma2(sv[2 * e], sv[2 * e + 1], sc, nmu);
            sv[2 * e] = ex2(sv[2 * e]);
            sv[2 * e + 1] = ex2(sv[2 * e + 1]);
            add2(s8[(e & 3) * 2], s8[(e & 3) * 2 + 1], sv[2 * e], sv[2 * e + 1]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < HK; ++c) {
            sv[c] = ex2(fmaf(sv[c], sc, nmu));
            s8[c & 7] += sv[c];
          }
        }
        lh += ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
        uint32_t pk[HK / 2];
#pragma unroll
        for (int e = 0; e < HK / 2; ++e) pk[e] = pack_p<F8>(sv[2 * e], sv[2 * e + 1]);
        // O_w and the P buffer are reused once this warpgroup's previous P V is complete.
        // Its barrier cannot be two phases behind: that tile's P was stored only after
        // the P V before it had completed.
        if (it >= 1) {
          if (!(good = wwait(&bars->o_done[wg], (it - 1) & 1))) continue;
          fence_after();
        }
        if (__any_sync(0xffffffffu, grow)) {  // (never on a unit's first tile)
#pragma unroll 1
          for (int c = 0; c < HD / 16; ++c) {  // 16 columns at a time: P stays in registers
            uint32_t ro[16];
            tmem_ld16(tq + COL_O + wg * 128 + c * 16, ro);
            tmem_wait_ld();
            reg_fence16(ro);
#pragma unroll
            for (int e = 0; e < 16; ++e) ro[e] = __float_as_uint(__uint_as_float(ro[e]) * alpha);
            tmem_st16(tq + COL_O + wg * 128 + c * 16, ro);
          }
        }
        tmem_st32(tq + COL_P + wg * (HK / 2), pk);
        tmem_wait_st();
        bool zeroed = false;
        // under a sliding window, keys before T - window + 1 left every row's window
        const int kvis = WIN ? T + 1 - window : -1;
        if (!F8 && (key0 + HK > nkeys || key0 < kvis)) {
          // clear this half's V rows past the sequence's end (they may hold the next
          // sequence or unwritten memory) and, under a sliding window, before the first
          // visible key (left the window: any bits), so that P = 0 never meets non-finite
          // data
          const uint32_t st = it % L::NRV;
          if (!(good = wwait(&bars->v_full[st], (it / L::NRV) & 1))) continue;
          uint8_t* vt = smem + L::VRING + st * L::VSTEP;
          auto clear_rows = [&](int first, int end) {  // tile rows [first, end)
            const int chunks = (end - first) * 8;  // 16-byte chunks per column block
            for (int q = r; q < chunks * L::NBLK; q += NSOFT / 2) {
              const int blk = q / chunks, rem = q % chunks;
              *reinterpret_cast<uint4*>(vt + blk * L::BLK + (first + rem / 8) * 128 + (rem % 8) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
          };
          const int h0 = wg * HK, h1 = h0 + HK;  // this half's rows of the tile
          const int lo_end = min(max(kvis - key0, 0), HK) + h0;
          const int hi_first = max(min(nkeys - key0, HK), 0) + h0;
          if (lo_end > h0) clear_rows(h0, lo_end);
          if (hi_first < h1) clear_rows(max(hi_first, lo_end), h1);
          zeroed = true;
        }
        if (zeroed) fence_proxy_async();
        fence_before();
        mbar_arrive(&bars->p_full[wg]);
      }
      // this warpgroup's last P V of the unit (and with it every earlier one) is complete
      if (good) {
        good = wwait(&bars->o_done[wg], it_last & 1);
        if (good) fence_after();
      }
      bars->xm[wg][r] = m_ref;
      bars->xl[wg][r] = lh;
      if (!softmax_pair_and(good)) {
        ok = false;
        break;
      }
      fence_after();  // the other warpgroup's accumulator is complete too

      // ---- epilogue: merge the two accumulators; this warpgroup's half of the columns
      const float m0 = bars->xm[0][r], m1 = bars->xm[1][r];
      const float m = fmaxf(m0, m1);
      const float a0 = m0 == -INFINITY ? 0.f : ex2(m0 - m);
      const float a1 = m1 == -INFINITY ? 0.f : ex2(m1 - m);
      const float l = a0 * bars->xl[0][r] + a1 * bars->xl[1][r];
      const bool whole = s.whole;
      const float inv = whole ? vs / l : 1.f;
      auto merged = [&](uint32_t o0, uint32_t o1) {  // an accumulator without tiles is skipped
        return (a0 != 0.f ? a0 * __uint_as_float(o0) : 0.f) +
               (a1 != 0.f ? a1 * __uint_as_float(o1) : 0.f);
      };
#pragma unroll 1
      for (int c = 0; c < OC / 16; ++c) {
        uint32_t r0[16], r1[16];
        tmem_ld16(tq + COL_O + wg * OC + c * 16, r0);
        tmem_ld16(tq + COL_O + 128 + wg * OC + c * 16, r1);
        tmem_wait_ld();
        reg_fence16(r0);
        reg_fence16(r1);
        if (live) {
          if (whole) {
            __nv_bfloat16* dst = (__nv_bfloat16*)p.out +
                                 ((pl.q_off(s.b) + i_row) * p.Hq + (int64_t)s.g * p.G + hl) * HD +
                                 wg * OC + c * 16;
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              pk[e] = pack_bf16(merged(r0[2 * e], r1[2 * e]) * inv,
                                merged(r0[2 * e + 1], r1[2 * e + 1]) * inv);
            uint4* d4 = reinterpret_cast<uint4*>(dst);
            d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          } else {
            const size_t slot = (size_t)blockIdx.x + s.u;
            float4* d4 = reinterpret_cast<float4*>(p.part_o + (slot * MT + r) * HD + wg * OC + c * 16);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              d4[e] = make_float4(merged(r0[4 * e], r1[4 * e]), merged(r0[4 * e + 1], r1[4 * e + 1]),
                                  merged(r0[4 * e + 2], r1[4 * e + 2]),
                                  merged(r0[4 * e + 3], r1[4 * e + 3]));
          }
        }
      }
      if (!whole && live && wg == 0) p.part_ml[((size_t)blockIdx.x + s.u) * MT + r] = make_float2(m, l);
      fence_before();  // TMEM reads above complete before the next unit's MMAs
    }
  }

  if constexpr (F8) {
    if (warp >= CONV_WARP0) {
      // ---------------------------------------------------------- E4M3 -> f16 V decoding
      // Raw 128-byte swizzled rows in, the 16-bit MN-major operand layout of the bf16 path
      // (two 64-column swizzled blocks) out. Thread ct owns 16-byte chunk column c = ct & 7
      // of rows rw + 16k, rw = (ct >> 3) ^ (c >> 2): each group of eight lanes takes the
      // eight chunk columns from two rows of opposite parity, so its 16-byte loads and
      // stores fall in eight different bank groups. Rows past the sequence's last key, and
      // rows before its first visible key under a sliding window, are written as zeros (P
      // is zero there, and 0 x NaN would not be).
      const int ct = (warp - CONV_WARP0) * 32 + lane;
      const int c = ct & 7;
      const int rw = (ct >> 3) ^ (c >> 2);
      const int ph = rw & 7;  // swizzle phase of rows rw + 16k
      const uint32_t src_off = rw * 128 + ((c ^ ph) << 4);
      const uint32_t dst_off = (c >> 2) * L::BLK + rw * 128;
      const uint32_t w0 = ((2 * (c & 3)) ^ ph) << 4, w1 = ((2 * (c & 3) + 1) ^ ph) << 4;
      constexpr int RSTEP = 16 * 128;  // bytes between a thread's rows
      int64_t t = t_begin;
      int u = u_first;
      Seg s;
      uint32_t it = 0;
      bool ok = true;
      while (ok && seg_next<WIN>(pl, num_units, t, t_end, u, s)) {
        // cache positions relative to the unit's first tile
        const int T = pl.T(s.b) - s.kbase;
        const int nkeys = T + pl.D(s.b) + 1;
        const int kvis = WIN ? T + 1 - window : -1;
        for (int j = s.j0; j < s.j1; ++j, ++it) {
          const uint32_t rs = it % L::NR, cs = it % NCV;
          if (!mbar_wait(&bars->v_full[rs], (it / L::NR) & 1, wt) ||
              (it >= NCV && !mbar_wait(&bars->vc_empty[cs], ((it / NCV) - 1) & 1, wt))) {
            ok = false;
            break;
          }
          fence_after();
          const uint8_t* rsrc = smem + L::RV + rs * L::RAW + src_off;
          uint8_t* cdst = smem + L::CV + cs * L::TILE + dst_off;
          uint4 w[KT / 16];
#pragma unroll
          for (int k = 0; k < KT / 16; ++k)
            w[k] = *reinterpret_cast<const uint4*>(rsrc + k * RSTEP);
          mbar_arrive(&bars->kv_empty[rs]);  // the raw V tile is read
          const int lim = nkeys - j * KT;    // rows >= lim lie past the sequence's end
          const int low = kvis - j * KT;     // rows < low left the sliding window
#pragma unroll
          for (int k = 0; k < KT / 16; ++k) {
            uint32_t h[8];
            e4m3x4_to_f16x4(w[k].x, h[0], h[1]);
            e4m3x4_to_f16x4(w[k].y, h[2], h[3]);
            e4m3x4_to_f16x4(w[k].z, h[4], h[5]);
            e4m3x4_to_f16x4(w[k].w, h[6], h[7]);
            if (rw + 16 * k >= lim || rw + 16 * k < low) {
#pragma unroll
              for (int e = 0; e < 8; ++e) h[e] = 0u;
            }
            uint8_t* row = cdst + k * RSTEP;
            *reinterpret_cast<uint4*>(row + w0) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(row + w1) = make_uint4(h[4], h[5], h[6], h[7]);
          }
          fence_proxy_async();
          mbar_arrive(&bars->vc_full[cs]);
        }
      }
    }
  }

  fence_before();
  __syncthreads();
  fence_after();
  // The next kernel (the split-KV combine) may launch once every CTA is here or gone:
  // released at the start instead, its CTAs and the acceptance kernel's after it took SMs
  // during this kernel (same box, steps: c3 147.3 vs 146.6 us, c2 with host lengths 116.2
  // vs 115.4 us, c2 122.5 either way).
  pdl_trigger();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// Device-planned launch: the plan in the workspace, written by the planning kernel.
template <int HD, bool F8, bool WIN, bool SPLIT>
__global__ void __launch_bounds__(F8 ? NTHREADS + 128 : NTHREADS, 1)
    attn_tc_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv) {
  attn_tc_body<HD, F8, WIN, SPLIT>(p, tmk, tmv, WsPlan{p});
}

// Host-planned launch: the plan travels with the launch. CTA 0 also copies what the
// combine kernel reads (unit list, unit starts, query offsets, counts) into the workspace.
template <int HD, bool F8, bool WIN, bool SPLIT>
__global__ void __launch_bounds__(F8 ? NTHREADS + 128 : NTHREADS, 1)
    attn_tc_kernel_hp(const AttnParams p, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv,
                      const __grid_constant__ HostPlan hp) {
  if (blockIdx.x == 0) {
    pdl_wait();  // the previous call's combine has read the workspace
    for (int u = threadIdx.x; u <= hp.num_units; u += blockDim.x) {
      if (u < hp.num_units) p.units[u] = hp.units[u];
      p.ubeg[u] = hp.ubeg[u];
    }
    for (int b = threadIdx.x; b <= p.B; b += blockDim.x) p.q_off[b] = hp.q_off[b];
    if (threadIdx.x == 0) {
      p.hdr->num_units = hp.num_units;
      p.hdr->total_tiles = hp.total_tiles;
      p.hdr->unit_ctas = hp.unit_ctas;
    }
  }
  attn_tc_body<HD, F8, WIN, SPLIT>(p, tmk, tmv, ParamPlan{hp});
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)f;
  }
  return fn;
}

// [kv_rows, Hkv, HD] -> boxes of 128 bytes x 1 head x KT rows, 128-byte swizzle: 64 bf16
// columns, or 128 one-byte E4M3 codes.
// Rows of `box_rows` cache positions of one KV head (box_rows: KT, or a paged cache's
// block size when that is smaller; a multiple of 8 keeps every box on a whole 1 KiB
// swizzle period in shared memory).
bool make_kv_map(CUtensorMap* map, const void* base, int64_t kv_rows, int hkv, int hd, bool fp8,
                 int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t es = fp8 ? 1 : 2;
  const cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)hkv, (cuuint64_t)kv_rows};
  const cuuint64_t strides[2] = {(cuuint64_t)hd * es, (cuuint64_t)hkv * hd * es};
  const cuuint32_t box[3] = {(cuuint32_t)(128 / es), 1, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B,
            // promote L2 fills to the bytes of one (row, head): 256 B of bf16, 128 B of E4M3;
            // wider fills would pull in the neighbouring head and double the DRAM traffic
            fp8 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int HD, bool F8, bool WIN, bool SPLIT>
cudaError_t launch_hd(const AttnParams& p, cudaStream_t s) {
  using L = TcLayout<HD, F8, SPLIT>;
  CUtensorMap mk, mv;
  const int box = p.block_size > 0 ? min(p.block_size, KT) : KT;
  if (!make_kv_map(&mk, p.k, p.kv_rows, p.Hkv, HD, F8, box) ||
      !make_kv_map(&mv, p.v, p.kv_rows, p.Hkv, HD, F8, box))
    return cudaErrorInvalidValue;
  auto kernel = attn_tc_kernel<HD, F8, WIN, SPLIT>;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::SMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, dim3(p.n_ctas), dim3(L::THREADS), L::SMEM, s, p, mk, mv);
}

template <int HD, bool F8, bool WIN>
cudaError_t launch_hd(const AttnParams& p, cudaStream_t s) {
  if constexpr (F8)
    return launch_hd<HD, F8, WIN, false>(p, s);
  else
    return p.kv_rings ? launch_hd<HD, F8, WIN, true>(p, s) : launch_hd<HD, F8, WIN, false>(p, s);
}

template <int HD, bool F8>
cudaError_t launch_hd(const AttnParams& p, cudaStream_t s) {
  return p.window > 0 ? launch_hd<HD, F8, true>(p, s) : launch_hd<HD, F8, false>(p, s);
}

template <int HD, bool F8, bool WIN, bool SPLIT>
cudaError_t launch_hd_hp(const AttnParams& p, const HostPlan& hp, cudaStream_t s) {
  using L = TcLayout<HD, F8, SPLIT>;
  CUtensorMap mk, mv;
  if (!make_kv_map(&mk, p.k, p.kv_rows, p.Hkv, HD, F8, KT) ||
      !make_kv_map(&mv, p.v, p.kv_rows, p.Hkv, HD, F8, KT))
    return cudaErrorInvalidValue;
  auto kernel = attn_tc_kernel_hp<HD, F8, WIN, SPLIT>;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::SMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, dim3(p.n_ctas), dim3(L::THREADS), L::SMEM, s, p, mk, mv, hp);
}

template <int HD, bool F8, bool WIN>
cudaError_t launch_hd_hp(const AttnParams& p, const HostPlan& hp, cudaStream_t s) {
  if constexpr (F8)
    return launch_hd_hp<HD, F8, WIN, false>(p, hp, s);
  else
    return p.kv_rings ? launch_hd_hp<HD, F8, WIN, true>(p, hp, s)
                      : launch_hd_hp<HD, F8, WIN, false>(p, hp, s);
}

template <int HD, bool F8>
cudaError_t launch_hd_hp(const AttnParams& p, const HostPlan& hp, cudaStream_t s) {
  return p.window > 0 ? launch_hd_hp<HD, F8, true>(p, hp, s)
                      : launch_hd_hp<HD, F8, false>(p, hp, s);
}

}  // namespace

bool kv_tensor_map(CUtensorMap* map, const void* base, int64_t kv_rows, int hkv, int hd,
                   bool fp8, int box_rows) {
  return make_kv_map(map, base, kv_rows, hkv, hd, fp8, box_rows);
}

bool attn_tc_available() { return encode_fn() != nullptr; }
int attn_tc_kt() { return KT; }

bool attn_tc_supports(int head_dim, bool fp8) { return head_dim == 128 || !fp8; }

cudaError_t launch_attn_tc_hp(const AttnParams& p, bool fp8, const HostPlan& hp,
                              cudaStream_t s) {
  if (!attn_tc_supports(p.d, fp8) || p.kv_rows <= 0 || p.kv_rows > 0x7fffffffLL ||
      p.block_size != 0)
    return cudaErrorNotSupported;
  if (fp8) return launch_hd_hp<128, true>(p, hp, s);
  return p.d == 128 ? launch_hd_hp<128, false>(p, hp, s) : launch_hd_hp<64, false>(p, hp, s);
}

cudaError_t launch_attn_tc(const AttnParams& p, bool fp8, cudaStream_t s) {
  if (!attn_tc_supports(p.d, fp8) || p.kv_rows <= 0 || p.kv_rows > 0x7fffffffLL)
    return cudaErrorNotSupported;
  if (fp8) return launch_hd<128, true>(p, s);
  return p.d == 128 ? launch_hd<128, false>(p, s) : launch_hd<64, false>(p, s);
}

}  // namespace sv

// internal.cuh -- shared declarations of libspecverify's kernels and host code.
//
// Work decomposition of verify attention (plan, attention, combine):
//   unit  = (sequence b, KV head g, row tile mt): up to 128 of the G*(1+D_b) query rows
//           that share KV head g ("GQA", "GPU and LLM, chapter 5"; guideline 2 of the
//           co-design summary: G*(1+D) rows per KV head, M = 128 fills a tile).
//   tile  = KT consecutive cache positions of one unit's key range. Tiles are aligned to
//           multiples of KT from the sequence's first position; a unit's tiles run from
//           the one holding its first visible key (0, or under a sliding window of W
//           positions the oldest key of its first window row, T_b + i_lo - W + 1) to the
//           one holding T_b + D_b.
//   Units are laid end to end on one global tile line; persistent CTAs process contiguous
//   ranges of it. Starting a unit costs a CTA about `switch_tiles` tiles' worth of time
//   (epilogue of the previous unit, loading and splitting Q, refilling the pipeline), so
//   the split is made on a virtual line on which every unit is preceded by switch_tiles
//   virtual tiles: CTA c owns the virtual range [c*VT/C, (c+1)*VT/C), VT = TT +
//   U * switch_tiles, and with it the real tiles whose virtual positions fall inside. A
//   CTA whose range crosses into a unit therefore gets fewer real tiles. The plan kernel
//   tabulates each CTA's first real tile and unit. A CTA that covers a whole unit writes
//   the normalised output itself; otherwise each CTA covering part of the unit
//   writes a partial (O unnormalised, running max m, running sum l) to slot c + u and the
//   combine kernel merges them with the same rescaling rule as the online softmax.
//   When there are no more units than CTAs, the plan may instead give each unit k CTAs
//   (k <= C / U), CTA u*k + i taking the i-th of k equal parts of unit u's tiles: no unit
//   starts inside a range, and only k partials per unit are combined (none for k = 1),
//   at the price of idle CTAs. It does so when a per-tile time model says so: a tile
//   takes max(tile_floor, n) time units while n CTAs stream at once (their share of HBM
//   bandwidth, or the tile's compute time), so the split line takes (TT + U *
//   switch_tiles) / C * max(tile_floor, C) and k CTAs per unit ceil(the longest unit's
//   tiles / k) * max(tile_floor, U * k).
//   Unit order on the line: by sequence, then KV head, then row tile; but when every
//   sequence has the same number (> 1) of row tiles, row-tile-major (all row tiles 0,
//   then all row tiles 1, ...), so that the CTAs of each row-tile slice of the split line
//   read the same K/V at the same time and share it through L2.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/specverify.h"

namespace sv {

constexpr uint32_t FLAG_ATTN_SHAPE = 1u;
constexpr uint32_t FLAG_TIMEOUT = 2u;
constexpr uint32_t FLAG_ACCEPT_SHAPE = 4u;

constexpr int MT = 128;  // query rows per unit (one tensor-core M tile)

// Plan header written by the plan kernel.
struct PlanHdr {
  int32_t num_units;
  int32_t total_tiles;
  int32_t kt;
  int32_t unit_ctas;  // k > 0: CTA u*k + i covers the i-th of k equal parts of unit u
                      // (k = 1: nothing to combine); 0: the split tile line
  int64_t sum_w;
  int64_t sum_kv;
};

// Byte offsets inside a spec_verify_attn workspace.
struct AttnWs {
  size_t ctrl, hdr, q_off, kv_off, units, ubeg, cta_tab, part_o, part_ml, total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline int max_units_for(int B, int Hkv, int G, int max_draft) {
  const int rows = G * (1 + max_draft);
  return B * Hkv * ((rows + MT - 1) / MT);
}

inline AttnWs attn_ws_layout(int B, int Hkv, int G, int d, int max_draft, int n_ctas) {
  AttnWs w;
  const size_t U = (size_t)max_units_for(B, Hkv, G, max_draft);
  const size_t slots = (size_t)n_ctas + U;
  size_t o = 0;
  w.ctrl = o;    o += 256;
  w.hdr = o;     o += 256;
  w.q_off = o;   o = align_up(o + sizeof(int64_t) * (B + 1), 256);
  w.kv_off = o;  o = align_up(o + sizeof(int64_t) * (B + 1), 256);
  w.units = o;   o = align_up(o + sizeof(int4) * U, 256);
  w.ubeg = o;    o = align_up(o + sizeof(int32_t) * (U + 1), 256);
  w.cta_tab = o; o = align_up(o + sizeof(int2) * ((size_t)n_ctas + 1), 256);
  w.part_o = o;  o = align_up(o + sizeof(float) * slots * MT * d, 256);
  w.part_ml = o; o = align_up(o + sizeof(float2) * slots * MT, 256);
  w.total = o;
  return w;
}

struct AttnParams {
  const void* q;
  const void* k;               // packed cache [kv_rows, Hkv, d], or the block pool
  const void* v;               // [num_blocks * block_size, Hkv, d] of a paged cache
  void* out;
  const float* kv_scale;      // [2, Hkv] or nullptr
  const int32_t* seq_lens;    // [B]
  const int32_t* draft_len;   // [B]
  uint32_t* flags;            // workspace control word
  PlanHdr* hdr;
  int64_t* q_off;             // [B+1]
  int64_t* kv_off;            // [B+1]
  int4* units;                // [U] (b, kv head, row tile, first cache position of the
                              // unit's first tile)
  int32_t* ubeg;              // [U+1] first global tile of each unit (unit u has
                              // ubeg[u+1] - ubeg[u] tiles)
  int2* cta_tab;              // [n_ctas+1] (first real tile, its unit) of each CTA's range
  float* part_o;              // [slots, MT, d]
  float2* part_ml;            // [slots, MT] (m in log2 units, l)
  int B, Hq, Hkv, G, d;
  int max_draft, max_seq;
  int64_t q_rows, kv_rows;
  int max_units;
  int n_ctas;
  int switch_tiles;           // virtual tiles charged for starting a unit
  int tile_floor;             // CTAs streaming at once at which a tile's share of HBM time
                              // equals its compute time (0: the model keeps the split line)
  int unit_ctas_mode;         // -1: choose by the cost model; 0: never; k > 0: k CTAs per
                              // unit whenever U * k <= CTAs
  const int32_t* block_table;  // paged cache: [B, bt_stride] physical block of each logical
                               // block (position j of sequence b: row j % block_size of
                               // block block_table[b * bt_stride + j / block_size])
  int bt_stride;
  int block_size;             // positions per block, a power of two; 0: packed cache
  int bs_log2;
  int64_t num_blocks;
  int window;                 // sliding window in positions (0: every earlier key); set to 0
                              // when it covers max_seq + max_draft + 1 positions
  float scale_log2;           // softmax_scale * log2(e)
  int kv_rings;               // tcgen05 kernel, bf16 K/V: 1 separate K and V rings (K loads
                              // run further ahead), 0 paired K + V stages
  long long wait_limit;       // tcgen05 kernel: clock cycles a barrier wait may take before
                              // it gives up (0: the default, about 2 s)
  int stall_first_tile;       // test hook: every CTA's producer withholds the K and V loads
                              // of the first tile of its range, so the waits for it run out
};

// First key tile of row tile mt of a sequence with T cached keys. Window row i sees keys
// max(0, T + i - window + 1) .. T + i ("GPU and LLM, chapter 5", "Sliding window": only the
// W most recent positions); the tile's smallest window row is mt * MT / G.
// (32-bit arithmetic: T <= 2^31 - 1025 and the window row mt * MT / G <= 255.)
__host__ __device__ inline int unit_first_tile(int T, int mt, int G, int window, int kt) {
  if (window <= 0) return 0;
  const int lo = T + mt * MT / G + 1 - window;
  return lo > 0 ? lo / kt : 0;
}
// First cache position whose K/V rows a sequence's window rows can see: positions before
// it may hold any bits (their V rows are zeroed on the chip before they meet P = 0).
__host__ __device__ inline int first_visible_key(int T, int window) {
  return window > 0 && T - window + 1 > 0 ? T - window + 1 : 0;
}

// Virtual-line position of real tile t of unit u (u * switch_tiles virtual tiles precede
// unit u's start, and switch_tiles more its first real tile).
__host__ __device__ inline int64_t vpos_of_tile(int64_t t, int u, int switch_tiles) {
  return t + (int64_t)(u + 1) * switch_tiles;
}

// The CTA whose range [c*TT/C, (c+1)*TT/C) of a line of TT positions contains position t.
__host__ __device__ inline int cta_of_tile(int64_t t, int64_t TT, int C) {
  return (int)(((t + 1) * (int64_t)C - 1) / TT);
}
// Whether CTA c's range of a line of TT positions is not empty (with fewer positions than
// CTAs some ranges are empty).
__host__ __device__ inline bool cta_has_tiles(int c, int64_t TT, int C) {
  return (int64_t)(c + 1) * TT / C > (int64_t)c * TT / C;
}

// Programmatic dependent launch: every kernel of the library is launched so that it may
// start while the previous kernel on the stream drains; it lets its own dependents launch
// (pdl_trigger: at once, except the tcgen05 attention kernel, whose CTAs release them when
// their work is done) and waits for the previous grid's results (pdl_wait) before it reads
// any input, so results are those of ordinary stream order.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Host-side fault injection (sv_inject_launch_failure): counts a launch, and returns true
// for the one that was armed to fail.
bool take_injected_launch_failure();

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  if (take_injected_launch_failure()) return cudaErrorLaunchFailure;  // nothing launched
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// A work plan computed on the host from host copies of the lengths, passed by value with
// the attention launch (a kernel parameter, read through the constant cache), so that no
// planning kernel runs. The same plan as the planning kernel's: unit list and starts,
// offsets, the unit-to-CTA policy and each CTA's range.
constexpr int HP_MAX_B = 256;   // sequences
constexpr int HP_MAX_U = 640;   // units
constexpr int HP_MAX_C = 192;   // CTAs
struct HostPlan {
  int32_t num_units, total_tiles, unit_ctas, pad;
  int32_t T[HP_MAX_B], D[HP_MAX_B];
  int64_t q_off[HP_MAX_B + 1], kv_off[HP_MAX_B + 1];
  int4 units[HP_MAX_U];
  int32_t ubeg[HP_MAX_U + 1];
  int2 cta_tab[HP_MAX_C + 1];
};
// Fills `hp` for the call `p` (kt: the attention kernel's tile) from host lengths T[B],
// D[B]. Returns SV_OK, SV_ERR_SHAPE for lengths out of range or packed sizes beyond the
// buffers, or SV_ERR_WORKSPACE when the plan does not fit a HostPlan.
sv_status host_plan(const AttnParams& p, int kt, const int32_t* T, const int32_t* D,
                    HostPlan* hp);

// Launchers (each returns the cudaGetLastError() of its launch).
cudaError_t launch_plan(const AttnParams& p, int kt, cudaStream_t s);
cudaError_t launch_combine(const AttnParams& p, cudaStream_t s);
cudaError_t launch_attn_mma(const AttnParams& p, bool fp8, cudaStream_t s);
int attn_mma_kt();
bool attn_tc_available();
bool attn_tc_supports(int head_dim, bool fp8);
int attn_tc_kt();
cudaError_t launch_attn_tc(const AttnParams& p, bool fp8, cudaStream_t s);
cudaError_t launch_attn_tc_hp(const AttnParams& p, bool fp8, const HostPlan& hp, cudaStream_t s);
// Row pairs (attn_pair.cu): one CTA per (sequence, KV head) holding both 128-row tiles when
// 128 < G (1 + max_draft) <= 256; bf16 K/V, d = 128, packed cache, no sliding window, and
// at most one CTA per SM. The CTAs check the lengths and work out the offsets themselves.
bool attn_pair_applies(const AttnParams& p, bool fp8, int sms);
cudaError_t launch_attn_pair(const AttnParams& p, cudaStream_t s);

// Acceptance.
struct AcceptWs {
  size_t ctrl, key, amax, total;
  int nctas;  // persistent argmax CTAs
};
AcceptWs accept_ws_layout(int B, int max_draft, int vocab, int num_sms);
cudaError_t launch_accept(int B, int max_draft, int vocab, int dtype, const void* logits,
                          const int32_t* draft_tokens, const int32_t* draft_len,
                          int32_t* accept_len, int32_t* next_token, int32_t* target_tokens,
                          void* ws, const AcceptWs& lay, cudaStream_t s);

// Stochastic acceptance (workspace: the flag word only).
cudaError_t launch_accept_stochastic(int B, int max_draft, int vocab, int dtype,
                                     const void* target, const void* draft,
                                     const int32_t* draft_tokens, const int32_t* draft_len,
                                     const float* u_accept, const float* u_sample,
                                     float inv_temp, int32_t* accept_len, int32_t* next_token,
                                     void* ws, cudaStream_t s);

// Draft signals.
struct SigWs {
  size_t ctrl, part, total;
  int nctas;
};
SigWs signals_ws_layout(int64_t rows, int vocab, int num_sms);
cudaError_t launch_signals(int64_t rows, int vocab, int dtype, const void* logits,
                           float* confidence, float* entropy, void* ws, const SigWs& lay,
                           cudaStream_t s);

}  // namespace sv

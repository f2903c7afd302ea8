// api.cu -- the C ABI of libspecverify: argument checks, workspace layout, launches.
// Every entry point is declared and documented in include/specverify.h.
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "internal.cuh"

using namespace sv;

namespace {

#ifndef SV_SWITCH_F8
#define SV_SWITCH_F8 9
#endif
#ifndef SV_SWITCH_BF16
#define SV_SWITCH_BF16 5
#endif
// Virtual tiles charged for starting a unit (see internal.cuh), per attention kernel.
constexpr int SWITCH_TILES_TC_FP8 = SV_SWITCH_F8;
constexpr int SWITCH_TILES_TC_BF16 = SV_SWITCH_BF16;
constexpr int SWITCH_TILES_MMA = 2;
// Per-tile compute floor of each kernel, in CTAs streaming at once (a 128-key tile's
// compute time x HBM bandwidth / the tile's bytes: bf16 about 0.9 us x 6.8 TB/s / 64 KB,
// E4M3 about 0.89 us x 6.8 TB/s / 32 KB). The cost model is not applied to the mma.sync
// kernel (it keeps the split line unless a policy is forced).
#ifndef SV_TILE_FLOOR_BF16
#define SV_TILE_FLOOR_BF16 93
#endif
#ifndef SV_TILE_FLOOR_F8
#define SV_TILE_FLOOR_F8 185
#endif
#ifndef SV_UNIT_CTAS
#define SV_UNIT_CTAS -1
#endif

// Positions and cache rows are 32-bit on the device (tile arithmetic, TMA coordinates).
constexpr int32_t MAX_SEQ_LEN = 0x7fffffff - 1024;
constexpr int64_t MAX_KV_ROWS = 0x7fffffff - 1024;

// Launches until the armed failure, plus one (0: nothing armed). Tests only.
std::atomic<int> g_fail_countdown{0};
// Wait limit of the next tcgen05 attention launch that withholds a tile (0: none). Tests.
std::atomic<long long> g_stall_limit{0};
int g_attn_kernel = 0;  // 0 automatic, 1 mma.sync, 2 tcgen05
int g_unit_ctas = SV_UNIT_CTAS;  // -1 cost model, 0 split tile line, k > 0 k CTAs per unit
int g_row_pairs = 0;  // 1: the row-pair kernel whenever it applies; 0: never (default)
// bf16 K/V on the tcgen05 kernel: -1 by the call's shape (default), 0 paired K + V stages,
// 1 separate K and V rings.
int g_kv_rings = -1;
// Split rings let the K loads run further ahead of the score MMAs. Measured attention time
// (us, paired / split): c2 92.2 / 89.3; c4 (T = 16384, G = 8) with D = 0, 1, 3, 7, 15:
// 166.5 / 162.0, 167.8 / 161.3, 168.0 / 162.7, 168.2 / 162.2, 169.3 / 164.0; D = 31
// 257.0 / 247.8. Paired stages measured faster where a KV head's second row tile is partial
// (D = 16: 247.1 / 259.3, D = 23: 250.7 / 255.8, although their whole steps ran faster
// split) and on the ragged c5 batch, whose CTAs each stream about 900 tiles (1286 / 1315).
constexpr int64_t KV_RINGS_MAX_TILES_PER_CTA = 1024;
cudaEvent_t g_ev_start = nullptr;
cudaEvent_t g_ev_stop = nullptr;

int current_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

sv_status check_desc(const sv_attn_desc* d) {
  if (!d) return SV_ERR_NULL;
  if (d->batch < 0 || d->num_kv_heads < 1 || d->num_q_heads < 1 ||
      d->num_q_heads % d->num_kv_heads != 0 || d->num_q_heads > 4096 ||
      d->max_draft_len < 0 || d->max_draft_len > 255 || d->max_seq_len < 0 ||
      d->max_seq_len > MAX_SEQ_LEN || d->q_rows < 0 || d->kv_rows < 0 ||
      d->kv_rows > MAX_KV_ROWS || d->sliding_window < 0)
    return SV_ERR_SHAPE;
  if (d->head_dim != 64 && d->head_dim != 128) return SV_ERR_SHAPE;
  if (!(d->softmax_scale >= 0.f) || isinf(d->softmax_scale)) return SV_ERR_SHAPE;
  if (d->kv_dtype != SV_BF16 && d->kv_dtype != SV_FP8_E4M3) return SV_ERR_DTYPE;
  return SV_OK;
}

AttnWs layout_for(const sv_attn_desc* d, int sms) {
  return attn_ws_layout(d->batch, d->num_kv_heads, d->num_q_heads / d->num_kv_heads,
                        d->head_dim, d->max_draft_len, sms);
}

// 1 = mma.sync, 2 = tcgen05
int pick_kernel(const sv_attn_desc* d) {
  const bool tc_ok =
      attn_tc_available() && attn_tc_supports(d->head_dim, d->kv_dtype == SV_FP8_E4M3);
  if (g_attn_kernel == 1) return 1;
  if (g_attn_kernel == 2) return tc_ok ? 2 : 1;
  return tc_ok ? 2 : 1;
}

}  // namespace

bool sv::take_injected_launch_failure() {
  int n = g_fail_countdown.load(std::memory_order_relaxed);
  while (n > 0)
    if (g_fail_countdown.compare_exchange_weak(n, n - 1, std::memory_order_relaxed))
      return n == 1;
  return false;
}

extern "C" {

SV_API int sv_inject_launch_failure(int after) {
  const int prev = g_fail_countdown.exchange(after >= 0 && after < (1 << 30) ? after + 1 : 0);
  return prev - 1;
}

SV_API int sv_inject_wait_timeout(int64_t limit_cycles) {
  return g_stall_limit.exchange(limit_cycles > 0 ? (long long)limit_cycles : 0) > 0 ? 1 : 0;
}

SV_API int sv_version(void) { return 400; }  // 0.4.0: wait-timeout injection

SV_API const char* sv_status_string(sv_status s) {
  switch (s) {
    case SV_OK: return "ok";
    case SV_ERR_NULL: return "null pointer";
    case SV_ERR_SHAPE: return "invalid shape";
    case SV_ERR_DTYPE: return "unsupported dtype";
    case SV_ERR_ALIGN: return "misaligned pointer";
    case SV_ERR_WORKSPACE: return "workspace too small";
    case SV_ERR_CUDA: return "CUDA error";
    case SV_ERR_TIMEOUT: return "device-side wait timed out";
    case SV_ERR_DEVICE_SHAPE: return "device-side length check failed";
  }
  return "unknown status";
}

SV_API int sv_set_attn_kernel(int which) {
  if (which < 0 || which > 2) return -1;
  if (which == 2 && !attn_tc_available()) return -1;
  const int prev = g_attn_kernel;
  g_attn_kernel = which;
  return prev;
}

SV_API int sv_set_unit_ctas(int mode) {
  if (mode < -1 || mode > 1024) return -2;
  const int prev = g_unit_ctas;
  g_unit_ctas = mode;
  return prev;
}

SV_API int sv_set_row_pairs(int mode) {
  if (mode < 0 || mode > 1) return -2;
  const int prev = g_row_pairs;
  g_row_pairs = mode;
  return prev;
}

SV_API int sv_set_kv_rings(int mode) {
  if (mode < -1 || mode > 1) return -2;
  const int prev = g_kv_rings;
  g_kv_rings = mode;
  return prev;
}

SV_API void sv_set_profile_events(void* start_event, void* stop_event) {
  if (start_event && stop_event) {
    g_ev_start = (cudaEvent_t)start_event;
    g_ev_stop = (cudaEvent_t)stop_event;
  } else {
    g_ev_start = g_ev_stop = nullptr;
  }
}

SV_API size_t spec_verify_attn_workspace_size(const sv_attn_desc* desc) {
  if (check_desc(desc) != SV_OK) return 0;
  const int sms = current_sms();
  if (sms <= 0) return 0;
  return layout_for(desc, sms).total;
}

}  // extern "C"

namespace {

// A paged cache (block_size 0: the packed layout).
struct PagedArgs {
  const int32_t* table;
  int32_t stride;
  int32_t block_size;
  int64_t num_blocks;
};

// The sizes, limits and work-distribution policy of one attention call on `sms` SMs with
// kernel `which` (1 mma.sync, 2 tcgen05); every pointer is left null.
AttnParams shape_params(const sv_attn_desc* desc, const PagedArgs& pg, int which, int sms) {
  const bool fp8 = desc->kv_dtype == SV_FP8_E4M3;
  const int kt = which == 2 ? attn_tc_kt() : attn_mma_kt();
  const int G = desc->num_q_heads / desc->num_kv_heads;
  const int64_t rows_per_kv = (int64_t)G * (1 + desc->max_draft_len);
  const int64_t max_tiles = (int64_t)desc->batch * desc->num_kv_heads * ((rows_per_kv + MT - 1) / MT) *
                            ((desc->max_seq_len + 1 + desc->max_draft_len + kt - 1) / kt);
  AttnParams p = {};
  p.B = desc->batch;
  p.Hq = desc->num_q_heads;
  p.Hkv = desc->num_kv_heads;
  p.G = G;
  p.d = desc->head_dim;
  p.max_draft = desc->max_draft_len;
  p.max_seq = desc->max_seq_len;
  // a window covering every position of the longest sequence is no window
  p.window = (int64_t)desc->sliding_window > (int64_t)desc->max_seq_len + desc->max_draft_len
                 ? 0
                 : desc->sliding_window;
  p.q_rows = desc->q_rows;
  p.kv_rows = pg.block_size > 0 ? pg.num_blocks * pg.block_size : desc->kv_rows;
  p.bt_stride = pg.stride;
  p.block_size = pg.block_size;
  p.bs_log2 = 0;
  while (pg.block_size > 0 && (1 << p.bs_log2) < pg.block_size) ++p.bs_log2;
  p.num_blocks = pg.num_blocks;
  p.max_units = max_units_for(p.B, p.Hkv, G, p.max_draft);
  p.n_ctas = (int)(max_tiles < sms ? (max_tiles > 0 ? max_tiles : 1) : sms);
  // measured cost of starting a unit inside a CTA's range, in tiles of that kernel
  p.switch_tiles = which == 2 ? (fp8 ? SWITCH_TILES_TC_FP8 : SWITCH_TILES_TC_BF16) : SWITCH_TILES_MMA;
  // The same model for a paged cache: with its block-table entries read a group of tiles
  // ahead, a CTA streams 16-position blocks at nearly the packed rate (c2: 97.5 us with
  // one CTA per unit against 115.3 us on the split tile line, packed 95.1 us).
  p.tile_floor = which == 2 ? (fp8 ? SV_TILE_FLOOR_F8 : SV_TILE_FLOOR_BF16) : 0;
  p.unit_ctas_mode = g_unit_ctas;
  const bool partial_row_tile = rows_per_kv > MT && rows_per_kv % MT != 0;
  const bool long_stream = max_tiles > KV_RINGS_MAX_TILES_PER_CTA * p.n_ctas;
  p.kv_rings = g_kv_rings >= 0 ? g_kv_rings : (partial_row_tile || long_stream ? 0 : 1);
  const float scale = desc->softmax_scale > 0.f ? desc->softmax_scale
                                                : 1.f / sqrtf((float)desc->head_dim);
  p.scale_log2 = scale * 1.4426950408889634f;
  return p;
}

// Whether a call of kernel `which` with these parameters runs the row-pair kernel: it is
// switched on and applies (see attn_pair_applies). Off by default: on every workload
// measured, the unit plan (each row tile streaming the keys, the second from L2) is faster.
bool use_row_pairs(const AttnParams& p, bool fp8, int which, int sms) {
  return which == 2 && g_row_pairs == 1 && attn_pair_applies(p, fp8, sms);
}

sv_status verify_impl(const sv_attn_desc* desc, const void* q, const void* k_cache,
                      const void* v_cache, const PagedArgs& pg, const int32_t* seq_lens,
                      const int32_t* draft_len, const float* kv_scale, void* out,
                      void* workspace, size_t workspace_bytes, void* stream,
                      const int32_t* seq_lens_host = nullptr,
                      const int32_t* draft_len_host = nullptr) {
  sv_status st = check_desc(desc);
  if (st != SV_OK) return st;
  if (desc->batch == 0) return SV_OK;
  if (!q || !k_cache || !v_cache || !seq_lens || !draft_len || !out || !workspace)
    return SV_ERR_NULL;
  if (pg.block_size > 0 && !pg.table) return SV_ERR_NULL;
  if (pg.block_size > 0 && !aligned(pg.table, 4)) return SV_ERR_ALIGN;
  if (seq_lens_host && draft_len_host)  // host copies of the lengths: checked here, at once
    for (int b = 0; b < desc->batch; ++b)
      if (seq_lens_host[b] < 0 || seq_lens_host[b] > desc->max_seq_len || draft_len_host[b] < 0 ||
          draft_len_host[b] > desc->max_draft_len)
        return SV_ERR_SHAPE;
  const bool fp8 = desc->kv_dtype == SV_FP8_E4M3;
  if (fp8 && !kv_scale) return SV_ERR_NULL;
  if (!fp8 && kv_scale) return SV_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(workspace, 256) || !aligned(seq_lens, 4) || !aligned(draft_len, 4) ||
      (kv_scale && !aligned(kv_scale, 4)))
    return SV_ERR_ALIGN;
  const int sms = current_sms();
  if (sms <= 0) return SV_ERR_CUDA;
  const AttnWs lay = layout_for(desc, sms);
  if (workspace_bytes < lay.total) return SV_ERR_WORKSPACE;

  const int which = pick_kernel(desc);
  const int kt = which == 2 ? attn_tc_kt() : attn_mma_kt();
  AttnParams p = shape_params(desc, pg, which, sms);
  if (which == 2) {  // a pending wait-timeout injection applies to this launch
    const long long lim = g_stall_limit.exchange(0);
    if (lim > 0) {
      p.wait_limit = lim;
      p.stall_first_tile = 1;
    }
  }
  uint8_t* ws = (uint8_t*)workspace;
  p.q = q;
  p.k = k_cache;
  p.v = v_cache;
  p.out = out;
  p.kv_scale = kv_scale;
  p.seq_lens = seq_lens;
  p.draft_len = draft_len;
  p.flags = (uint32_t*)(ws + lay.ctrl);
  p.hdr = (PlanHdr*)(ws + lay.hdr);
  p.q_off = (int64_t*)(ws + lay.q_off);
  p.kv_off = (int64_t*)(ws + lay.kv_off);
  p.units = (int4*)(ws + lay.units);
  p.ubeg = (int32_t*)(ws + lay.ubeg);
  p.cta_tab = (int2*)(ws + lay.cta_tab);
  p.part_o = (float*)(ws + lay.part_o);
  p.part_ml = (float2*)(ws + lay.part_ml);
  p.block_table = pg.table;

  cudaStream_t s = (cudaStream_t)stream;
  if (use_row_pairs(p, fp8, which, sms)) {  // one launch: no plan, nothing to combine
    if (g_ev_start && cudaEventRecord(g_ev_start, s) != cudaSuccess) return SV_ERR_CUDA;
    if (launch_attn_pair(p, s) != cudaSuccess) return SV_ERR_CUDA;
    if (g_ev_stop && cudaEventRecord(g_ev_stop, s) != cudaSuccess) return SV_ERR_CUDA;
    return SV_OK;
  }
  // Host lengths: plan on the host and pass the plan with the attention launch (tcgen05
  // kernel, packed cache), unless it does not fit a HostPlan.
  static thread_local HostPlan hp;
  bool host_planned = false;
  if (seq_lens_host && draft_len_host && which == 2 && pg.block_size == 0) {
    const sv_status hs = host_plan(p, kt, seq_lens_host, draft_len_host, &hp);
    if (hs == SV_ERR_SHAPE) return SV_ERR_SHAPE;
    host_planned = hs == SV_OK;
  }
  if (!host_planned && launch_plan(p, kt, s) != cudaSuccess) return SV_ERR_CUDA;
  if (g_ev_start && cudaEventRecord(g_ev_start, s) != cudaSuccess) return SV_ERR_CUDA;
  const cudaError_t e = host_planned ? launch_attn_tc_hp(p, fp8, hp, s)
                        : which == 2 ? launch_attn_tc(p, fp8, s)
                                     : launch_attn_mma(p, fp8, s);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  if (g_ev_stop && cudaEventRecord(g_ev_stop, s) != cudaSuccess) return SV_ERR_CUDA;
  if (launch_combine(p, s) != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}

}  // namespace

extern "C" {

SV_API sv_status spec_verify_attn(const sv_attn_desc* desc, const void* q, const void* k_cache,
                                  const void* v_cache, const int32_t* seq_lens,
                                  const int32_t* draft_len, const float* kv_scale, void* out,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  const PagedArgs packed = {nullptr, 0, 0, 0};
  return verify_impl(desc, q, k_cache, v_cache, packed, seq_lens, draft_len, kv_scale, out,
                     workspace, workspace_bytes, stream);
}

SV_API sv_status spec_verify_attn_host_lengths(const sv_attn_desc* desc, const void* q,
                                               const void* k_cache, const void* v_cache,
                                               const int32_t* seq_lens,
                                               const int32_t* draft_len,
                                               const int32_t* seq_lens_host,
                                               const int32_t* draft_len_host,
                                               const float* kv_scale, void* out,
                                               void* workspace, size_t workspace_bytes,
                                               void* stream) {
  if (desc && desc->batch > 0 && (!seq_lens_host || !draft_len_host)) return SV_ERR_NULL;
  const PagedArgs packed = {nullptr, 0, 0, 0};
  return verify_impl(desc, q, k_cache, v_cache, packed, seq_lens, draft_len, kv_scale, out,
                     workspace, workspace_bytes, stream, seq_lens_host, draft_len_host);
}

SV_API sv_status spec_verify_attn_paged(const sv_attn_desc* desc, const void* q,
                                        const void* k_pages, const void* v_pages,
                                        int64_t num_blocks, int32_t block_size,
                                        const int32_t* block_table, int32_t max_blocks_per_seq,
                                        const int32_t* seq_lens, const int32_t* draft_len,
                                        const float* kv_scale, void* out, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  if (block_size < 8 || block_size > (1 << 16) || (block_size & (block_size - 1)) != 0 ||
      num_blocks < 1 || num_blocks > MAX_KV_ROWS / block_size || max_blocks_per_seq < 1)
    return SV_ERR_SHAPE;
  const PagedArgs pg = {block_table, max_blocks_per_seq, block_size, num_blocks};
  return verify_impl(desc, q, k_pages, v_pages, pg, seq_lens, draft_len, kv_scale, out,
                     workspace, workspace_bytes, stream);
}

SV_API sv_status sv_plan_preview(const sv_attn_desc* desc, int32_t block_size,
                                 const int32_t* seq_lens_host, const int32_t* draft_len_host,
                                 int32_t num_sms, int32_t attn_kernel, sv_plan_info* info,
                                 int32_t* units, int32_t* unit_begin, int32_t* cta_begin,
                                 int32_t capacity_units) {
  sv_status st = check_desc(desc);
  if (st != SV_OK) return st;
  if (!info) return SV_ERR_NULL;
  if (desc->batch > 0 && (!seq_lens_host || !draft_len_host)) return SV_ERR_NULL;
  if (num_sms < 1 || capacity_units < 0 || (attn_kernel != 1 && attn_kernel != 2) ||
      (block_size != 0 &&
       (block_size < 8 || block_size > (1 << 16) || (block_size & (block_size - 1)) != 0)))
    return SV_ERR_SHAPE;
  if (attn_kernel == 2 && !attn_tc_supports(desc->head_dim, desc->kv_dtype == SV_FP8_E4M3))
    return SV_ERR_SHAPE;
  // a paged pool's size does not enter the plan: the largest pool the limits allow
  const PagedArgs pg = {nullptr, 1 << 30, block_size,
                        block_size > 0 ? MAX_KV_ROWS / block_size : 0};
  const AttnParams p = shape_params(desc, pg, attn_kernel, num_sms);
  const int kt = attn_kernel == 2 ? attn_tc_kt() : attn_mma_kt();
  *info = sv_plan_info{0, 0, kt, p.n_ctas, 0, p.switch_tiles};
  if (desc->batch == 0) return SV_OK;
  static thread_local HostPlan hp;
  st = host_plan(p, kt, seq_lens_host, draft_len_host, &hp);
  if (st != SV_OK) return st;
  info->num_units = hp.num_units;
  info->total_tiles = hp.total_tiles;
  info->unit_ctas = hp.unit_ctas;
  if ((units || unit_begin) && hp.num_units > capacity_units) return SV_ERR_WORKSPACE;
  for (int u = 0; units && u < hp.num_units; ++u) {
    units[4 * u] = hp.units[u].x;
    units[4 * u + 1] = hp.units[u].y;
    units[4 * u + 2] = hp.units[u].z;
    units[4 * u + 3] = hp.units[u].w;
  }
  for (int u = 0; unit_begin && u <= hp.num_units; ++u) unit_begin[u] = hp.ubeg[u];
  for (int c = 0; cta_begin && c <= p.n_ctas; ++c) {
    cta_begin[2 * c] = hp.cta_tab[c].x;
    cta_begin[2 * c + 1] = hp.cta_tab[c].y;
  }
  return SV_OK;
}

SV_API int sv_row_pair_mode(const sv_attn_desc* desc, int32_t block_size, int32_t num_sms,
                           int32_t attn_kernel) {
  if (check_desc(desc) != SV_OK || num_sms < 1 || (attn_kernel != 1 && attn_kernel != 2) ||
      block_size < 0)
    return -1;
  const PagedArgs pg = {nullptr, 1 << 30, block_size,
                        block_size > 0 ? MAX_KV_ROWS / block_size : 0};
  const AttnParams p = shape_params(desc, pg, attn_kernel, num_sms);
  return use_row_pairs(p, desc->kv_dtype == SV_FP8_E4M3, attn_kernel, num_sms) ? 1 : 0;
}

SV_API size_t spec_accept_workspace_size(int32_t batch, int32_t max_draft_len, int32_t vocab) {
  if (batch < 0 || max_draft_len < 0 || max_draft_len > 255 || vocab <= 0) return 0;
  const int sms = current_sms();
  if (sms <= 0) return 0;
  return accept_ws_layout(batch, max_draft_len, vocab, sms).total;
}

SV_API sv_status spec_accept(int32_t batch, int32_t max_draft_len, int32_t vocab,
                             int32_t logits_dtype, const void* logits,
                             const int32_t* draft_tokens, const int32_t* draft_len,
                             int32_t* accept_len, int32_t* next_token, int32_t* target_tokens,
                             void* workspace, size_t workspace_bytes, void* stream) {
  if (batch < 0 || max_draft_len < 0 || max_draft_len > 255 || vocab <= 0) return SV_ERR_SHAPE;
  if (logits_dtype != SV_BF16 && logits_dtype != SV_FP32) return SV_ERR_DTYPE;
  if (batch == 0) return SV_OK;
  if (!logits || !draft_len || !accept_len || !next_token || !workspace) return SV_ERR_NULL;
  if (max_draft_len > 0 && !draft_tokens) return SV_ERR_NULL;
  const uintptr_t es = logits_dtype == SV_BF16 ? 2 : 4;
  if (!aligned(logits, es) || !aligned(draft_len, 4) || !aligned(accept_len, 4) ||
      !aligned(next_token, 4) || (draft_tokens && !aligned(draft_tokens, 4)) ||
      (target_tokens && !aligned(target_tokens, 4)) || !aligned(workspace, 256))
    return SV_ERR_ALIGN;
  const int sms = current_sms();
  if (sms <= 0) return SV_ERR_CUDA;
  const AcceptWs lay = accept_ws_layout(batch, max_draft_len, vocab, sms);
  if (workspace_bytes < lay.total) return SV_ERR_WORKSPACE;
  const cudaError_t e = launch_accept(batch, max_draft_len, vocab, logits_dtype, logits,
                                      draft_tokens, draft_len, accept_len, next_token,
                                      target_tokens, workspace, lay, (cudaStream_t)stream);
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

SV_API size_t spec_accept_stochastic_workspace_size(int32_t batch, int32_t max_draft_len,
                                                   int32_t vocab) {
  if (batch < 0 || max_draft_len < 0 || max_draft_len > 255 || vocab <= 0 ||
      vocab > (1 << 30))
    return 0;
  return 256;  // the flag word
}

SV_API sv_status spec_accept_stochastic(int32_t batch, int32_t max_draft_len, int32_t vocab,
                                        int32_t logits_dtype, const void* target_logits,
                                        const void* draft_logits, const int32_t* draft_tokens,
                                        const int32_t* draft_len, const float* u_accept,
                                        const float* u_sample, float temperature,
                                        int32_t* accept_len, int32_t* next_token,
                                        void* workspace, size_t workspace_bytes, void* stream) {
  if (batch < 0 || max_draft_len < 0 || max_draft_len > 255 || vocab <= 0 ||
      vocab > (1 << 30) || !(temperature > 0.f) || isinf(temperature))
    return SV_ERR_SHAPE;
  if (logits_dtype != SV_BF16 && logits_dtype != SV_FP32) return SV_ERR_DTYPE;
  if (batch == 0) return SV_OK;
  if (!target_logits || !draft_len || !u_sample || !accept_len || !next_token || !workspace)
    return SV_ERR_NULL;
  if (max_draft_len > 0 && (!draft_logits || !draft_tokens || !u_accept)) return SV_ERR_NULL;
  const uintptr_t es = logits_dtype == SV_BF16 ? 2 : 4;
  if (!aligned(target_logits, es) || (draft_logits && !aligned(draft_logits, es)) ||
      !aligned(draft_len, 4) || (draft_tokens && !aligned(draft_tokens, 4)) ||
      (u_accept && !aligned(u_accept, 4)) || !aligned(u_sample, 4) ||
      !aligned(accept_len, 4) || !aligned(next_token, 4) || !aligned(workspace, 256))
    return SV_ERR_ALIGN;
  if (workspace_bytes < 256) return SV_ERR_WORKSPACE;
  const cudaError_t e = launch_accept_stochastic(
      batch, max_draft_len, vocab, logits_dtype, target_logits, draft_logits, draft_tokens,
      draft_len, u_accept, u_sample, 1.f / temperature, accept_len, next_token, workspace,
      (cudaStream_t)stream);
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

SV_API size_t spec_draft_signals_workspace_size(int32_t rows, int32_t vocab) {
  if (rows < 0 || vocab <= 0) return 0;
  const int sms = current_sms();
  if (sms <= 0) return 0;
  return signals_ws_layout(rows, vocab, sms).total;
}

SV_API sv_status spec_draft_signals(int32_t rows, int32_t vocab, int32_t logits_dtype,
                                    const void* logits, float* confidence, float* entropy,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  if (rows < 0 || vocab <= 0) return SV_ERR_SHAPE;
  if (logits_dtype != SV_BF16 && logits_dtype != SV_FP32) return SV_ERR_DTYPE;
  if (rows == 0) return SV_OK;
  if (!logits || !confidence || !entropy || !workspace) return SV_ERR_NULL;
  const uintptr_t es = logits_dtype == SV_BF16 ? 2 : 4;
  if (!aligned(logits, es) || !aligned(confidence, 4) || !aligned(entropy, 4) ||
      !aligned(workspace, 256))
    return SV_ERR_ALIGN;
  const int sms = current_sms();
  if (sms <= 0) return SV_ERR_CUDA;
  const SigWs lay = signals_ws_layout(rows, vocab, sms);
  if (workspace_bytes < lay.total) return SV_ERR_WORKSPACE;
  const cudaError_t e = launch_signals(rows, vocab, logits_dtype, logits, confidence, entropy,
                                       workspace, lay, (cudaStream_t)stream);
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

SV_API sv_status sv_workspace_status(void* workspace, int clear, void* stream) {
  if (!workspace) return SV_ERR_NULL;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t flags = 0;
  if (cudaMemcpyAsync(&flags, workspace, sizeof flags, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SV_ERR_CUDA;
  if (clear && cudaMemsetAsync(workspace, 0, sizeof flags, s) != cudaSuccess) return SV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SV_ERR_CUDA;
  if (flags & FLAG_TIMEOUT) return SV_ERR_TIMEOUT;
  if (flags & (FLAG_ATTN_SHAPE | FLAG_ACCEPT_SHAPE)) return SV_ERR_DEVICE_SHAPE;
  return SV_OK;
}

}  // extern "C"

/*
 * oracle.c -- plain fp64 CPU oracle for the speculative-decoding verification step.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load this library. It shares no code, header, table or constant with the
 * CUDA library; it is written straight from the definitions it cites and is slow on
 * purpose: every score table is materialised, every argmax is a naive loop.
 *
 * Sources (page title, then section):
 *   [P2] "Co-Designing AI Models Using Speculative Decoding ..." (summary page),
 *        section "basic structure of speculative decoding": draft length D, acceptance
 *        length AL in [1, 1+D], accept draft tokens up to the first mismatch.
 *   [P3] "GPU and LLM, chapter 5", sections "Online softmax: carry the max and the sum"
 *        (the m / l / O update, exact rather than approximate), "GQA: several Q heads share
 *        one K/V head", "Speculative decoding (2): verify together" (3 accepted, the 4th
 *        rejected, the target's own token inserted; one forward over k+1 positions).
 *   [P4] "SpecKV: Adaptive Speculative Decoding with Compression-Aware Gamma Selection"
 *        (summary page), section "technical core", item 1: the draft model's confidence
 *        and entropy, the inputs of the gamma controller.
 *
 * Readings where the pages are silent:
 *   - The 1+D window rows' K/V are already in the cache at positions T..T+D; window row i
 *     sees keys 0..T+i inclusive (T+i+1 keys).
 *   - Query head h uses KV head h / G (consecutive groups of G query heads).
 *   - FP8 values are OCP E4M3 codes times a per-KV-head fp32 scale (kv_scale[0][g] for K,
 *     kv_scale[1][g] for V).
 *   - Argmax ties go to the lowest index; -0.0 equals +0.0.
 *   - Draft signals: confidence = the largest probability of the row's softmax (the first
 *     of the page's two options); entropy = the Shannon entropy of that softmax in nats.
 *   - Sliding window ([P3] "Sliding window: do not keep the distant past"): with a window
 *     of W >= 1 positions the query at position p sees only the W most recent positions,
 *     itself included, i.e. keys max(0, p - W + 1) .. p; for window row i, p = T + i.
 *     W = 0 means no window (every earlier key).
 *   - Stochastic acceptance ([P3] "Speculative decoding (2)": the acceptance rule keeps
 *     the distribution of the output exactly that of the large model alone; the rule
 *     itself is not printed). The rule with that property from the paper the page cites
 *     (Leviathan, Kalman and Matias, "Fast Inference from Transformers via Speculative
 *     Decoding", 2023): with p the target's and q the drafter's softmax (logits divided
 *     by a temperature) at a draft position, the draft x is kept with probability
 *     min(1, p(x) / q(x)); at the first rejection the emitted token is drawn from the
 *     normalised max(0, p - q); with every draft kept, from the target's last row. The
 *     uniform draws are inputs: draft x_j is kept iff u_j q(x_j) < p(x_j), and a token is
 *     drawn as the smallest index k whose running sum of weights exceeds u times their
 *     total. If every weight of max(0, p - q) is 0 (p = q, so the rejected draft had
 *     q(x) = 0), the token is drawn from p.
 *
 * Layouts (packed ragged batch): q and out [sum_b W_b, Hq, d]; k and v
 * [sum_b (T_b + W_b), Hkv, d]; W_b = 1 + D_b; sequences in batch order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bfloat16 is the upper half of an IEEE-754 binary32 word. */
double orc_bf16_to_f64(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP 8-bit floating point, E4M3 variant: 1 sign bit, 4 exponent bits (bias 7),
 * 3 mantissa bits, no infinities; S.1111.111 is NaN. */
double orc_e4m3_to_f64(uint8_t bits) {
  int s = (bits >> 7) & 1;
  int e = (bits >> 3) & 15;
  int m = bits & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, 1 - 7);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

double orc_f32_to_f64(float f) { return (double)f; }

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

typedef struct {
  int B, Hq, Hkv, d, G;
  int kv_fp8;
  const uint16_t* q;
  const void* k;
  const void* v;
  const float* kv_scale;
  double scale;
  int64_t* q_off;   /* [B+1] prefix sums of W_b */
  int64_t* kv_off;  /* [B+1] prefix sums of T_b + W_b */
  const int32_t* seq_lens;
  const int32_t* draft_len;
  int window;      /* 0: none; W >= 1: only the W most recent positions are visible */
  double lut[256]; /* e4m3 code -> value, from orc_e4m3_to_f64 */
} orc_ctx;

static double kv_elem(const orc_ctx* c, const void* base, int which, int64_t row, int g,
                      int col) {
  int64_t idx = (row * c->Hkv + g) * (int64_t)c->d + col;
  if (c->kv_fp8)
    return c->lut[((const uint8_t*)base)[idx]] * (double)c->kv_scale[which * c->Hkv + g];
  return orc_bf16_to_f64(((const uint16_t*)base)[idx]);
}

static int setup(orc_ctx* c, int B, int Hq, int Hkv, int d, const int32_t* seq_lens,
                 const int32_t* draft_len, int kv_fp8, const uint16_t* q, const void* k,
                 const void* v, const float* kv_scale, double scale, int window) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0 || window < 0) return 1;
  c->window = window;
  if (kv_fp8 && !kv_scale) return 1;
  c->B = B; c->Hq = Hq; c->Hkv = Hkv; c->d = d; c->G = Hq / Hkv;
  c->kv_fp8 = kv_fp8; c->q = q; c->k = k; c->v = v; c->kv_scale = kv_scale;
  c->scale = scale; c->seq_lens = seq_lens; c->draft_len = draft_len;
  c->q_off = (int64_t*)malloc(sizeof(int64_t) * (B + 1));
  c->kv_off = (int64_t*)malloc(sizeof(int64_t) * (B + 1));
  c->q_off[0] = 0; c->kv_off[0] = 0;
  for (int b = 0; b < B; ++b) {
    if (seq_lens[b] < 0 || draft_len[b] < 0) return 1;
    c->q_off[b + 1] = c->q_off[b] + 1 + draft_len[b];
    c->kv_off[b + 1] = c->kv_off[b] + seq_lens[b] + 1 + draft_len[b];
  }
  for (int i = 0; i < 256; ++i) c->lut[i] = orc_e4m3_to_f64((uint8_t)i);
  return 0;
}

static void teardown(orc_ctx* c) { free(c->q_off); free(c->kv_off); }

/* First key visible to window row i of sequence b: 0, or with a sliding window of W
 * positions the oldest of the W positions ending at T + i. */
static int64_t first_key(const orc_ctx* c, int b, int i) {
  if (c->window <= 0) return 0;
  int64_t lo = (int64_t)c->seq_lens[b] + i - c->window + 1;
  return lo > 0 ? lo : 0;
}

/* One output row, materialised softmax ([P3] attention = softmax(q K^T) V over the
 * visible keys; the window-causal mask keeps keys first_key .. T+i, and s[n] holds the
 * score of key first_key + n). */
static void row_materialised(const orc_ctx* c, int b, int h, int i, double* s,
                             double* out_row) {
  const int g = h / c->G, d = c->d;
  const int64_t j_lo = first_key(c, b, i);
  const int64_t nkeys = (int64_t)c->seq_lens[b] + i + 1;
  const int64_t qrow = c->q_off[b] + i;
  const uint16_t* qv = c->q + (qrow * c->Hq + h) * (int64_t)d;
  double mx = -INFINITY;
  for (int64_t j = j_lo; j < nkeys; ++j) {
    double acc = 0.0;
    for (int col = 0; col < d; ++col)
      acc += orc_bf16_to_f64(qv[col]) * kv_elem(c, c->k, 0, c->kv_off[b] + j, g, col);
    s[j - j_lo] = acc * c->scale;
    if (s[j - j_lo] > mx) mx = s[j - j_lo];
  }
  double denom = 0.0;
  for (int64_t j = j_lo; j < nkeys; ++j) {
    s[j - j_lo] = exp(s[j - j_lo] - mx);
    denom += s[j - j_lo];
  }
  for (int col = 0; col < d; ++col) out_row[col] = 0.0;
  for (int64_t j = j_lo; j < nkeys; ++j) {
    double p = s[j - j_lo] / denom;
    for (int col = 0; col < d; ++col)
      out_row[col] += p * kv_elem(c, c->v, 1, c->kv_off[b] + j, g, col);
  }
}

/* One output row with the online-softmax update of [P3] "Online softmax", applied tile by
 * tile: m_new = max(m, max s); l_new = l*exp(m - m_new) + sum exp(s - m_new);
 * O_new = O*exp(m - m_new) + sum exp(s - m_new) v; finally O / l. */
static void row_online(const orc_ctx* c, int b, int h, int i, int tile, double* s,
                       double* out_row) {
  const int g = h / c->G, d = c->d;
  const int64_t nkeys = (int64_t)c->seq_lens[b] + i + 1;
  const int64_t qrow = c->q_off[b] + i;
  const uint16_t* qv = c->q + (qrow * c->Hq + h) * (int64_t)d;
  double m = -INFINITY, l = 0.0;
  for (int col = 0; col < d; ++col) out_row[col] = 0.0;
  for (int64_t j0 = first_key(c, b, i); j0 < nkeys; j0 += tile) {
    int64_t j1 = j0 + tile < nkeys ? j0 + tile : nkeys;
    double tmax = -INFINITY;
    for (int64_t j = j0; j < j1; ++j) {
      double acc = 0.0;
      for (int col = 0; col < d; ++col)
        acc += orc_bf16_to_f64(qv[col]) * kv_elem(c, c->k, 0, c->kv_off[b] + j, g, col);
      s[j - j0] = acc * c->scale;
      if (s[j - j0] > tmax) tmax = s[j - j0];
    }
    double m_new = m > tmax ? m : tmax;
    double alpha = exp(m - m_new); /* exp(-inf) = 0 on the first tile */
    l *= alpha;
    for (int col = 0; col < d; ++col) out_row[col] *= alpha;
    for (int64_t j = j0; j < j1; ++j) {
      double p = exp(s[j - j0] - m_new);
      l += p;
      for (int col = 0; col < d; ++col)
        out_row[col] += p * kv_elem(c, c->v, 1, c->kv_off[b] + j, g, col);
    }
    m = m_new;
  }
  for (int col = 0; col < d; ++col) out_row[col] /= l;
}

static int run_attn(int B, int Hq, int Hkv, int d, const int32_t* seq_lens,
                    const int32_t* draft_len, int kv_fp8, const uint16_t* q, const void* k,
                    const void* v, const float* kv_scale, double scale,
                    const uint8_t* unit_mask, const uint8_t* row_mask, double* out,
                    int nthreads, int tile, int window) {
  orc_ctx c;
  if (setup(&c, B, Hq, Hkv, d, seq_lens, draft_len, kv_fp8, q, k, v, kv_scale, scale,
            window)) {
    return 1;
  }
  int64_t max_keys = 1;
  for (int b = 0; b < B; ++b) {
    int64_t n = (int64_t)seq_lens[b] + 1 + draft_len[b];
    if (n > max_keys) max_keys = n;
  }
  /* packed query row -> sequence */
  const int64_t qrows = c.q_off[B];
  int32_t* row_b = (int32_t*)malloc(sizeof(int32_t) * (size_t)(qrows > 0 ? qrows : 1));
  for (int b = 0; b < B; ++b)
    for (int64_t r = c.q_off[b]; r < c.q_off[b + 1]; ++r) row_b[r] = b;
  const int64_t total = qrows * Hq; /* one task per (query row, head) */
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(tile > 0 ? tile : max_keys));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
    for (int64_t task = 0; task < total; ++task) {
      if (row_mask && !row_mask[task]) continue;
      const int64_t qrow = task / Hq;
      const int h = (int)(task % Hq);
      const int b = row_b[qrow];
      if (unit_mask && !unit_mask[(int64_t)b * Hkv + h / c.G]) continue;
      const int i = (int)(qrow - c.q_off[b]);
      double* o = out + task * (int64_t)d;
      if (tile > 0)
        row_online(&c, b, h, i, tile, s, o);
      else
        row_materialised(&c, b, h, i, s, o);
    }
    free(s);
  }
  free(row_b);
  teardown(&c);
  return 0;
}

/* Verify attention, materialised softmax. unit_mask [B*Hkv] selects (b, kv-head) units and
 * row_mask [sum W * Hq] selects (query row, head) outputs to compute (NULL: all); outputs
 * not selected are left untouched. kv_fp8 = 0: k/v are bf16 bit patterns; 1: E4M3 codes
 * with kv_scale [2, Hkv]. window = 0: every earlier key; W >= 1: a sliding window of the W
 * most recent positions. Returns 0 on success. */
int orc_verify_attn(int B, int Hq, int Hkv, int d, const int32_t* seq_lens,
                    const int32_t* draft_len, int kv_fp8, const uint16_t* q, const void* k,
                    const void* v, const float* kv_scale, double scale,
                    const uint8_t* unit_mask, const uint8_t* row_mask, double* out,
                    int nthreads, int window) {
  return run_attn(B, Hq, Hkv, d, seq_lens, draft_len, kv_fp8, q, k, v, kv_scale, scale,
                  unit_mask, row_mask, out, nthreads, 0, window);
}

/* The same attention through the tile-by-tile online-softmax update (tile >= 1 keys). */
int orc_verify_attn_online(int B, int Hq, int Hkv, int d, const int32_t* seq_lens,
                           const int32_t* draft_len, int kv_fp8, const uint16_t* q,
                           const void* k, const void* v, const float* kv_scale,
                           double scale, const uint8_t* unit_mask, const uint8_t* row_mask,
                           double* out, int nthreads, int tile, int window) {
  if (tile < 1) return 1;
  return run_attn(B, Hq, Hkv, d, seq_lens, draft_len, kv_fp8, q, k, v, kv_scale, scale,
                  unit_mask, row_mask, out, nthreads, tile, window);
}

/* Row-wise argmax, naive loop, first index wins ties (strict '>' keeps the earliest).
 * dtype 0: bf16 bit patterns (uint16); 2: fp32. Values are compared exactly in fp64. */
int orc_argmax_rows(int64_t rows, int64_t vocab, int dtype, const void* logits,
                    int32_t* amax, int nthreads) {
  if (rows < 0 || vocab <= 0 || (dtype != 0 && dtype != 2)) return 1;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for num_threads(nthreads) schedule(static)
#endif
  for (int64_t r = 0; r < rows; ++r) {
    double best = 0.0;
    int64_t arg = 0;
    for (int64_t j = 0; j < vocab; ++j) {
      double x = dtype == 0 ? orc_bf16_to_f64(((const uint16_t*)logits)[r * vocab + j])
                            : (double)((const float*)logits)[r * vocab + j];
      if (j == 0 || x > best) { best = x; arg = j; }
    }
    amax[r] = (int32_t)arg;
  }
  return 0;
}

/* Greedy acceptance ([P2] "accept tokens until the first mismatch"; [P3] the target's own
 * token replaces the first rejected draft, and with all k drafts accepted the step yields
 * k+1 tokens). amax holds the target's argmax for every window row [sum_b W_b];
 * draft_tokens is packed [sum_b D_b]. For sequence b: n = number of leading positions j
 * with draft[j] == amax[j]; AL = n + 1; next_token = amax[n]. */
int orc_accept(int B, const int32_t* draft_len, const int32_t* draft_tokens,
               const int32_t* amax, int32_t* accept_len, int32_t* next_token) {
  int64_t q_off = 0, d_off = 0;
  for (int b = 0; b < B; ++b) {
    int D = draft_len[b];
    if (D < 0) return 1;
    int n = 0;
    while (n < D && draft_tokens[d_off + n] == amax[q_off + n]) ++n;
    accept_len[b] = n + 1;
    next_token[b] = amax[q_off + n];
    q_off += 1 + D;
    d_off += D;
  }
  return 0;
}

/* Draft signals of every row ([P4] "technical core", item 1). The softmax of the row is
 * materialised in fp64, p_j = exp(x_j - m) / sum_k exp(x_k - m) with m the row maximum;
 * confidence = max_j p_j; entropy = -sum_j p_j ln p_j over the p_j > 0 (0 ln 0 = 0).
 * dtype 0: bf16 bit patterns; 2: fp32. Rows must hold at least one finite value. */
int orc_draft_signals(int64_t rows, int64_t vocab, int dtype, const void* logits,
                      double* confidence, double* entropy, int nthreads) {
  if (rows < 0 || vocab <= 0 || (dtype != 0 && dtype != 2)) return 1;
  int bad = 0;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for num_threads(nthreads) schedule(static) reduction(| : bad)
#endif
  for (int64_t r = 0; r < rows; ++r) {
    double* p = (double*)malloc(sizeof(double) * (size_t)vocab);
    if (!p) {
      bad = 1;
      continue;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < vocab; ++j) {
      p[j] = dtype == 0 ? orc_bf16_to_f64(((const uint16_t*)logits)[r * vocab + j])
                        : (double)((const float*)logits)[r * vocab + j];
      if (p[j] > m) m = p[j];
    }
    double z = 0.0;
    for (int64_t j = 0; j < vocab; ++j) {
      p[j] = exp(p[j] - m);
      z += p[j];
    }
    double pmax = 0.0, h = 0.0;
    for (int64_t j = 0; j < vocab; ++j) {
      const double pj = p[j] / z;
      if (pj > pmax) pmax = pj;
      if (pj > 0.0) h -= pj * log(pj);
    }
    confidence[r] = pmax;
    entropy[r] = h;
    free(p);
  }
  return bad;
}

/* Logit j of row r divided by the temperature, in fp64 (dtype 0: bf16 bits; 2: fp32). */
static double scaled_logit(const void* base, int dtype, int64_t r, int64_t vocab, int64_t j,
                           double inv_temp) {
  const double x = dtype == 0 ? orc_bf16_to_f64(((const uint16_t*)base)[r * vocab + j])
                              : (double)((const float*)base)[r * vocab + j];
  return x * inv_temp;
}

/* The softmax of one row, materialised: p[j] = exp(x_j - m) / sum_k exp(x_k - m), with
 * x = logits / temperature and m the row maximum. Returns 1 if the row has no finite
 * value. */
static int softmax_row(const void* base, int dtype, int64_t r, int64_t vocab, double inv_temp,
                       double* p) {
  double m = -INFINITY;
  for (int64_t j = 0; j < vocab; ++j) {
    p[j] = scaled_logit(base, dtype, r, vocab, j, inv_temp);
    if (p[j] > m) m = p[j];
  }
  if (!isfinite(m)) return 1;
  double z = 0.0;
  for (int64_t j = 0; j < vocab; ++j) {
    p[j] = exp(p[j] - m);
    z += p[j];
  }
  for (int64_t j = 0; j < vocab; ++j) p[j] /= z;
  return 0;
}

/* Inverse CDF of the distribution proportional to w >= 0 at u in [0, 1): the smallest k
 * whose running sum w[0] + ... + w[k] exceeds u * sum(w). *margin receives the distance of
 * u * sum(w) from the nearer end of k's interval, relative to sum(w). Returns -1 if every
 * weight is 0. */
static int64_t inverse_cdf(const double* w, int64_t vocab, double u, double* margin) {
  double total = 0.0;
  for (int64_t k = 0; k < vocab; ++k) total += w[k];
  if (!(total > 0.0)) return -1;
  const double t = u * total;
  double cum = 0.0;
  int64_t last = -1;
  for (int64_t k = 0; k < vocab; ++k) {
    if (w[k] > 0.0) last = k;
    const double prev = cum;
    cum += w[k];
    if (cum > t) {
      const double a = t - prev, b = cum - t;
      *margin = (a < b ? a : b) / total;
      return k;
    }
  }
  *margin = 0.0;  /* rounding left t at the end: the last token of positive weight */
  return last;
}

/* Stochastic acceptance of every sequence (see the reading above). target: [sum_b W_b,
 * vocab] logits, the target's rows of each window; draft: [sum_b D_b, vocab], the
 * drafter's logits at each draft position; draft_tokens [sum_b D_b]; u_accept [sum_b D_b]
 * and u_sample [B] uniform in [0, 1). Writes accept_len, next_token and, per sequence,
 * two decision margins: margin_accept, the smallest |u q(x) - p(x)| / max(u q(x), p(x))
 * over the drafts examined (1 without drafts), and margin_sample, the inverse-CDF margin
 * of the drawn token (a result decided by floating point within such a margin may
 * legitimately differ in another precision). */
int orc_accept_stochastic(int B, int64_t vocab, int dtype, const void* target,
                          const void* draft, const int32_t* draft_tokens,
                          const int32_t* draft_len, const float* u_accept,
                          const float* u_sample, double temperature, int32_t* accept_len,
                          int32_t* next_token, double* margin_accept, double* margin_sample) {
  if (B < 0 || vocab <= 0 || (dtype != 0 && dtype != 2) || !(temperature > 0.0)) return 1;
  const double inv_temp = 1.0 / temperature;
  double* p = (double*)malloc(sizeof(double) * (size_t)vocab);
  double* q = (double*)malloc(sizeof(double) * (size_t)vocab);
  if (!p || !q) {
    free(p);
    free(q);
    return 1;
  }
  int bad = 0;
  int64_t q_off = 0, d_off = 0;
  for (int b = 0; b < B && !bad; ++b) {
    const int D = draft_len[b];
    if (D < 0) {
      bad = 1;
      break;
    }
    double mg = 1.0;
    int n = D;  /* drafts kept */
    for (int j = 0; j < D; ++j) {
      const int32_t x = draft_tokens[d_off + j];
      if (x < 0 || x >= vocab || softmax_row(target, dtype, q_off + j, vocab, inv_temp, p) ||
          softmax_row(draft, dtype, d_off + j, vocab, inv_temp, q)) {
        bad = 1;
        break;
      }
      const double lhs = (double)u_accept[d_off + j] * q[x], rhs = p[x];
      const double den = lhs > rhs ? lhs : rhs;
      const double m = den > 0.0 ? fabs(lhs - rhs) / den : 0.0;
      if (m < mg) mg = m;
      if (!(lhs < rhs)) {
        n = j;
        break;
      }
    }
    if (bad) break;
    if (n < D) {  /* p and q hold row n: draw from max(0, p - q) */
      for (int64_t k = 0; k < vocab; ++k) p[k] = p[k] > q[k] ? p[k] - q[k] : 0.0;
    } else if (softmax_row(target, dtype, q_off + D, vocab, inv_temp, p)) {
      bad = 1;
      break;
    }
    double m2 = 0.0;
    int64_t k = inverse_cdf(p, vocab, (double)u_sample[b], &m2);
    if (k < 0 && n < D) {
      /* every residual weight is 0 (p = q; a rejection then needs q(x) = 0): draw from
       * the target's row instead */
      if (softmax_row(target, dtype, q_off + n, vocab, inv_temp, p)) {
        bad = 1;
        break;
      }
      k = inverse_cdf(p, vocab, (double)u_sample[b], &m2);
    }
    if (k < 0) {
      bad = 1;
      break;
    }
    accept_len[b] = n + 1;
    next_token[b] = (int32_t)k;
    margin_accept[b] = mg;
    margin_sample[b] = m2;
    q_off += 1 + D;
    d_off += D;
  }
  free(p);
  free(q);
  return bad;
}

/* Every keep / reject decision of stochastic acceptance, whether or not the sequence's
 * acceptance reaches it: for draft position j of sequence b (row d_off + j of the
 * drafter's logits, d_off = D_0 + ... + D_(b-1); row q_off + j of the target's, q_off =
 * d_off + b), with x = draft_tokens[d_off + j], lhs = u_accept[d_off + j] q(x) and rhs =
 * p(x), decision[d_off + j] = (rhs - lhs) / max(lhs, rhs), or 0 when both are 0. The draft
 * is kept iff the value is positive (u q(x) < p(x), the rule of orc_accept_stochastic), and
 * its magnitude is the decision's relative margin: a value within a small margin of 0 may
 * come out either way in another precision. [P3] "Speculative decoding (2)"; the rule of
 * Leviathan et al. (2023) as above. */
int orc_stochastic_decisions(int B, int64_t vocab, int dtype, const void* target,
                             const void* draft, const int32_t* draft_tokens,
                             const int32_t* draft_len, const float* u_accept,
                             double temperature, double* decision) {
  if (B < 0 || vocab <= 0 || (dtype != 0 && dtype != 2) || !(temperature > 0.0)) return 1;
  const double inv_temp = 1.0 / temperature;
  double* p = (double*)malloc(sizeof(double) * (size_t)vocab);
  double* q = (double*)malloc(sizeof(double) * (size_t)vocab);
  if (!p || !q) {
    free(p);
    free(q);
    return 1;
  }
  int bad = 0;
  int64_t d_off = 0;
  for (int b = 0; b < B && !bad; ++b) {
    const int D = draft_len[b];
    if (D < 0) {
      bad = 1;
      break;
    }
    const int64_t q_off = d_off + b;
    for (int j = 0; j < D; ++j) {
      const int32_t x = draft_tokens[d_off + j];
      if (x < 0 || x >= vocab || softmax_row(target, dtype, q_off + j, vocab, inv_temp, p) ||
          softmax_row(draft, dtype, d_off + j, vocab, inv_temp, q)) {
        bad = 1;
        break;
      }
      const double lhs = (double)u_accept[d_off + j] * q[x], rhs = p[x];
      const double den = lhs > rhs ? lhs : rhs;
      decision[d_off + j] = den > 0.0 ? (rhs - lhs) / den : 0.0;
    }
    d_off += D;
  }
  free(p);
  free(q);
  return bad;
}

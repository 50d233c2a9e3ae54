/*
 * CPU oracle of the per-layer causal grouped-query attention step.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the timed CPU
 * baseline of the benchmark load this library.  It shares no code, header,
 * table or constant with the CUDA path and never calls it.
 *
 * It computes the plain definition of the step in fp64, one (token, head)
 * row at a time, with no blocking, fusion or online softmax:
 *
 *   1. split the packed qkv row into Q, K and V heads
 *      (zero-to-sglang Ch.3 code walkthrough, section 3.3; transformer-basics
 *      "Attention calculation: part 1": [1,12,4096] -> [1,12,32,128]);
 *   2. RMSNorm over each Q and K head's last dimension with a learned weight
 *      (code walkthrough section 3.3; part 1's q_norm / k_norm after .view);
 *   3. RoPE on Q and K at each token's position (concept chapter section 2.2
 *      and its section 2.6 table; the RoFormer paper they cite), V untouched;
 *   4. append K (rounded once to bf16) and V (bit copy) to the cache
 *      (transformer-basics "Prefill vs Decode": DynamicCache.update, 0 -> 12 -> 13);
 *   5. causal GQA: query head h reads KV head h / (Hq/Hkv) (repeat_interleave),
 *      scores q.k / sqrt(D), future keys excluded, softmax, weighted sum of V
 *      (code walkthrough section 3.3 teaching snippet; transformer-basics
 *      "Attention calculation: part 1", scaling = head_dim ** -0.5).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - RMSNorm: y = w * x / sqrt(mean(x^2) + eps);
 *   - RoPE: rotate-half pairing (i, i + D/2), frequency theta^(-2i/D),
 *     rotation [[cos, -sin], [sin, cos]] applied to (x_i, x_{i+D/2});
 *     the pairing convention is "parity unpinned": the pages fix no pairing;
 *   - norm before RoPE; position of new token j of request b is c_b + j;
 *   - Q stays in fp64; K is rounded to bf16 (round to nearest even) once,
 *     when it is written to the cache; softmax and P.V in fp64.
 *
 * One-byte cache entries (kv_fp8 != 0): the concept chapter's section 4.3
 * (decode is bound by memory bandwidth) and its section 2.6 (KV-cache
 * reduction among the modern variants) motivate them; the pages fix no
 * format, so the reading is OCP FP8 E4M3 with one scale per cache: the
 * stored byte of x is e4m3(fp32(x) * fp32(1 / scale)), the product taken in
 * fp32 because that is the precision the stored code is decided in, rounded
 * to nearest even with magnitudes beyond 448 clamped to 448; an entry reads
 * as byte * scale.  Attention then runs in fp64 on those values.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a double to the nearest bf16 (ties to even) directly, without an
 * intermediate float rounding: scale the significand so that the last kept
 * bit is the unit, round with nearbyint (the default rounding mode is
 * round-to-nearest-even), scale back.  The result is exactly representable in
 * float, so the final conversion and bit extraction are exact. */
uint16_t oracle_bf16_round(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80;
  int e;
  double m = frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
  /* normal bf16 keeps 8 significant bits; below 2^-126 the quantum is 2^-133 */
  int shift = (e >= -125) ? 8 : e + 133;
  double r = nearbyint(ldexp(m, shift));
  double y = ldexp(r, e - shift);
  if (y >= ldexp(1.0, 128)) return sign | 0x7F80;
  float f = (float)y;
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return sign | (uint16_t)(u >> 16);
}

/*
 * OCP FP8 E4M3: sign bit, 4 exponent bits (bias 7), 3 mantissa bits.  Code
 * (E, M) with E >= 1 is (8 + M) * 2^(E - 10); E = 0 is M * 2^-9 (subnormal);
 * E = 15, M = 7 is NaN; there is no infinity, so 448 (E = 15, M = 6) is the
 * largest finite value.
 */
double oracle_e4m3_decode(uint8_t b) {
  int E = (b >> 3) & 15, M = b & 7;
  if (E == 15 && M == 7) return NAN;
  double v = E == 0 ? ldexp((double)M, -9) : ldexp((double)(8 + M), E - 10);
  return (b & 0x80) ? -v : v;
}

/* Nearest E4M3 code to x, ties to even; finite magnitudes at or beyond 448
 * give 448 (the saturating conversion).  The quantum of the binade
 * [2^e, 2^(e+1)) is 2^(e-3), and 2^-9 below 2^-6 (subnormals); dividing by
 * it is exact, nearbyint rounds to nearest even, and the rounded value is
 * then exactly one code (it may be the bottom of the next binade). */
uint8_t oracle_e4m3_encode(double x) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0;
  double a = fabs(x);
  if (a >= 448.0) return sign | 0x7E;
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e); /* a in [2^(e-1), 2^e) */
  int lo = e - 1 < -6 ? -6 : e - 1;
  double quantum = ldexp(1.0, lo - 3);
  double r = nearbyint(a / quantum) * quantum; /* <= 448 since a < 448 = 14 * 32 */
  if (r < ldexp(1.0, -6)) return sign | (uint8_t)(r / ldexp(1.0, -9));
  int er;
  double f = frexp(r, &er); /* r = f * 2^er, f in [0.5, 1) */
  int E = er - 1 + 7;
  int M = (int)((2.0 * f - 1.0) * 8.0);
  return sign | (uint8_t)(E << 3) | (uint8_t)M;
}

/* Code stored for value x under a cache scale: e4m3(fp32(x) * fp32(1/scale)),
 * both roundings to fp32 and the product in fp32 (C evaluates float * float
 * in float on the targets this builds for). */
static uint8_t e4m3_store(double x, float scale) {
  const float r = 1.0f / scale;
  const float t = (float)x * r;
  return oracle_e4m3_encode((double)t);
}

/* Weighted RMSNorm of one head vector (step 2). */
void oracle_rmsnorm(const double* x, const double* w, int D, double eps, double* y) {
  double ss = 0.0;
  for (int i = 0; i < D; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / (double)D + eps);
  for (int i = 0; i < D; ++i) y[i] = w[i] * (x[i] * inv);
}

/* RoPE of one head vector at position pos, in place (step 3). */
void oracle_rope(double* x, int D, double pos, double theta) {
  int half = D / 2;
  for (int i = 0; i < half; ++i) {
    double freq = pow(theta, -2.0 * (double)i / (double)D);
    double a = pos * freq;
    double c = cos(a), s = sin(a);
    double x1 = x[i], x2 = x[i + half];
    x[i] = x1 * c - x2 * s;
    x[i + half] = x2 * c + x1 * s;
  }
}

static int find_request(const int32_t* cu, int B, int64_t t) {
  int lo = 0, hi = B; /* cu[lo] <= t < cu[hi] */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (cu[mid] <= t) lo = mid; else hi = mid;
  }
  return lo;
}

/*
 * Slot of the entry at position pos of request b.  page_size == 0: the
 * request's contiguous region, slot_base[b] + pos.  Otherwise the paged
 * layout: page page_table[b * pages_per_req + pos / page_size], entry
 * pos % page_size of that page.
 */
static int64_t slot_of(const int64_t* slot_base, const int32_t* page_table, int page_size,
                       int pages_per_req, int b, int64_t pos) {
  if (page_size == 0) return slot_base[b] + pos;
  return (int64_t)page_table[(int64_t)b * pages_per_req + pos / page_size] * page_size +
         pos % page_size;
}

static void load_head(const uint16_t* row, int64_t col0, int D, double* out) {
  for (int i = 0; i < D; ++i) out[i] = bf16_bits_to_double(row[col0 + i]);
}

/* Head vector of token t from the packed qkv: bf16 bits, or (row64 != NULL)
 * the fp64 output of the projection itself, never rounded. */
static void load_src(const uint16_t* qkv, const double* qkv64, int64_t t, int64_t W, int64_t col0,
                     int D, double* out) {
  if (qkv64) {
    for (int i = 0; i < D; ++i) out[i] = qkv64[t * W + col0 + i];
  } else {
    load_head(qkv + t * W, col0, D, out);
  }
}

/*
 * The merged Q/K/V projection in front of the step and the output projection
 * behind it (walkthrough section 3.3: qkv_proj, then o_proj on the attention
 * output): y[n][o] = sum_c x[n][c] * w[o][c], x fp64 [N, C], w bf16 bits
 * [O, C] (the nn.Linear weight layout), y fp64 [N, O]; plain loops, fp64 sums
 * in index order.
 */
void oracle_linear(int64_t N, int64_t C, int64_t O, const double* x, const uint16_t* w, double* y) {
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n)
    for (int64_t o = 0; o < O; ++o) {
      double acc = 0.0;
      for (int64_t c = 0; c < C; ++c) acc += x[n * C + c] * bf16_bits_to_double(w[o * C + c]);
      y[n * O + o] = acc;
    }
}

/*
 * Steps 1-4 for all N tokens.  The cache (k_cache, v_cache: bf16 bits, or
 * E4M3 bytes when kv_fp8, [num_slots, Hkv, D]) is updated in place: token j
 * of request b goes to the slot of position cache_lens[b] + j (slot_of).  Q rows (normed, rotated, fp64) are written
 * to q_out: all N*Hq rows as [N, Hq, D] when nq < 0, otherwise the nq rows
 * (q_tok[r], q_head[r]) as [nq, D].  Returns the number of requests whose
 * region cannot hold cache_lens + new tokens (those write nothing).
 */
static int prologue_impl(int Hq, int Hkv, int D, double eps, double theta,
                    const uint16_t* qkv, const double* qkv64, int64_t N, const uint16_t* q_norm_w,
                    const uint16_t* k_norm_w, int B, const int32_t* cu_seqlens,
                    const int32_t* cache_lens, const int64_t* slot_base,
                    const int32_t* slot_capacity, const int32_t* page_table, int page_size,
                    int pages_per_req, int64_t num_slots, void* k_cache,
                    void* v_cache, int kv_fp8, float k_scale, float v_scale, int64_t nq,
                    const int32_t* q_tok, const int32_t* q_head, double* q_out) {
  const int64_t W = (int64_t)(Hq + 2 * Hkv) * D;
  double* qw = malloc(sizeof(double) * D);
  double* kw = malloc(sizeof(double) * D);
  load_head(q_norm_w, 0, D, qw);
  load_head(k_norm_w, 0, D, kw);
  int bad = 0;
  for (int b = 0; b < B; ++b) {
    int64_t n = cu_seqlens[b + 1] - cu_seqlens[b];
    int64_t end = (int64_t)cache_lens[b] + n;
    int fits = n >= 0 && end <= slot_capacity[b];
    if (fits && page_size == 0) fits = slot_base[b] >= 0 && slot_base[b] + end <= num_slots;
    if (fits && page_size != 0) {
      fits = end <= (int64_t)pages_per_req * page_size;
      for (int64_t pg = 0; fits && pg * page_size < end; ++pg) {
        int64_t page = page_table[(int64_t)b * pages_per_req + pg];
        fits = page >= 0 && (page + 1) * page_size <= num_slots;
      }
    }
    if (!fits) {
      ++bad;
      continue;
    }
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) {
      int64_t t = cu_seqlens[b] + j;
      double pos = (double)cache_lens[b] + (double)j;
      int64_t slot = slot_of(slot_base, page_table, page_size, pages_per_req, b, cache_lens[b] + j);
      double x[256], y[256], v[256];
      for (int kh = 0; kh < Hkv; ++kh) {
        load_src(qkv, qkv64, t, W, (int64_t)(Hq + kh) * D, D, x);
        oracle_rmsnorm(x, kw, D, eps, y);
        oracle_rope(y, D, pos, theta);
        const int64_t e0 = (slot * Hkv + kh) * D;
        load_src(qkv, qkv64, t, W, (int64_t)(Hq + Hkv + kh) * D, D, v);
        if (kv_fp8) {
          uint8_t* kd = (uint8_t*)k_cache + e0;
          uint8_t* vd = (uint8_t*)v_cache + e0;
          for (int i = 0; i < D; ++i) {
            kd[i] = e4m3_store(y[i], k_scale);
            vd[i] = e4m3_store(v[i], v_scale);
          }
        } else {
          uint16_t* kd = (uint16_t*)k_cache + e0;
          uint16_t* vd = (uint16_t*)v_cache + e0;
          for (int i = 0; i < D; ++i) {
            kd[i] = oracle_bf16_round(y[i]);
            vd[i] = oracle_bf16_round(v[i]);  /* a bf16 input rounds to itself */
          }
        }
      }
    }
  }
  int64_t rows = nq < 0 ? N * Hq : nq;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    int64_t t = nq < 0 ? r / Hq : q_tok[r];
    int h = nq < 0 ? (int)(r % Hq) : q_head[r];
    int b = find_request(cu_seqlens, B, t);
    double pos = (double)cache_lens[b] + (double)(t - cu_seqlens[b]);
    double x[256];
    load_src(qkv, qkv64, t, W, (int64_t)h * D, D, x);
    oracle_rmsnorm(x, qw, D, eps, q_out + r * D);
    oracle_rope(q_out + r * D, D, pos, theta);
  }
  free(qw);
  free(kw);
  return bad;
}

int oracle_prologue(int Hq, int Hkv, int D, double eps, double theta,
                    const uint16_t* qkv, int64_t N, const uint16_t* q_norm_w,
                    const uint16_t* k_norm_w, int B, const int32_t* cu_seqlens,
                    const int32_t* cache_lens, const int64_t* slot_base,
                    const int32_t* slot_capacity, const int32_t* page_table, int page_size,
                    int pages_per_req, int64_t num_slots, void* k_cache,
                    void* v_cache, int kv_fp8, float k_scale, float v_scale, int64_t nq,
                    const int32_t* q_tok, const int32_t* q_head, double* q_out) {
  return prologue_impl(Hq, Hkv, D, eps, theta, qkv, NULL, N, q_norm_w, k_norm_w, B, cu_seqlens,
                       cache_lens, slot_base, slot_capacity, page_table, page_size, pages_per_req,
                       num_slots, k_cache, v_cache, kv_fp8, k_scale, v_scale, nq, q_tok, q_head,
                       q_out);
}

/*
 * The same steps fed by the projection's own output qkv64 (fp64 [N, W], as
 * oracle_linear gives it) instead of bf16 qkv: what a projection kernel that
 * hands its accumulators straight to the norm, the rotation and the cache
 * computes.  V is then rounded once, like K, when it enters the cache.
 */
int oracle_prologue_projected(int Hq, int Hkv, int D, double eps, double theta,
                              const double* qkv64, int64_t N, const uint16_t* q_norm_w,
                              const uint16_t* k_norm_w, int B, const int32_t* cu_seqlens,
                              const int32_t* cache_lens, const int64_t* slot_base,
                              const int32_t* slot_capacity, const int32_t* page_table,
                              int page_size, int pages_per_req, int64_t num_slots, void* k_cache,
                              void* v_cache, int kv_fp8, float k_scale, float v_scale, int64_t nq,
                              const int32_t* q_tok, const int32_t* q_head, double* q_out) {
  return prologue_impl(Hq, Hkv, D, eps, theta, NULL, qkv64, N, q_norm_w, k_norm_w, B, cu_seqlens,
                       cache_lens, slot_base, slot_capacity, page_table, page_size, pages_per_req,
                       num_slots, k_cache, v_cache, kv_fp8, k_scale, v_scale, nq, q_tok, q_head,
                       q_out);
}

/*
 * Step 5 for nrows (token, head) rows: out[r] = softmax(q_r . K^T / sqrt(D)) V
 * over the keys at positions 0 .. c_b + j of the row's request (the query's
 * own key included; later keys excluded), read from the cache (E4M3 entries
 * when kv_fp8: byte * scale).
 */
static double cache_entry(const void* cache, int kv_fp8, float scale, int64_t idx) {
  if (kv_fp8) return oracle_e4m3_decode(((const uint8_t*)cache)[idx]) * (double)scale;
  return bf16_bits_to_double(((const uint16_t*)cache)[idx]);
}

void oracle_attention(int Hq, int Hkv, int D, const void* k_cache, const void* v_cache,
                      int kv_fp8, float k_scale, float v_scale,
                      int B, const int32_t* cu_seqlens, const int32_t* cache_lens,
                      const int64_t* slot_base, const int32_t* page_table, int page_size,
                      int pages_per_req, int64_t nrows, const int32_t* tok,
                      const int32_t* head, const double* q, double* out) {
  const int G = Hq / Hkv;
  const double scale = 1.0 / sqrt((double)D);
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t t = tok[r];
    int h = head[r];
    int b = find_request(cu_seqlens, B, t);
    int64_t pos = (int64_t)cache_lens[b] + (t - cu_seqlens[b]);
    int kvh = h / G;
    int64_t nkeys = pos + 1;
    double* s = malloc(sizeof(double) * (size_t)nkeys);
    const double* qr = q + r * D;
    for (int64_t u = 0; u < nkeys; ++u) {
      const int64_t k0 = (slot_of(slot_base, page_table, page_size, pages_per_req, b, u) * Hkv + kvh) * D;
      double acc = 0.0;
      for (int i = 0; i < D; ++i) acc += qr[i] * cache_entry(k_cache, kv_fp8, k_scale, k0 + i);
      s[u] = acc * scale;
    }
    /* softmax(s) = exp(s - max) / sum exp(s - max): the shift leaves it unchanged */
    double m = -INFINITY;
    for (int64_t u = 0; u < nkeys; ++u) m = s[u] > m ? s[u] : m;
    double z = 0.0;
    for (int64_t u = 0; u < nkeys; ++u) {
      s[u] = exp(s[u] - m);
      z += s[u];
    }
    double* o = out + r * D;
    for (int i = 0; i < D; ++i) o[i] = 0.0;
    for (int64_t u = 0; u < nkeys; ++u) {
      double p = s[u] / z;
      const int64_t v0 = (slot_of(slot_base, page_table, page_size, pages_per_req, b, u) * Hkv + kvh) * D;
      for (int i = 0; i < D; ++i) o[i] += p * cache_entry(v_cache, kv_fp8, v_scale, v0 + i);
    }
    free(s);
  }
}

/*
 * Token sampling from one row of logits (concept chapter section 3.2: greedy
 * decoding, temperature, top-k and top-p; the walkthrough's section 4.3:
 * greedy batches take the argmax, the others temperature + top-k/top-p).
 *
 *   temperature <= 0: greedy, the smallest index holding the largest logit.
 *   Otherwise the distribution is softmax(logits / temperature) (section
 *   3.2.2's formula), truncated (section 3.2.3) to the tokens whose logit is
 *   at least lambda = max(lambda_k, lambda_p):
 *     top-k (0 < top_k < V): lambda_k = the top_k-th largest logit (ties
 *       with it are kept);
 *     top-p (top_p < 1): walking the tokens from the most probable down,
 *       lambda_p = the logit at which the cumulative probability first
 *       reaches top_p (tokens of equal logit enter together);
 *   then renormalised and sampled by the inverse distribution function in
 *   vocabulary order with the given uniform u in [0, 1): the token is the
 *   smallest kept index whose cumulative kept probability exceeds u.
 *
 * Returns the token.  *margin (not for greedy rows: +inf) is the smallest
 * relative distance of the row's two real-valued decisions from a boundary:
 * the top-p crossing (cumulative mass against top_p, as a fraction of the
 * total) and the sampled position (u against the cumulative kept fractions).
 * A result whose margin is below the device's rounding error may validly
 * differ on the device.
 */
/* qsort order: larger logit first, then smaller index (one row at a time). */
static const float* g_sort_logits;
static int cmp_desc_logit(const void* a, const void* b) {
  const float* l = g_sort_logits;
  int64_t i = *(const int64_t*)a, j = *(const int64_t*)b;
  if (l[i] != l[j]) return l[i] > l[j] ? -1 : 1;
  return i < j ? -1 : (i > j);
}

/* The truncation step for one row: weights w_i = exp(l_i / T - max / T),
 * their total *W, the kept threshold *lambda (logits >= *lambda are kept)
 * and the relative distance *margin_p of top_p from the crossing (inf when
 * top-p does not truncate).  Returns w (malloc'd). */
static double* truncate_row(int64_t V, const float* logits, double temperature, int64_t top_k,
                            double top_p, double* lambda, double* W, double* margin_p) {
  int64_t arg = 0;
  for (int64_t i = 1; i < V; ++i)
    if (logits[i] > logits[arg]) arg = i;
  double m = (double)logits[arg] / temperature;
  double* w = malloc(sizeof(double) * (size_t)V);
  *W = 0.0;
  for (int64_t i = 0; i < V; ++i) {
    w[i] = exp((double)logits[i] / temperature - m);
    *W += w[i];
  }
  int64_t* order = malloc(sizeof(int64_t) * (size_t)V);
  for (int64_t i = 0; i < V; ++i) order[i] = i;
  g_sort_logits = logits;
  qsort(order, (size_t)V, sizeof(int64_t), cmp_desc_logit);
  *lambda = -INFINITY;
  *margin_p = INFINITY;
  if (top_k > 0 && top_k < V) *lambda = logits[order[top_k - 1]];
  if (top_p < 1.0) {
    double cum = 0.0, target = top_p * *W;
    for (int64_t n = 0; n < V;) {
      int64_t e = n;
      double group = 0.0;
      while (e < V && logits[order[e]] == logits[order[n]]) group += w[order[e++]];
      double before = cum;
      cum += group;
      if (cum >= target || e == V) {
        double lp = logits[order[n]];
        if (lp > *lambda) *lambda = lp;
        *margin_p = fmin(cum - target, target - before) / *W;
        break;
      }
      n = e;
    }
  }
  free(order);
  return w;
}

int64_t oracle_sample(int64_t V, const float* logits, double temperature, int64_t top_k,
                      double top_p, double u, double* margin) {
  *margin = INFINITY;
  if (!(temperature > 0.0)) {
    int64_t arg = 0;
    for (int64_t i = 1; i < V; ++i)
      if (logits[i] > logits[arg]) arg = i;
    return arg;
  }
  double lambda, W, margin_p;
  double* w = truncate_row(V, logits, temperature, top_k, top_p, &lambda, &W, &margin_p);
  *margin = margin_p;
  double S = 0.0;
  for (int64_t i = 0; i < V; ++i)
    if (logits[i] >= lambda) S += w[i];
  double t = u * S, cum = 0.0;
  int64_t token = -1, last = -1;
  for (int64_t i = 0; i < V; ++i) {
    if (!(logits[i] >= lambda)) continue;
    last = i;
    double before = cum;
    cum += w[i];
    if (w[i] > 0.0) {
      double d = fmin(fabs(cum - t), fabs(before - t)) / S;
      if (d < *margin) *margin = d;
    }
    if (token < 0 && cum > t) token = i;
  }
  if (token < 0) token = last;
  free(w);
  return token;
}

/* For a non-greedy row: whether `token` is kept, and the kept cumulative
 * fractions just before (*lo) and after (*hi) it in vocabulary order (the
 * range of u that selects it). */
int oracle_sample_bracket(int64_t V, const float* logits, double temperature, int64_t top_k,
                          double top_p, int64_t token, double* lo, double* hi) {
  double lambda, W, margin_p;
  double* w = truncate_row(V, logits, temperature, top_k, top_p, &lambda, &W, &margin_p);
  double S = 0.0, before = 0.0;
  for (int64_t i = 0; i < V; ++i)
    if (logits[i] >= lambda) {
      if (i < token) before += w[i];
      S += w[i];
    }
  int kept = token >= 0 && token < V && logits[token] >= lambda;
  *lo = before / S;
  *hi = (before + (kept ? w[token] : 0.0)) / S;
  free(w);
  return kept;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * moe_oracle.c -- plain fp64 CPU oracle for the forward pass of a
 * Mixture-of-Experts FFN layer:
 *
 *     y[t] = g_t * shared(x[t]) + sum_s w[t,s] * SwiGLU-expert_{idx[t,s]}(x[t])
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may build and run it.  It shares no code, header, table or
 * helper with the CUDA path; the two meet only in the seeded input generators.
 *
 * Every quantity is computed in double precision, one token at a time, in the
 * order the definitions state.  Inputs stored as bf16 or fp32 are widened to
 * double exactly before use (a bf16 value is the top 16 bits of an fp32).
 *
 * Passages followed (page title, section):
 *  - "MoE: shared experts, arbitrary V_TOPK expert shapes, and an enforced
 *    stage-marker contract", Group A (packed routing shape word) and Group C
 *    (shared expert summed unweighted; Qwen2-MoE sigmoid gate; fused shared
 *    width = moe_inter x n_shared).
 *  - "MoE: timing-replay harnesses, shared experts, parameterized V_TOPK
 *    routing", Part 2 (topk_softmax generic in (num_experts, top_k); a missing
 *    shape word is an error, never top_k = 0; SwiGLU = silu(g) * u).
 *  - "MoE: shared experts, arbitrary V_TOPK expert shapes, and an enforced
 *    stage-marker contract", Group E (residual_setup: the residual copy, the
 *    input RMSNorm and its norm-weight multiply before the MoE FFN).
 *  - "Fused MoE Kernel Notes", Scatter/gather layout (scatter_index maps each
 *    (token, slot) into the expert-grouped [tokens*topk, hidden] buffer;
 *    gather sums the routed outputs back), Duplicate top-k routes (one expert
 *    group may exceed the token count).
 *
 * Readings where the pages are silent (each is listed with the design notes):
 *  - top-k order: descending logit, equal logits -> lower expert index first;
 *    slot s holds the (s+1)-th largest.
 *  - weights: norm_topk = 1 -> softmax over the k selected logits;
 *    norm_topk = 0 -> full softmax over all E logits, taken at the selected k.
 *  - rows inside an expert group are in row-major (token, slot) order.
 *  - silu(g) = g / (1 + exp(-g)); sigmoid gate = 1 / (1 + exp(-z)).
 *  - input RMSNorm: x / sqrt(mean(x^2) + eps) * w, rounded once to the
 *    activation type; the residual added after the combine is x itself.
 *  - weight shapes follow the [out, in] convention: router [E(+1), H],
 *    gate/up [E, I, H] (expert stride given), down [E, H, I], shared gate/up
 *    [I_sh, H], shared down [H, I_sh]; the shared-gate logit weight is row E
 *    of the router matrix.
 *
 * All functions are pinned by tests that do not reuse this code (worked values
 * printed on the pages, brute force on tiny inputs, closed forms, and library
 * routines in special cases); none is "parity unpinned".
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define OR_F32 0
#define OR_BF16 1

/* Widen element i of a bf16 or fp32 array to double, exactly. */
static double ld(const void *p, int dtype, int64_t i) {
  if (dtype == OR_BF16) {
    uint32_t bits = ((uint32_t)((const uint16_t *)p)[i]) << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
  }
  return (double)((const float *)p)[i];
}

/* ---------------------------------------------------------------------------
 * Packed routing-shape word.  Group A of the PLENA compiler page: the control
 * register holds (num_experts << 8) | top_k; the 8-bit shift keeps every shape
 * up to 16383 experts inside a 22-bit immediate and bounds top_k at 255.
 * Returns 0 (never a valid word) when the shape does not fit.
 * ------------------------------------------------------------------------- */
uint32_t oracle_topk_pack(int32_t num_experts, int32_t top_k) {
  if (num_experts < 1 || num_experts > 16383) return 0;
  if (top_k < 1 || top_k > 255) return 0;
  return ((uint32_t)num_experts << 8) | (uint32_t)top_k;
}

/* Inverse of oracle_topk_pack.  A zero word is the "shape register was never
 * set" case the simulator page traps on: it is an error (-1), not top_k = 0. */
int32_t oracle_topk_unpack(uint32_t word, int32_t *num_experts, int32_t *top_k) {
  if (word == 0 || word > 0x3FFFFFu) return -1;
  int32_t e = (int32_t)(word >> 8), k = (int32_t)(word & 0xFFu);
  if (e < 1 || k < 1) return -1;
  *num_experts = e;
  *top_k = k;
  return 0;
}

/* ---------------------------------------------------------------------------
 * Thread pool helper: run body(lo, hi, ctx) over [0, n) split in nthreads.
 * ------------------------------------------------------------------------- */
typedef void (*range_fn)(int64_t lo, int64_t hi, void *ctx);
typedef struct {
  range_fn fn;
  void *ctx;
  int64_t lo, hi;
} range_job;

static void *range_thread(void *arg) {
  range_job *j = (range_job *)arg;
  j->fn(j->lo, j->hi, j->ctx);
  return NULL;
}

static int resolve_threads(int nthreads) {
  if (nthreads > 0) return nthreads;
  long c = sysconf(_SC_NPROCESSORS_ONLN);
  return c > 0 ? (int)c : 1;
}

static void parallel_range(int64_t n, int nthreads, range_fn fn, void *ctx) {
  nthreads = resolve_threads(nthreads);
  if (nthreads > n) nthreads = (int)(n > 0 ? n : 1);
  if (nthreads <= 1) {
    fn(0, n, ctx);
    return;
  }
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
  range_job *jobs = (range_job *)malloc(sizeof(range_job) * nthreads);
  for (int i = 0; i < nthreads; i++) {
    jobs[i].fn = fn;
    jobs[i].ctx = ctx;
    jobs[i].lo = n * i / nthreads;
    jobs[i].hi = n * (i + 1) / nthreads;
    pthread_create(&th[i], NULL, range_thread, &jobs[i]);
  }
  for (int i = 0; i < nthreads; i++) pthread_join(th[i], NULL);
  free(th);
  free(jobs);
}

/* ---------------------------------------------------------------------------
 * Router GEMM: logits[t, c] = sum_h x[tok(t), h] * w_router[c, h] for every
 * router row c < ncols (ncols = E, or E + 1 when row E is the shared-gate
 * weight).  Router logits are the "router_topk" stage of the PLENA compiler
 * page, Group E.  tokens == NULL means tokens 0..n-1.
 * ------------------------------------------------------------------------- */
typedef struct {
  int64_t H, ncols;
  const void *x;
  int xdt;
  const void *wr;
  int wdt;
  const int64_t *tokens;
  double *logits;
} logits_ctx;

static void logits_body(int64_t lo, int64_t hi, void *p) {
  logits_ctx *c = (logits_ctx *)p;
  for (int64_t i = lo; i < hi; i++) {
    int64_t t = c->tokens ? c->tokens[i] : i;
    for (int64_t col = 0; col < c->ncols; col++) {
      double acc = 0.0;
      for (int64_t h = 0; h < c->H; h++)
        acc += ld(c->x, c->xdt, t * c->H + h) * ld(c->wr, c->wdt, col * c->H + h);
      c->logits[i * c->ncols + col] = acc;
    }
  }
}

void oracle_router_logits(int64_t n, const int64_t *tokens, int64_t H, int64_t ncols,
                          const void *x, int32_t x_dtype, const void *w_router,
                          int32_t w_dtype, double *logits, int32_t nthreads) {
  logits_ctx c = {.H = H, .ncols = ncols, .x = x, .xdt = x_dtype, .wr = w_router,
                  .wdt = w_dtype, .tokens = tokens, .logits = logits};
  parallel_range(n, nthreads, logits_body, &c);
}

/* ---------------------------------------------------------------------------
 * Top-k selection and routing weights for one token.  topk_softmax is generic
 * in (num_experts, top_k) (simulator page, C_SET_TOPK_REG section).
 *   selection: k rounds, each taking the largest logit not yet taken, equal
 *              logits resolved to the lower expert index;
 *   weights:   norm_topk = 1: exp(l_s - m) / sum over the selected k;
 *              norm_topk = 0: exp(l_s - m) / sum over all E  (m = max logit);
 *   gap:       smallest difference between neighbours in the sorted top-(k+1)
 *              list (infinity when k == E): a gap near zero marks a near-tie
 *              that may legitimately reorder slots or swap set membership.
 * Returns -1 on a bad shape word.
 * ------------------------------------------------------------------------- */
int32_t oracle_topk_softmax(int64_t n, uint32_t shape_word, int32_t norm_topk,
                            const double *logits, int64_t ld_logits, int32_t *idx,
                            double *weights, double *gap) {
  int32_t E, k;
  if (oracle_topk_unpack(shape_word, &E, &k) != 0) return -1;
  if (k > E) return -1;
  char *taken = (char *)malloc((size_t)E);
  int32_t *order = (int32_t *)malloc(sizeof(int32_t) * (size_t)(k + 1));
  for (int64_t t = 0; t < n; t++) {
    const double *l = logits + t * ld_logits;
    memset(taken, 0, (size_t)E);
    int32_t rounds = (k < E) ? k + 1 : k; /* one extra round for the gap */
    for (int32_t r = 0; r < rounds; r++) {
      int32_t best = -1;
      for (int32_t e = 0; e < E; e++) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e; /* strict '>' keeps lower index */
      }
      taken[best] = 1;
      order[r] = best;
    }
    double m = l[order[0]];
    double denom = 0.0;
    if (norm_topk) {
      for (int32_t s = 0; s < k; s++) denom += exp(l[order[s]] - m);
    } else {
      for (int32_t e = 0; e < E; e++) denom += exp(l[e] - m);
    }
    double g = INFINITY;
    for (int32_t r = 0; r + 1 < rounds; r++) {
      double d = l[order[r]] - l[order[r + 1]];
      if (d < g) g = d;
    }
    for (int32_t s = 0; s < k; s++) {
      idx[t * k + s] = order[s];
      weights[t * k + s] = exp(l[order[s]] - m) / denom;
    }
    if (gap) gap[t] = g;
  }
  free(taken);
  free(order);
  return 0;
}

/* Qwen2-MoE shared-expert gate: sigmoid(z) = 1 / (1 + exp(-z)), one scalar per
 * token (PLENA compiler page, Group C: the S_SUB/S_EXP/S_ADD/S_RECI sequence
 * computes exactly this). */
void oracle_sigmoid(int64_t n, const double *z, int64_t ld_z, double *gate) {
  for (int64_t t = 0; t < n; t++) gate[t] = 1.0 / (1.0 + exp(-z[t * ld_z]));
}

/* ---------------------------------------------------------------------------
 * Rounding of a double to the activation type, round to nearest, ties to
 * even: what the layer stores its activations in.  bf16 keeps 8 significant
 * bits with fp32's exponent range; a value is written as its bf16 bit pattern
 * (the top 16 bits of the fp32 with that value).  fp32 values are written as
 * fp32 (C's double -> float conversion rounds to nearest even).
 * ------------------------------------------------------------------------- */
static void st_act(void *p, int dtype, int64_t i, double v) {
  if (dtype != OR_BF16) {
    ((float *)p)[i] = (float)v;
    return;
  }
  double r;
  if (isnan(v)) {
    ((uint16_t *)p)[i] = 0x7FC0;   /* the canonical quiet NaN */
    return;
  } else if (v == 0.0 || isinf(v)) {
    r = v;
  } else {
    const double a = fabs(v);
    double q;   /* the spacing of bf16 values around a */
    if (a < ldexp(1.0, -126)) {
      q = ldexp(1.0, -133);   /* subnormal range: fixed spacing */
    } else {
      int e;
      frexp(a, &e);           /* a = m 2^e, 0.5 <= m < 1 */
      q = ldexp(1.0, e - 8);  /* 8 significant bits */
    }
    r = rint(a / q) * q;      /* rint: nearest, ties to even */
    if (r > ldexp(255.0, 120)) r = INFINITY;   /* beyond the largest finite bf16 */
    r = copysign(r, v);
  }
  const float f = (float)r;   /* exact: r has at most 8 significant bits */
  uint32_t bits;
  memcpy(&bits, &f, 4);
  ((uint16_t *)p)[i] = (uint16_t)(bits >> 16);
}

/* One value, for tests of the rounding rule: the activation-type value
 * nearest to v (ties to even), returned as a double. */
double oracle_round_act(double v, int32_t dtype) {
  if (dtype == OR_BF16) {
    uint16_t b;
    st_act(&b, OR_BF16, 0, v);
    return ld(&b, OR_BF16, 0);
  }
  float f;
  st_act(&f, OR_F32, 0, v);
  return (double)f;
}

/* ---------------------------------------------------------------------------
 * Input preparation of the MoE sublayer (Group E of the PLENA compiler page:
 * the "residual_setup" stage -- residual copy, input RMSNorm and its
 * norm-weight multiply; the residual itself is x):
 *   x_norm[t, h] = x[t, h] / sqrt((1/H) sum_h' x[t, h']^2 + eps) * w[h]
 * in double, then rounded once to the activation type (`out`, [T, H], same
 * type as x).  The router and the experts then see exactly these values, as
 * on the GPU, so both sides decide the routing on the same inputs.
 * ------------------------------------------------------------------------- */
void oracle_rmsnorm(int64_t T, int64_t H, const void *x, int32_t dtype, const void *w,
                    double eps, void *out) {
  for (int64_t t = 0; t < T; t++) {
    double ss = 0.0;
    for (int64_t h = 0; h < H; h++) {
      const double v = ld(x, dtype, t * H + h);
      ss += v * v;
    }
    const double inv = 1.0 / sqrt(ss / (double)H + eps);
    for (int64_t h = 0; h < H; h++)
      st_act(out, dtype, t * H + h, ld(x, dtype, t * H + h) * inv * ld(w, dtype, h));
  }
}

/* ---------------------------------------------------------------------------
 * Expert histogram and scatter_index ("Fused MoE Kernel Notes", Scatter/gather
 * layout and Duplicate top-k routes).
 *   counts[e]            number of (token, slot) pairs routed to expert e
 *                        (a duplicate slot counts again);
 *   offsets[e]           sum of counts[e'] for e' < e; offsets[E] = T*k;
 *   scatter_index[t,s]   offsets[e] + number of pairs (t', s') routed to e
 *                        that come before (t, s) in row-major order;
 *   row_token[r]         the token whose row lands at grouped row r.
 * Returns -1 when a route is outside [0, E).
 * ------------------------------------------------------------------------- */
int32_t oracle_permute(int64_t T, int32_t k, int32_t E, const int32_t *idx,
                       int32_t *counts, int32_t *offsets, int32_t *scatter_index,
                       int32_t *row_token) {
  for (int64_t p = 0; p < T * k; p++)
    if (idx[p] < 0 || idx[p] >= E) return -1;
  for (int32_t e = 0; e < E; e++) counts[e] = 0;
  for (int64_t p = 0; p < T * k; p++) counts[idx[p]]++;
  offsets[0] = 0;
  for (int32_t e = 0; e < E; e++) offsets[e + 1] = offsets[e] + counts[e];
  int32_t *next = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
  for (int32_t e = 0; e < E; e++) next[e] = offsets[e];
  for (int64_t t = 0; t < T; t++) {
    for (int32_t s = 0; s < k; s++) {
      int32_t e = idx[t * k + s];
      int32_t r = next[e]++;
      scatter_index[t * k + s] = r;
      row_token[r] = (int32_t)t;
    }
  }
  free(next);
  return 0;
}

/* ---------------------------------------------------------------------------
 * One SwiGLU FFN applied to one token row (routed expert or shared MLP):
 *   g_j = sum_h x_h * Wg[j, h],  u_j = sum_h x_h * Wu[j, h]   (j < I)
 *   a_j = silu(g_j) * u_j
 *   o_h = sum_j a_j * Wd[h, j]                               (h < H)
 * silu(g) * u is the activation of the PLENA simulator page's shared-expert
 * tests; the shared branch is a dense FFN over every row (compiler page,
 * Group C).  o is accumulated into out with factor scale.
 * ------------------------------------------------------------------------- */
static void swiglu_ffn(int64_t H, int64_t I, const double *x, const void *wg,
                       const void *wu, const void *wd, int wdt, double scale,
                       double *a_scratch, double *out) {
  for (int64_t j = 0; j < I; j++) {
    double g = 0.0, u = 0.0;
    for (int64_t h = 0; h < H; h++) {
      g += x[h] * ld(wg, wdt, j * H + h);
      u += x[h] * ld(wu, wdt, j * H + h);
    }
    a_scratch[j] = g / (1.0 + exp(-g)) * u;
  }
  for (int64_t h = 0; h < H; h++) {
    double o = 0.0;
    for (int64_t j = 0; j < I; j++) o += a_scratch[j] * ld(wd, wdt, h * I + j);
    out[h] += scale * o;
  }
}

/* ---------------------------------------------------------------------------
 * Expert FFNs and combine for a list of tokens, routes given:
 *   y[i] = gate[i] * shared(x[tok_i]) + sum_s w[i,s] * expert_{idx[i,s]}(x[tok_i])
 * (y = shared(x) + sum_k route_weight_k * routed_expert_k(x): both PLENA
 * pages, shared-expert sections; gate = 1 when the shared expert is ungated).
 *
 * Routed weights: expert e's gate/up matrices start at e * gate_stride /
 * e * up_stride elements (split or merged fc1 layouts) and its down matrix at
 * e * down_stride.  I_sh = 0 means no shared expert.  gate == NULL means 1.
 * idx/w are [n, k] for the listed tokens.  y is [n, H], overwritten.
 * ------------------------------------------------------------------------- */
typedef struct {
  int64_t H, I, I_sh;
  int32_t k;
  const void *x;
  int xdt;
  int wdt;
  const int64_t *tokens;
  const int32_t *idx;
  const double *w;
  const double *gate;
  const void *wg, *wu, *wd;
  int64_t sg, su, sd;
  const void *shg, *shu, *shd;
  double *y;
} ffn_ctx;

static void ffn_body(int64_t lo, int64_t hi, void *p) {
  ffn_ctx *c = (ffn_ctx *)p;
  int64_t amax = c->I > c->I_sh ? c->I : c->I_sh;
  double *xr = (double *)malloc(sizeof(double) * (size_t)c->H);
  double *a = (double *)malloc(sizeof(double) * (size_t)(amax > 0 ? amax : 1));
  for (int64_t i = lo; i < hi; i++) {
    int64_t t = c->tokens ? c->tokens[i] : i;
    for (int64_t h = 0; h < c->H; h++) xr[h] = ld(c->x, c->xdt, t * c->H + h);
    double *yr = c->y + i * c->H;
    for (int64_t h = 0; h < c->H; h++) yr[h] = 0.0;
    if (c->I_sh > 0) {
      double g = c->gate ? c->gate[i] : 1.0;
      swiglu_ffn(c->H, c->I_sh, xr, c->shg, c->shu, c->shd, c->wdt, g, a, yr);
    }
    for (int32_t s = 0; s < c->k; s++) {
      int64_t e = c->idx[i * c->k + s];
      const char *base_g = (const char *)c->wg;
      const char *base_u = (const char *)c->wu;
      const char *base_d = (const char *)c->wd;
      int64_t esz = (c->wdt == OR_BF16) ? 2 : 4;
      swiglu_ffn(c->H, c->I, xr, base_g + e * c->sg * esz, base_u + e * c->su * esz,
                 base_d + e * c->sd * esz, c->wdt, c->w[i * c->k + s], a, yr);
    }
  }
  free(xr);
  free(a);
}

void oracle_moe_ffn(int64_t n, const int64_t *tokens, int64_t H, int64_t I,
                    int64_t I_sh, int32_t k, const void *x, int32_t x_dtype,
                    int32_t w_dtype, const int32_t *idx, const double *w,
                    const double *gate, const void *w_gate, int64_t gate_stride,
                    const void *w_up, int64_t up_stride, const void *w_down,
                    int64_t down_stride, const void *sh_gate, const void *sh_up,
                    const void *sh_down, double *y, int32_t nthreads) {
  ffn_ctx c = {.H = H, .I = I, .I_sh = I_sh, .k = k, .x = x, .xdt = x_dtype,
               .wdt = w_dtype, .tokens = tokens, .idx = idx, .w = w, .gate = gate,
               .wg = w_gate, .wu = w_up, .wd = w_down, .sg = gate_stride,
               .su = up_stride, .sd = down_stride, .shg = sh_gate, .shu = sh_up,
               .shd = sh_down, .y = y};
  parallel_range(n, nthreads, ffn_body, &c);
}

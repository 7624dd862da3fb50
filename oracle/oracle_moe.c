/*
 * oracle_moe.c -- plain, slow, fp64 reference of the quantized sparse MoE layer
 * forward.  TEST INFRASTRUCTURE ONLY: only the tests, the package smoke check
 * and the benchmark's CPU-baseline leg may load it.  It shares no code, header
 * or table with the CUDA library; it reads the same packed bytes with its own
 * unpacking code.
 *
 * What it computes, step by step, and where the pages state it:
 *
 *  1. Router logits z[t][e] = sum_i x[t][i] * Wr[e][i], then s = sigmoid(z).
 *     "25GB RAM runs 744B GLM-5.2" page (pwwt.cn), section 3.1: a DeepSeek-V3
 *     style sigmoid router picks 8 of 256 experts per token.
 *  2. Selection score u = s + b[e]; the bias only steers which experts are
 *     chosen (same page, section 4.3: auxiliary-loss-free balancing adjusts an
 *     expert bias; the engine must reproduce sigmoid routing, expert selection
 *     and the scaling semantics exactly).  The k largest u are chosen, a tie
 *     going to the lower expert id.
 *  3. Gate weights g_j = rho * s_j / sum_{selected} s  (renormalised over the
 *     unbiased sigmoid scores, times the routed scaling factor rho).
 *  4. Batch-union grouping (same page, section 3.4): (token, slot) pairs are
 *     grouped by expert so each selected expert is visited once for all of its
 *     tokens.  Here: a counting sort by expert id, stable in t*k + j.
 *  5. Per pair, the expert's SwiGLU FFN on dequantised weights
 *     w = (q - zero_point) * scale ("Colibri walkthrough" page (discosf.com),
 *     section 3.4: per-output-channel scale and zero_point, int8 or int4):
 *        a = Wg x, c = Wu x, h = silu(a) * c, y = Wd h.
 *  6. Optional always-on shared expert ("25GB RAM" page, section 2: shared
 *     experts stay resident), weight 1.
 *  7. out[t] = sum_j g_j * y_j (j ascending) + y_shared.
 *
 * Readings where the pages are silent: the selected set is reported in
 * ascending expert id order; renormalisation uses the unbiased s; the shared
 * expert has weight 1; RMSNorm (stacked layers) is h / sqrt(mean(h^2) + eps)
 * with unit gain and its result is rounded to bf16, the layer's input type.
 *
 * Everything accumulates in double, in the index order written here.  x, the
 * router weights and the scales are read exactly (bf16/fp16/fp32 -> double).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_Q_INT4_G128 0
#define ORC_Q_INT8_PC 1
#define ORC_X_BF16 0
#define ORC_X_F32 1

typedef struct {
  const uint8_t* q;   /* int4: [N][K/2], low nibble = even k ; int8: [N][K] */
  const void* s;      /* int4: fp16 bits [N][K/128]          ; int8: float [N] */
  const uint8_t* z;   /* int4: [N][ceil(K/256)], low nibble = even group ; int8: [N] */
} orc_qmat;

typedef struct {
  orc_qmat gate, up, down;
} orc_expert;

typedef struct {
  int d, F, E, k;
  double rho;
  int qtype;
  int xtype;
  int has_shared;
  int F_shared;
  int qtype_shared;
} orc_desc;

/* ---------------------------------------------------------------- number formats */

/* bfloat16: the top 16 bits of an IEEE binary32 */
double orc_bf16_to_double(uint16_t h) {
  uint32_t x = (uint32_t)h << 16;
  float f;
  memcpy(&f, &x, 4);
  return (double)f;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits */
double orc_f16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp(1024.0 + (double)m, e - 25);
  return sign ? -v : v;
}

/* double -> nearest bfloat16 (ties to even), returned as a double */
double orc_round_to_bf16(double v) {
  if (v == 0.0 || !isfinite(v)) return v;
  int e;
  frexp(v, &e);                       /* |v| in [2^(e-1), 2^e) */
  if (e - 1 < -126) e = -125;         /* bf16 subnormal range keeps a fixed quantum */
  double quantum = ldexp(1.0, e - 1 - 7);
  return nearbyint(v / quantum) * quantum;  /* default rounding mode: ties to even */
}

static double x_at(int xtype, const void* x, size_t i) {
  if (xtype == ORC_X_BF16) return orc_bf16_to_double(((const uint16_t*)x)[i]);
  return (double)((const float*)x)[i];
}

/* ---------------------------------------------------------------- dequantisation */

/* row n of a quantised [N][K] matrix as doubles: w = (q - zero_point) * scale */
void orc_dequant_row(const orc_qmat* m, int qtype, int K, int n, double* w) {
  if (qtype == ORC_Q_INT4_G128) {
    int G = K / 128, ZB = (G + 1) / 2;
    const uint8_t* qr = m->q + (size_t)n * (size_t)(K / 2);
    const uint16_t* sr = (const uint16_t*)m->s + (size_t)n * (size_t)G;
    const uint8_t* zr = m->z + (size_t)n * (size_t)ZB;
    for (int k = 0; k < K; ++k) {
      uint8_t byte = qr[k / 2];
      int code = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
      int g = k / 128;
      uint8_t zb = zr[g / 2];
      int zero = (g % 2 == 0) ? (zb & 15) : (zb >> 4);
      w[k] = (double)(code - zero) * orc_f16_to_double(sr[g]);
    }
  } else {
    const uint8_t* qr = m->q + (size_t)n * (size_t)K;
    double scale = (double)((const float*)m->s)[n];
    int zero = m->z[n];
    for (int k = 0; k < K; ++k) w[k] = (double)((int)qr[k] - zero) * scale;
  }
}

static double silu(double a) { return a / (1.0 + exp(-a)); }

/*
 * One token through one SwiGLU expert: y[d] = Wd (silu(Wg x) * (Wu x)).
 * scratch: at least max(d, F) + F doubles.
 */
void orc_expert_ffn(int qtype, int d, int F, const orc_expert* ex, const double* x, double* y, double* scratch) {
  double* w = scratch;          /* one dequantised row */
  double* h = scratch + (d > F ? d : F);
  for (int n = 0; n < F; ++n) {
    double a = 0.0, c = 0.0;
    orc_dequant_row(&ex->gate, qtype, d, n, w);
    for (int i = 0; i < d; ++i) a += w[i] * x[i];
    orc_dequant_row(&ex->up, qtype, d, n, w);
    for (int i = 0; i < d; ++i) c += w[i] * x[i];
    h[n] = silu(a) * c;
  }
  for (int m = 0; m < d; ++m) {
    double acc = 0.0;
    orc_dequant_row(&ex->down, qtype, F, m, w);
    for (int n = 0; n < F; ++n) acc += w[n] * h[n];
    y[m] = acc;
  }
}

/* ---------------------------------------------------------------- routing */

/*
 * Route one token.  xt: the token's activations as doubles.
 * Outputs: sel[k] (ascending expert id), g[k], gap = u_(k) - u_(k+1) (u sorted
 * descending; +inf when k == E), s_all[E] (sigmoid scores, nullable).
 */
static void route_token(int d, int E, int k, double rho, const double* xt, const float* Wr, const float* b,
                        int32_t* sel, double* g, double* gap, double* s_all, double* u, unsigned char* taken) {
  double* s = s_all;
  for (int e = 0; e < E; ++e) {
    double z = 0.0;
    const float* we = Wr + (size_t)e * (size_t)d;
    for (int i = 0; i < d; ++i) z += xt[i] * (double)we[i];
    s[e] = 1.0 / (1.0 + exp(-z));
    u[e] = s[e] + (double)b[e];
    taken[e] = 0;
  }
  double kth = 0.0;
  for (int j = 0; j < k; ++j) {     /* pick the largest remaining u; ties -> lower e */
    int best = -1;
    for (int e = 0; e < E; ++e)
      if (!taken[e] && (best < 0 || u[e] > u[best])) best = e;
    taken[best] = 1;
    kth = u[best];
  }
  if (k < E) {
    int nxt = -1;
    for (int e = 0; e < E; ++e)
      if (!taken[e] && (nxt < 0 || u[e] > u[nxt])) nxt = e;
    *gap = kth - u[nxt];
  } else {
    *gap = INFINITY;
  }
  int j = 0;
  double ssum = 0.0;
  for (int e = 0; e < E; ++e)
    if (taken[e]) { sel[j++] = e; ssum += s[e]; }
  for (j = 0; j < k; ++j) g[j] = rho * s[sel[j]] / ssum;
}

/*
 * Route T tokens.  topk_idx[T][k] ascending expert ids, topk_w[T][k], gap[T],
 * scores[T][E] (sigmoid s, nullable).  Returns 0, or -1 on bad arguments.
 */
int orc_route(const orc_desc* D, int T, const void* x, const float* Wr, const float* b, int32_t* topk_idx,
              double* topk_w, double* gap, double* scores, int nthreads) {
  if (D->k < 1 || D->k > D->E || T < 0) return -1;
  int d = D->d, E = D->E, k = D->k;
  int bad = 0;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : 1)
  {
    double* xt = (double*)malloc(sizeof(double) * (size_t)d);
    double* s = (double*)malloc(sizeof(double) * (size_t)E);
    double* u = (double*)malloc(sizeof(double) * (size_t)E);
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    if (!xt || !s || !u || !taken) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int t = 0; t < T; ++t) {
        for (int i = 0; i < d; ++i) xt[i] = x_at(D->xtype, x, (size_t)t * (size_t)d + (size_t)i);
        route_token(d, E, k, D->rho, xt, Wr, b, topk_idx + (size_t)t * k, topk_w + (size_t)t * k, gap + t, s, u,
                    taken);
        if (scores) memcpy(scores + (size_t)t * (size_t)E, s, sizeof(double) * (size_t)E);
      }
    }
    free(xt); free(s); free(u); free(taken);
  }
  return bad ? -1 : 0;
}

/*
 * Batch-union grouping: counting sort of the T*k (token, slot) pairs by expert
 * id, stable in the flat index t*k + j.  offsets[E+1] is the exclusive prefix
 * sum of the per-expert counts; pair_token/pair_slot[T*k] list the pairs in
 * grouped order; pair_of[T*k] gives each (t, j)'s position in that order.
 */
int orc_permute(int T, int k, int E, const int32_t* topk_idx, int32_t* offsets, int32_t* pair_token,
                int32_t* pair_slot, int32_t* pair_of) {
  int32_t* fill = (int32_t*)calloc((size_t)E + 1, sizeof(int32_t));
  if (!fill) return -1;
  for (int e = 0; e <= E; ++e) offsets[e] = 0;
  for (long f = 0; f < (long)T * k; ++f) {
    int e = topk_idx[f];
    if (e < 0 || e >= E) { free(fill); return -1; }
    offsets[e + 1] += 1;
  }
  for (int e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
  for (long f = 0; f < (long)T * k; ++f) {
    int e = topk_idx[f];
    int pos = offsets[e] + fill[e]++;
    pair_token[pos] = (int32_t)(f / k);
    pair_slot[pos] = (int32_t)(f % k);
    pair_of[f] = pos;
  }
  free(fill);
  return 0;
}

/* ---------------------------------------------------------------- the layer */

/*
 * MoE layer output for a subset of tokens (tokens are independent, so any
 * subset is exact).  tokens[n_tok] index rows of x; out[n_tok][d].
 * sel_override[n_tok][k] (nullable, ascending ids, -1 in [0] = no override)
 * replaces the selected set of a token; its gate weights are then rho*s/sum(s)
 * over the given set with the oracle's own s.  Shared expert: `shared`
 * (nullable) with F = D->F_shared.  Returns 0, or -1 on allocation failure.
 */
int orc_moe_forward(const orc_desc* D, const void* x, const float* Wr, const float* b, const orc_expert* experts,
                    const orc_expert* shared, const int32_t* tokens, int n_tok, const int32_t* sel_override,
                    double* out, int nthreads) {
  int d = D->d, E = D->E, k = D->k, F = D->F;
  int Fmax = F > D->F_shared ? F : D->F_shared;
  int bad = 0;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : 1)
  {
    double* xt = (double*)malloc(sizeof(double) * (size_t)d);
    double* y = (double*)malloc(sizeof(double) * (size_t)d);
    double* scratch = (double*)malloc(sizeof(double) * ((size_t)(d > Fmax ? d : Fmax) + (size_t)Fmax));
    double* s = (double*)malloc(sizeof(double) * (size_t)E);
    double* u = (double*)malloc(sizeof(double) * (size_t)E);
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    int32_t* sel = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
    double* g = (double*)malloc(sizeof(double) * (size_t)k);
    if (!xt || !y || !scratch || !s || !u || !taken || !sel || !g) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int n = 0; n < n_tok; ++n) {
        int t = tokens[n];
        double gap;
        for (int i = 0; i < d; ++i) xt[i] = x_at(D->xtype, x, (size_t)t * (size_t)d + (size_t)i);
        route_token(d, E, k, D->rho, xt, Wr, b, sel, g, &gap, s, u, taken);
        if (sel_override && sel_override[(size_t)n * k] >= 0) {
          double ssum = 0.0;
          for (int j = 0; j < k; ++j) { sel[j] = sel_override[(size_t)n * k + j]; ssum += s[sel[j]]; }
          for (int j = 0; j < k; ++j) g[j] = D->rho * s[sel[j]] / ssum;
        }
        double* o = out + (size_t)n * (size_t)d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        for (int j = 0; j < k; ++j) {
          orc_expert_ffn(D->qtype, d, F, &experts[sel[j]], xt, y, scratch);
          for (int i = 0; i < d; ++i) o[i] += g[j] * y[i];
        }
        if (D->has_shared && shared) {
          orc_expert_ffn(D->qtype_shared, d, D->F_shared, shared, xt, y, scratch);
          for (int i = 0; i < d; ++i) o[i] += y[i];
        }
      }
    }
    free(xt); free(y); free(scratch); free(s); free(u); free(taken); free(sel); free(g);
  }
  return bad ? -1 : 0;
}

/*
 * RMSNorm with unit gain, rounded to bf16 (returned as doubles):
 * n = bf16(h / sqrt(mean(h^2) + eps)).
 */
void orc_rmsnorm_bf16(int d, const double* h, double eps, double* n) {
  double ss = 0.0;
  for (int i = 0; i < d; ++i) ss += h[i] * h[i];
  double r = sqrt(ss / (double)d + eps);
  for (int i = 0; i < d; ++i) n[i] = orc_round_to_bf16(h[i] / r);
}

/* ---------------------------------------------------------------- integer-dot variant (IDOT) */

/*
 * "25GB RAM runs 744B GLM-5.2" page (pwwt.cn), section 6 (reproducibility): the
 * engine has integer-dot kernels (switch IDOT) whose rounding depends on the
 * batch shape, so their output may differ slightly from the single-token path.
 * The pages do not give the activation format.  Reading: the inputs of every
 * quantised matrix-vector product (x for gate and up, h for down) are cut into
 * blocks of 32 consecutive values; a block shares the scale 2^(e-6) with
 * e = floor(log2(max |v|)) over the block (e at least -100, so that the scale
 * stays a normal single-precision number; an all-zero block has e = -100), and
 * each value becomes the integer
 * q = round-half-even(v / 2^(e-6)) clamped to [-127, 127] (an 8-bit integer
 * with a shared power-of-two exponent, as in the OCP microscaling MXINT8
 * format).  The weights are unchanged, so every product (c - z) * q is an
 * integer.  Routing reads x itself.
 *
 * orc_mx8_block: n values -> vq = q * 2^(e-6).  With tau > 0, amb[i] bounds
 * |vq' - vq[i]| for a quantisation of a value within the kernel's rounding
 * error of v[i] (a near tie): one step 2^(e-6) where |v| / 2^(e-6) lies within
 * tau of a half-integer, and 1.5 steps for the whole block where max |v| lies
 * within a relative tau/64 of a power of two (the exponent may differ by one);
 * zero elsewhere.  Returns e.
 */
int orc_mx8_block(int n, const double* v, double tau, double* vq, double* amb) {
  double m = 0.0;
  for (int i = 0; i < n; ++i) m = fabs(v[i]) > m ? fabs(v[i]) : m;
  int e = -100;
  if (m > 0.0) {
    int ex;
    frexp(m, &ex);                  /* m = f * 2^ex, f in [0.5, 1) */
    e = ex - 1 > -100 ? ex - 1 : -100;
  }
  double step = ldexp(1.0, e - 6);
  int block_amb = 0;
  if (tau > 0.0 && m > 0.0) {
    double r = m / ldexp(1.0, e);   /* in [1, 2) unless e was clamped */
    block_amb = (r - 1.0 < tau / 64.0) || (2.0 - r < tau / 64.0);
  }
  for (int i = 0; i < n; ++i) {
    double s = v[i] / step;         /* exact: a power-of-two scale */
    double q = nearbyint(s);        /* the default rounding mode: half to even */
    if (q > 127.0) q = 127.0;
    if (q < -127.0) q = -127.0;
    vq[i] = q * step;
    if (amb) {
      double a = 0.0;
      double fr = fabs(s) - floor(fabs(s));
      if (tau > 0.0 && fabs(fr - 0.5) < tau && fabs(s) < 127.5) a = step;
      if (block_amb) a = 1.5 * step;
      amb[i] = a;
    }
  }
  return e;
}

/*
 * The down projection's input of one token in one expert with IDOT inputs:
 * x -> blocks of 32 (exact decisions: x is read exactly and the scale is a
 * power of two), the gate/up products and h[F] in double, then h -> blocks of
 * 32: hq[F] (the values q * 2^(e-6)) and amb[F] (near-tie bounds, tau as in
 * orc_mx8_block).  scratch: at least 2 * max(d, F) doubles.
 */
void orc_idot_hidden(int qtype, int d, int F, const orc_expert* ex, const double* x, double tau, double* h,
                     double* hq, double* amb, double* scratch) {
  int mx = d > F ? d : F;
  double* w = scratch;
  double* xq = scratch + mx;
  for (int b = 0; b < d; b += 32) orc_mx8_block(32, x + b, 0.0, xq + b, NULL);
  for (int n = 0; n < F; ++n) {
    double a = 0.0, c = 0.0;
    orc_dequant_row(&ex->gate, qtype, d, n, w);
    for (int i = 0; i < d; ++i) a += w[i] * xq[i];
    orc_dequant_row(&ex->up, qtype, d, n, w);
    for (int i = 0; i < d; ++i) c += w[i] * xq[i];
    h[n] = c * silu(a);
  }
  for (int b = 0; b < F; b += 32) orc_mx8_block(32, h + b, tau, hq + b, amb + b);
}

/*
 * One token through one SwiGLU expert with IDOT inputs: orc_idot_hidden, then
 * y = Wd hq and ybound[m] = sum_n |Wd[m][n]| * amb[n].  scratch: at least
 * 2 * max(d, F) + 3 * F doubles.
 */
void orc_expert_ffn_idot(int qtype, int d, int F, const orc_expert* ex, const double* x, double tau, double* y,
                         double* ybound, double* scratch) {
  int mx = d > F ? d : F;
  double* w = scratch;
  double* h = scratch + 2 * (size_t)mx;
  double* hq = h + F;
  double* amb = hq + F;
  orc_idot_hidden(qtype, d, F, ex, x, tau, h, hq, amb, scratch);
  for (int m = 0; m < d; ++m) {
    double acc = 0.0, bnd = 0.0;
    orc_dequant_row(&ex->down, qtype, F, m, w);
    for (int n = 0; n < F; ++n) {
      acc += w[n] * hq[n];
      bnd += fabs(w[n]) * amb[n];
    }
    y[m] = acc;
    ybound[m] = bnd;
  }
}

/*
 * The layer with IDOT expert products, for a subset of tokens (as
 * orc_moe_forward): routing on x itself, out[n][d] = sum_j g_j y_j + y_shared
 * with the IDOT expert outputs, bound[n][d] = sum_j g_j ybound_j + ybound_shared
 * (the near-tie allowance of each output).  Returns 0, or -1 on allocation
 * failure.
 */
int orc_moe_forward_idot(const orc_desc* D, const void* x, const float* Wr, const float* b, const orc_expert* experts,
                         const orc_expert* shared, const int32_t* tokens, int n_tok, double tau, double* out,
                         double* bound, int nthreads) {
  int d = D->d, E = D->E, k = D->k, F = D->F;
  int Fmax = F > D->F_shared ? F : D->F_shared;
  int mx = d > Fmax ? d : Fmax;
  int bad = 0;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : 1)
  {
    double* xt = (double*)malloc(sizeof(double) * (size_t)d);
    double* y = (double*)malloc(sizeof(double) * (size_t)d);
    double* yb = (double*)malloc(sizeof(double) * (size_t)d);
    double* scratch = (double*)malloc(sizeof(double) * (2 * (size_t)mx + 3 * (size_t)Fmax));
    double* s = (double*)malloc(sizeof(double) * (size_t)E);
    double* u = (double*)malloc(sizeof(double) * (size_t)E);
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    int32_t* sel = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
    double* g = (double*)malloc(sizeof(double) * (size_t)k);
    if (!xt || !y || !yb || !scratch || !s || !u || !taken || !sel || !g) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int n = 0; n < n_tok; ++n) {
        int t = tokens[n];
        double gap;
        for (int i = 0; i < d; ++i) xt[i] = x_at(D->xtype, x, (size_t)t * (size_t)d + (size_t)i);
        route_token(d, E, k, D->rho, xt, Wr, b, sel, g, &gap, s, u, taken);
        double* o = out + (size_t)n * (size_t)d;
        double* ob = bound + (size_t)n * (size_t)d;
        for (int i = 0; i < d; ++i) { o[i] = 0.0; ob[i] = 0.0; }
        for (int j = 0; j < k; ++j) {
          orc_expert_ffn_idot(D->qtype, d, F, &experts[sel[j]], xt, tau, y, yb, scratch);
          for (int i = 0; i < d; ++i) { o[i] += g[j] * y[i]; ob[i] += g[j] * yb[i]; }
        }
        if (D->has_shared && shared) {
          orc_expert_ffn_idot(D->qtype_shared, d, D->F_shared, shared, xt, tau, y, yb, scratch);
          for (int i = 0; i < d; ++i) { o[i] += y[i]; ob[i] += yb[i]; }
        }
      }
    }
    free(xt); free(y); free(yb); free(scratch); free(s); free(u); free(taken); free(sel); free(g);
  }
  return bad ? -1 : 0;
}

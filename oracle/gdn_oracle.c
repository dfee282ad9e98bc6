/*
 * gdn_oracle.c -- plain fp64 CPU oracle for the Gated DeltaNet token mixer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the yardstick the CUDA path is
 * checked against.  Only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark may load it; the product library never links or calls it,
 * and it shares no code, header or table with the CUDA sources.
 *
 * What it computes, per (sequence b, value head h), token by token, in fp64:
 *
 *   1. causal depthwise conv (width 4) + SiLU on every q|k|v channel
 *        page "Qwen3.8-27B" (docs.theformalera.com), node gdn.conv:
 *        y[t,c] = silu( sum_{j<4} w[c,j] * x[t+j-3, c] ),  w[c,3] is the
 *        current token; missing left context comes from the carried conv
 *        window (zeros when there is none).
 *   2. L2 normalisation of q and k with eps inside the root, q then scaled
 *        page "How Qwen3.5 works" (azmle112.github.io), section 9.4;
 *        the 27B node gdn.core fixes qk_l2norm_eps = 1e-6, scale 1/sqrt(128).
 *   3. the gated delta rule, decay -> predict -> correct -> read
 *        "How Qwen3.5 works" section 9.6 (written there for the k x v
 *        orientation); node gdn.core writes the same update for the
 *        v x k orientation used here:
 *          S_t = e^{g_t} S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *          o_t = S_t q_t,    value head h reads key head floor(h / (Hv/Hk)).
 *   4. the per-head gated RMSNorm
 *        node gdn.norm: y = w * x / sqrt(mean(x^2) + eps) * silu(z);
 *        section 9.9 of "How Qwen3.5 works" (scale applied directly, SiLU
 *        gate after normalising).
 *   0. optionally, the gates from their raw projections
 *        "How Qwen3.5 works" section 9.5: beta = sigmoid(b),
 *        g = -exp(A_log) * softplus(a + dt_bias), per value head.
 *
 * State layout: S[b][h][i][j], i = value index (row), j = key index
 * (contiguous), i.e. the node gdn.core orientation.  Dimensions are generic
 * (the worked 2x2 example of section 9.8 runs with Dk = Dv = 2).
 *
 * Every input arrives as float (bf16 values are exact in float); every
 * intermediate and every output is double.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int B, T, Hk, Hv, Dk, Dv;
  double eps_l2;   /* epsilon inside the L2-norm root */
  double eps_norm; /* epsilon of the gated RMSNorm */
  double q_scale;  /* applied to the normalised query */
} oracle_shape;

int oracle_abi_version(void) { return 1; }

/* silu(x) = x * sigmoid(x) = x / (1 + e^{-x}). */
double oracle_silu(double x) { return x / (1.0 + exp(-x)); }

/* Step 1 for one channel at one token.  window[0..3] are the raw inputs of
 * tokens t-3, t-2, t-1, t (oldest first); taps[3] multiplies token t. */
double oracle_conv_silu_one(const double *window, const double *taps) {
  double acc = 0.0;
  for (int j = 0; j < 4; ++j) acc += taps[j] * window[j];
  return oracle_silu(acc);
}

/* Step 2: y = scale * x / sqrt(sum x^2 + eps). */
void oracle_l2norm(int n, const double *x, double eps, double scale, double *y) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss + eps);
  for (int i = 0; i < n; ++i) y[i] = x[i] * inv * scale;
}

/* Step 3, one token on one head.  S is Dv x Dk, row i holds the value
 * component i for every key direction j.  Order: decay, predict, correct,
 * read.  Row i only ever interacts with v[i], so each row is finished
 * before the next is touched. */
void oracle_core_step(int Dk, int Dv, double *S, const double *q, const double *k,
                      const double *v, double g, double beta, double *o) {
  double alpha = exp(g); /* g = -inf gives exactly 0: a reset */
  for (int i = 0; i < Dv; ++i) {
    double *row = S + (size_t)i * Dk;
    for (int j = 0; j < Dk; ++j) row[j] *= alpha;          /* decay   */
    double pred = 0.0;
    for (int j = 0; j < Dk; ++j) pred += row[j] * k[j];     /* predict */
    double delta = beta * (v[i] - pred);
    for (int j = 0; j < Dk; ++j) row[j] += delta * k[j];    /* correct */
    double out = 0.0;
    for (int j = 0; j < Dk; ++j) out += row[j] * q[j];      /* read    */
    o[i] = out;
  }
}

/* Step 3 over a whole sequence for one head: q,k [T][Dk], v [T][Dv],
 * g,beta [T], S in/out [Dv][Dk], o [T][Dv]. */
void oracle_core_recurrent(int T, int Dk, int Dv, const double *q, const double *k,
                           const double *v, const double *g, const double *beta,
                           double *S, double *o) {
  for (int t = 0; t < T; ++t)
    oracle_core_step(Dk, Dv, S, q + (size_t)t * Dk, k + (size_t)t * Dk,
                     v + (size_t)t * Dv, g[t], beta[t], o + (size_t)t * Dv);
}

/* Step 0 ("How Qwen3.5 works" section 9.5): the write gate and the log
 * decay of one token on one value head from the raw projections a, b and
 * the head's parameters A_log, dt_bias. */
double oracle_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* softplus(x) = log(1 + e^x), evaluated without overflow for large x. */
double oracle_softplus(double x) { return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x)); }

void oracle_gates(double a, double b, double A_log, double dt_bias, double *g, double *beta) {
  *beta = oracle_sigmoid(b);
  *g = -exp(A_log) * oracle_softplus(a + dt_bias);
}

/* Step 4 for one head: y = w * x / sqrt(mean(x^2) + eps) * silu(z). */
void oracle_gated_norm(int n, const double *x, const double *z, const double *w,
                       double eps, double *y) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / n + eps);
  for (int i = 0; i < n; ++i) y[i] = w[i] * (x[i] * inv) * oracle_silu(z[i]);
}

/* Channel numbering of the conv input (q | k | v, "How Qwen3.5 works"
 * section 9.2 and the gdn.conv / gdn.core tensor table of the 27B spec). */
static size_t chan_q(const oracle_shape *s, int kh, int i) { return (size_t)kh * s->Dk + i; }
static size_t chan_k(const oracle_shape *s, int kh, int i) {
  return (size_t)s->Hk * s->Dk + (size_t)kh * s->Dk + i;
}
static size_t chan_v(const oracle_shape *s, int h, int i) {
  return 2 * (size_t)s->Hk * s->Dk + (size_t)h * s->Dv + i;
}

/* Raw conv input of channel c at extended time e in [0, T+3):
 * e < 3 is the carried window (oldest first), e >= 3 is token e-3. */
static double xext(const oracle_shape *s, const float *qkv_pre, const float *conv0, int b,
                   int e, size_t c) {
  size_t C = 2 * (size_t)s->Hk * s->Dk + (size_t)s->Hv * s->Dv;
  if (e < 3) return conv0 ? (double)conv0[((size_t)b * 3 + e) * C + c] : 0.0;
  return (double)qkv_pre[((size_t)b * s->T + (e - 3)) * C + c];
}

static double conv_at(const oracle_shape *s, const float *qkv_pre, const float *conv_w,
                      const float *conv0, int b, int t, size_t c) {
  double window[4], taps[4];
  for (int j = 0; j < 4; ++j) {
    window[j] = xext(s, qkv_pre, conv0, b, t + j, c);
    taps[j] = (double)conv_w[c * 4 + j];
  }
  return oracle_conv_silu_one(window, taps);
}

/* Raw gate inputs: a, b [B][T][Hv]; A_log, dt_bias [Hv]. */
typedef struct {
  const float *a, *b, *A_log, *dt_bias;
} oracle_raw_gates;

/*
 * The whole mixer for a list of (b, h) units.
 *
 *   qkv_pre [B][T][C], C = 2*Hk*Dk + Hv*Dv     z [B][T][Hv*Dv]
 *   g, beta [B][T][Hv], or NULL with `raw` giving the gates' projections
 *   conv_w [C][4]     norm_w [Dv]
 *   S0 [B][Hv][Dv][Dk] or NULL (zeros)         conv0 [B][3][C] or NULL (zeros)
 *   units[n_units] = b*Hv + h, or NULL for all B*Hv units in order
 *   y      [n_units][T][Dv]   gated-norm output (the mixer output)
 *   core_o [n_units][T][Dv]   core output before the norm, or NULL
 *   S_T    [n_units][Dv][Dk]  final state
 *   S_snap [n_units][T][Dv][Dk] or NULL: the state after each token
 *   conv_T [B][3][C] or NULL  last three raw rows of (conv0 ++ qkv_pre)
 *
 * Returns 0, or -1 for a shape the method does not define (T < 1,
 * Hv not a multiple of Hk, non-positive sizes), a unit out of range, or
 * neither (g, beta) nor raw gates given.
 */
int oracle_gdn_prefill_ex(const oracle_shape *s, const float *qkv_pre, const float *z,
                          const float *g, const float *beta, const oracle_raw_gates *raw,
                          const float *conv_w, const float *norm_w, const float *S0,
                          const float *conv0, int n_units, const int *units, double *y,
                          double *core_o, double *S_T, double *S_snap, double *conv_T,
                          int n_threads) {
  if (s->B < 1 || s->T < 1 || s->Hk < 1 || s->Hv < 1 || s->Dk < 1 || s->Dv < 1) return -1;
  if (!(g && beta) && !(raw && raw->a && raw->b && raw->A_log && raw->dt_bias)) return -1;
  if (s->Hv % s->Hk != 0) return -1;
  int total = s->B * s->Hv;
  if (!units) n_units = total;
  for (int u = 0; u < n_units; ++u) {
    int id = units ? units[u] : u;
    if (id < 0 || id >= total) return -1;
  }
  const int r = s->Hv / s->Hk;
  const int T = s->T, Dk = s->Dk, Dv = s->Dv;
  const size_t C = 2 * (size_t)s->Hk * Dk + (size_t)s->Hv * Dv;

  if (conv_T) {
    for (int b = 0; b < s->B; ++b)
      for (int e = 0; e < 3; ++e)
        for (size_t c = 0; c < C; ++c)
          conv_T[((size_t)b * 3 + e) * C + c] = xext(s, qkv_pre, conv0, b, T + e, c);
  }

  int failed = 0;
#ifdef _OPENMP
  if (n_threads < 1) n_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
#endif
  for (int u = 0; u < n_units; ++u) {
    int id = units ? units[u] : u;
    int b = id / s->Hv, h = id % s->Hv, kh = h / r;
    double *S = (double *)malloc(sizeof(double) * ((size_t)Dv * Dk + 4 * (size_t)Dk + 4 * (size_t)Dv));
    if (!S) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      failed = 1;
      continue;
    }
    double *qraw = S + (size_t)Dv * Dk, *kraw = qraw + Dk, *qh = kraw + Dk, *kh_ = qh + Dk;
    double *vv = kh_ + Dk, *o = vv + Dv, *zz = o + Dv, *ww = zz + Dv;
    for (size_t i = 0; i < (size_t)Dv * Dk; ++i)
      S[i] = S0 ? (double)S0[((size_t)b * s->Hv + h) * Dv * Dk + i] : 0.0;
    for (int i = 0; i < Dv; ++i) ww[i] = (double)norm_w[i];

    for (int t = 0; t < T; ++t) {
      for (int i = 0; i < Dk; ++i) {
        qraw[i] = conv_at(s, qkv_pre, conv_w, conv0, b, t, chan_q(s, kh, i));
        kraw[i] = conv_at(s, qkv_pre, conv_w, conv0, b, t, chan_k(s, kh, i));
      }
      for (int i = 0; i < Dv; ++i) vv[i] = conv_at(s, qkv_pre, conv_w, conv0, b, t, chan_v(s, h, i));
      oracle_l2norm(Dk, qraw, s->eps_l2, s->q_scale, qh);
      oracle_l2norm(Dk, kraw, s->eps_l2, 1.0, kh_);
      size_t gi = ((size_t)b * T + t) * s->Hv + h;
      double gt, bt;
      if (g && beta) {
        gt = (double)g[gi];
        bt = (double)beta[gi];
      } else {
        oracle_gates((double)raw->a[gi], (double)raw->b[gi], (double)raw->A_log[h],
                     (double)raw->dt_bias[h], &gt, &bt);
      }
      oracle_core_step(Dk, Dv, S, qh, kh_, vv, gt, bt, o);
      if (S_snap)
        memcpy(S_snap + ((size_t)u * T + t) * Dv * Dk, S, sizeof(double) * (size_t)Dv * Dk);
      if (core_o) memcpy(core_o + ((size_t)u * T + t) * Dv, o, sizeof(double) * Dv);
      const float *zt = z + ((size_t)b * T + t) * ((size_t)s->Hv * Dv) + (size_t)h * Dv;
      for (int i = 0; i < Dv; ++i) zz[i] = (double)zt[i];
      oracle_gated_norm(Dv, o, zz, ww, s->eps_norm, y + ((size_t)u * T + t) * Dv);
    }
    memcpy(S_T + (size_t)u * Dv * Dk, S, sizeof(double) * (size_t)Dv * Dk);
    free(S);
  }
  return failed ? -1 : 0;
}

/* The mixer with precomputed gates and no snapshots. */
int oracle_gdn_prefill(const oracle_shape *s, const float *qkv_pre, const float *z,
                       const float *g, const float *beta, const float *conv_w,
                       const float *norm_w, const float *S0, const float *conv0, int n_units,
                       const int *units, double *y, double *core_o, double *S_T,
                       double *conv_T, int n_threads) {
  if (!g || !beta) return -1;
  return oracle_gdn_prefill_ex(s, qkv_pre, z, g, beta, NULL, conv_w, norm_w, S0, conv0, n_units,
                               units, y, core_o, S_T, NULL, conv_T, n_threads);
}

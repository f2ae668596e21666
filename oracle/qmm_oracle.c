/*
 * qmm_oracle.c -- plain, slow, single-threaded CPU oracle for the group-wise
 * quantised linear layer and the routed MoE feed-forward layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this code.  It shares no code, header,
 * table or helper with the CUDA library, and it never reads anything the
 * CUDA library produced.
 *
 * Sources (the three web pages this project restates):
 *  [P1] "Why I hand-wrote a DeepSeek inference engine in pure C" (hnwysp.cn,
 *       news 134870): section 2.3 (group-wise INT8/INT4 scheme, dequantise as
 *       (q - zero_point) * scale), section 3.2 (quantize_group: per-group
 *       min/max, scale = (max-min)/(2^bits-1), zp = round(-min/scale),
 *       q = clamp(round(v/scale)+zp, 0, 255) stored as q-128; dequantise
 *       (q + 128 - zp) * scale; fuse dequantisation into the matmul inner
 *       loop; INT4 stores two codes per byte), section 3.3 (the fp32 matmul),
 *       section 3.4 (softmax subtracts the maximum first) and section 3.5 (the
 *       MoE router is a linear layer, a softmax and a top-k; tokens are grouped
 *       by expert; expert outputs are combined by a weighted sum).
 *  [P2] "ds4 code walkthrough" (ds4-learning.pages.dev), Trace 2: DeepSeek V4
 *       Flash has 256 experts, 6 used per token, embedding width 4096.
 *  [P3] "I ran a 284B-parameter LLM from 3.2GB of RAM in plain C"
 *       (feinterview.poetries.top): CPU paths made bit-identical by a fixed
 *       accumulator tree and -ffp-contract=off.
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *  - groups are `group` consecutive elements along K of one row of W[N,K];
 *  - zero points are int32 (never narrowed);
 *  - rounding is C roundf (half away from zero), division is IEEE fp32 `/`;
 *  - float->int conversions saturate to int32 and the code sum is formed in
 *    64-bit before the clamp, so every input has a defined result;
 *  - when (max-min)/(2^bits-1) is zero (a constant group) the scale becomes
 *    max(|min|,|max|), or 1 if that is zero, and the same formulas follow;
 *  - INT4: low nibble holds the even column, no -128 shift;
 *  - router logits: 128 fp32 partial sums (partial p accumulates columns
 *    p, p+128, ... with correctly rounded fmaf), combined by a fixed tree,
 *    then the bias is added;
 *  - top-k compares logits, larger first, equal logits -> lower index first;
 *  - weights are renormalised over the selected k: w_i = p_i / sum_j p_j;
 *  - the expert FFN is SwiGLU: silu(x Wg^T) * (x Wu^T), then Wd.
 * Accumulation of linear / FFN outputs is in double ("truth"); quantisation
 * and router selection are in fp32 because they must be bit-exact.
 *
 * Compile with -O2 -ffp-contract=off and without -ffast-math.
 */
#include "qmm_oracle.h"

#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Quantisation [P1 section 3.2]                                       */
/* ------------------------------------------------------------------ */

/* roundf, then a saturating conversion to int32 (NaN -> 0). */
static int32_t sat_round_i32(float v) {
  const float r = roundf(v);
  if (r != r) return 0;
  if (r >= 2147483648.0f) return INT32_MAX;
  if (r <= -2147483648.0f) return INT32_MIN;
  return (int32_t)r;
}

int orc_quantize(const float *w, int64_t N, int64_t K, int bits, int group,
                 void *codes, float *scales, int32_t *zps) {
  if (!w || !codes || !scales || !zps) return -1;
  if (bits != 8 && bits != 4) return -1;
  if (group <= 0 || N < 0 || K <= 0 || K % group != 0) return -1;
  if (bits == 4 && (group % 2 != 0)) return -1;
  const int32_t qmax = (1 << bits) - 1;
  const int64_t G = K / group;
  uint8_t *c8 = (uint8_t *)codes;
  if (bits == 4) memset(c8, 0, (size_t)(N * K / 2));
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t j = 0; j < G; ++j) {
      const float *src = w + n * K + j * group;
      /* per-group min and max */
      float mn = FLT_MAX, mx = -FLT_MAX;
      for (int i = 0; i < group; ++i) {
        if (src[i] < mn) mn = src[i];
        if (src[i] > mx) mx = src[i];
      }
      /* scale = (max - min) / (2^bits - 1), in fp32 */
      float s = (mx - mn) / (float)qmax;
      if (s == 0.0f) { /* constant group (reading: see header) */
        const float amn = fabsf(mn), amx = fabsf(mx);
        s = amn > amx ? amn : amx;
        if (s == 0.0f) s = 1.0f;
      }
      /* zero point = round(-min / scale) */
      const int32_t zp = sat_round_i32(-mn / s);
      scales[n * G + j] = s;
      zps[n * G + j] = zp;
      for (int i = 0; i < group; ++i) {
        int64_t t = (int64_t)sat_round_i32(src[i] / s) + (int64_t)zp;
        if (t < 0) t = 0;
        if (t > qmax) t = qmax;
        const int64_t k = j * group + i;
        if (bits == 8) {
          c8[n * K + k] = (uint8_t)(int8_t)(t - 128); /* stored q - 128 */
        } else {
          const int64_t byte = (n * K + k) / 2;
          c8[byte] |= (uint8_t)(t << (4 * (k & 1))); /* low nibble = even k */
        }
      }
    }
  }
  return 0;
}

int32_t orc_code_at(const orc_qweight *w, int64_t n, int64_t k) {
  const uint8_t *c8 = (const uint8_t *)w->codes;
  if (w->bits == 8) {
    return (int32_t)(int8_t)c8[n * w->K + k] + 128; /* q = stored + 128 */
  }
  const uint8_t b = c8[(n * w->K + k) / 2];
  return (k & 1) ? (int32_t)(b >> 4) : (int32_t)(b & 0x0F);
}

/* Dequantised weight as the pages define it: (q - zp) * scale, the integer
 * difference converted to fp32 and then one fp32 multiply. */
static float dequant_one(int32_t q, int32_t zp, float s) {
  return (float)((int64_t)q - (int64_t)zp) * s;
}

void orc_dequantize(const orc_qweight *w, float *out) {
  const int64_t G = w->K / w->group;
  for (int64_t n = 0; n < w->N; ++n) {
    for (int64_t k = 0; k < w->K; ++k) {
      const int64_t gi = n * G + k / w->group;
      out[n * w->K + k] = dequant_one(orc_code_at(w, n, k), w->zps[gi], w->scales[gi]);
    }
  }
}

/* ------------------------------------------------------------------ */
/* Linear layer y[m,n] = sum_k x[m,k] * W^[n,k]  [P1 sections 3.2, 3.3] */
/* ------------------------------------------------------------------ */

/* Fused form: the codes are unpacked and dequantised inside the k loop
 * (the P1 section 3.2 performance tip), accumulation in double. */
void orc_linear_fused(const float *x, int64_t M, const orc_qweight *w, double *y) {
  const int64_t K = w->K, G = K / w->group;
  const uint8_t *c8 = (const uint8_t *)w->codes;
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < w->N; ++n) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        int32_t q;
        if (w->bits == 8) {
          q = (int32_t)(int8_t)c8[n * K + k] + 128;
        } else {
          const uint8_t b = c8[(n * K + k) >> 1];
          q = (k & 1) ? (b >> 4) : (b & 0x0F);
        }
        const int64_t gi = n * G + k / w->group;
        const float wh = (float)((int64_t)q - (int64_t)w->zps[gi]) * w->scales[gi];
        acc += (double)x[m * K + k] * (double)wh;
      }
      y[m * w->N + n] = acc;
    }
  }
}

/* Unfused form: dequantise the whole matrix first, then an i-k-j matmul
 * (the P1 section 3.3 loop order) with double accumulators. */
void orc_linear_two_step(const float *x, int64_t M, const orc_qweight *w, double *y) {
  const int64_t N = w->N, K = w->K;
  float *wh = (float *)malloc((size_t)(N * K) * sizeof(float));
  if (!wh) return;
  orc_dequantize(w, wh);
  for (int64_t i = 0; i < M; ++i) {
    double *c = y + i * N;
    for (int64_t j = 0; j < N; ++j) c[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double a = (double)x[i * K + k];
      for (int64_t j = 0; j < N; ++j) c[j] += a * (double)wh[j * K + k];
    }
  }
  free(wh);
}

/* Per-output tolerance of an fp32 implementation: 1e-5 * sum_k |x_k w^_k| + 1e-6. */
void orc_linear_bound(const float *x, int64_t M, const orc_qweight *w, double *bound) {
  const int64_t K = w->K, G = K / w->group;
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < w->N; ++n) {
      double a = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const int64_t gi = n * G + k / w->group;
        const float wh = dequant_one(orc_code_at(w, n, k), w->zps[gi], w->scales[gi]);
        a += fabs((double)x[m * K + k] * (double)wh);
      }
      bound[m * w->N + n] = 1e-5 * a + 1e-6;
    }
  }
}

/* ------------------------------------------------------------------ */
/* Router [P1 sections 3.4, 3.5]                                       */
/* ------------------------------------------------------------------ */

#define ORC_ROUTER_PARTIALS 128

/* One router logit in fp32 with the fixed summation order. */
static float router_dot(const float *x, const float *wr, int64_t H) {
  float part[ORC_ROUTER_PARTIALS];
  for (int p = 0; p < ORC_ROUTER_PARTIALS; ++p) {
    float acc = 0.0f;
    for (int64_t k = p; k < H; k += ORC_ROUTER_PARTIALS) acc = fmaf(x[k], wr[k], acc);
    part[p] = acc;
  }
  /* level 1: 32 sums of 4 adjacent partials, (a + b) + (c + d) */
  float t[32];
  for (int l = 0; l < 32; ++l) {
    t[l] = (part[4 * l] + part[4 * l + 1]) + (part[4 * l + 2] + part[4 * l + 3]);
  }
  /* levels 2..6: halving tree t[l] = t[l] + t[l + o], o = 16, 8, 4, 2, 1 */
  for (int o = 16; o >= 1; o >>= 1) {
    for (int l = 0; l < o; ++l) t[l] = t[l] + t[l + o];
  }
  return t[0];
}

void orc_router_logits(const float *x, int64_t M, int64_t H, const float *wr,
                       const float *bias, int32_t E, float *logits) {
  for (int64_t m = 0; m < M; ++m) {
    for (int32_t e = 0; e < E; ++e) {
      float l = router_dot(x + m * H, wr + (int64_t)e * H, H);
      if (bias) l = l + bias[e];
      logits[m * E + e] = l;
    }
  }
}

/* a beats b: larger logit first, equal logits -> lower expert index first. */
static int beats(float la, int32_t a, float lb, int32_t b) {
  return (la > lb) || (la == lb && a < b);
}

void orc_topk(const float *logits, int64_t M, int32_t E, int32_t k,
              int32_t *idx, float *w) {
  char *taken = (char *)malloc((size_t)E);
  double *p = (double *)malloc((size_t)E * sizeof(double));
  if (!taken || !p) { free(taken); free(p); return; }
  for (int64_t m = 0; m < M; ++m) {
    const float *l = logits + m * E;
    /* selection by repeated best-of-remaining with the comparator above */
    memset(taken, 0, (size_t)E);
    for (int32_t i = 0; i < k; ++i) {
      int32_t best = -1;
      for (int32_t e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || beats(l[e], e, l[best], best)) best = e;
      }
      taken[best] = 1;
      idx[m * k + i] = best;
    }
    /* softmax over all E experts, maximum subtracted first, in double */
    double mx = -INFINITY;
    for (int32_t e = 0; e < E; ++e) if ((double)l[e] > mx) mx = (double)l[e];
    double z = 0.0;
    for (int32_t e = 0; e < E; ++e) { p[e] = exp((double)l[e] - mx); z += p[e]; }
    for (int32_t e = 0; e < E; ++e) p[e] /= z;
    /* renormalise over the selected experts */
    double ps = 0.0;
    for (int32_t i = 0; i < k; ++i) ps += p[idx[m * k + i]];
    for (int32_t i = 0; i < k; ++i) w[m * k + i] = (float)(p[idx[m * k + i]] / ps);
  }
  free(taken);
  free(p);
}

/* Routing load check [P1 section 3.5, last paragraph: when one expert is
 * chosen more often than a threshold the engine warns, because grouped expert
 * work then degenerates towards serial work].  Counts how often each expert
 * appears among the M x k selected indices (indices outside [0, E) are not
 * counted), then stats = {largest count, the lowest expert index with that
 * count, number of experts chosen at least once, number of counted
 * selections}.  Returns 1 when the largest count exceeds `threshold`. */
int orc_load_stats(const int32_t *idx, int64_t M, int32_t k, int32_t E,
                   int64_t threshold, int64_t *stats) {
  int64_t *count = (int64_t *)calloc((size_t)E, sizeof(int64_t));
  if (!count) return -1;
  for (int64_t a = 0; a < M * k; ++a)
    if (idx[a] >= 0 && idx[a] < E) count[idx[a]] += 1;
  int64_t best = 0, total = 0, touched = 0;
  int32_t arg = 0;
  for (int32_t e = 0; e < E; ++e) {
    if (count[e] > best) { best = count[e]; arg = e; }
    if (count[e] > 0) touched += 1;
    total += count[e];
  }
  free(count);
  stats[0] = best;
  stats[1] = arg;
  stats[2] = touched;
  stats[3] = total;
  return best > threshold ? 1 : 0;
}

/* ------------------------------------------------------------------ */
/* Routed SwiGLU MoE FFN [P1 section 3.5, P2 Trace 2]                  */
/* ------------------------------------------------------------------ */

static double silu(double a) { return a / (1.0 + exp(-a)); }

static double silu_grad(double a) {
  const double sg = 1.0 / (1.0 + exp(-a));
  return sg * (1.0 + a * (1.0 - sg));
}

/* row n of x . W^T in double, plus sum |x_k W^[n,k]| for the bound */
static void dot_row(const double *x, const orc_qweight *w, int64_t n,
                    double *val, double *absval, double *absw) {
  const int64_t K = w->K, G = K / w->group;
  double acc = 0.0, a = 0.0, aw = 0.0;
  for (int64_t k = 0; k < K; ++k) {
    const int64_t gi = n * G + k / w->group;
    const double wh = (double)dequant_one(orc_code_at(w, n, k), w->zps[gi], w->scales[gi]);
    acc += x[k] * wh;
    a += fabs(x[k] * wh);
    aw += fabs(wh);
  }
  *val = acc;
  if (absval) *absval = a;
  if (absw) *absw = aw;
}

int orc_moe_ffn(const float *x, int64_t M, int64_t H, int64_t I,
                const int32_t *idx, const float *tw, int32_t k, int32_t E,
                const orc_qweight *gate, const orc_qweight *up,
                const orc_qweight *down, double dw, double *y, double *bound) {
  double *xd = (double *)malloc((size_t)H * sizeof(double));
  double *h = (double *)malloc((size_t)I * sizeof(double));
  double *dh = (double *)malloc((size_t)I * sizeof(double));
  if (!xd || !h || !dh) { free(xd); free(h); free(dh); return -1; }
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < H; ++n) { y[m * H + n] = 0.0; if (bound) bound[m * H + n] = 1e-6; }
    for (int64_t c = 0; c < H; ++c) xd[c] = (double)x[m * H + c];
    for (int32_t i = 0; i < k; ++i) {
      const int32_t e = idx[m * k + i];
      if (e < 0 || e >= E || !gate[e].codes || !up[e].codes || !down[e].codes) {
        free(xd); free(h); free(dh); return -2;
      }
      const double wt = (double)tw[m * k + i];
      /* gate and up projections, SwiGLU */
      for (int64_t j = 0; j < I; ++j) {
        double g, u, ag, au;
        dot_row(xd, &gate[e], j, &g, &ag, NULL);
        dot_row(xd, &up[e], j, &u, &au, NULL);
        h[j] = silu(g) * u;
        const double Dg = 1e-5 * ag + 1e-6, Du = 1e-5 * au + 1e-6;
        dh[j] = fabs(silu_grad(g) * u) * Dg + fabs(silu(g)) * Du + 1e-6 * fabs(h[j]);
      }
      /* down projection and weighted combine */
      for (int64_t n = 0; n < H; ++n) {
        double o, ao;
        dot_row(h, &down[e], n, &o, &ao, NULL);
        y[m * H + n] += wt * o;
        if (bound) {
          /* sum_j |W^d[n,j]| * dh_j */
          const int64_t G = I / down[e].group;
          double prop = 0.0;
          for (int64_t j = 0; j < I; ++j) {
            const int64_t gi = n * G + j / down[e].group;
            prop += fabs((double)dequant_one(orc_code_at(&down[e], n, j), down[e].zps[gi],
                                             down[e].scales[gi])) * dh[j];
          }
          bound[m * H + n] += fabs(wt) * (1e-5 * ao + prop + 1e-6) + dw * fabs(o);
        }
      }
    }
  }
  free(xd);
  free(h);
  free(dh);
  return 0;
}

/* ------------------------------------------------------------------ */
/* Decode attention with rotary positions [P1 section 3.4]             */
/* ------------------------------------------------------------------ */
/*
 * Readings where the page is silent (listed in the design notes):
 *  - a "pair of dimensions" is (2i, 2i+1) of a head vector, rotated by the
 *    angle pos * theta_i with theta_i = base^(-2i/head_dim); base 10000 is
 *    the caller's choice, not the page's;
 *  - the table holds cos and sin of those angles rounded to fp32, and the
 *    rotation is (a, b) -> (a cos - b sin, a sin + b cos);
 *  - query head h reads key/value head h / (n_head / n_kv) (n_kv = n_head:
 *    the page's multi-head attention; fewer: grouped heads as in the ds4
 *    walkthrough's 64 query heads over one key/value head);
 *  - the KV cache of one layer is [2][n_kv][max_seq][head_dim] fp32 (keys,
 *    then values), the page's [layers, 2, heads, max_seq, head_dim] for one
 *    layer; the decode step writes row pos and attends over rows 0..pos.
 */

void orc_rope_table(int64_t max_seq, int32_t head_dim, double base, float *cos_t, float *sin_t) {
  const int32_t hp = head_dim / 2;
  for (int64_t p = 0; p < max_seq; ++p) {
    for (int32_t i = 0; i < hp; ++i) {
      const double theta = pow(base, -2.0 * (double)i / (double)head_dim);
      const double ang = (double)p * theta;
      cos_t[p * hp + i] = (float)cos(ang);
      sin_t[p * hp + i] = (float)sin(ang);
    }
  }
}

void orc_rope_apply(const double *x, int32_t n_vec, int32_t head_dim, int64_t pos,
                    const float *cos_t, const float *sin_t, double *out) {
  const int32_t hp = head_dim / 2;
  for (int32_t v = 0; v < n_vec; ++v) {
    for (int32_t i = 0; i < hp; ++i) {
      const double c = (double)cos_t[pos * hp + i], s = (double)sin_t[pos * hp + i];
      const double a = x[v * head_dim + 2 * i], b = x[v * head_dim + 2 * i + 1];
      out[v * head_dim + 2 * i] = a * c - b * s;
      out[v * head_dim + 2 * i + 1] = a * s + b * c;
    }
  }
}

/* Bound of the rotated values from bounds da of the inputs: the rotation in
 * fp32 (|err| <= 1e-5 (|a c| + |b s|) + 1e-6, the fp32 rule of a two-term
 * dot product) plus |c| da + |s| db. */
static void rope_bound(const double *x, const double *dx, int32_t n_vec, int32_t head_dim,
                       int64_t pos, const float *cos_t, const float *sin_t, double *bound) {
  const int32_t hp = head_dim / 2;
  for (int32_t v = 0; v < n_vec; ++v) {
    for (int32_t i = 0; i < hp; ++i) {
      const double c = fabs((double)cos_t[pos * hp + i]), s = fabs((double)sin_t[pos * hp + i]);
      const double a = fabs(x[v * head_dim + 2 * i]), b = fabs(x[v * head_dim + 2 * i + 1]);
      const double da = dx ? dx[v * head_dim + 2 * i] : 0.0;
      const double db = dx ? dx[v * head_dim + 2 * i + 1] : 0.0;
      bound[v * head_dim + 2 * i] = 1e-5 * (a * c + b * s) + 1e-6 + c * da + s * db;
      bound[v * head_dim + 2 * i + 1] = 1e-5 * (a * s + b * c) + 1e-6 + s * da + c * db;
    }
  }
}

void orc_attention(const double *q, const double *dq, const float *k_cache, const float *v_cache,
                   const double *k_last, const double *v_last, const double *dk_last,
                   const double *dv_last, int32_t n_head, int32_t n_kv, int32_t head_dim,
                   int64_t max_seq, int64_t T, double *out, double *bound) {
  const int32_t grp = n_head / n_kv;
  const double scale = 1.0 / sqrt((double)head_dim);
  double *s = (double *)malloc((size_t)T * sizeof(double));
  double *ds = (double *)malloc((size_t)T * sizeof(double));
  double *p = (double *)malloc((size_t)T * sizeof(double));
  if (!s || !ds || !p) { free(s); free(ds); free(p); return; }
  for (int32_t h = 0; h < n_head; ++h) {
    const int32_t kvh = h / grp;
    const double *qh = q + (int64_t)h * head_dim;
    /* row t of the keys / values of head kvh: the cache, or row T-1 from
     * k_last / v_last when given (the row this decode step writes) */
    for (int64_t t = 0; t < T; ++t) {
      double dot = 0.0, adot = 0.0, prop = 0.0;
      for (int32_t i = 0; i < head_dim; ++i) {
        const int64_t ci = ((int64_t)kvh * max_seq + t) * head_dim + i;
        const int last = (t == T - 1) && k_last;
        const double kv = last ? k_last[(int64_t)kvh * head_dim + i] : (double)k_cache[ci];
        dot += qh[i] * kv;
        adot += fabs(qh[i] * kv);
        if (dq) prop += fabs(kv) * dq[(int64_t)h * head_dim + i];
        if (last && dk_last) prop += fabs(qh[i]) * dk_last[(int64_t)kvh * head_dim + i];
      }
      s[t] = dot * scale;
      ds[t] = (1e-5 * adot + prop) * scale + 1e-6;
    }
    /* softmax with the maximum subtracted first */
    double mx = s[0];
    for (int64_t t = 1; t < T; ++t) mx = s[t] > mx ? s[t] : mx;
    double z = 0.0;
    for (int64_t t = 0; t < T; ++t) { p[t] = exp(s[t] - mx); z += p[t]; }
    double mean_ds = 0.0;
    for (int64_t t = 0; t < T; ++t) { p[t] /= z; mean_ds += p[t] * ds[t]; }
    for (int32_t d = 0; d < head_dim; ++d) {
      double acc = 0.0, b = 0.0, apv = 0.0;
      for (int64_t t = 0; t < T; ++t) {
        const int64_t ci = ((int64_t)kvh * max_seq + t) * head_dim + d;
        const int last = (t == T - 1) && v_last;
        const double vv = last ? v_last[(int64_t)kvh * head_dim + d] : (double)v_cache[ci];
        acc += p[t] * vv;
        apv += p[t] * fabs(vv);
        /* first order: dp_t <= p_t (ds_t + sum_u p_u ds_u + 1e-6) */
        b += p[t] * (ds[t] + mean_ds + 1e-6) * fabs(vv);
        if (last && dv_last) b += p[t] * dv_last[(int64_t)kvh * head_dim + d];
      }
      out[(int64_t)h * head_dim + d] = acc;
      if (bound) bound[(int64_t)h * head_dim + d] = b + 1e-5 * apv + 1e-6;
    }
  }
  free(s);
  free(ds);
  free(p);
}

int orc_attn_decode(const float *x, int64_t pos, int32_t n_head, int32_t n_kv, int32_t head_dim,
                    int64_t max_seq, const orc_qweight *wq, const orc_qweight *wk,
                    const orc_qweight *wv, const orc_qweight *wo, const float *cos_t,
                    const float *sin_t, const float *cache_in, double *kv_new, double *kv_bound,
                    double *y, double *bound) {
  const int64_t D = wq->K, nq = (int64_t)n_head * head_dim, nk = (int64_t)n_kv * head_dim;
  if (wk->K != D || wv->K != D || wq->N != nq || wk->N != nk || wv->N != nk || wo->K != nq)
    return -1;
  double *xd = (double *)malloc((size_t)D * sizeof(double));
  double *q = (double *)malloc((size_t)(4 * nq + 4 * nk) * sizeof(double));
  if (!xd || !q) { free(xd); free(q); return -2; }
  double *dq = q + nq, *qr = dq + nq, *dqr = qr + nq;
  double *k = dqr + nq, *dk = k + nk, *v = dk + nk, *dv = v + nk;
  double *a = (double *)malloc((size_t)(2 * nq + 2 * nk) * sizeof(double));
  if (!a) { free(xd); free(q); return -2; }
  double *da = a + nq, *kr = da + nq, *dkr = kr + nk;
  for (int64_t c = 0; c < D; ++c) xd[c] = (double)x[c];
  /* the three projections (fused dequantised linear layers) */
  for (int64_t n = 0; n < nq; ++n) {
    double val, av;
    dot_row(xd, wq, n, &val, &av, NULL);
    q[n] = val;
    dq[n] = 1e-5 * av + 1e-6;
  }
  for (int64_t n = 0; n < nk; ++n) {
    double val, av;
    dot_row(xd, wk, n, &val, &av, NULL);
    k[n] = val;
    dk[n] = 1e-5 * av + 1e-6;
    dot_row(xd, wv, n, &val, &av, NULL);
    v[n] = val;
    dv[n] = 1e-5 * av + 1e-6;
  }
  /* rotary positions for the query and the new key */
  orc_rope_apply(q, n_head, head_dim, pos, cos_t, sin_t, qr);
  rope_bound(q, dq, n_head, head_dim, pos, cos_t, sin_t, dqr);
  orc_rope_apply(k, n_kv, head_dim, pos, cos_t, sin_t, kr);
  rope_bound(k, dk, n_kv, head_dim, pos, cos_t, sin_t, dkr);
  if (kv_new) {
    memcpy(kv_new, kr, (size_t)nk * sizeof(double));
    memcpy(kv_new + nk, v, (size_t)nk * sizeof(double));
  }
  if (kv_bound) {
    memcpy(kv_bound, dkr, (size_t)nk * sizeof(double));
    memcpy(kv_bound + nk, dv, (size_t)nk * sizeof(double));
  }
  /* attention over cache rows 0..pos, row pos being this step's key/value */
  const float *kc = cache_in, *vc = cache_in + (int64_t)n_kv * max_seq * head_dim;
  orc_attention(qr, dqr, kc, vc, kr, v, dkr, dv, n_head, n_kv, head_dim, max_seq, pos + 1, a, da);
  /* output projection, with the propagated bound sum_j |Wo[n,j]| da_j */
  const int64_t G = nq / wo->group;
  for (int64_t n = 0; n < wo->N; ++n) {
    double val, av;
    dot_row(a, wo, n, &val, &av, NULL);
    y[n] = val;
    if (bound) {
      double prop = 0.0;
      for (int64_t j = 0; j < nq; ++j) {
        const int64_t gi = n * G + j / wo->group;
        prop += fabs((double)dequant_one(orc_code_at(wo, n, j), wo->zps[gi], wo->scales[gi])) *
                da[j];
      }
      bound[n] = 1e-5 * av + prop + 1e-6;
    }
  }
  free(xd);
  free(q);
  free(a);
  return 0;
}

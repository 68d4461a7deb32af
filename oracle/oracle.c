/*
 * Flint-shaped sparse MoE layer: plain fp64 CPU oracle (TEST INFRASTRUCTURE ONLY).
 * See oracle.h for what it computes and which readings it takes.  Single-threaded,
 * no blocking, no fusion, no reordering beyond the definitions written below.
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared oracle.c -lm
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

double oracle_bf16_to_f64(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* Router scoring: a linear map to one logit per expert, plus the optional bias, then a
 * sigmoid per expert (the serving-kit post, "The architecture, from the config": sigmoid
 * router scoring, not softmax routing). */
int oracle_router(const double* x, int T, int H, int E, const uint16_t* w_router,
                  const float* bias, double* logits, double* scores) {
  if (!x || !w_router || T < 0 || H <= 0 || E <= 0) return ORACLE_EINVAL;
  double* l = (double*)malloc(sizeof(double) * (size_t)E);
  if (!l) return ORACLE_EINVAL;
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) l[e] = 0.0;
    for (int h = 0; h < H; ++h) {
      const double xv = x[(size_t)t * H + h];
      const uint16_t* row = w_router + (size_t)h * E;
      for (int e = 0; e < E; ++e) l[e] += xv * oracle_bf16_to_f64(row[e]);
    }
    for (int e = 0; e < E; ++e) {
      double z = l[e] + (bias ? (double)bias[e] : 0.0);
      if (logits) logits[(size_t)t * E + e] = z;
      if (scores) scores[(size_t)t * E + e] = sigmoid(z);
    }
  }
  free(l);
  return ORACLE_OK;
}

/* "a before b" in the ranking: higher score first, lower index on equal scores. */
static int ranks_before(double sa, int a, double sb, int b) {
  if (sa > sb) return 1;
  if (sa < sb) return 0;
  return a < b;
}

/* Normalised top-k (the serving-kit post, "The architecture, from the config": 6 of 256
 * routed experts per token, normalised top-k).  Selection by k passes of "best remaining
 * expert" under the (score desc, index asc) ranking; the gates are the chosen scores
 * divided by their sum. */
int oracle_select(const double* s, int E, int k, int32_t* idx, double* gates, double* gaps) {
  if (!s || k <= 0 || k > E) return ORACLE_EINVAL;
  char* taken = (char*)calloc((size_t)E, 1);
  if (!taken) return ORACLE_EINVAL;
  double* sel = (double*)malloc(sizeof(double) * (size_t)(k + 1));
  int n_rank = (k < E) ? k + 1 : k; /* also find the (k+1)-th for the gap */
  int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)n_rank);
  for (int j = 0; j < n_rank; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      if (best < 0 || ranks_before(s[e], e, s[best], best)) best = e;
    }
    taken[best] = 1;
    order[j] = best;
    sel[j] = s[best];
  }
  double sum = 0.0;
  for (int j = 0; j < k; ++j) sum += sel[j];
  for (int j = 0; j < k; ++j) {
    if (idx) idx[j] = order[j];
    if (gates) gates[j] = sel[j] / sum;
  }
  if (gaps) {
    for (int j = 0; j < k; ++j) {
      if (j + 1 < n_rank)
        gaps[j] = sel[j] - sel[j + 1];
      else
        gaps[j] = INFINITY;
    }
  }
  free(order);
  free(sel);
  free(taken);
  return ORACLE_OK;
}

/* A SwiGLU MLP: out = (silu(x Wg) elementwise-times (x Wu)) Wd, with the products
 * accumulated over the contraction index in ascending order. */
void oracle_swiglu(const double* x, int H, int I, const uint16_t* wg, const uint16_t* wu,
                   const uint16_t* wd, double* out, double* hbuf) {
  double* g = hbuf;
  double* u = (double*)malloc(sizeof(double) * (size_t)I);
  for (int i = 0; i < I; ++i) {
    g[i] = 0.0;
    u[i] = 0.0;
  }
  for (int h = 0; h < H; ++h) {
    const double xv = x[h];
    const uint16_t* rg = wg + (size_t)h * I;
    const uint16_t* ru = wu + (size_t)h * I;
    for (int i = 0; i < I; ++i) {
      g[i] += xv * oracle_bf16_to_f64(rg[i]);
      u[i] += xv * oracle_bf16_to_f64(ru[i]);
    }
  }
  for (int i = 0; i < I; ++i) g[i] = silu(g[i]) * u[i];
  for (int h = 0; h < H; ++h) out[h] = 0.0;
  for (int i = 0; i < I; ++i) {
    const double hv = g[i];
    const uint16_t* rd = wd + (size_t)i * H;
    for (int h = 0; h < H; ++h) out[h] += hv * oracle_bf16_to_f64(rd[h]);
  }
  free(u);
}

static int check_layer(const oracle_layer* L) {
  if (!L || L->H <= 0 || L->E <= 0 || L->k <= 0 || L->k > L->E || L->I <= 0 || L->Is <= 0)
    return ORACLE_EINVAL;
  if (!L->w_router || !L->w_gate || !L->w_up || !L->w_down || !L->ws_gate || !L->ws_up ||
      !L->ws_down)
    return ORACLE_EINVAL;
  return ORACLE_OK;
}

/* y[t] = shared(x[t]) + sum_j gates[j] * E_{idx[j]}(x[t]), the sum taken in slot order. */
static int combine_token(const oracle_layer* L, const double* xt, const int32_t* sel,
                         const double* g, double* yt, double* tmp, double* hbuf) {
  const int H = L->H;
  oracle_swiglu(xt, H, L->Is, L->ws_gate, L->ws_up, L->ws_down, yt, hbuf);
  for (int j = 0; j < L->k; ++j) {
    int e = sel[j];
    if (e < 0 || e >= L->E) return ORACLE_EINVAL;
    if (!L->w_gate[e] || !L->w_up[e] || !L->w_down[e]) return ORACLE_EMISSING_EXPERT;
    oracle_swiglu(xt, H, L->I, L->w_gate[e], L->w_up[e], L->w_down[e], tmp, hbuf);
    for (int h = 0; h < H; ++h) yt[h] += g[j] * tmp[h];
  }
  return ORACLE_OK;
}

int oracle_moe_forward(const oracle_layer* L, const double* x, int T, double* y, int32_t* idx,
                       double* gates, double* gaps, double* scores) {
  int rc = check_layer(L);
  if (rc) return rc;
  if (!x || !y || T < 0) return ORACLE_EINVAL;
  const int H = L->H, E = L->E, k = L->k;
  int imax = L->I > L->Is ? L->I : L->Is;
  double* s = (double*)malloc(sizeof(double) * (size_t)E);
  double* tmp = (double*)malloc(sizeof(double) * (size_t)H);
  double* hbuf = (double*)malloc(sizeof(double) * (size_t)imax);
  int32_t* sel = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
  double* g = (double*)malloc(sizeof(double) * (size_t)k);
  double* gp = (double*)malloc(sizeof(double) * (size_t)k);
  for (int t = 0; t < T && rc == ORACLE_OK; ++t) {
    const double* xt = x + (size_t)t * H;
    rc = oracle_router(xt, 1, H, E, L->w_router, L->router_bias, NULL, s);
    if (rc) break;
    rc = oracle_select(s, E, k, sel, g, gp);
    if (rc) break;
    rc = combine_token(L, xt, sel, g, y + (size_t)t * H, tmp, hbuf);
    for (int j = 0; j < k; ++j) {
      if (idx) idx[(size_t)t * k + j] = sel[j];
      if (gates) gates[(size_t)t * k + j] = g[j];
      if (gaps) gaps[(size_t)t * k + j] = gp[j];
    }
    if (scores) memcpy(scores + (size_t)t * E, s, sizeof(double) * (size_t)E);
  }
  free(gp);
  free(g);
  free(sel);
  free(hbuf);
  free(tmp);
  free(s);
  return rc;
}

int oracle_moe_forward_given(const oracle_layer* L, const double* x, int T, const int32_t* idx,
                             double* y) {
  int rc = check_layer(L);
  if (rc) return rc;
  if (!x || !y || !idx || T < 0) return ORACLE_EINVAL;
  const int H = L->H, E = L->E, k = L->k;
  int imax = L->I > L->Is ? L->I : L->Is;
  double* s = (double*)malloc(sizeof(double) * (size_t)E);
  double* tmp = (double*)malloc(sizeof(double) * (size_t)H);
  double* hbuf = (double*)malloc(sizeof(double) * (size_t)imax);
  double* g = (double*)malloc(sizeof(double) * (size_t)k);
  for (int t = 0; t < T && rc == ORACLE_OK; ++t) {
    const double* xt = x + (size_t)t * H;
    const int32_t* sel = idx + (size_t)t * k;
    rc = oracle_router(xt, 1, H, E, L->w_router, L->router_bias, NULL, s);
    if (rc) break;
    double sum = 0.0;
    for (int j = 0; j < k; ++j) {
      if (sel[j] < 0 || sel[j] >= E) {
        rc = ORACLE_EINVAL;
        break;
      }
      sum += s[sel[j]];
    }
    if (rc) break;
    for (int j = 0; j < k; ++j) g[j] = s[sel[j]] / sum;
    rc = combine_token(L, xt, sel, g, y + (size_t)t * H, tmp, hbuf);
  }
  free(g);
  free(hbuf);
  free(tmp);
  free(s);
  return rc;
}

/* Counting sort: count pairs per expert, exclusive scan, then place pairs in (t, j)
 * order, which keeps the sort stable. */
int oracle_permute(const int32_t* idx, int T, int k, int E, int32_t* counts, int32_t* offsets,
                   int32_t* perm, int32_t* inv) {
  if (!idx || T < 0 || k <= 0 || E <= 0 || !counts || !offsets) return ORACLE_EINVAL;
  const long n = (long)T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (long p = 0; p < n; ++p) {
    if (idx[p] < 0 || idx[p] >= E) return ORACLE_EINVAL;
    counts[idx[p]] += 1;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  for (int e = 0; e < E; ++e) fill[e] = offsets[e];
  for (long p = 0; p < n; ++p) {
    int32_t row = fill[idx[p]]++;
    if (perm) perm[row] = (int32_t)p;
    if (inv) inv[p] = row;
  }
  free(fill);
  return ORACLE_OK;
}

/* Round to the nearest bfloat16 value, ties to even (normal range; the layer's values are
 * far from bf16's subnormal and overflow limits). */
double oracle_round_bf16(double v) {
  if (v == 0.0 || !isfinite(v)) return v;
  int e;
  const double m = frexp(v, &e);       /* v = m * 2^e, 0.5 <= |m| < 1 */
  const double q = nearbyint(m * 256.0); /* 8 significant bits; default mode: ties to even */
  return ldexp(q, e - 8);
}

/* RMSNorm with a unit weight. */
void oracle_rmsnorm(const double* x, int T, int H, double eps, double* r) {
  for (int t = 0; t < T; ++t) {
    const double* xt = x + (size_t)t * H;
    double ss = 0.0;
    for (int h = 0; h < H; ++h) ss += xt[h] * xt[h];
    const double d = sqrt(ss / (double)H + eps);
    for (int h = 0; h < H; ++h) r[(size_t)t * H + h] = xt[h] / d;
  }
}

/* Decode attention with a learned sink per head, over each sequence's ring of W cached tokens. */
int oracle_swa_decode(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* sinks,
                      const int32_t* pos, int B, int nh, int nkv, int d, int W, double* out) {
  if (!q || !k || !v || !sinks || !pos || !out || B < 0 || nh <= 0 || nkv <= 0 || nh % nkv || d <= 0 || W <= 0)
    return ORACLE_EINVAL;
  const int group = nh / nkv;
  const double scale = 1.0 / sqrt((double)d);
  double* s = (double*)malloc(sizeof(double) * (size_t)W);
  if (!s) return ORACLE_EINVAL;
  for (int b = 0; b < B; ++b) {
    if (pos[b] < 0) {
      free(s);
      return ORACLE_EINVAL;
    }
    const int n = pos[b] + 1 < W ? pos[b] + 1 : W;
    for (int h = 0; h < nh; ++h) {
      const int g = h / group;
      const uint16_t* qh = q + ((size_t)b * nh + h) * d;
      double m = (double)sinks[h];
      for (int j = 0; j < n; ++j) {
        const uint16_t* kj = k + (((size_t)b * W + j) * nkv + g) * d;
        double dot = 0.0;
        for (int i = 0; i < d; ++i) dot += oracle_bf16_to_f64(qh[i]) * oracle_bf16_to_f64(kj[i]);
        s[j] = dot * scale;
        if (s[j] > m) m = s[j];
      }
      double den = exp((double)sinks[h] - m);
      for (int j = 0; j < n; ++j) den += exp(s[j] - m);
      double* o = out + ((size_t)b * nh + h) * d;
      for (int i = 0; i < d; ++i) o[i] = 0.0;
      for (int j = 0; j < n; ++j) {
        const double p = exp(s[j] - m) / den;
        const uint16_t* vj = v + (((size_t)b * W + j) * nkv + g) * d;
        for (int i = 0; i < d; ++i) o[i] += p * oracle_bf16_to_f64(vj[i]);
      }
    }
  }
  free(s);
  return ORACLE_OK;
}

/* FP4 E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa; exponent 0 is subnormal. */
double oracle_e2m1_to_f64(unsigned code) {
  const unsigned sign = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
  const double mag = e == 0 ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
  return sign ? -mag : mag;
}

/* FP8 E4M3 (the variant without infinities): bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0
 * mantissa; exponent 0 is subnormal; exponent 15 with mantissa 7 is NaN. */
double oracle_e4m3_to_f64(unsigned byte) {
  const unsigned sign = (byte >> 7) & 1u, e = (byte >> 3) & 15u, m = byte & 7u;
  if (e == 15u && m == 7u) return NAN;
  const double mag = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, (int)e - 7);
  return sign ? -mag : mag;
}

int oracle_nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, float tensor_scale, int K, int N,
                         double* out) {
  if (!codes || !scales || !out || K <= 0 || N <= 0 || K % 16) return ORACLE_EINVAL;
  for (int k = 0; k < K; ++k)
    for (int n = 0; n < N; ++n) {
      const uint8_t byte = codes[(size_t)n * (K / 2) + k / 2];
      const unsigned code = (k % 2) ? (byte >> 4) : (byte & 15u);
      const double s = oracle_e4m3_to_f64(scales[(size_t)n * (K / 16) + k / 16]);
      out[(size_t)k * N + n] = oracle_e2m1_to_f64(code) * s * (double)tensor_scale;
    }
  return ORACLE_OK;
}

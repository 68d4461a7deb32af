/*
 * Flint-shaped sparse MoE layer: plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the slow, obviously-correct definition that the
 * CUDA path is checked against.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline / reference leg may load it; the product library never does,
 * and it shares no code, header or constant table with the CUDA sources.
 *
 * What it computes (sources: the Recursive Flint serving-kit post, section "The
 * architecture, from the config", and the news article "Recursive opens Flint, a 40B
 * coding model with 2.5B active", section "What runs on each token"):
 *   - every MoE layer has 256 routed experts, 6 chosen per token, and one shared
 *     expert that runs on every token; expert width 512, shared width 1024, hidden 2048;
 *   - router scores are sigmoids of the router logits, and the chosen experts' weights
 *     are those scores normalised over the chosen set (not a softmax).
 * Readings where the pages are silent (each one is listed in the design notes):
 *   - experts are SwiGLU MLPs: E(x) = (silu(x Wg) * (x Wu)) Wd, silu(z) = z / (1 + e^-z);
 *   - an optional per-expert router bias is added to the logit before the sigmoid and is
 *     used both for selection and for the gate values; routed scaling factor is 1;
 *   - ties in score are broken by the lower expert index, for membership and for order;
 *     the chosen experts are listed in (score descending, index ascending) order;
 *   - y = shared(x) + sum_j g_j E_{sel_j}(x).
 * Everything is evaluated in IEEE double with no rounding of intermediates; bf16 inputs
 * are widened exactly.
 */
#ifndef FLINT_MOE_ORACLE_H
#define FLINT_MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int H;                          /* hidden size */
  int E;                          /* routed experts */
  int k;                          /* experts chosen per token */
  int I;                          /* routed expert width */
  int Is;                         /* shared expert width */
  const uint16_t* w_router;       /* bf16 bits [H][E] */
  const float* router_bias;       /* [E] or NULL */
  const uint16_t* const* w_gate;  /* E pointers, each bf16 [H][I]; NULL = not supplied */
  const uint16_t* const* w_up;    /* E pointers, each bf16 [H][I] */
  const uint16_t* const* w_down;  /* E pointers, each bf16 [I][H] */
  const uint16_t* ws_gate;        /* bf16 [H][Is] */
  const uint16_t* ws_up;          /* bf16 [H][Is] */
  const uint16_t* ws_down;        /* bf16 [Is][H] */
} oracle_layer;

/* Error codes (0 = ok). */
#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_EMISSING_EXPERT 2

double oracle_bf16_to_f64(uint16_t bits);

/* logits[t][e] = sum_h x[t][h] Wr[h][e] + b[e];  s[t][e] = 1 / (1 + exp(-logits)). */
int oracle_router(const double* x, int T, int H, int E, const uint16_t* w_router,
                  const float* bias, double* logits, double* scores);

/* One token: the first k experts in (score desc, index asc) order, their normalised
 * gates, and gaps[j] = s_(j) - s_(j+1) for j = 0..k-1 (gaps[k-1] is the k-th minus the
 * (k+1)-th score, or +inf when k == E). */
int oracle_select(const double* scores, int E, int k, int32_t* idx, double* gates, double* gaps);

/* One SwiGLU MLP on one row: out = (silu(x Wg) * (x Wu)) Wd.  Wg, Wu: [H][I]; Wd: [I][H].
 * hbuf: scratch of I doubles. */
void oracle_swiglu(const double* x, int H, int I, const uint16_t* wg, const uint16_t* wu,
                   const uint16_t* wd, double* out, double* hbuf);

/* The whole layer on T rows of x ([T][H], double).  y: [T][H].  Optional outputs (may be
 * NULL): idx [T][k], gates [T][k], gaps [T][k], scores [T][E]. */
int oracle_moe_forward(const oracle_layer* L, const double* x, int T, double* y,
                       int32_t* idx, double* gates, double* gaps, double* scores);

/* Same layer with the chosen experts given (idx [T][k]) instead of selected: gates are the
 * fp64 scores of the given experts normalised over them.  Used to re-evaluate tokens whose
 * top-k is decided by a near tie. */
int oracle_moe_forward_given(const oracle_layer* L, const double* x, int T, const int32_t* idx,
                             double* y);

/* Stable counting sort of the (token, slot) pairs by expert.  idx: [T][k].
 * counts[E]; offsets[E+1] (exclusive scan); perm[T*k]: sorted row -> pair t*k+j;
 * inv[T*k]: pair -> sorted row.  Pairs of one expert keep (t, j) order. */
int oracle_permute(const int32_t* idx, int T, int k, int E, int32_t* counts, int32_t* offsets,
                   int32_t* perm, int32_t* inv);

/* v rounded to the nearest bfloat16 value (ties to even). */
double oracle_round_bf16(double v);

/* r[t] = x[t] / sqrt(mean_h x[t][h]^2 + eps)  (unit weight). */
void oracle_rmsnorm(const double* x, int T, int H, double eps, double* r);

/* NVFP4 weights (the pages' four-bit builds: news article "Recursive opens Flint, a 40B coding
 * model with 2.5B active", section "Built with the Eureka Machine"; the format's published
 * definition): every element is an FP4 E2M1 code (sign, 2 exponent bits with bias 1, 1 mantissa
 * bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), every 16 consecutive elements along the
 * contraction dimension share one FP8 E4M3 scale (sign, 4 exponent bits with bias 7, 3 mantissa
 * bits; no infinities, 0x7F / 0xFF are NaN; largest 448), and the tensor has one fp32 scale:
 * value = e2m1 * e4m3 * tensor_scale. */
double oracle_e2m1_to_f64(unsigned code);  /* low 4 bits */
double oracle_e4m3_to_f64(unsigned byte);
/* W [K][N] (the math orientation y = x W) from the K-major encoding: codes [N][K/2] (byte
 * (n, j): W[2j][n] in the low nibble, W[2j+1][n] in the high), scales [N][K/16] (E4M3 bytes; the
 * scale of W[16g .. 16g+15][n]) and the tensor scale; out [K][N].  K % 16 == 0. */
int oracle_nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, float tensor_scale, int K, int N,
                         double* out);

/* Decode attention of one sliding-window layer (serving-kit post, "The architecture, from the
 * config": 32 query heads, 4 KV heads, head dimension 128; sliding-window layers attend to a
 * 513-token window, the current token plus 512 back; learned per-head attention sinks; news
 * article "Recursive opens Flint, a 40B coding model with 2.5B active", section "What runs on
 * each token": a sink is a slot that can take attention no real token needs).  Readings: the
 * sink of head h is a logit that joins the softmax denominator and carries no value; scores
 * are q.k / sqrt(head_dim); query head h reads KV head h / (n_heads / n_kv); q and k arrive
 * normalised and rotated (the per-head QK RMSNorm and RoPE belong to the projections).
 * The cache of each sequence is a ring of W slots holding its last W tokens (position p in
 * slot p mod W); with pos[b] the position of the sequence's current token (its K and V
 * already stored), the valid slots are 0 .. min(pos[b] + 1, W) - 1.
 *   q [B][nh][d], k, v [B][W][nkv][d] (bf16 bits), sinks [nh], pos [B]; out [B][nh][d]:
 *   out[b][h] = sum_j e^(s_j - m) v_j / (e^(sink_h - m) + sum_j e^(s_j - m)), m = max(sink_h, s_j). */
int oracle_swa_decode(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* sinks,
                      const int32_t* pos, int B, int nh, int nkv, int d, int W, double* out);

#ifdef __cplusplus
}
#endif
#endif

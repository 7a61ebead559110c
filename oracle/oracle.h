/*
 * Oracle of the routed mixture-of-experts feed-forward step over Q8_0 weights.
 *
 * TEST INFRASTRUCTURE ONLY. This plain, single-threaded C code in fp64 is what
 * the CUDA library is checked against. Only the tests, the smoke check and the
 * bench's CPU-baseline leg may load it; the library never does, and the two
 * share no source, header, table or helper.
 *
 * What the step computes. The pages (the Flyweight README, "flyweight-llm"
 * 0.2.0 and 0.5.1, §Features "sparse MoE execution" and §Quantization, and
 * the vOOM README's notes on routers, top-k and SwiGLU experts) name the
 * pieces but print no formula. The plainest reading, used throughout:
 *
 *   router      z[t,e] = sum_h x[t,h] * Wr[e,h] + b[e]           (fp32 inputs)
 *   selection   the k largest z[t,.], ties to the lower expert id, ordered by
 *               descending z (equal z: lower id first)
 *   gates       g[t,j] = softmax over all E of z[t,.], restricted to the k
 *               selected experts and renormalised to sum to 1
 *   expert e    y_e(x) = Wd_e ( SiLU(Wg_e x) * (Wu_e x) ),  SiLU(a) = a/(1+e^-a)
 *   output      out[t] = sum_j g[t,j] * y_{ids[t,j]}(x_t)  (+ y_shared(x_t))
 *
 * Q8_0 (named on the pages as a GGUF tensor format, §Quantization): each row of
 * a weight matrix is cut along its input (reduction) dimension into blocks of
 * 32 values stored as a little-endian IEEE binary16 scale d followed by 32
 * signed bytes q; the weight is d*q. Quantising: amax = max|w| over the block,
 * d = amax/127, q = round-half-away-from-zero(w/d) clamped to [-127, 127]; an
 * all-zero block stores d = 0 and q = 0.
 *
 * All arithmetic is fp64 and follows the definitions' own order (sums in
 * natural index order); every input (bf16, fp32, fp16*int8) converts to fp64
 * exactly.
 */
#ifndef FW_ORACLE_H
#define FW_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_Q8_0_BLOCK 32
#define ORACLE_Q8_0_BYTES 34

/* IEEE 754 binary16 and bfloat16 conversions, from the formats' definitions. */
double oracle_half_to_double(uint16_t h);
uint16_t oracle_double_to_half(double x); /* round to nearest even; subnormals kept; overflow -> inf */
double oracle_bf16_to_double(uint16_t b);

/* Q8_0: w is [rows][K] row-major fp32, K % 32 == 0; blocks is rows*(K/32)*34 bytes.
 * Returns 0, or -1 on bad sizes. */
int oracle_q8_0_quantize(const float *w, int64_t rows, int64_t K, uint8_t *blocks);
int oracle_q8_0_dequantize(const uint8_t *blocks, int64_t rows, int64_t K, double *w);

/* z [T][E] = x [T][H] (bf16 bits) * Wr[E][H]^T + bias[E] (bias may be NULL). */
void oracle_router_logits(const uint16_t *x, int64_t T, int64_t H, const float *Wr, const float *bias,
                          int64_t E, double *z);

/* ids [T][k], gates [T][k] from logits z [T][E]. */
void oracle_topk_gates(const double *z, int64_t T, int64_t E, int64_t k, int32_t *ids, double *gates);

/* The same gates by the literal route: full softmax over E, pick ids, divide by their sum. */
void oracle_gates_full_softmax(const double *z, int64_t T, int64_t E, int64_t k, const int32_t *ids,
                               double *gates);

/* Token-to-expert grouping of the T*k (token, slot) pairs, slot id s = t*k + j:
 * offsets [E+1] exclusive prefix sum of per-expert counts; perm [T*k] lists the
 * slot ids grouped by expert, ascending expert, and within an expert by
 * ascending token; inv [T*k] is the inverse (inv[perm[p]] = p). */
void oracle_permutation(const int32_t *ids, int64_t T, int64_t k, int64_t E, int32_t *offsets, int32_t *perm,
                        int32_t *inv);

/* One expert on one token: y[H] = Wd (SiLU(Wg x) * (Wu x)); wg, wu are [I][H]
 * Q8_0, wd is [H][I] Q8_0; x is fp64 [H]. */
void oracle_expert_ffn(const uint8_t *wg, const uint8_t *wu, const uint8_t *wd, int64_t H, int64_t I,
                       const double *x, double *y);

/* The whole step for T tokens. w_gate/w_up/w_down hold E+S pointers (S shared
 * experts at indices E..E+S-1); a routed entry may be NULL when no token selects
 * that expert. ids/gates may be NULL. out is fp64 [T][H].
 * Returns 0; -1 on bad sizes; -2 when a selected expert's weights are NULL. */
int oracle_moe_forward(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k, int64_t S, const uint16_t *x,
                       const float *Wr, const float *bias, const uint8_t *const *w_gate,
                       const uint8_t *const *w_up, const uint8_t *const *w_down, int32_t *ids, double *gates,
                       double *out);

/* The same output given already-made routing (ids, gates): used to time and to
 * check only the expert part. */
int oracle_moe_experts(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k, int64_t S, const uint16_t *x,
                       const int32_t *ids, const double *gates, const uint8_t *const *w_gate,
                       const uint8_t *const *w_up, const uint8_t *const *w_down, double *out);

/* Q8 activations (the Flyweight README, 0.2.0, §Quantization: Q8-activation
 * dp4a group-decode kernels, and §Current limitations: the int8 MMQ path;
 * the pages give no formula, and the reading used here is the Q8_0 rule
 * applied to an activation vector in fp32): v [n] fp32 is cut into blocks of
 * blk values (n % blk == 0); per block d = amax/127 and q =
 * round-half-away-from-zero(v/d) clamped to [-127, 127], the division and d
 * both in fp32 (an all-zero block: d = 0, q = 0). out [n] = q*d (exact in fp64);
 * q [n] and d [n/blk] may be NULL. Returns 0, -1 on bad sizes. */
int oracle_q8_activations(const float *v, int64_t n, int64_t blk, double *out, int8_t *q, float *d);

/* The expert part with Q8 activations: each token's x (bf16 -> fp32) through
 * oracle_q8_activations in blocks of 32 before the gate/up projections, and
 * each expert's h = SiLU(g)*u (rounded to fp32) in blocks of 16 before the
 * down projection; otherwise as oracle_moe_experts. */
int oracle_moe_experts_q8act(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k, int64_t S, const uint16_t *x,
                             const int32_t *ids, const double *gates, const uint8_t *const *w_gate,
                             const uint8_t *const *w_up, const uint8_t *const *w_down, double *out);

#ifdef __cplusplus
}
#endif
#endif

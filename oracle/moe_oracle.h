/*
 * moe_oracle.h -- plain fp64 CPU oracle of the MoE-layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  It shares no code with the GPU path.
 *
 * Every function is the plain definition of its step, written as sequential
 * loops in double precision (compiled with -ffp-contract=off, no SIMD
 * intrinsics).  Inputs are read-only host arrays owned by the caller; outputs
 * are caller-allocated host arrays.  Functions return 0 on success and a
 * negative code on bad arguments (-1) or a missing expert record (-2).
 *
 * Sources (page title, section):
 *   LazyLoRA README, "The engine": top-16 routing over 896 routed experts,
 *     MXFP4 experts, fp32 (here: fp64) expert accumulation;
 *   LazyLoRA README, "The engine": 2 shared experts in each MoE layer beside
 *     the routed ones;
 *   LazyLoRA README, "File map": the router (top-16 gating with a
 *     score-correction bias) and SiTU 4*tanh(g/4)*sigmoid(g) x 25*tanh(u/25);
 *   WASTE README, "3 bits per expert weight": RVQ with 3 stages of 256-entry
 *     codebooks over 8-dim vectors;
 *   "Running a 2.78-Trillion-Parameter Model Across Two Desks", Act II: the
 *     MoE layer returns the gate-weighted sum of the selected experts' outputs.
 *   MXFP4 element and scale encodings (E2M1, E8M0, blocks of 32) follow the OCP
 *   Microscaling Formats (MX) v1.0 specification; the pages only name MXFP4.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { OR_F32 = 0, OR_BF16 = 1, OR_F64 = 2 };
enum { OR_ACT_SWIGLU = 0, OR_ACT_SITU = 1 };

/* ---- element decodes ---------------------------------------------------- */
double or_e2m1(int code);            /* E2M1 code 0..15 -> value (code 8 is -0.0) */
double or_e8m0(int byte);            /* 2^(byte-127); byte 255 -> NaN            */
double or_bf16(uint16_t bits);       /* bfloat16 bit pattern -> value           */
double or_f16(uint16_t bits);        /* IEEE binary16 bit pattern -> value      */

/* ---- weight decodes ----------------------------------------------------- */
/* MXFP4 matrix [rows][K]: codes [rows][K/2] (low nibble = even column),
 * scales [rows][K/32] (one E8M0 per 32 consecutive columns).  Row r -> w[K]. */
void or_mxfp4_row(const uint8_t* codes, const uint8_t* scales, int K, int r, double* w);
/* RVQ3 matrix [rows][K]: codes [3][K/8][rows] (stage-planar, position-major:
 * code[s][v][r]), codebooks cb fp16 [3][256][8];
 * w[r][8v+i] = sum over stages s of cb[s][code[s][v][r]][i]. */
void or_rvq3_row(const uint8_t* codes, const uint16_t* cb, int rows, int K, int r, double* w);
/* The same weights from codes stored row by row, [3][rows][K/8] (the
 * row-major record layout, converted on the GPU side by moe_rvq3_repack):
 * stage s's code for weights r, 8v..8v+7 is codes[(s * rows + r) * (K/8) + v]. */
void or_rvq3_row_rowmajor(const uint8_t* codes, const uint16_t* cb, int rows, int K, int r, double* w);

/* Byte offsets of the three matrices inside one expert record. */
size_t or_mxfp4_record_bytes(int d, int ff);
size_t or_rvq3_record_bytes(int d, int ff);

/* ---- record checksum ------------------------------------------------------
 * CRC-32 (IEEE 802.3 generator, reflected, initial value and final xor all
 * ones: the zlib/PNG/Ethernet checksum) of n bytes.  WASTE README, "How it
 * works": every expert record carries a CRC32 of its payload, checked when
 * asked to verify. */
uint32_t or_crc32(const uint8_t* p, size_t n);

/* ---- router --------------------------------------------------------------
 * l[t][e] = sum_i W[e][i] x[t][i] (ascending i) + bias[e];
 * top-k by (l descending, e ascending); g_j = exp(l_j - l_max) / sum_sel exp(.)
 * logits (nullable) [T][E]; topk_idx [T][k]; gates [T][k]. */
int or_router(const void* x, int x_dtype, const void* w, int w_dtype, const float* bias, int T, int d, int E,
              int k, double* logits, int32_t* topk_idx, double* gates);
/* The same with a choice of where the bias enters: bias_mode 0 adds it to the
 * logits used for both the selection and the gates (or_router); bias_mode 1
 * (the score-correction reading: the bias steers which experts are chosen, not
 * how much they weigh) selects on l + bias but takes the gates from l alone,
 * g_j = exp(l_j - max_sel l) / sum_sel exp(l - max_sel l).  logits (nullable)
 * receives the selection keys l + bias. */
int or_router_mode(const void* x, int x_dtype, const void* w, int w_dtype, const float* bias, int bias_mode, int T,
                   int d, int E, int k, double* logits, int32_t* topk_idx, double* gates);
/* The top-k/gate step alone, on given fp64 logits [T][E]. */
int or_topk_gates(const double* logits, int T, int E, int k, int32_t* topk_idx, double* gates);

/* ---- bucketing -----------------------------------------------------------
 * Stable counting sort of pair ids p = t*k + j by expert topk_idx[p]:
 * counts [E], offsets [E+1] (exclusive scan), pair_ids [T*k]. */
int or_bucket(const int32_t* topk_idx, int T, int k, int E, int32_t* counts, int32_t* offsets,
              int32_t* pair_ids);

/* ---- one expert FFN for one token ---------------------------------------
 * g = Wg x, u = Wu x, h = act(g, u), y = Wd h; x [d] and y [d] in fp64. */
int or_expert_mxfp4(const double* x, const uint8_t* rec, int d, int ff, int act, double* y);
int or_expert_rvq3(const double* x, const uint8_t* rec, const uint16_t* cb_gate, const uint16_t* cb_up,
                   const uint16_t* cb_down, int d, int ff, int act, double* y);
/* The same expert on a record whose nine code planes are stored row by row:
 * gate [3][ff][d/8] | up [3][ff][d/8] | down [3][d][ff/8]. */
int or_expert_rvq3_rowmajor(const double* x, const uint8_t* rec, const uint16_t* cb_gate, const uint16_t* cb_up,
                            const uint16_t* cb_down, int d, int ff, int act, double* y);
double or_act(double g, double u, int act);

/* ---- combine ------------------------------------------------------------
 * out[t] = x[t] + sum_{j ascending, g[t][j] != 0} g[t][j] * y_pairs[t*k + j];
 * x_resid nullable (then out is the MoE delta alone). */
int or_combine(const double* x_resid, const double* y_pairs, const double* gates, int T, int k, int d,
               double* out);

/* ---- whole layer ---------------------------------------------------------
 * quant 0 = MXFP4, 1 = RVQ3.  records: array [E] of host pointers (NULL = the
 * expert's record is absent; routing a pair to it is an error, -2).
 * Outputs (each nullable): topk_idx [T][k], gates [T][k], y_delta [T][d] (the
 * MoE delta, combine with no residual) and out [T][d] (= x + delta).
 * Only tokens with token_mask[t] != 0 get expert outputs (token_mask nullable =
 * all tokens); rows of y_delta/out for other tokens are left untouched.
 * nthreads > 1 runs the independent (token, slot) pairs on that many OpenMP
 * threads; the arithmetic of each pair is unchanged. */
int or_layer_forward(const void* x, int x_dtype, const void* router_w, int w_dtype, const float* bias, int T,
                     int d, int ff, int E, int k, int act, int quant, const uint8_t* const* records,
                     const uint16_t* cb_gate, const uint16_t* cb_up, const uint16_t* cb_down,
                     const uint8_t* token_mask, int nthreads, int32_t* topk_idx, double* gates, double* y_delta,
                     double* out);

/* or_layer_forward with the bias mode of or_router_mode and n_shared shared
 * experts: records has E + n_shared entries, and records[E + s] is shared
 * expert s, which every token passes through with weight 1:
 *   out[t] = x[t] + sum_{j < k} g[t][j] y_{e_j}(x[t]) + sum_{s < n_shared} y_{E+s}(x[t]).
 * topk_idx and gates stay [T][k] (the routed part). */
int or_layer_forward_ex(const void* x, int x_dtype, const void* router_w, int w_dtype, const float* bias,
                        int bias_mode, int T, int d, int ff, int E, int k, int n_shared, int act, int quant,
                        const uint8_t* const* records, const uint16_t* cb_gate, const uint16_t* cb_up,
                        const uint16_t* cb_down, const uint8_t* token_mask, int nthreads, int32_t* topk_idx,
                        double* gates, double* y_delta, double* out);

/* Expert-parallel partial: like or_layer_forward's delta but summing only the
 * pairs whose expert lies in [e_begin, e_end), given the routing. */
int or_partial_delta(const void* x, int x_dtype, const int32_t* topk_idx, const double* gates, int T, int d,
                     int ff, int k, int act, int quant, const uint8_t* const* records, const uint16_t* cb_gate,
                     const uint16_t* cb_up, const uint16_t* cb_down, int e_begin, int e_end, double* delta);

/* ---- latent projections ---------------------------------------------------
 * LazyLoRA README, "The engine": the routed experts work in a latent space of
 * width d = 3584, entered by a projection from the model's hidden width and
 * left by a projection back; the page does not state K3's model width, so D
 * is a parameter.
 *   or_project: y[t][n] = sum_k W[n][k] * x[t][k], summed in ascending k in
 *     fp64 (W row-major [N][K]).
 *   or_round_bf16: the bf16 value nearest to v, ties to the even significand
 *     (bit pattern); overflow to infinity, NaN kept NaN.
 *   or_latent_forward: z = bf16(W_in x) (the latent activation enters the
 *     experts in bf16, as every layer input does), u = the MoE delta of z
 *     (or_layer_forward_ex without the residual), out = x + W_out u, for
 *     W_in [d][D] and W_out [D][d].  z_bits (nullable) receives z's bf16
 *     bits [T][d], out (nullable) the result [T][D]. */
int or_project(const void* x, int x_dtype, const void* w, int w_dtype, int T, int K, int N, double* y);
uint16_t or_round_bf16(double v);
int or_latent_forward(const void* x, int x_dtype, const void* w_in, const void* w_out, int w_dtype, int D,
                      const void* router_w, int router_dtype, const float* bias, int bias_mode, int T, int d, int ff,
                      int E, int k, int n_shared, int act, int quant, const uint8_t* const* records,
                      const uint16_t* cb_gate, const uint16_t* cb_up, const uint16_t* cb_down, int nthreads,
                      uint16_t* z_bits, double* out);

#ifdef __cplusplus
}
#endif
#endif /* MOE_ORACLE_H */

/*
 * moe_oracle.c -- plain fp64 CPU oracle of the MoE-layer forward.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product path.  See moe_oracle.h
 * for the definitions and their sources.  Build: gcc -std=c11 -O2
 * -ffp-contract=off [-fopenmp]; no SIMD intrinsics.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Element decodes                                                           */
/* ------------------------------------------------------------------------ */

/* OCP MX v1.0 E2M1: sign s = bit 3, exponent e = bits 2..1 (bias 1), mantissa
 * m = bit 0.  e == 0 is subnormal: 0.5*m; otherwise 2^(e-1) * (1 + m/2).
 * Magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}. */
double or_e2m1(int code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* OCP MX v1.0 E8M0 scale: 2^(byte - 127); 0xFF encodes NaN. */
double or_e8m0(int byte) { return byte == 255 ? NAN : ldexp(1.0, byte - 127); }

double or_bf16(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

double or_f16(uint16_t bits) {
  int s = bits >> 15, e = (bits >> 10) & 31, m = bits & 1023;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp(1024.0 + m, e - 25);
  return s ? -v : v;
}

static double load_val(const void* p, int dtype, size_t i) {
  if (dtype == OR_BF16) return or_bf16(((const uint16_t*)p)[i]);
  if (dtype == OR_F64) return ((const double*)p)[i];
  return (double)((const float*)p)[i];
}

/* ------------------------------------------------------------------------ */
/* Weight decodes                                                            */
/* ------------------------------------------------------------------------ */

void or_mxfp4_row(const uint8_t* codes, const uint8_t* scales, int K, int r, double* w) {
  const uint8_t* cr = codes + (size_t)r * (size_t)(K / 2);
  const uint8_t* sr = scales + (size_t)r * (size_t)(K / 32);
  for (int c = 0; c < K; ++c) {
    uint8_t byte = cr[c / 2];
    int code = (c % 2 == 0) ? (byte & 15) : (byte >> 4);
    w[c] = or_e2m1(code) * or_e8m0(sr[c / 32]);
  }
}

void or_rvq3_row(const uint8_t* codes, const uint16_t* cb, int rows, int K, int r, double* w) {
  int nv = K / 8;
  for (int v = 0; v < nv; ++v) {
    for (int i = 0; i < 8; ++i) {
      double acc = 0.0;
      for (int s = 0; s < 3; ++s) {
        int c = codes[((size_t)s * nv + v) * rows + r];
        acc += or_f16(cb[((size_t)s * 256 + c) * 8 + i]);
      }
      w[8 * v + i] = acc;
    }
  }
}

/* The same weights when each stage's codes are stored row by row: plane
 * [3][rows][K/8], stage s's code for weights r, 8v..8v+7 at
 * codes[(s * rows + r) * nv + v]. */
void or_rvq3_row_rowmajor(const uint8_t* codes, const uint16_t* cb, int rows, int K, int r, double* w) {
  int nv = K / 8;
  for (int v = 0; v < nv; ++v) {
    for (int i = 0; i < 8; ++i) {
      double acc = 0.0;
      for (int s = 0; s < 3; ++s) {
        int c = codes[((size_t)s * rows + r) * nv + v];
        acc += or_f16(cb[((size_t)s * 256 + c) * 8 + i]);
      }
      w[8 * v + i] = acc;
    }
  }
}

size_t or_mxfp4_record_bytes(int d, int ff) {
  return 3 * ((size_t)ff * d / 2 + (size_t)ff * d / 32);
}

size_t or_rvq3_record_bytes(int d, int ff) { return 9 * (size_t)ff * d / 8; }

/* ------------------------------------------------------------------------ */
/* Record checksum                                                           */
/* ------------------------------------------------------------------------ */

/* CRC-32 of the IEEE 802.3 / zlib kind: the bytes enter least significant bit
 * first into a 32-bit register that starts as all ones; each bit shifts the
 * register right and, when the bit shifted out differs from the input bit,
 * xors in the reflected generator 0xEDB88320; the result is the register
 * complemented.  One bit at a time, exactly as defined. */
uint32_t or_crc32(const uint8_t* p, size_t n) {
  uint32_t reg = 0xFFFFFFFFu;
  for (size_t i = 0; i < n; ++i) {
    for (int b = 0; b < 8; ++b) {
      const uint32_t in = (p[i] >> b) & 1u;
      const uint32_t out = reg & 1u;
      reg >>= 1;
      if (in != out) reg ^= 0xEDB88320u;
    }
  }
  return reg ^ 0xFFFFFFFFu;
}

/* ------------------------------------------------------------------------ */
/* Router                                                                    */
/* ------------------------------------------------------------------------ */

/* Top-k on the selection keys, gates from gate_logits (the same array unless
 * the bias takes part in the selection only). */
static int topk_select_gates(const double* keys, const double* gate_logits, int T, int E, int k, int32_t* topk_idx,
                             double* gates) {
  if (T < 0 || E <= 0 || k <= 0 || k > E) return -1;
  unsigned char* taken = (unsigned char*)malloc((size_t)E);
  if (!taken) return -1;
  for (int t = 0; t < T; ++t) {
    const double* l = keys + (size_t)t * E;
    const double* gl = gate_logits + (size_t)t * E;
    int32_t* sel = topk_idx + (size_t)t * k;
    memset(taken, 0, (size_t)E);
    /* k rounds of arg-max; a strictly greater value wins, so among equal values
     * the lowest expert index (scanned first) is kept. */
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e;
      }
      taken[best] = 1;
      sel[j] = best;
    }
    /* Softmax over all E experts restricted to the selected ones and
     * renormalised equals the softmax over the selected logits alone; the
     * largest selected gate logit is subtracted before exp. */
    double lmax = gl[sel[0]];
    for (int j = 1; j < k; ++j)
      if (gl[sel[j]] > lmax) lmax = gl[sel[j]];
    double den = 0.0;
    for (int j = 0; j < k; ++j) den += exp(gl[sel[j]] - lmax);
    for (int j = 0; j < k; ++j) gates[(size_t)t * k + j] = exp(gl[sel[j]] - lmax) / den;
  }
  free(taken);
  return 0;
}

int or_topk_gates(const double* logits, int T, int E, int k, int32_t* topk_idx, double* gates) {
  return topk_select_gates(logits, logits, T, E, k, topk_idx, gates);
}

int or_router_mode(const void* x, int x_dtype, const void* w, int w_dtype, const float* bias, int bias_mode, int T,
                   int d, int E, int k, double* logits, int32_t* topk_idx, double* gates) {
  if (T < 0 || d <= 0 || E <= 0 || k <= 0 || k > E || (bias_mode != 0 && bias_mode != 1)) return -1;
  const size_t n = (size_t)(T > 0 ? T : 1) * E;
  double* l = logits ? logits : (double*)malloc(sizeof(double) * n);
  double* plain = bias_mode == 1 ? (double*)malloc(sizeof(double) * n) : NULL;
  int rc = -1;
  if (!l || (bias_mode == 1 && !plain)) goto done;
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double s = 0.0;
      for (int i = 0; i < d; ++i)
        s += load_val(w, w_dtype, (size_t)e * d + i) * load_val(x, x_dtype, (size_t)t * d + i);
      if (plain) plain[(size_t)t * E + e] = s;
      if (bias) s += (double)bias[e];
      l[(size_t)t * E + e] = s;
    }
  }
  rc = topk_select_gates(l, plain ? plain : l, T, E, k, topk_idx, gates);
done:
  if (!logits) free(l);
  free(plain);
  return rc;
}

int or_router(const void* x, int x_dtype, const void* w, int w_dtype, const float* bias, int T, int d, int E,
              int k, double* logits, int32_t* topk_idx, double* gates) {
  return or_router_mode(x, x_dtype, w, w_dtype, bias, 0, T, d, E, k, logits, topk_idx, gates);
}

/* ------------------------------------------------------------------------ */
/* Bucketing                                                                 */
/* ------------------------------------------------------------------------ */

int or_bucket(const int32_t* topk_idx, int T, int k, int E, int32_t* counts, int32_t* offsets,
              int32_t* pair_ids) {
  int P = T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int p = 0; p < P; ++p) {
    int e = topk_idx[p];
    if (e < 0 || e >= E) return -1;
    counts[e] += 1;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  if (!fill) return -1;
  for (int e = 0; e < E; ++e) fill[e] = offsets[e];
  for (int p = 0; p < P; ++p) pair_ids[fill[topk_idx[p]]++] = p; /* ascending p: stable */
  free(fill);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Expert FFN                                                                */
/* ------------------------------------------------------------------------ */

static double sigmoid(double g) { return 1.0 / (1.0 + exp(-g)); }

double or_act(double g, double u, int act) {
  if (act == OR_ACT_SITU) /* LazyLoRA README, "File map": SiTU */
    return 4.0 * tanh(g / 4.0) * sigmoid(g) * 25.0 * tanh(u / 25.0);
  return g * sigmoid(g) * u; /* SwiGLU: silu(g) * u */
}

static double dot(const double* a, const double* b, int n) {
  double s = 0.0;
  for (int i = 0; i < n; ++i) s += a[i] * b[i];
  return s;
}

int or_expert_mxfp4(const double* x, const uint8_t* rec, int d, int ff, int act, double* y) {
  if (!rec) return -2;
  size_t cb = (size_t)ff * d / 2, sb = (size_t)ff * d / 32;
  const uint8_t* g_codes = rec;
  const uint8_t* g_scales = g_codes + cb;
  const uint8_t* u_codes = g_scales + sb;
  const uint8_t* u_scales = u_codes + cb;
  const uint8_t* d_codes = u_scales + sb;
  const uint8_t* d_scales = d_codes + cb;
  int n = d > ff ? d : ff;
  double* w = (double*)malloc(sizeof(double) * (size_t)n);
  double* h = (double*)malloc(sizeof(double) * (size_t)ff);
  if (!w || !h) {
    free(w);
    free(h);
    return -1;
  }
  for (int r = 0; r < ff; ++r) {
    or_mxfp4_row(g_codes, g_scales, d, r, w);
    double g = dot(w, x, d);
    or_mxfp4_row(u_codes, u_scales, d, r, w);
    double u = dot(w, x, d);
    h[r] = or_act(g, u, act);
  }
  for (int r = 0; r < d; ++r) {
    or_mxfp4_row(d_codes, d_scales, ff, r, w);
    y[r] = dot(w, h, ff);
  }
  free(w);
  free(h);
  return 0;
}

/* The RVQ3 expert on a record whose planes are stored position-major
 * (row_major == 0) or row by row (row_major == 1). */
static int expert_rvq3_layout(const double* x, const uint8_t* rec, const uint16_t* cb_gate, const uint16_t* cb_up,
                              const uint16_t* cb_down, int d, int ff, int act, int row_major, double* y) {
  if (!rec) return -2;
  size_t mb = 3 * (size_t)ff * d / 8;
  const uint8_t* g_codes = rec;
  const uint8_t* u_codes = rec + mb;
  const uint8_t* d_codes = rec + 2 * mb;
  void (*row)(const uint8_t*, const uint16_t*, int, int, int, double*) = row_major ? or_rvq3_row_rowmajor : or_rvq3_row;
  int n = d > ff ? d : ff;
  double* w = (double*)malloc(sizeof(double) * (size_t)n);
  double* h = (double*)malloc(sizeof(double) * (size_t)ff);
  if (!w || !h) {
    free(w);
    free(h);
    return -1;
  }
  for (int r = 0; r < ff; ++r) {
    row(g_codes, cb_gate, ff, d, r, w);
    double g = dot(w, x, d);
    row(u_codes, cb_up, ff, d, r, w);
    double u = dot(w, x, d);
    h[r] = or_act(g, u, act);
  }
  for (int r = 0; r < d; ++r) {
    row(d_codes, cb_down, d, ff, r, w);
    y[r] = dot(w, h, ff);
  }
  free(w);
  free(h);
  return 0;
}

int or_expert_rvq3(const double* x, const uint8_t* rec, const uint16_t* cb_gate, const uint16_t* cb_up,
                   const uint16_t* cb_down, int d, int ff, int act, double* y) {
  return expert_rvq3_layout(x, rec, cb_gate, cb_up, cb_down, d, ff, act, 0, y);
}

int or_expert_rvq3_rowmajor(const double* x, const uint8_t* rec, const uint16_t* cb_gate, const uint16_t* cb_up,
                            const uint16_t* cb_down, int d, int ff, int act, double* y) {
  return expert_rvq3_layout(x, rec, cb_gate, cb_up, cb_down, d, ff, act, 1, y);
}

/* ------------------------------------------------------------------------ */
/* Combine                                                                   */
/* ------------------------------------------------------------------------ */

int or_combine(const double* x_resid, const double* y_pairs, const double* gates, int T, int k, int d,
               double* out) {
  for (int t = 0; t < T; ++t) {
    for (int i = 0; i < d; ++i) {
      double s = 0.0;
      for (int j = 0; j < k; ++j) {
        double g = gates[(size_t)t * k + j];
        if (g != 0.0) s += g * y_pairs[((size_t)t * k + j) * d + i];
      }
      out[(size_t)t * d + i] = (x_resid ? x_resid[(size_t)t * d + i] : 0.0) + s;
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Whole layer                                                               */
/* ------------------------------------------------------------------------ */

static int run_expert(const double* xt, int quant, const uint8_t* rec, const uint16_t* cbg, const uint16_t* cbu,
                      const uint16_t* cbd, int d, int ff, int act, double* y) {
  if (quant == 0) return or_expert_mxfp4(xt, rec, d, ff, act, y);
  return or_expert_rvq3(xt, rec, cbg, cbu, cbd, d, ff, act, y);
}

/* Per-pair expert outputs for the given pairs; a pair with gate 0 contributes
 * nothing to the combine, so its expert is not evaluated (its record may be
 * absent or hold anything). */
static int pair_outputs(const void* x, int x_dtype, const int32_t* topk_idx, const double* gates, int T, int d,
                        int ff, int k, int act, int quant, const uint8_t* const* records, const uint16_t* cbg,
                        const uint16_t* cbu, const uint16_t* cbd, const uint8_t* token_mask, int e_begin,
                        int e_end, int nthreads, double* y_pairs) {
  int P = T * k;
  int rc = 0;
  (void)nthreads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1) reduction(min : rc)
  for (int p = 0; p < P; ++p) {
    int t = p / k;
    int e = topk_idx[p];
    double* y = y_pairs + (size_t)p * d;
    for (int i = 0; i < d; ++i) y[i] = 0.0;
    if ((token_mask && !token_mask[t]) || gates[p] == 0.0 || e < e_begin || e >= e_end) continue;
    double* xt = (double*)malloc(sizeof(double) * (size_t)d);
    if (!xt) {
      rc = -1;
      continue;
    }
    for (int i = 0; i < d; ++i) xt[i] = load_val(x, x_dtype, (size_t)t * d + i);
    int r = run_expert(xt, quant, records[e], cbg, cbu, cbd, d, ff, act, y);
    if (r < rc) rc = r;
    free(xt);
  }
  return rc;
}

int or_layer_forward_ex(const void* x, int x_dtype, const void* router_w, int w_dtype, const float* bias,
                        int bias_mode, int T, int d, int ff, int E, int k, int n_shared, int act, int quant,
                        const uint8_t* const* records, const uint16_t* cb_gate, const uint16_t* cb_up,
                        const uint16_t* cb_down, const uint8_t* token_mask, int nthreads, int32_t* topk_idx,
                        double* gates, double* y_delta, double* out) {
  if (T < 0 || d <= 0 || ff <= 0 || E <= 0 || k <= 0 || k > E || n_shared < 0 || (d % 32) || (ff % 32)) return -1;
  /* Every token's pairs: the k routed experts with their gates, then the
   * n_shared shared experts (records E .. E + n_shared - 1) with weight 1. */
  const int ks = k + n_shared;
  size_t P = (size_t)T * k, Ps = (size_t)T * ks;
  int32_t* idx = topk_idx ? topk_idx : (int32_t*)malloc(sizeof(int32_t) * (P ? P : 1));
  double* g = gates ? gates : (double*)malloc(sizeof(double) * (P ? P : 1));
  int32_t* idx_s = (int32_t*)malloc(sizeof(int32_t) * (Ps ? Ps : 1));
  double* g_s = (double*)malloc(sizeof(double) * (Ps ? Ps : 1));
  double* yp = (double*)malloc(sizeof(double) * (Ps ? Ps : 1) * d);
  double* delta = (double*)malloc(sizeof(double) * (size_t)(T ? T : 1) * d);
  int rc = -1;
  if (!idx || !g || !idx_s || !g_s || !yp || !delta) goto done;
  rc = or_router_mode(x, x_dtype, router_w, w_dtype, bias, bias_mode, T, d, E, k, NULL, idx, g);
  if (rc) goto done;
  for (int t = 0; t < T; ++t) {
    for (int j = 0; j < ks; ++j) {
      idx_s[(size_t)t * ks + j] = j < k ? idx[(size_t)t * k + j] : E + (j - k);
      g_s[(size_t)t * ks + j] = j < k ? g[(size_t)t * k + j] : 1.0;
    }
  }
  rc = pair_outputs(x, x_dtype, idx_s, g_s, T, d, ff, ks, act, quant, records, cb_gate, cb_up, cb_down, token_mask,
                    0, E + n_shared, nthreads, yp);
  if (rc) goto done;
  or_combine(NULL, yp, g_s, T, ks, d, delta);
  for (int t = 0; t < T; ++t) {
    if (token_mask && !token_mask[t]) continue;
    for (int i = 0; i < d; ++i) {
      double dv = delta[(size_t)t * d + i];
      if (y_delta) y_delta[(size_t)t * d + i] = dv;
      if (out) out[(size_t)t * d + i] = load_val(x, x_dtype, (size_t)t * d + i) + dv;
    }
  }
done:
  if (!topk_idx) free(idx);
  if (!gates) free(g);
  free(idx_s);
  free(g_s);
  free(yp);
  free(delta);
  return rc;
}

int or_layer_forward(const void* x, int x_dtype, const void* router_w, int w_dtype, const float* bias, int T,
                     int d, int ff, int E, int k, int act, int quant, const uint8_t* const* records,
                     const uint16_t* cb_gate, const uint16_t* cb_up, const uint16_t* cb_down,
                     const uint8_t* token_mask, int nthreads, int32_t* topk_idx, double* gates, double* y_delta,
                     double* out) {
  return or_layer_forward_ex(x, x_dtype, router_w, w_dtype, bias, 0, T, d, ff, E, k, 0, act, quant, records, cb_gate,
                             cb_up, cb_down, token_mask, nthreads, topk_idx, gates, y_delta, out);
}

int or_partial_delta(const void* x, int x_dtype, const int32_t* topk_idx, const double* gates, int T, int d,
                     int ff, int k, int act, int quant, const uint8_t* const* records, const uint16_t* cb_gate,
                     const uint16_t* cb_up, const uint16_t* cb_down, int e_begin, int e_end, double* delta) {
  size_t P = (size_t)T * k;
  double* yp = (double*)malloc(sizeof(double) * (P ? P : 1) * d);
  if (!yp) return -1;
  int rc = pair_outputs(x, x_dtype, topk_idx, gates, T, d, ff, k, act, quant, records, cb_gate, cb_up, cb_down,
                        NULL, e_begin, e_end, 1, yp);
  if (!rc) or_combine(NULL, yp, gates, T, k, d, delta);
  free(yp);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Latent projections                                                        */
/* ------------------------------------------------------------------------ */

int or_project(const void* x, int x_dtype, const void* w, int w_dtype, int T, int K, int N, double* y) {
  if (T < 0 || K <= 0 || N <= 0 || !x || !w || !y) return -1;
  for (int t = 0; t < T; ++t) {
    for (int n = 0; n < N; ++n) {
      double s = 0.0;
      for (int k = 0; k < K; ++k) s += load_val(w, w_dtype, (size_t)n * K + k) * load_val(x, x_dtype, (size_t)t * K + k);
      y[(size_t)t * N + n] = s;
    }
  }
  return 0;
}

/* bf16 keeps the sign, the 8 exponent bits and 7 fraction bits of a float:
 * the representable values around v are found from v's binary exponent, and
 * the nearer one is taken, the one with an even last bit on a tie. */
uint16_t or_round_bf16(double v) {
  if (v != v) return 0x7FC0;
  const int neg = v < 0 || (v == 0 && 1.0 / v < 0);
  double a = neg ? -v : v;
  uint16_t bits;
  if (a == 0.0) {
    bits = 0;
  } else {
    int e;
    frexp(a, &e);                    /* a = f * 2^e, f in [0.5, 1) */
    int q = e - 8;                   /* 8 significant bits: the spacing is 2^(e-8) */
    if (q < -133) q = -133;          /* below the normal range: the subnormal spacing 2^-133 */
    const double ulp = ldexp(1.0, q);
    double m = floor(a / ulp);       /* a / ulp is exact (a power of two divides) */
    const double rem = a - m * ulp;  /* exact */
    if (rem > 0.5 * ulp || (rem == 0.5 * ulp && fmod(m, 2.0) != 0.0)) m += 1.0;
    const double r = m * ulp;        /* the rounded magnitude */
    if (r >= ldexp(1.0, 128)) {
      bits = 0x7F80;                 /* infinity */
    } else {
      float f = (float)r;            /* r has at most 8 significant bits and is in range: exact */
      uint32_t u;
      memcpy(&u, &f, sizeof u);
      bits = (uint16_t)(u >> 16);
    }
  }
  return (uint16_t)(bits | (neg ? 0x8000 : 0));
}

int or_latent_forward(const void* x, int x_dtype, const void* w_in, const void* w_out, int w_dtype, int D,
                      const void* router_w, int router_dtype, const float* bias, int bias_mode, int T, int d, int ff,
                      int E, int k, int n_shared, int act, int quant, const uint8_t* const* records,
                      const uint16_t* cb_gate, const uint16_t* cb_up, const uint16_t* cb_down, int nthreads,
                      uint16_t* z_bits, double* out) {
  if (T < 0 || D <= 0 || d <= 0) return -1;
  const size_t nz = (size_t)(T ? T : 1) * d, nd = (size_t)(T ? T : 1) * D;
  double* z = (double*)malloc(sizeof(double) * nz);
  uint16_t* zb = (uint16_t*)malloc(sizeof(uint16_t) * nz);
  double* u = (double*)malloc(sizeof(double) * nz);
  double* back = (double*)malloc(sizeof(double) * nd);
  int rc = -1;
  if (!z || !zb || !u || !back) goto done;
  if ((rc = or_project(x, x_dtype, w_in, w_dtype, T, D, d, z)) != 0) goto done;
  for (size_t i = 0; i < (size_t)T * d; ++i) zb[i] = or_round_bf16(z[i]);
  if (z_bits) memcpy(z_bits, zb, sizeof(uint16_t) * (size_t)T * d);
  rc = or_layer_forward_ex(zb, OR_BF16, router_w, router_dtype, bias, bias_mode, T, d, ff, E, k, n_shared, act, quant,
                           records, cb_gate, cb_up, cb_down, NULL, nthreads, NULL, NULL, u, NULL);
  if (rc) goto done;
  if ((rc = or_project(u, OR_F64, w_out, w_dtype, T, d, D, back)) != 0) goto done;
  if (out)
    for (size_t i = 0; i < (size_t)T * D; ++i) out[i] = load_val(x, x_dtype, i) + back[i];
done:
  free(z);
  free(zb);
  free(u);
  free(back);
  return rc;
}
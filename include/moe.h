/*
 * moe.h -- C ABI of the GB300 (sm_103a) MoE-layer forward library, libmoe_gb300.so.
 *
 * The layer (Kimi-K3 shape: d = 3584 latent, ff = 3072, E = 896 routed experts,
 * top-16) runs in five steps, each one entry point below:
 *
 *   moe_route_topk       router logits, top-k selection, renormalised gates
 *   moe_bucket_tokens    group the (token, slot) pairs by expert
 *   moe_expert_ffn_mxfp4 / moe_expert_ffn_rvq3
 *                        decode each selected expert's gate/up/down matrices
 *                        from their compressed form inside the kernel and run
 *                        the SwiGLU (or SiTU) FFN with fp32 accumulation
 *   moe_combine          gate-weighted sum of the expert outputs, added to the
 *                        residual
 *   moe_layer_forward    the four steps chained on one stream
 *   moe_stack_forward    several layers chained, bf16 activations in between
 *
 * Sources (page title, section):
 *   - "Running a 2.78-Trillion-Parameter Model Across Two Desks", Act II: one
 *     activation vector per MoE layer goes in and the weighted sum of the
 *     selected experts' outputs comes back; 17.55 MB per MXFP4 expert; fp32
 *     compute with bf16 storage after a bf16 path failed its tolerance gate.
 *   - LazyLoRA README, "The engine": 896 routed experts per layer, top-16
 *     routing, MXFP4 expert weights, a fused decode-and-dot that never widens
 *     the packed weights, expert sums accumulated in fp32; "File map": the
 *     router's top-16 gating with a score-correction bias, and SiTU.
 *   - WASTE README, "3 bits per expert weight": residual vector quantisation
 *     with 3 stages of 256-entry codebooks over 8-dim vectors; "How it works":
 *     gate, up and down of one expert adjacent in one record; "What is this":
 *     an embeddable C API with an init-able config and status codes.
 *   - MXFP4 encodings follow the OCP Microscaling Formats (MX) v1.0
 *     specification (E2M1 elements, E8M0 scale per 32 elements).
 *
 * Conventions that hold for every call:
 *   - Every data pointer is a DEVICE pointer owned by the caller unless a
 *     comment says otherwise.  The library allocates nothing per call: scratch
 *     memory is the caller's workspace `ws` of `ws_bytes` bytes (256-byte
 *     aligned), sized with the matching moe_*_ws_bytes query.
 *   - Calls are asynchronous on `stream` and do not synchronise the host.
 *     They must be made with the context's device current.
 *   - Arguments are validated on the host first; a bad argument returns a
 *     status at once and launches nothing.  Problems only visible on the device
 *     (an out-of-range expert index in caller-supplied routing, a NULL record
 *     for an expert that tokens were routed to, a pipeline wait that timed out)
 *     set the context's device error word; the affected work is skipped, the
 *     call's outputs are then undefined, and moe_ctx_check reports the error.
 *     No weight is ever replaced by zeros or random values.
 *   - Activations (x, out), router weights and fp32 pair buffers must be
 *     16-byte aligned (they are read with vector loads); records and codebooks
 *     too.  A misaligned pointer is MOE_ERR_INVALID_ARG.
 *   - T = 0 is valid and launches nothing.
 *   - Limits: d and ff multiples of 32, 32 <= d, ff <= 4096; 1 <= k <= 32,
 *     k <= E <= 2048; T * k <= 2^24.  Larger shapes return MOE_ERR_UNSUPPORTED.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,      /* NULL pointer, bad shape, bad enum        */
  MOE_ERR_UNSUPPORTED = 2,      /* shape outside the limits above           */
  MOE_ERR_WORKSPACE = 3,        /* ws NULL, misaligned or too small         */
  MOE_ERR_CUDA = 4,             /* a CUDA runtime call failed               */
  MOE_ERR_BAD_EXPERT_INDEX = 5, /* routing named an expert outside [0, E)   */
  MOE_ERR_MISSING_EXPERT = 6,   /* a routed expert's record pointer is NULL */
  MOE_ERR_TIMEOUT = 7,          /* a bounded device-side wait gave up       */
  MOE_ERR_BAD_RECORD = 8        /* a record failed its check (moe_records_check) */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;
typedef enum { MOE_ACT_SWIGLU = 0, MOE_ACT_SITU = 1 } moe_act;
typedef enum { MOE_QUANT_MXFP4 = 0, MOE_QUANT_RVQ3 = 1 } moe_quant;
/* Where the router's score-correction bias enters (LazyLoRA README, "File
 * map": top-16 gating with a score-correction bias).  LOGIT: added to the
 * logits, so it moves both the selection and the gates.  SELECT: added to the
 * selection keys only; the gates are the renormalised softmax of the logits
 * without it. */
typedef enum { MOE_BIAS_LOGIT = 0, MOE_BIAS_SELECT = 1 } moe_bias_mode;

typedef struct moe_ctx moe_ctx;

/*
 * MXFP4 expert bank.  records: device array [E] of device pointers, one per
 * expert (NULL = absent), each 16-byte aligned, pointing at one contiguous
 * record of moe_mxfp4_record_bytes(d, ff) bytes laid out as
 *   gate.codes [ff][d/2] | gate.scales [ff][d/32] | up.codes [ff][d/2] |
 *   up.scales [ff][d/32] | down.codes [d][ff/2]   | down.scales [d][ff/32]
 * Matrices are row-major with the contraction axis contiguous: column c of a
 * row is the low nibble of byte c/2 when c is even and the high nibble when c
 * is odd; scale byte c/32 of the row (E8M0, value 2^(byte-127), 0xFF = NaN)
 * multiplies the 32 columns of that block.  Gate and up map d -> ff, down maps
 * ff -> d.  For d = 3584, ff = 3072 a record is 17,547,264 bytes and every
 * region starts on a 4 KiB multiple.
 */
typedef struct {
  const uint8_t* const* records;
  int d, ff, E;
} moe_mxfp4_experts;

/*
 * RVQ3 expert bank.  records: as above, each record moe_rvq3_record_bytes(d, ff)
 * bytes laid out stage-planar and position-major:
 *   gate.codes [3][d/8][ff] | up.codes [3][d/8][ff] | down.codes [3][ff/8][d]
 * i.e. code[s][v][r] is stage s's codebook index for weights r, 8v..8v+7 of
 * the matrix (rows contiguous for a fixed vector position).  codebooks[m] for
 * m = gate, up, down: device fp16 [3][256][8] (stage, entry, component).  The
 * weight is the sum of the three stages' codewords:
 *   w[r][8v+i] = cb[0][code[0][v][r]][i] + cb[1][code[1][v][r]][i] + cb[2][code[2][v][r]][i].
 * The three pointers may be equal (one codebook set per layer).
 */
typedef struct {
  const uint8_t* const* records;
  const uint16_t* codebooks[3];
  int d, ff, E;
} moe_rvq3_experts;

/* One MoE layer: router (W [E][d] row-major, optional fp32 score-correction
 * bias [E] entering as bias_mode says) and its expert bank.  The bank holds
 * E + n_shared records: records[0 .. E) are the routed experts and records[E + s]
 * is shared expert s, which every token passes through with weight 1
 * (LazyLoRA README, "The engine": 896 routed and 2 shared experts in each MoE
 * layer).  The bank's E field is E + n_shared; k + n_shared <= 32.  The shared
 * experts use the bank's quantisation (and, for RVQ3, its codebooks). */
typedef struct {
  int d, ff, E, k;
  moe_act act;
  moe_quant quant;
  const void* router_w;
  moe_dtype router_w_dtype;
  const float* router_bias; /* nullable */
  moe_mxfp4_experts mxfp4;  /* used when quant == MOE_QUANT_MXFP4 */
  moe_rvq3_experts rvq3;    /* used when quant == MOE_QUANT_RVQ3  */
  int n_shared;             /* shared experts after the routed ones (0: none) */
  moe_bias_mode bias_mode;  /* MOE_BIAS_LOGIT unless the bias steers the selection only */
} moe_layer;

/* ---- context ------------------------------------------------------------- */

MOE_API const char* moe_status_str(moe_status s);

/* Creates a context on `device` (allocates a 16-byte device error word; this and
 * moe_ctx_destroy are the only calls that allocate).  The caller's current
 * device is left unchanged. */
MOE_API moe_status moe_ctx_create(moe_ctx** ctx, int device);
MOE_API void moe_ctx_destroy(moe_ctx* ctx);

/* Synchronises `stream`, reads and clears the device error word.  Returns
 * MOE_OK or the first device-detected error since the last check; *detail (if
 * non-NULL) receives its detail (the offending expert index, or -1). */
MOE_API moe_status moe_ctx_check(moe_ctx* ctx, cudaStream_t stream, int* detail);

/* Router diagnostics: synchronises `stream` and returns (then clears) the
 * number of tokens whose top-k needed the fp64 recheck and the number of
 * logits that were recomputed by the sequential fp64 sum since the last call. */
MOE_API moe_status moe_ctx_stats(moe_ctx* ctx, cudaStream_t stream, long long* fp64_tokens, long long* seq_logits);

/* Per-launch timing, a diagnostic for benchmarks.  moe_ctx_profile(ctx, n)
 * with n > 0 creates 2n CUDA events (this allocates) and from then on every
 * kernel the context's calls launch is bracketed by an event pair on its
 * stream, up to n launches between reads; n = 0 turns it off and frees the
 * events.  moe_ctx_profile_read synchronises `stream`, then writes, per kernel
 * name in order of first launch, the name (NUL-terminated, 32 bytes per entry
 * in `names`), the launch count and the summed milliseconds, for at most
 * max_entries names; it clears the records and returns the number of entries
 * written, or minus a moe_status on error.  The event records sit between
 * launches, so the timed launches do not overlap their neighbours. */
MOE_API moe_status moe_ctx_profile(moe_ctx* ctx, int n);
MOE_API int moe_ctx_profile_read(moe_ctx* ctx, cudaStream_t stream, int max_entries, char* names, int* launches,
                                 double* total_ms);

/* Limit of the kernels' pipeline waits (a stage of weights arriving, a
 * partial sum being consumed), in nanoseconds; 0 restores the default of 2 s.
 * Values below 1000 are raised to 1000.  A wait that runs out records
 * MOE_ERR_TIMEOUT on the error word, the kernel skips its remaining work and
 * returns, and moe_ctx_check reports it; the context stays usable.  Waits
 * for a CTA's own copies and tensor-core operations in flight before it
 * leaves keep the 2 s limit whatever this setting.  Synchronous (it writes
 * the setting to the device); it applies to launches made after it returns.
 * Failure detection in the spirit of the pages' fail-loud checks (WASTE
 * README, "How it works"; LazyLoRA README, "How you know this is real"). */
MOE_API moe_status moe_ctx_set_wait_limit_ns(moe_ctx* ctx, unsigned long long ns);

/* Diagnostic: launches one wait on a barrier that nothing completes, through
 * the same bounded-wait helper as every pipeline wait, so that it runs out
 * after the context's wait limit and records MOE_ERR_TIMEOUT (detail -1).
 * Lets a caller check that timed-out waits return and are reported, without
 * any fault or hang.  Asynchronous on `stream`. */
MOE_API moe_status moe_ctx_wait_selftest(moe_ctx* ctx, cudaStream_t stream);

/* Library version string and the SM count the context sizes its grids for. */
MOE_API const char* moe_version(void);
MOE_API int moe_ctx_num_sms(const moe_ctx* ctx);

/* MXFP4 expert kernels (OCP MX v1.0 E2M1 codes with E8M0 scales per 32; the
 * pages' MXFP4 experts, LazyLoRA README "The engine"; batching, not caching,
 * is the lever, "Cost, measured").
 *   MOE_MXFP4_BLOCK_SCALED: every routed expert on the block-scaled tensor-core
 *     MMA: the record's codes and scale bytes are the A operand as stored; the
 *     activations enter as a sum of E4M3 terms with their own E8M0 scales (x:
 *     two terms, exactly the bf16 value; h: three terms, about 12 significant
 *     bits); products and sums in fp32.  Used when the activations are bf16,
 *     d and ff are multiples of 512, E <= 4096, the device has at most 160
 *     SMs and every routed record is 32-byte aligned (a misaligned record sets
 *     MOE_ERR_INVALID_ARG on the error word); otherwise the call falls back to
 *     the GEMV pair below.
 *   MOE_MXFP4_GEMV: every routed expert on the streaming GEMV pair (gate/up,
 *     then down): the weights are decoded in registers and multiplied on the
 *     warp-level MMA (bf16 activations) or by fused multiply-adds (fp32
 *     activations), every product exact and summed in fp32.
 *   MOE_MXFP4_AUTO (default): the GEMV pair for calls of one token, the
 *     block-scaled kernel for more (the faster of the two on a GB300 for
 *     each case).
 * All compute the same layer within the fp32 tolerance.  Other values return
 * MOE_ERR_INVALID_ARG.  moe_ctx_mxfp4_kernel returns the setting, or -1 for a
 * NULL context. */
typedef enum { MOE_MXFP4_BLOCK_SCALED = 0, MOE_MXFP4_GEMV = 1, MOE_MXFP4_AUTO = 2 } moe_mxfp4_kernel;
MOE_API moe_status moe_ctx_set_mxfp4_kernel(moe_ctx* ctx, int kernel);
MOE_API int moe_ctx_mxfp4_kernel(const moe_ctx* ctx);

/* ---- sizes ----------------------------------------------------------------- */

MOE_API size_t moe_mxfp4_record_bytes(int d, int ff);
MOE_API size_t moe_rvq3_record_bytes(int d, int ff);

/* Workspace bytes each call needs (0 if the shape is invalid). */
MOE_API size_t moe_route_topk_ws_bytes(int T, int d, int E, int k);
MOE_API size_t moe_bucket_tokens_ws_bytes(int T, int k, int E);
MOE_API size_t moe_expert_ffn_ws_bytes(int T, int k, int d, int ff, int E, moe_quant quant);
MOE_API size_t moe_layer_forward_ws_bytes(const moe_layer* L, int T);
MOE_API size_t moe_stack_forward_ws_bytes(const moe_layer* layers, int n_layers, int T);

/* ---- the steps ----------------------------------------------------------- */

/*
 * Router and top-k.  x [T][d] (x_dtype), router_w [E][d] (w_dtype), bias [E]
 * fp32 or NULL.  Writes topk_idx [T][k] (int32) and gates [T][k] (fp32).
 *   l[t][e] = sum_i W[e][i] * x[t][i] + bias[e]
 *   topk_idx[t][0..k) = the k largest l[t][.] ordered by (l descending, e
 *   ascending): an exact tie goes to the lower expert index;
 *   gates[t][j] = exp(l_j - l_0) / sum_j' exp(l_j' - l_0)  (softmax over all E
 *   experts restricted to the selected ones and renormalised).
 * Logits are accumulated in fp32 with a rigorous error bound per logit; where
 * the bound leaves the order of the selected experts or the k-th/(k+1)-th
 * boundary undecided, the candidates are recomputed in fp64 (and, if still
 * undecided, by a sequential fp64 sum in ascending i), so the selection equals
 * the one made on exact fp64 logits summed in ascending i.
 */
MOE_API moe_status moe_route_topk(moe_ctx* ctx, const void* x, moe_dtype x_dtype, const void* router_w, moe_dtype w_dtype,
                          const float* bias, int T, int d, int E, int k, int32_t* topk_idx, float* gates, void* ws,
                          size_t ws_bytes, cudaStream_t stream);

/*
 * moe_route_topk with a choice of bias mode (same arguments and workspace
 * otherwise).  MOE_BIAS_LOGIT is moe_route_topk.  MOE_BIAS_SELECT ranks the
 * experts by the key l[t][e] + bias[e] (ties to the lower index, certified as
 * above against keys summed in fp64 in ascending i and then biased) and sets
 *   gates[t][j] = exp(l_j - m) / sum_j' exp(l_j' - m),  m = max over the
 *   selected j of l_j,
 * with l the logits WITHOUT the bias.  An invalid bias_mode returns
 * MOE_ERR_INVALID_ARG.
 */
MOE_API moe_status moe_route_topk_ex(moe_ctx* ctx, const void* x, moe_dtype x_dtype, const void* router_w,
                                     moe_dtype w_dtype, const float* bias, moe_bias_mode bias_mode, int T, int d, int E,
                                     int k, int32_t* topk_idx, float* gates, void* ws, size_t ws_bytes,
                                     cudaStream_t stream);

/*
 * Bucketing: a stable counting sort of the pairs p = t*k + j by expert
 * topk_idx[p].  Writes counts [E] (pairs per expert), offsets [E+1] (exclusive
 * prefix sum, offsets[E] = T*k) and pair_ids [T*k] (pair ids grouped by expert
 * in ascending expert order, ascending p within an expert).  Counts come from
 * warp-aggregated shared-memory atomics; the slot order is deterministic.
 */
MOE_API moe_status moe_bucket_tokens(moe_ctx* ctx, const int32_t* topk_idx, int T, int k, int E, int32_t* counts,
                             int32_t* offsets, int32_t* pair_ids, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Expert FFN for every routed pair.  x [T][d] (x_dtype); offsets/pair_ids as
 * written by moe_bucket_tokens.  For the pair in slot s of expert e (token
 * t = pair_ids[s] / k):  g = Wg_e x_t, u = Wu_e x_t, h = act(g, u),
 * y = Wd_e h, written to y_pairs [T*k][d] (fp32) at row pair_ids[s].
 * act: SwiGLU h = silu(g) * u; SiTU h = 4 tanh(g/4) sigmoid(g) * 25 tanh(u/25).
 * Weights are decoded in registers / shared memory and never written back;
 * products and sums are fp32.
 */
MOE_API moe_status moe_expert_ffn_mxfp4(moe_ctx* ctx, const void* x, moe_dtype x_dtype, int T, int k,
                                const moe_mxfp4_experts* experts, moe_act act, const int32_t* offsets,
                                const int32_t* pair_ids, float* y_pairs, void* ws, size_t ws_bytes,
                                cudaStream_t stream);
MOE_API moe_status moe_expert_ffn_rvq3(moe_ctx* ctx, const void* x, moe_dtype x_dtype, int T, int k,
                               const moe_rvq3_experts* experts, moe_act act, const int32_t* offsets,
                               const int32_t* pair_ids, float* y_pairs, void* ws, size_t ws_bytes,
                               cudaStream_t stream);

/*
 * moe_expert_ffn_mxfp4 without a workspace, for callers that cannot allocate
 * device memory (an embedding framework or server that owns the allocator,
 * or code that must not allocate after start-up).  Same arguments as
 * moe_expert_ffn_mxfp4 minus the workspace.  Whatever the context's
 * moe_ctx_set_mxfp4_kernel setting, this call always runs the streaming GEMV
 * pair (MOE_MXFP4_GEMV), for any number of tokens; its outputs agree with
 * moe_expert_ffn_mxfp4's within the fp32 tolerance, and are bit-identical to
 * it when that call also runs the GEMV pair.  The scratch the GEMV pair keeps
 * between launches (the active-expert list, a per-token scale and the hidden
 * activations h, T*k*ff floats) lives in a static device array inside the
 * library, moe_expert_ffn_mxfp4_static_max_bytes() bytes (4 MiB) that every
 * GPU using the library reserves until the process exits.  Calls whose
 * scratch would not fit (about T*k*ff > 1,040,000; at ff = 3072 up to
 * T*k = 340 pairs) return MOE_ERR_UNSUPPORTED.  This call allocates nothing:
 * the first call on a device looks up the array's device address (once per
 * device), so make that first call before any stream capture.  Every call, on
 * every stream of a device, shares the one array and it keeps the last call's
 * contents: calls that overlap on the GPU race and give undefined results;
 * serialise them.  The source pages have no counterpart to this entry point.
 */
MOE_API moe_status moe_expert_ffn_mxfp4_static(moe_ctx* ctx, const void* x, moe_dtype x_dtype, int T, int k,
                                               const moe_mxfp4_experts* experts, moe_act act, const int32_t* offsets,
                                               const int32_t* pair_ids, float* y_pairs, cudaStream_t stream);
MOE_API size_t moe_expert_ffn_mxfp4_static_max_bytes(void);

/*
 * Combine: out[t][i] = x_resid[t][i] + sum over j ascending with gates[t][j] != 0
 * of gates[t][j] * y_pairs[t*k + j][i].  x_resid [T][d] (x_dtype) may be NULL
 * (out is then the MoE delta alone).  out [T][d] in out_dtype (bf16: the fp32
 * sum rounded to nearest even).  A pair with gate 0 never enters the sum, whatever
 * its row of y_pairs holds (NaN included); every row of y_pairs [T*k][d] may be read.
 */
MOE_API moe_status moe_combine(moe_ctx* ctx, const void* x_resid, moe_dtype x_dtype, const float* y_pairs,
                       const float* gates, int T, int k, int d, void* out, moe_dtype out_dtype, cudaStream_t stream);

/*
 * The whole layer: route, bucket, expert FFN, combine (with x as residual).
 * x [T][d] (x_dtype), out [T][d] (out_dtype; may not alias x).
 *   out[t] = x[t] + sum_{j < k} g[t][j] y_{e_j}(x[t]) + sum_{s < n_shared} y_{E+s}(x[t])
 * The optional outputs receive the pairs the layer evaluated when non-NULL:
 * topk_idx_out [T][k + n_shared] and gates_out [T][k + n_shared] (the routed
 * selection, then the shared experts E .. E + n_shared - 1 with gate 1) and
 * counts_out [E + n_shared] (tokens per expert).
 */
MOE_API moe_status moe_layer_forward(moe_ctx* ctx, const moe_layer* L, const void* x, moe_dtype x_dtype, int T, void* out,
                             moe_dtype out_dtype, int32_t* topk_idx_out, float* gates_out, int32_t* counts_out,
                             void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Several layers in sequence: layer l's output, rounded to bf16 (nearest
 * even), is layer l+1's input.  x [T][d] (x_dtype) feeds layer 0; out [T][d]
 * receives the last layer's output in out_dtype.  All layers share d.
 */
MOE_API moe_status moe_stack_forward(moe_ctx* ctx, const moe_layer* layers, int n_layers, const void* x, moe_dtype x_dtype,
                             int T, void* out, moe_dtype out_dtype, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Layer stack with its routing trace (LazyLoRA README, "How you know this is
 * real": the routing a run took is recorded so it can be checked; WASTE
 * README, "How it works").  As moe_stack_forward, and when non-NULL:
 *   topk_trace, gates_trace: layer l's pairs [T][k_l + n_shared_l] (routed
 *     selection, then the shared experts with gate 1), as moe_layer_forward's
 *     topk_idx_out / gates_out, concatenated over the layers in order (layer l
 *     starts at T * sum over l' < l of (k_l' + n_shared_l'));
 *   counts_trace: layer l's tokens per expert [E_l + n_shared_l], concatenated
 *     likewise.
 * Device buffers owned by the caller; every layer's part is written.
 */
MOE_API moe_status moe_stack_forward_ex(moe_ctx* ctx, const moe_layer* layers, int n_layers, const void* x,
                                        moe_dtype x_dtype, int T, void* out, moe_dtype out_dtype, int32_t* topk_trace,
                                        float* gates_trace, int32_t* counts_trace, void* ws, size_t ws_bytes,
                                        cudaStream_t stream);

/*
 * RVQ3 records from the row-major code layout to the position-major one that
 * moe_rvq3_experts reads (WASTE README, "3 bits per expert weight": three
 * 8-bit codes per 8 consecutive weights of a row).  Row-major record, each
 * plane [rows][K/8] with a row's codes contiguous:
 *   gate.codes [3][ff][d/8] | up.codes [3][ff][d/8] | down.codes [3][d][ff/8]
 * Each of the 9 planes is transposed to [K/8][rows]; the size,
 * moe_rvq3_record_bytes(d, ff), is unchanged.  src, dst: device arrays [n] of
 * device pointers to records (a record may not be converted in place: src[i]
 * == dst[i] sets MOE_ERR_INVALID_ARG on the error word with detail i, a NULL
 * pointer MOE_ERR_MISSING_EXPERT; that record is skipped).  Meant for load
 * time, outside any timed region; reads and writes every byte once.  n = 0 is
 * a no-op.
 */
MOE_API moe_status moe_rvq3_repack(moe_ctx* ctx, const uint8_t* const* src, uint8_t* const* dst, int n, int d, int ff,
                                   cudaStream_t stream);

/*
 * Experts beyond HBM ("Running a 2.78-Trillion-Parameter Model Across Two
 * Desks", Act II: experts split into tiers ranked by how often they are used;
 * Act III: an expert in no tier comes back as missing, never substituted;
 * WASTE README, "How it works": a bounded expert cache in front of the slow
 * store).  A tier owns one layer's record table: the hottest experts sit in
 * HBM slots, the others are read in place from page-locked host (Grace)
 * memory over NVLink-C2C by the same expert kernels (direct_host = 1), or
 * their table entry is NULL and a layer that routes to them reports
 * MOE_ERR_MISSING_EXPERT (direct_host = 0).
 *   E            records in the bank (a layer's E + n_shared)
 *   record_bytes bytes per record (a multiple of 16)
 *   host_records HOST array [E] of pointers to each expert's record in
 *                page-locked, mapped host memory (cudaHostAlloc, or
 *                cudaHostRegister with cudaHostRegisterMapped), 256-byte
 *                aligned; NULL: the expert has no host copy (it can only be
 *                resident if it is already in a slot -- it never is, so it
 *                is absent)
 *   slots        device memory for n_slots records, slot_stride bytes apart
 *                (a multiple of 256 >= record_bytes; 256-byte aligned)
 *   records      DEVICE array [E] the tier writes: the layer's record table
 *                (moe_mxfp4_experts.records / moe_rvq3_experts.records)
 *   direct_host  1: a non-resident expert's entry is its host copy; 0: NULL
 *   decay        heat[e] <- decay * heat[e] + counts[e] per observation, 0 < decay <= 1
 * All of this memory is the caller's and must outlive the tier.  moe_tier_create
 * allocates the tier's own bookkeeping (a device heat array [E] and page-locked
 * host staging), and writes the initial table (nothing resident).
 */
typedef struct moe_tier moe_tier;
typedef struct {
  int E;
  size_t record_bytes;
  const uint8_t* const* host_records;
  uint8_t* slots;
  int n_slots;
  size_t slot_stride;
  const uint8_t** records;
  int direct_host;
  float decay;
} moe_tier_desc;

MOE_API moe_status moe_tier_create(moe_ctx* ctx, const moe_tier_desc* desc, moe_tier** tier);
MOE_API void moe_tier_destroy(moe_tier* tier);

/* Adds one step's tokens per expert (device counts [E], as moe_layer_forward's
 * counts_out) into the decayed heat.  Asynchronous on `stream`. */
MOE_API moe_status moe_tier_observe(moe_tier* tier, const int32_t* counts, cudaStream_t stream);

/* Ranks the experts by heat (ties: an already resident expert, then the lower
 * id; see moe_tier_plan), keeps the n_slots hottest that have a host copy or
 * are resident, copies the newcomers into slots (evicting the coldest) and
 * rewrites the table.  Synchronises `stream` to read the heat, then enqueues
 * on it: the table entries of moved experts switched away from their slots,
 * one cudaMemcpyAsync per newcomer, the final table.  Run it on the stream the
 * layer runs on (or order the two with events): the copies overwrite evicted
 * slots.  *n_moved (nullable) receives the number of records copied. */
MOE_API moe_status moe_tier_rebalance(moe_tier* tier, cudaStream_t stream, int* n_moved);

/* Makes the n <= n_slots listed experts (host array) resident ahead of any
 * heat, in list order (a warm start, e.g. from an earlier run's counts);
 * experts already in other slots stay where those slots are free.
 * Synchronises `stream`, then enqueues as moe_tier_rebalance. */
MOE_API moe_status moe_tier_pin(moe_tier* tier, const int32_t* experts, int n, cudaStream_t stream);

/* Host copies of the residency (slot of each expert or -1; host [E], nullable)
 * and of the heat (host [E] floats, nullable; synchronous). */
MOE_API moe_status moe_tier_residency(const moe_tier* tier, int32_t* slot_of_expert, float* heat);

/* The ranking moe_tier_rebalance applies, as a pure host function: experts
 * that have a host copy (has_host[e] != 0) or a slot (slot_of[e] in [0,
 * n_slots)) are ordered by heat descending, then resident first, then id
 * ascending; the first n_slots are kept.  Kept residents stay in their slot;
 * the others take the free slots in ascending order.  Writes new_slot_of [E]
 * (slot or -1) and returns the number of experts that move into a slot, or -1
 * for a bad argument.  No GPU is used. */
MOE_API int moe_tier_plan(int E, int n_slots, const float* heat, const uint8_t* has_host, const int32_t* slot_of,
                          int32_t* new_slot_of);

/*
 * Latent projections (LazyLoRA README, "The engine": the routed experts work
 * in a latent space of width d = 3584, entered by a projection from the
 * model's hidden width D and left by a projection back; the page does not
 * state K3's hidden width, so D is a parameter).
 *
 * moe_project: y[t][n] = resid[t][n] + sum_k W[n][k] x[t][k] for t < T, n < N.
 *   x [T][K] (x_dtype), W [N][K] row-major (w_dtype), resid [T][N] (nullable,
 *   resid_dtype), y [T][N] (fp32, or bf16 rounded to nearest even).  Sums in
 *   fp32 (bf16 x bf16 products are exact in fp32).  K a multiple of 32; x and W
 *   16-byte aligned.  K, N <= 65536.
 *
 * moe_latent_layer_forward: the layer L run in its latent space (L->d is the
 * latent width) for a hidden-width input:
 *   z   = bf16(W_in x)                       W_in [d][D], the experts' input
 *   u   = the MoE delta of z: sum_j g_j y_j(z) + the shared experts (fp32)
 *   out = x + W_out u                        W_out [D][d]
 * x and out [T][D]; w_dtype bf16 or fp32 for both matrices; latent_out
 * (nullable, 16-byte aligned) receives z's bf16 bits [T][d].  ws:
 * moe_latent_layer_forward_ws_bytes(L, D, T) bytes.  D a multiple of 32.
 */
MOE_API moe_status moe_project(moe_ctx* ctx, const void* x, moe_dtype x_dtype, int T, int K, const void* w,
                               moe_dtype w_dtype, int N, const void* resid, moe_dtype resid_dtype, void* y,
                               moe_dtype y_dtype, cudaStream_t stream);
MOE_API size_t moe_latent_layer_forward_ws_bytes(const moe_layer* L, int D, int T);
MOE_API moe_status moe_latent_layer_forward(moe_ctx* ctx, const moe_layer* L, const void* w_in, const void* w_out,
                                            moe_dtype w_dtype, int D, const void* x, moe_dtype x_dtype, int T,
                                            void* out, moe_dtype out_dtype, uint16_t* latent_out, void* ws,
                                            size_t ws_bytes, cudaStream_t stream);

/*
 * Record check (WASTE README, "How it works": every expert record carries a
 * CRC32 of its payload, verified on request, so that a truncated or spliced
 * bank names the bad record instead of answering from wrong bytes).
 * records: device array [n] of device pointers to records of record_bytes
 * bytes each (a multiple of 16; every record 16-byte aligned).  Computes the
 * CRC-32 of each record (IEEE 802.3 generator, reflected, initial value and
 * final xor all ones: the value zlib's crc32 gives) into crc_out [n] (device,
 * nullable) and, when expected [n] (device) is given, compares.  A NULL record
 * sets MOE_ERR_MISSING_EXPERT, a misaligned one or a mismatch
 * MOE_ERR_BAD_RECORD on the context's error word (detail: the record's
 * index; with several bad records, one of them); moe_ctx_check reports it.
 * crc_out of a NULL or misaligned record is 0.  Reads every byte once (an
 * HBM-bound pass, meant for load time: a 15.7 GB bank of 896 K3 experts).
 * ws: moe_records_check_ws_bytes(n, record_bytes) bytes (one word per 4 KiB
 * of every record).  n = 0 is a no-op; n times the record's 4 KiB units at or
 * above 2^31 returns MOE_ERR_UNSUPPORTED.
 */
MOE_API size_t moe_records_check_ws_bytes(int n, size_t record_bytes);
MOE_API moe_status moe_records_check(moe_ctx* ctx, const uint8_t* const* records, int n, size_t record_bytes,
                                     const uint32_t* expected, uint32_t* crc_out, void* ws, size_t ws_bytes,
                                     cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */

// moe_internal.cuh -- device helpers and kernel launcher declarations shared by
// the translation units of libmoe_gb300.so.  Not part of the public ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe.h"

namespace moe {

constexpr int kMaxK = 32;          // top-k limit
constexpr int kMaxE = 2048;        // expert-count limit
constexpr int kMaxDim = 4096;      // d, ff limit
constexpr int kRowsPerHalf = 16;   // GEMV tile: rows per half-warp
constexpr int kTokChunk = 2;       // GEMV: tokens per pass over a weight tile
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded device waits: 2 s

// ---------------------------------------------------------------- error word
// err[0] = first status code, err[1] = its detail.  First error wins.
__device__ __forceinline__ void dev_error(int* err, int code, int detail) {
  if (atomicCAS(err, 0, code) == 0) atomicExch(err + 1, detail);
}

// ---------------------------------------------------------------- PDL
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- timers
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// err[4..5] of the context's error word hold the limit of pipeline waits in
// ns, set by moe_ctx_set_wait_limit_ns (0: kWaitLimitNs).
__device__ __forceinline__ uint64_t wait_limit_ns(const int* err) {
  const uint64_t v = *reinterpret_cast<const volatile uint64_t*>(err + 4);
  return v != 0 ? v : kWaitLimitNs;
}

// Spins on the phase with the given parity for at most limit_ns.  Returns
// false (and records MOE_ERR_TIMEOUT) if it gave up.
static __device__ __noinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, int* err, uint64_t limit_ns) {
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) {
      dev_error(err, MOE_ERR_TIMEOUT, -1);
      return false;
    }
  }
}

// A pipeline wait: bounded by the context's wait limit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_for(bar, parity, err, wait_limit_ns(err));
}

// A drain wait (copies or MMAs of this CTA still in flight before it leaves):
// always the fixed kWaitLimitNs, so that a short pipeline limit never lets a
// CTA exit while its copies can still write its shared memory.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_for(bar, parity, err, kWaitLimitNs);
}

// 1-D bulk copy global -> shared, completing `bytes` of transaction on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Named barrier among `nthreads` threads (a multiple of 32) with id `id` (1..15).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- numeric helpers
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// E8M0 scale byte -> 2^(b-127) as fp32 (0 -> 2^-127 subnormal, 255 -> NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
  if (b == 255u) return __uint_as_float(0x7FC00000u);
  if (b == 0u) return __uint_as_float(0x00400000u);
  return __uint_as_float(b << 23);
}

// Four bytes of packed E2M1 codes (low nibble = even column) -> four f16x2
// (exact: every E2M1 value is an f16), byte b -> h[b], even column in the low half.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

__device__ __forceinline__ float act_fn(float g, float u, int act) {
  float sig = 1.0f / (1.0f + expf(-g));
  if (act == MOE_ACT_SITU) return 4.0f * tanhf(g * 0.25f) * sig * 25.0f * tanhf(u * 0.04f);
  return g * sig * u;
}

// The activation with the hardware exponential and an approximate divide
// (relative error about 1e-6, far inside the fp32 path's error budget).
__device__ __forceinline__ float act_fast(float g, float u, int act) {
  if (act == MOE_ACT_SITU) return act_fn(g, u, act);
  return __fdividef(g * u, 1.0f + __expf(-g));
}

__device__ __forceinline__ float load_act(const void* p, int dtype, size_t i) {
  if (dtype == MOE_BF16) return bf16_bits_to_f32(static_cast<const uint16_t*>(p)[i]);
  return static_cast<const float*>(p)[i];
}

// ---------------------------------------------------------------- launchers
// Each returns cudaSuccess or the launch error.  All pointers are device pointers.

struct BucketArgs {
  const int32_t* topk_idx;
  int T, k, E;
  int32_t* counts;
  int32_t* offsets;
  int32_t* pair_ids;
  int32_t* active;  // [E+1] workspace: active[0] = n_active, active[1..] = experts in ascending order
  int* err;
};
cudaError_t launch_bucket(const BucketArgs& a, bool pdl, cudaStream_t s);

struct RouteArgs {
  const void* x;
  int x_dtype;
  const void* w;
  int w_dtype;
  const float* bias;      // added to the logits by the router kernels (selection and gates), or null
  const float* sel_bias;  // added by the top-k to the selection keys only (gates without it), or null
  int T, d, E, k;
  int n_shared;   // shared experts E .. E + n_shared - 1 appended to every token's row (gate 1)
  float* logits;  // [T][E]   workspace
  float* nrm_w;   // [E]      workspace: ||W_e||_2
  float* nrm_x;   // [T]      workspace: ||x_t||_2
  float* max_x;   // [T]      workspace: max_i |x_t[i]|
  float* absdot;  // [T][E]   workspace: sum_i |W[e][i] x[t][i]| (compensated logits only)
  int comp;       // logits by compensated (Dot2) sums; bounds from absdot
  float gamma;    // error-bound coefficient (see router_gamma / router_gamma_comp)
  float gamma_comp;  // the compensated sums' coefficient (router_gamma_comp), for the top-k's recheck
  double gamma_fp64;  // the warp-parallel fp64 sums' coefficient (router_gamma_fp64), for the recheck
  int32_t* topk_idx;  // [T][k + n_shared]
  float* gates;       // [T][k + n_shared]
  int* err;
  int fuse_bucket;    // one token: the top-k kernel also buckets the pairs (with `bucket`)
  BucketArgs bucket;
};
cudaError_t launch_route_topk(const RouteArgs& a, int num_sms, cudaStream_t s);

struct CombineArgs {
  const void* x;
  int x_dtype;
  const float* y_pairs;  // [T*k][d], or with nparts > 1 [T*k][nparts][d] partial sums added in ascending order
  const float* gates;
  int T, k, d;
  void* out;
  int out_dtype;
  int nparts;
};

struct FfnArgs {
  const uint8_t* const* records;
  const uint16_t* cb[3];  // RVQ3 codebooks
  int d, ff, E, k, T;
  int act;
  const void* x;
  int x_dtype;
  const int32_t* offsets;
  const int32_t* pair_ids;
  const int32_t* active;  // active[0] = n_active, then the expert ids
  const float* max_x;     // [T] max_i |x_t[i]| (bf16 activations are rescaled by a power of two from it)
  float* h;               // [T*k][ff] workspace, slot order
  float* y_pairs;         // [T*k][d] by pair id
  float* partial;         // RVQ3 only: K-slice partial sums (workspace)
  int* err;
  // 1 when x and max_x were complete before the kernel launched just ahead of
  // the expert kernels started (the layer path: the router wrote max_x two
  // launches earlier), so that the one-token GEMV may stage x before its wait;
  // 0 when the launch just ahead writes them (the standalone expert calls)
  int x_early;
};
cudaError_t launch_active_from_offsets(const int32_t* offsets, int E, int32_t* active, bool pdl, cudaStream_t s);
cudaError_t launch_mxfp4_ffn(const FfnArgs& a, int num_sms, bool pdl, cudaStream_t s);
// The FFN on the block-scaled tensor-core MMA (mxfp4_bs.cu): every expert
// with tokens (active[] lists them all), bf16 activations, d and ff multiples
// of 512.  ws: mxfp4_bs_ws_bytes(T, k, d, ff, num_sms) bytes, 256-byte aligned.
struct BsLaunch {
  const uint8_t* const* records;
  int d, ff, E, k, T;
  int act;
  const void* x;
  const int32_t* offsets;
  const int32_t* pair_ids;
  const int32_t* active;
  float* y_pairs;
  void* ws;
  int* err;
};
bool mxfp4_bs_supported(int d, int ff, int E, int x_dtype);
size_t mxfp4_bs_ws_bytes(int T, int k, int d, int ff, int max_sms);
cudaError_t launch_mxfp4_bs(const BsLaunch& L, int num_sms, bool pdl, cudaStream_t s);
// The same FFN with the inner products on mma.sync (mxfp4_mma_gemv.cu); bf16 activations.
bool mxfp4_mma_gemv_supported(int d, int ff, int x_dtype);
cudaError_t launch_mxfp4_ffn_mma(const FfnArgs& a, int num_sms, bool pdl, cudaStream_t s);
cudaError_t launch_token_absmax(const void* x, int x_dtype, int T, int d, float* max_x, bool pdl, cudaStream_t s);
// RVQ3 FFN (rvq3_gemv.cu).  a.partial: rvq3_partial_floats(T, k, d, ff)
// floats.  pair_expert: the expert of each pair p = t * k + j ([T][k], e.g. the
// routing), or null to derive it from a.offsets / a.pair_ids.  y_out: also sum
// the down kernel's slice partials into a.y_pairs; otherwise they stay in
// rvq3_down_partials(a) as [T*k][rvq3_down_parts(d, ff)][d] for the combine.
cudaError_t launch_rvq3_ffn(const FfnArgs& a, const int32_t* pair_expert, bool y_out, int num_sms, bool pdl,
                            cudaStream_t s);
size_t rvq3_partial_floats(int T, int k, int d, int ff);
int rvq3_down_parts(int d, int ff);
float* rvq3_down_partials(const FfnArgs& a);

cudaError_t launch_combine(const CombineArgs& a, bool pdl, cudaStream_t s);

// CRC-32 of n records of record_bytes (a multiple of 16) each; checks them
// against expected[] when given (records_check.cu).  unit_ws holds one word
// per 4 KiB unit of every record: n * records_crc_units(record_bytes) words.
int records_crc_units(size_t record_bytes);
cudaError_t launch_records_check(const uint8_t* const* records, int n, size_t record_bytes, const uint32_t* expected,
                                 uint32_t* crc_out, uint32_t* unit_ws, int* err, int num_sms, cudaStream_t s);

// y[t][n] = resid[t][n] (optional) + sum_k W[n][k] x[t][k] (project.cu); W
// [N][K] bf16 or fp32 with K a multiple of 32, every pointer 16-byte aligned.
cudaError_t launch_project(const void* x, int x_dtype, const void* w, int w_dtype, const void* resid, int resid_dtype,
                           void* y, int y_dtype, int T, int K, int N, bool pdl, cudaStream_t s);

// A wait that nothing completes, for testing the timeout path (selftest.cu).
cudaError_t launch_wait_selftest(int* err, cudaStream_t s);

// Row-major to position-major RVQ3 records (rvq3_repack.cu): n records of
// moe_rvq3_record_bytes(d, ff) bytes; src[i] and dst[i] device pointers.
cudaError_t launch_rvq3_repack(const uint8_t* const* src, uint8_t* const* dst, int n, int d, int ff, int* err,
                               int num_sms, cudaStream_t s);

// ABI-layer helpers (abi.cu) shared with other translation units' entry points.
moe_status check_expert_ffn_call(const moe_ctx* ctx, const void* x, moe_dtype x_dtype, int T, int k, int d, int ff,
                                 int E, moe_act act, const int32_t* offsets, const int32_t* pair_ids,
                                 const float* y_pairs);
int* ctx_error_word(const moe_ctx* ctx);

// Raises a kernel's dynamic shared memory limit on the current device once,
// instead of before every launch (the driver call costs microseconds).
cudaError_t ensure_smem(const void* kernel, size_t bytes);
template <typename... KArgs>
cudaError_t ensure_smem(void (*kernel)(KArgs...), size_t bytes) {
  return ensure_smem(reinterpret_cast<const void*>(kernel), bytes);
}

// Per-launch event timing, active while an entry point of a context with
// profiling enabled runs (set by the ABI layer for the calling thread).
struct Profiler;
extern thread_local Profiler* tl_profiler;
void profiler_begin(Profiler* p, const char* name, cudaStream_t s);
void profiler_end(Profiler* p, cudaStream_t s);
Profiler* ctx_profiler(const moe_ctx* ctx);

// Makes the context's profiler current for the launches of one entry point.
struct ProfScope {
  Profiler* prev;
  explicit ProfScope(const moe_ctx* c) : prev(tl_profiler) { tl_profiler = c ? ctx_profiler(c) : nullptr; }
  ~ProfScope() { tl_profiler = prev; }
  ProfScope(const ProfScope&) = delete;
  ProfScope& operator=(const ProfScope&) = delete;
};

// Launch helper: optional programmatic dependent launch; `name` labels the
// launch for the profiler.
template <typename... KArgs, typename... Args>
cudaError_t launch(const char* name, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                   bool pdl, Args&&... args) {
  Profiler* prof = tl_profiler;
  if (prof) profiler_begin(prof, name, s);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (prof) profiler_end(prof, s);
  return err;
}

}  // namespace moe

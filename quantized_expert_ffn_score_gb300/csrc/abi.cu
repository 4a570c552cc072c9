// abi.cu -- the extern "C" entry points of libmoe_gb300.so (declared in
// include/moe.h): argument validation, workspace carving and the launch chains.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <utility>

#include "moe_internal.cuh"

#include <map>
#include <mutex>
#include <vector>

namespace moe {

// Event pairs recorded around each launch while profiling is on.
struct Profiler {
  struct Rec {
    const char* name;
    int ev0, ev1;
  };
  std::vector<cudaEvent_t> pool;
  std::vector<Rec> recs;
  int next = 0;
  int open = -1;
  const char* open_name = nullptr;
};

thread_local Profiler* tl_profiler = nullptr;

cudaError_t ensure_smem(const void* kernel, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> done;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(mu);
  size_t& cur = done[{dev, kernel}];
  if (bytes <= cur) return cudaSuccess;
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (err == cudaSuccess) cur = bytes;
  return err;
}

void profiler_begin(Profiler* p, const char* name, cudaStream_t s) {
  p->open = -1;
  if (p->next + 2 > (int)p->pool.size()) return;  // pool exhausted: launch not timed
  p->open = p->next;
  p->open_name = name;
  cudaEventRecord(p->pool[p->next++], s);
}

void profiler_end(Profiler* p, cudaStream_t s) {
  if (p->open < 0) return;
  cudaEventRecord(p->pool[p->next], s);
  p->recs.push_back({p->open_name, p->open, p->next});
  ++p->next;
  p->open = -1;
}

}  // namespace moe

struct moe_ctx {
  int device;
  int num_sms;
  int mxfp4_kernel;  // moe_mxfp4_kernel: block-scaled MMA path, the GEMV pair, or chosen by token count
  int* err;  // device: [0] status, [1] detail, [2..3] router recheck counters, [4..5] wait limit (ns, u64)
  moe::Profiler* prof;
};

namespace moe {
Profiler* ctx_profiler(const moe_ctx* ctx) { return ctx->prof; }
}  // namespace moe
using moe::ProfScope;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Sequential carving of a workspace into 256-byte aligned regions.
// Largest SM count the block-scaled path's per-CTA workspace is sized for.
constexpr int kMaxSms = 160;

struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  template <typename T>
  T* take(size_t count) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += align_up(count * sizeof(T));
    return p;
  }
};

bool dims_ok(int d, int ff) {
  return d >= 32 && ff >= 32 && d % 32 == 0 && ff % 32 == 0 && d <= moe::kMaxDim && ff <= moe::kMaxDim;
}

moe_status check_route_shape(int T, int d, int E, int k) {
  if (T < 0 || d <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
  if (k > E) return MOE_ERR_INVALID_ARG;
  if (d % 32 || d > moe::kMaxDim || E > moe::kMaxE || k > moe::kMaxK) return MOE_ERR_UNSUPPORTED;
  if ((long long)T * k > (1LL << 24)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

bool dtype_ok(int dt) { return dt == MOE_F32 || dt == MOE_BF16; }

// Activations, router weights and fp32 pair buffers are read with 16-byte vector loads.
bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status ws_check(void* ws, size_t ws_bytes, size_t need) {
  if (need == 0) return MOE_OK;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0 || ws_bytes < need) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

moe_status ctx_ok(const moe_ctx* ctx) {
  if (ctx == nullptr) return MOE_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  return dev == ctx->device ? MOE_OK : MOE_ERR_INVALID_ARG;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Router error-bound coefficient: summation-tree depth of the logits kernel
// (d / (32 N) chunks per lane + log2 N + 5 shuffle levels, N elements per 16-byte
// chunk; one more level when the products are not exact in fp32), as
// gamma_h = h u / (1 - h u), inflated for the fp32 evaluation of the norms, plus
// the fp64 reference's own error (about d * 2^-53).
float router_gamma(int d, moe_dtype x_dtype, moe_dtype w_dtype) {
  const int N = w_dtype == MOE_BF16 ? 8 : 4;
  int h = (d + 32 * N - 1) / (32 * N) + (N == 8 ? 3 : 2) + 5;
  if (!(x_dtype == MOE_BF16 && w_dtype == MOE_BF16)) h += 1;
  const double u = 5.9604644775390625e-8;  // 2^-24
  double g = h * u / (1.0 - h * u);
  g = g * 1.002 + 1e-12;
  return (float)(g * 1.0001);
}

// Small token counts (decode) compute the router logits with compensated sums:
// the logit kernel is memory-bound there, and the much tighter bound lets the
// top-k certify almost every token without the fp64 recheck.
constexpr int kCompensatedMaxT = 16;

// Bound coefficient of the compensated logits: |l32 - l_ref| <= K * sum|w x| +
// 4u |l32| with K = (gamma_n^2 (1 + gamma_n) + gamma64_{d+1}) * 1.01, n = d + 32.
float router_gamma_comp(int d) {
  const double u = 5.9604644775390625e-8, u64 = 1.1102230246251565e-16;
  const double n = d + 32.0, gn = n * u / (1.0 - n * u), g64 = (d + 1.0) * u64 / (1.0 - (d + 1.0) * u64);
  return (float)((gn * gn * (1.0 + gn) + g64) * 1.01);
}

// Bound coefficient of the top-k recheck's warp-parallel fp64 logits against the
// reference's sequential fp64 sum: gamma64(d/32 + 6) for the warp sum (lane
// chains of d/32 products plus a 5-level butterfly and the bias), gamma64(d + 1)
// for the reference, 1 % for the fp64 evaluation of sum|p|.
double router_gamma_fp64(int d) {
  const double u = 1.1102230246251565e-16;  // 2^-53
  auto g = [u](double n) { return n * u / (1.0 - n * u); };
  return (g(d / 32 + 6) + g(d + 1.0)) * 1.01;
}

struct RouteWs {
  float* logits;
  float* nrm_w;
  float* nrm_x;
  float* max_x;
  float* absdot;
};
RouteWs carve_route(Carver& c, int T, int E) {
  RouteWs r;
  r.logits = c.take<float>((size_t)T * E);
  r.nrm_w = c.take<float>(E);
  r.nrm_x = c.take<float>(T > 0 ? T : 1);
  r.max_x = c.take<float>(T > 0 ? T : 1);
  r.absdot = c.take<float>(T <= kCompensatedMaxT ? (size_t)T * E : 1);
  return r;
}

moe::RouteArgs route_args(const void* x, moe_dtype x_dtype, const void* w, moe_dtype w_dtype, const float* bias,
                          int bias_mode, int T, int d, int E, int k, int n_shared, const RouteWs& ws, int32_t* topk,
                          float* gates, int* err) {
  moe::RouteArgs ra;
  std::memset(&ra, 0, sizeof ra);
  ra.x = x;
  ra.x_dtype = x_dtype;
  ra.w = w;
  ra.w_dtype = w_dtype;
  ra.bias = bias_mode == MOE_BIAS_SELECT ? nullptr : bias;
  ra.sel_bias = bias_mode == MOE_BIAS_SELECT ? bias : nullptr;
  ra.T = T;
  ra.d = d;
  ra.E = E;
  ra.k = k;
  ra.n_shared = n_shared;
  ra.logits = ws.logits;
  ra.nrm_w = ws.nrm_w;
  ra.nrm_x = ws.nrm_x;
  ra.max_x = ws.max_x;
  ra.absdot = ws.absdot;
  ra.comp = T <= kCompensatedMaxT ? 1 : 0;
  ra.gamma = ra.comp ? router_gamma_comp(d) : router_gamma(d, x_dtype, w_dtype);
  ra.gamma_comp = router_gamma_comp(d);
  ra.gamma_fp64 = router_gamma_fp64(d);
  ra.topk_idx = topk;
  ra.gates = gates;
  ra.err = err;
  return ra;
}

struct FfnWs {
  int32_t* active;
  float* max_x;
  float* h;
  float* partial;
  void* bs;          // block-scaled path workspace (MXFP4, d and ff multiples of 512)
};
FfnWs carve_ffn(Carver& c, int T, int k, int d, int ff, int E, moe_quant q) {
  FfnWs f;
  f.active = c.take<int32_t>((size_t)E + 1);
  f.max_x = c.take<float>(T > 0 ? T : 1);
  f.h = c.take<float>((size_t)T * k * ff);
  f.partial = q == MOE_QUANT_RVQ3 ? c.take<float>(moe::rvq3_partial_floats(T, k, d, ff)) : nullptr;
  f.bs = nullptr;
  if (q == MOE_QUANT_MXFP4 && moe::mxfp4_bs_supported(d, ff, E, MOE_BF16))
    f.bs = c.take<uint8_t>(moe::mxfp4_bs_ws_bytes(T, k, d, ff, kMaxSms));
  return f;
}

// Whether this call's MXFP4 experts run on the block-scaled MMA path.
bool use_bs(const moe_ctx* ctx, const FfnWs& w, int T, int d, int ff, int E, moe_dtype x_dtype) {
  const bool want = ctx->mxfp4_kernel == MOE_MXFP4_BLOCK_SCALED || (ctx->mxfp4_kernel == MOE_MXFP4_AUTO && T >= 2);
  return want && w.bs != nullptr && moe::mxfp4_bs_supported(d, ff, E, x_dtype);
}

moe::BsLaunch bs_launch(const moe::FfnArgs& f, const FfnWs& w) {
  moe::BsLaunch b;
  b.records = f.records;
  b.d = f.d;
  b.ff = f.ff;
  b.E = f.E;
  b.k = f.k;
  b.T = f.T;
  b.act = f.act;
  b.x = f.x;
  b.offsets = f.offsets;
  b.pair_ids = f.pair_ids;
  b.active = f.active;
  b.y_pairs = f.y_pairs;
  b.ws = w.bs;
  b.err = f.err;
  return b;
}

struct LayerWs {
  RouteWs route;
  int32_t* topk;
  float* gates;
  int32_t* counts;
  int32_t* offsets;
  int32_t* pairs;
  FfnWs ffn;
  float* y_pairs;
};
// A layer's pairs: every token's k routed experts followed by its n_shared
// shared ones (expert ids E .. E + n_shared - 1, gate 1).
int layer_pairs_per_token(const moe_layer* L) { return L->k + L->n_shared; }
int layer_experts(const moe_layer* L) { return L->E + L->n_shared; }

LayerWs carve_layer(Carver& c, const moe_layer* L, int T) {
  LayerWs w;
  const int ks = layer_pairs_per_token(L), Es = layer_experts(L);
  const size_t P = (size_t)T * ks;
  w.route = carve_route(c, T, L->E);
  w.topk = c.take<int32_t>(P ? P : 1);
  w.gates = c.take<float>(P ? P : 1);
  w.counts = c.take<int32_t>(Es);
  w.offsets = c.take<int32_t>((size_t)Es + 1);
  w.pairs = c.take<int32_t>(P ? P : 1);
  w.ffn = carve_ffn(c, T, ks, L->d, L->ff, Es, L->quant);
  w.y_pairs = c.take<float>(P * L->d);
  return w;
}

moe_status check_layer(const moe_layer* L) {
  if (L == nullptr) return MOE_ERR_INVALID_ARG;
  moe_status st = check_route_shape(0, L->d, L->E, L->k);
  if (st != MOE_OK) return st;
  if (!dims_ok(L->d, L->ff)) return MOE_ERR_UNSUPPORTED;
  if (L->router_w == nullptr || !dtype_ok(L->router_w_dtype)) return MOE_ERR_INVALID_ARG;
  if (L->act != MOE_ACT_SWIGLU && L->act != MOE_ACT_SITU) return MOE_ERR_INVALID_ARG;
  if (L->bias_mode != MOE_BIAS_LOGIT && L->bias_mode != MOE_BIAS_SELECT) return MOE_ERR_INVALID_ARG;
  if (L->n_shared < 0) return MOE_ERR_INVALID_ARG;
  if (layer_pairs_per_token(L) > moe::kMaxK || layer_experts(L) > moe::kMaxE) return MOE_ERR_UNSUPPORTED;
  const int Es = layer_experts(L);
  if (L->quant == MOE_QUANT_MXFP4) {
    const moe_mxfp4_experts& m = L->mxfp4;
    if (m.records == nullptr || m.d != L->d || m.ff != L->ff || m.E != Es) return MOE_ERR_INVALID_ARG;
  } else if (L->quant == MOE_QUANT_RVQ3) {
    const moe_rvq3_experts& r = L->rvq3;
    if (r.records == nullptr || r.d != L->d || r.ff != L->ff || r.E != Es) return MOE_ERR_INVALID_ARG;
    for (int m = 0; m < 3; ++m)
      if (r.codebooks[m] == nullptr || (reinterpret_cast<uintptr_t>(r.codebooks[m]) & 15u)) return MOE_ERR_INVALID_ARG;
  } else {
    return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

moe::FfnArgs ffn_args(const moe_ctx* ctx, const void* x, moe_dtype x_dtype, int T, int k, int d, int ff, int E,
                      moe_act act, const int32_t* offsets, const int32_t* pair_ids, float* y_pairs, const FfnWs& w) {
  moe::FfnArgs a;
  std::memset(&a, 0, sizeof a);
  a.d = d;
  a.ff = ff;
  a.E = E;
  a.k = k;
  a.T = T;
  a.act = act;
  a.x = x;
  a.x_dtype = x_dtype;
  a.offsets = offsets;
  a.pair_ids = pair_ids;
  a.active = w.active;
  a.max_x = w.max_x;
  a.h = w.h;
  a.partial = w.partial;
  a.y_pairs = y_pairs;
  a.err = ctx->err;
  return a;
}

// residual = false: out is the MoE delta alone (the latent layer projects it back).
moe_status layer_forward_impl(moe_ctx* ctx, const moe_layer* L, const void* x, moe_dtype x_dtype, int T, void* out,
                              moe_dtype out_dtype, int32_t* topk_out, float* gates_out, int32_t* counts_out,
                              const LayerWs& w, cudaStream_t s, bool residual = true) {
  if (T == 0) return MOE_OK;
  const int ks = layer_pairs_per_token(L), Es = layer_experts(L);
  const int32_t* topk = topk_out ? topk_out : w.topk;
  const float* gates = gates_out ? gates_out : w.gates;
  int32_t* counts = counts_out ? counts_out : w.counts;
  moe::RouteArgs ra = route_args(x, x_dtype, L->router_w, L->router_w_dtype, L->router_bias, L->bias_mode, T, L->d,
                                 L->E, L->k, L->n_shared, w.route, const_cast<int32_t*>(topk),
                                 const_cast<float*>(gates), ctx->err);
  const bool bs = L->quant == MOE_QUANT_MXFP4 && use_bs(ctx, w.ffn, T, L->d, L->ff, Es, x_dtype);
  moe::BucketArgs ba{topk, T, ks, Es, counts, w.offsets, w.pairs, w.ffn.active, ctx->err};
  if (T == 1) {  // one token: the top-k kernel buckets its pairs itself
    ra.fuse_bucket = 1;
    ra.bucket = ba;
    ra.bucket.counts = counts_out;  // no later step reads the counts: only the caller's copy is written
  }
  moe_status st = cuda_status(moe::launch_route_topk(ra, ctx->num_sms, s));
  if (st != MOE_OK) return st;
  // the RVQ3 kernels work from the routing itself (pairs in token order); the
  // buckets are then only needed for the caller's counts
  const bool need_buckets = L->quant == MOE_QUANT_MXFP4 || counts_out != nullptr;
  if (T != 1 && need_buckets) {
    st = cuda_status(moe::launch_bucket(ba, true, s));
    if (st != MOE_OK) return st;
  }
  moe::FfnArgs fa = ffn_args(ctx, x, x_dtype, T, ks, L->d, L->ff, Es, L->act, w.offsets, w.pairs, w.y_pairs, w.ffn);
  fa.max_x = w.route.max_x;  // computed by the router kernel
  fa.x_early = 1;            // two launches before the expert kernels
  if (L->quant == MOE_QUANT_MXFP4 && bs) {
    fa.records = L->mxfp4.records;
    st = cuda_status(moe::launch_mxfp4_bs(bs_launch(fa, w.ffn), ctx->num_sms, true, s));
  } else if (L->quant == MOE_QUANT_MXFP4) {
    fa.records = L->mxfp4.records;
    st = cuda_status(moe::launch_mxfp4_ffn(fa, ctx->num_sms, true, s));
  } else {
    fa.records = L->rvq3.records;
    for (int m = 0; m < 3; ++m) fa.cb[m] = L->rvq3.codebooks[m];
    st = cuda_status(moe::launch_rvq3_ffn(fa, topk, false, ctx->num_sms, true, s));
    if (st != MOE_OK) return st;
    // the combine adds the down kernel's per-slice sums of each pair
    moe::CombineArgs ca{residual ? x : nullptr, x_dtype, moe::rvq3_down_partials(fa), gates, T, ks, L->d, out,
                        out_dtype, moe::rvq3_down_parts(L->d, L->ff)};
    return cuda_status(moe::launch_combine(ca, true, s));
  }
  if (st != MOE_OK) return st;
  moe::CombineArgs ca{residual ? x : nullptr, x_dtype, w.y_pairs, gates, T, ks, L->d, out, out_dtype, 1};
  return cuda_status(moe::launch_combine(ca, true, s));
}

}  // namespace

extern "C" {

const char* moe_status_str(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_BAD_EXPERT_INDEX: return "routing named an expert outside [0, E)";
    case MOE_ERR_MISSING_EXPERT: return "a routed expert's record is missing";
    case MOE_ERR_TIMEOUT: return "a bounded device wait timed out";
    case MOE_ERR_BAD_RECORD: return "a record failed its check (checksum mismatch or misaligned)";
  }
  return "unknown status";
}

const char* moe_version(void) { return "moe_gb300 0.1 (sm_103a)"; }

moe_status moe_ctx_create(moe_ctx** ctx, int device) {
  if (ctx == nullptr) return MOE_ERR_INVALID_ARG;
  *ctx = nullptr;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaSetDevice(device) != cudaSuccess) return MOE_ERR_CUDA;
  moe_ctx* c = static_cast<moe_ctx*>(std::calloc(1, sizeof(moe_ctx)));
  moe_status st = MOE_OK;
  if (c == nullptr) {
    st = MOE_ERR_CUDA;
  } else {
    c->device = device;
    c->mxfp4_kernel = MOE_MXFP4_AUTO;
    if (cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaMalloc(&c->err, 8 * sizeof(int)) != cudaSuccess || cudaMemset(c->err, 0, 8 * sizeof(int)) != cudaSuccess) {
      if (c->err) cudaFree(c->err);
      std::free(c);
      c = nullptr;
      st = MOE_ERR_CUDA;
    }
  }
  cudaSetDevice(prev);
  *ctx = c;
  return st;
}

void moe_ctx_destroy(moe_ctx* ctx) {
  if (ctx == nullptr) return;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(ctx->device);
  moe_ctx_profile(ctx, 0);
  cudaFree(ctx->err);
  cudaSetDevice(prev);
  std::free(ctx);
}

int moe_ctx_num_sms(const moe_ctx* ctx) { return ctx ? ctx->num_sms : 0; }

moe_status moe_ctx_set_wait_limit_ns(moe_ctx* ctx, unsigned long long ns) {
  moe_status st = ctx_ok(ctx);
  if (st != MOE_OK) return st;
  if (ns != 0 && ns < 1000ull) ns = 1000ull;
  const uint64_t v = ns;
  return cudaMemcpy(ctx->err + 4, &v, sizeof v, cudaMemcpyHostToDevice) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_ctx_wait_selftest(moe_ctx* ctx, cudaStream_t stream) {
  moe_status st = ctx_ok(ctx);
  if (st != MOE_OK) return st;
  ProfScope prof_scope(ctx);
  return cuda_status(moe::launch_wait_selftest(ctx->err, stream));
}

moe_status moe_rvq3_repack(moe_ctx* ctx, const uint8_t* const* src, uint8_t* const* dst, int n, int d, int ff,
                           cudaStream_t stream) {
  moe_status st = ctx_ok(ctx);
  if (st != MOE_OK) return st;
  ProfScope prof_scope(ctx);
  if (n < 0) return MOE_ERR_INVALID_ARG;
  if (!dims_ok(d, ff)) return d > 0 && ff > 0 && d % 32 == 0 && ff % 32 == 0 ? MOE_ERR_UNSUPPORTED : MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (src == nullptr || dst == nullptr) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_rvq3_repack(src, dst, n, d, ff, ctx->err, ctx->num_sms, stream));
}

moe_status moe_ctx_set_mxfp4_kernel(moe_ctx* ctx, int kernel) {
  if (ctx == nullptr || (kernel != MOE_MXFP4_BLOCK_SCALED && kernel != MOE_MXFP4_GEMV && kernel != MOE_MXFP4_AUTO))
    return MOE_ERR_INVALID_ARG;
  ctx->mxfp4_kernel = kernel;
  return MOE_OK;
}

int moe_ctx_mxfp4_kernel(const moe_ctx* ctx) { return ctx ? ctx->mxfp4_kernel : -1; }

moe_status moe_ctx_profile(moe_ctx* ctx, int capacity) {
  if (ctx == nullptr || capacity < 0) return MOE_ERR_INVALID_ARG;
  if (ctx->prof) {
    for (cudaEvent_t e : ctx->prof->pool) cudaEventDestroy(e);
    delete ctx->prof;
    ctx->prof = nullptr;
  }
  if (capacity == 0) return MOE_OK;
  moe::Profiler* p = new moe::Profiler();
  p->pool.resize(2 * (size_t)capacity);
  for (auto& e : p->pool) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      e = nullptr;
      for (cudaEvent_t x : p->pool)
        if (x) cudaEventDestroy(x);
      delete p;
      return MOE_ERR_CUDA;
    }
  }
  ctx->prof = p;
  return MOE_OK;
}

int moe_ctx_profile_read(moe_ctx* ctx, cudaStream_t stream, int max_entries, char* names, int* launches,
                         double* total_ms) {
  if (ctx == nullptr || ctx->prof == nullptr || max_entries < 0) return -(int)MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return -(int)MOE_ERR_CUDA;
  moe::Profiler* p = ctx->prof;
  int n = 0;
  std::vector<const char*> keys;
  for (const auto& r : p->recs) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, p->pool[r.ev0], p->pool[r.ev1]) != cudaSuccess) return -(int)MOE_ERR_CUDA;
    int i = 0;
    while (i < (int)keys.size() && std::strcmp(keys[i], r.name) != 0) ++i;
    if (i == (int)keys.size()) {
      keys.push_back(r.name);
      if (i < max_entries) {
        std::strncpy(names + 32 * i, r.name, 31);
        names[32 * i + 31] = 0;
        launches[i] = 0;
        total_ms[i] = 0.0;
      }
    }
    if (i < max_entries) {
      launches[i] += 1;
      total_ms[i] += ms;
    }
  }
  n = (int)keys.size() < max_entries ? (int)keys.size() : max_entries;
  p->recs.clear();
  p->next = 0;
  return n;
}

moe_status moe_ctx_check(moe_ctx* ctx, cudaStream_t stream, int* detail) {
  moe_status st = ctx_ok(ctx);
  if (st != MOE_OK) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  int h[2] = {0, 0};
  if (cudaMemcpy(h, ctx->err, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (h[0] != 0 && cudaMemset(ctx->err, 0, 2 * sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  if (detail) *detail = h[0] ? h[1] : -1;
  return static_cast<moe_status>(h[0]);
}

moe_status moe_ctx_stats(moe_ctx* ctx, cudaStream_t stream, long long* fp64_tokens, long long* seq_logits) {
  moe_status st = ctx_ok(ctx);
  if (st != MOE_OK) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  int h[2] = {0, 0};
  if (cudaMemcpy(h, ctx->err + 2, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(ctx->err + 2, 0, 2 * sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  if (fp64_tokens) *fp64_tokens = h[0];
  if (seq_logits) *seq_logits = h[1];
  return MOE_OK;
}

size_t moe_mxfp4_record_bytes(int d, int ff) {
  if (d <= 0 || ff <= 0 || d % 32 || ff % 32) return 0;
  return 3 * ((size_t)ff * d / 2 + (size_t)ff * d / 32);
}

size_t moe_rvq3_record_bytes(int d, int ff) {
  if (d <= 0 || ff <= 0 || d % 32 || ff % 32) return 0;
  return 9 * (size_t)ff * d / 8;
}

size_t moe_route_topk_ws_bytes(int T, int d, int E, int k) {
  if (check_route_shape(T, d, E, k) != MOE_OK) return 0;
  Carver c(nullptr);
  carve_route(c, T, E);
  return c.off;
}

size_t moe_bucket_tokens_ws_bytes(int T, int k, int E) {
  if (check_route_shape(T, 32, E, k) != MOE_OK) return 0;
  return align_up(((size_t)E + 1) * sizeof(int32_t));
}

size_t moe_expert_ffn_ws_bytes(int T, int k, int d, int ff, int E, moe_quant quant) {
  if (check_route_shape(T, d, E, k) != MOE_OK || !dims_ok(d, ff)) return 0;
  if (quant != MOE_QUANT_MXFP4 && quant != MOE_QUANT_RVQ3) return 0;
  Carver c(nullptr);
  carve_ffn(c, T, k, d, ff, E, quant);
  return c.off;
}

size_t moe_layer_forward_ws_bytes(const moe_layer* L, int T) {
  if (check_layer(L) != MOE_OK || check_route_shape(T, L->d, layer_experts(L), layer_pairs_per_token(L)) != MOE_OK) return 0;
  Carver c(nullptr);
  carve_layer(c, L, T);
  return c.off;
}

size_t moe_stack_forward_ws_bytes(const moe_layer* layers, int n_layers, int T) {
  if (layers == nullptr || n_layers <= 0) return 0;
  size_t mx = 0;
  for (int l = 0; l < n_layers; ++l) {
    size_t b = moe_layer_forward_ws_bytes(&layers[l], T);
    if (b == 0 || layers[l].d != layers[0].d) return 0;
    mx = b > mx ? b : mx;
  }
  return mx + 2 * align_up((size_t)T * layers[0].d * sizeof(uint16_t));
}

moe_status moe_route_topk(moe_ctx* ctx, const void* x, moe_dtype x_dtype, const void* router_w, moe_dtype w_dtype,
                          const float* bias, int T, int d, int E, int k, int32_t* topk_idx, float* gates, void* ws,
                          size_t ws_bytes, cudaStream_t stream) {
  return moe_route_topk_ex(ctx, x, x_dtype, router_w, w_dtype, bias, MOE_BIAS_LOGIT, T, d, E, k, topk_idx, gates, ws,
                           ws_bytes, stream);
}

moe_status moe_route_topk_ex(moe_ctx* ctx, const void* x, moe_dtype x_dtype, const void* router_w, moe_dtype w_dtype,
                             const float* bias, moe_bias_mode bias_mode, int T, int d, int E, int k, int32_t* topk_idx,
                             float* gates, void* ws, size_t ws_bytes, cudaStream_t stream) {
  moe_status st = ctx_ok(ctx);
  if (st != MOE_OK) return st;
  ProfScope prof_scope(ctx);
  if ((st = check_route_shape(T, d, E, k)) != MOE_OK) return st;
  if (!dtype_ok(x_dtype) || !dtype_ok(w_dtype)) return MOE_ERR_INVALID_ARG;
  if (bias_mode != MOE_BIAS_LOGIT && bias_mode != MOE_BIAS_SELECT) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !router_w || !topk_idx || !gates) return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(router_w)) return MOE_ERR_INVALID_ARG;
  if ((st = ws_check(ws, ws_bytes, moe_route_topk_ws_bytes(T, d, E, k))) != MOE_OK) return st;
  Carver c(ws);
  RouteWs w = carve_route(c, T, E);
  moe::RouteArgs ra = route_args(x, x_dtype, router_w, w_dtype, bias, bias_mode, T, d, E, k, 0, w, topk_idx, gates,
                                 ctx->err);
  return cuda_status(moe::launch_route_topk(ra, ctx->num_sms, stream));
}

size_t moe_records_check_ws_bytes(int n, size_t record_bytes) {
  if (n < 0 || record_bytes == 0 || record_bytes % 16) return 0;
  return align_up((size_t)(n > 0 ? n : 1) * moe::records_crc_units(record_bytes) * sizeof(uint32_t));
}

moe_status moe_records_check(moe_ctx* ctx, const uint8_t* const* records, int n, size_t record_bytes,
                             const uint32_t* expected, uint32_t* crc_out, void* ws, size_t ws_bytes,
                             cudaStream_t stream) {
  moe_status st = ctx_ok(ctx);
  if (st != MOE_OK) return st;
  ProfScope prof_scope(ctx);
  if (n < 0 || record_bytes == 0 || record_bytes % 16) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (records == nullptr) return MOE_ERR_INVALID_ARG;
  if ((long long)n * moe::records_crc_units(record_bytes) >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  if ((st = ws_check(ws, ws_bytes, moe_records_check_ws_bytes(n, record_bytes))) != MOE_OK) return st;
  return cuda_status(moe::launch_records_check(records, n, record_bytes, expected, crc_out,
                                               static_cast<uint32_t*>(ws), ctx->err, ctx->num_sms, stream));
}

moe_status moe_bucket_tokens(moe_ctx* ctx, const int32_t* topk_idx, int T, int k, int E, int32_t* counts,
                             int32_t* offsets, int32_t* pair_ids, void* ws, size_t ws_bytes, cudaStream_t stream) {
  moe_status st = ctx_ok(ctx);
  if (st != MOE_OK) return st;
  ProfScope prof_scope(ctx);
  if ((st = check_route_shape(T, 32, E, k)) != MOE_OK) return st;
  if (!counts || !offsets || (T > 0 && (!topk_idx || !pair_ids))) return MOE_ERR_INVALID_ARG;
  if ((st = ws_check(ws, ws_bytes, moe_bucket_tokens_ws_bytes(T, k, E))) != MOE_OK) return st;
  if (T == 0) {
    if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, stream) != cudaSuccess ||
        cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), stream) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  moe::BucketArgs ba{topk_idx, T, k, E, counts, offsets, pair_ids, static_cast<int32_t*>(ws), ctx->err};
  return cuda_status(moe::launch_bucket(ba, false, stream));
}

}  // extern "C"

namespace moe {

moe_status check_expert_ffn_call(const moe_ctx* ctx, const void* x, moe_dtype x_dtype, int T, int k, int d, int ff,
                                 int E, moe_act act, const int32_t* offsets, const int32_t* pair_ids,
                                 const float* y_pairs) {
  moe_status st = ctx_ok(ctx);
  if (st != MOE_OK) return st;
  if ((st = check_route_shape(T, d, E, k)) != MOE_OK) return st;
  if (!dims_ok(d, ff)) return MOE_ERR_UNSUPPORTED;
  if (!dtype_ok(x_dtype) || (act != MOE_ACT_SWIGLU && act != MOE_ACT_SITU)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !offsets || !pair_ids || !y_pairs) return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(y_pairs)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

int* ctx_error_word(const moe_ctx* ctx) { return ctx->err; }

}  // namespace moe

extern "C" {

static moe_status expert_ffn_common(moe_ctx* ctx, const void* x, moe_dtype x_dtype, int T, int k, int d, int ff,
                                    int E, moe_act act, moe_quant q, const int32_t* offsets, const int32_t* pair_ids,
                                    float* y_pairs, void* ws, size_t ws_bytes, moe::FfnArgs* out_args,
                                    FfnWs* out_ws) {
  moe_status st = ctx_ok(ctx);
  if (st != MOE_OK) return st;
  if ((st = check_route_shape(T, d, E, k)) != MOE_OK) return st;
  if (!dims_ok(d, ff)) return MOE_ERR_UNSUPPORTED;
  if (!dtype_ok(x_dtype) || (act != MOE_ACT_SWIGLU && act != MOE_ACT_SITU)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !offsets || !pair_ids || !y_pairs) return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(y_pairs)) return MOE_ERR_INVALID_ARG;
  if ((st = ws_check(ws, ws_bytes, moe_expert_ffn_ws_bytes(T, k, d, ff, E, q))) != MOE_OK) return st;
  Carver c(ws);
  FfnWs w = carve_ffn(c, T, k, d, ff, E, q);
  *out_args = ffn_args(ctx, x, x_dtype, T, k, d, ff, E, act, offsets, pair_ids, y_pairs, w);
  *out_ws = w;
  return MOE_OK;
}

moe_status moe_expert_ffn_mxfp4(moe_ctx* ctx, const void* x, moe_dtype x_dtype, int T, int k,
                                const moe_mxfp4_experts* experts, moe_act act, const int32_t* offsets,
                                const int32_t* pair_ids, float* y_pairs, void* ws, size_t ws_bytes,
                                cudaStream_t stream) {
  if (experts == nullptr || experts->records == nullptr) return MOE_ERR_INVALID_ARG;
  ProfScope prof_scope(ctx);
  moe::FfnArgs a;
  FfnWs w;
  moe_status st = expert_ffn_common(ctx, x, x_dtype, T, k, experts->d, experts->ff, experts->E, act,
                                    MOE_QUANT_MXFP4, offsets, pair_ids, y_pairs, ws, ws_bytes, &a, &w);
  if (st != MOE_OK || T == 0) return st;
  a.records = experts->records;
  st = cuda_status(
      moe::launch_active_from_offsets(offsets, experts->E, const_cast<int32_t*>(a.active), false, stream));
  if (st != MOE_OK) return st;
  if (use_bs(ctx, w, T, experts->d, experts->ff, experts->E, x_dtype))
    return cuda_status(moe::launch_mxfp4_bs(bs_launch(a, w), ctx->num_sms, true, stream));
  st = cuda_status(moe::launch_token_absmax(x, x_dtype, T, experts->d, const_cast<float*>(a.max_x), true, stream));
  if (st != MOE_OK) return st;
  return cuda_status(moe::launch_mxfp4_ffn(a, ctx->num_sms, true, stream));
}

moe_status moe_expert_ffn_rvq3(moe_ctx* ctx, const void* x, moe_dtype x_dtype, int T, int k,
                               const moe_rvq3_experts* experts, moe_act act, const int32_t* offsets,
                               const int32_t* pair_ids, float* y_pairs, void* ws, size_t ws_bytes,
                               cudaStream_t stream) {
  if (experts == nullptr || experts->records == nullptr) return MOE_ERR_INVALID_ARG;
  for (int m = 0; m < 3; ++m)
    if (experts->codebooks[m] == nullptr || (reinterpret_cast<uintptr_t>(experts->codebooks[m]) & 15u))
      return MOE_ERR_INVALID_ARG;
  ProfScope prof_scope(ctx);
  moe::FfnArgs a;
  FfnWs w;
  moe_status st = expert_ffn_common(ctx, x, x_dtype, T, k, experts->d, experts->ff, experts->E, act, MOE_QUANT_RVQ3,
                                    offsets, pair_ids, y_pairs, ws, ws_bytes, &a, &w);
  if (st != MOE_OK || T == 0) return st;
  a.records = experts->records;
  for (int m = 0; m < 3; ++m) a.cb[m] = experts->codebooks[m];
  return cuda_status(moe::launch_rvq3_ffn(a, nullptr, true, ctx->num_sms, false, stream));
}

moe_status moe_combine(moe_ctx* ctx, const void* x_resid, moe_dtype x_dtype, const float* y_pairs,
                       const float* gates, int T, int k, int d, void* out, moe_dtype out_dtype, cudaStream_t stream) {
  moe_status st = ctx_ok(ctx);
  if (st != MOE_OK) return st;
  ProfScope prof_scope(ctx);
  if (T < 0 || k <= 0 || k > moe::kMaxK || d <= 0 || d % 32) return MOE_ERR_INVALID_ARG;
  if (!dtype_ok(x_dtype) || !dtype_ok(out_dtype)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!y_pairs || !gates || !out) return MOE_ERR_INVALID_ARG;
  if (!al16(y_pairs) || !al16(out)) return MOE_ERR_INVALID_ARG;
  moe::CombineArgs ca{x_resid, x_dtype, y_pairs, gates, T, k, d, out, out_dtype, 1};
  return cuda_status(moe::launch_combine(ca, false, stream));
}

moe_status moe_layer_forward(moe_ctx* ctx, const moe_layer* L, const void* x, moe_dtype x_dtype, int T, void* out,
                             moe_dtype out_dtype, int32_t* topk_idx_out, float* gates_out, int32_t* counts_out,
                             void* ws, size_t ws_bytes, cudaStream_t stream) {
  moe_status st = ctx_ok(ctx);
  if (st != MOE_OK) return st;
  ProfScope prof_scope(ctx);
  if ((st = check_layer(L)) != MOE_OK) return st;
  if ((st = check_route_shape(T, L->d, layer_experts(L), layer_pairs_per_token(L))) != MOE_OK) return st;
  if (!dtype_ok(x_dtype) || !dtype_ok(out_dtype)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !out || x == out) return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(out) || !al16(L->router_w)) return MOE_ERR_INVALID_ARG;
  if ((st = ws_check(ws, ws_bytes, moe_layer_forward_ws_bytes(L, T))) != MOE_OK) return st;
  Carver c(ws);
  LayerWs w = carve_layer(c, L, T);
  return layer_forward_impl(ctx, L, x, x_dtype, T, out, out_dtype, topk_idx_out, gates_out, counts_out, w, stream);
}

moe_status moe_stack_forward(moe_ctx* ctx, const moe_layer* layers, int n_layers, const void* x, moe_dtype x_dtype,
                             int T, void* out, moe_dtype out_dtype, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return moe_stack_forward_ex(ctx, layers, n_layers, x, x_dtype, T, out, out_dtype, nullptr, nullptr, nullptr, ws,
                              ws_bytes, stream);
}

moe_status moe_stack_forward_ex(moe_ctx* ctx, const moe_layer* layers, int n_layers, const void* x, moe_dtype x_dtype,
                                int T, void* out, moe_dtype out_dtype, int32_t* topk_trace, float* gates_trace,
                                int32_t* counts_trace, void* ws, size_t ws_bytes, cudaStream_t stream) {
  moe_status st = ctx_ok(ctx);
  if (st != MOE_OK) return st;
  ProfScope prof_scope(ctx);
  if (layers == nullptr || n_layers <= 0) return MOE_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l) {
    if ((st = check_layer(&layers[l])) != MOE_OK) return st;
    if ((st = check_route_shape(T, layers[l].d, layer_experts(&layers[l]), layer_pairs_per_token(&layers[l]))) != MOE_OK) return st;
    if (layers[l].d != layers[0].d) return MOE_ERR_INVALID_ARG;
  }
  if (!dtype_ok(x_dtype) || !dtype_ok(out_dtype)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !out || x == out) return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(out)) return MOE_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l)
    if (!al16(layers[l].router_w)) return MOE_ERR_INVALID_ARG;
  if ((st = ws_check(ws, ws_bytes, moe_stack_forward_ws_bytes(layers, n_layers, T))) != MOE_OK) return st;
  size_t layer_ws = 0;
  for (int l = 0; l < n_layers; ++l) {
    size_t b = moe_layer_forward_ws_bytes(&layers[l], T);
    layer_ws = b > layer_ws ? b : layer_ws;
  }
  char* base = static_cast<char*>(ws);
  uint16_t* buf[2] = {reinterpret_cast<uint16_t*>(base + layer_ws),
                      reinterpret_cast<uint16_t*>(base + layer_ws + align_up((size_t)T * layers[0].d * 2))};
  size_t pair_off = 0, exp_off = 0;  // where layer l's trace starts
  for (int l = 0; l < n_layers; ++l) {
    const void* in = l == 0 ? x : buf[(l - 1) & 1];
    const moe_dtype in_dt = l == 0 ? x_dtype : MOE_BF16;
    const bool last = l == n_layers - 1;
    void* o = last ? out : buf[l & 1];
    Carver c(ws);
    LayerWs w = carve_layer(c, &layers[l], T);
    st = layer_forward_impl(ctx, &layers[l], in, in_dt, T, o, last ? out_dtype : MOE_BF16,
                            topk_trace ? topk_trace + pair_off : nullptr, gates_trace ? gates_trace + pair_off : nullptr,
                            counts_trace ? counts_trace + exp_off : nullptr, w, stream);
    if (st != MOE_OK) return st;
    pair_off += (size_t)T * layer_pairs_per_token(&layers[l]);
    exp_off += (size_t)layer_experts(&layers[l]);
  }
  return MOE_OK;
}

size_t moe_latent_layer_forward_ws_bytes(const moe_layer* L, int D, int T) {
  if (D <= 0 || D % 32 || D > 65536) return 0;
  const size_t lw = moe_layer_forward_ws_bytes(L, T);
  if (lw == 0) return 0;
  return lw + align_up((size_t)T * L->d * sizeof(uint16_t)) + align_up((size_t)T * L->d * sizeof(float));
}

moe_status moe_project(moe_ctx* ctx, const void* x, moe_dtype x_dtype, int T, int K, const void* w, moe_dtype w_dtype,
                       int N, const void* resid, moe_dtype resid_dtype, void* y, moe_dtype y_dtype,
                       cudaStream_t stream) {
  moe_status st = ctx_ok(ctx);
  if (st != MOE_OK) return st;
  ProfScope prof_scope(ctx);
  if (T < 0 || K <= 0 || N <= 0 || K % 32) return MOE_ERR_INVALID_ARG;
  if (K > 65536 || N > 65536 || (long long)T * (K > N ? K : N) > (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  if (!dtype_ok(x_dtype) || !dtype_ok(w_dtype) || !dtype_ok(y_dtype) || (resid && !dtype_ok(resid_dtype)))
    return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w || !y || !al16(x) || !al16(w)) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_project(x, x_dtype, w, w_dtype, resid, resid_dtype, y, y_dtype, T, K, N, false,
                                         stream));
}

moe_status moe_latent_layer_forward(moe_ctx* ctx, const moe_layer* L, const void* w_in, const void* w_out,
                                    moe_dtype w_dtype, int D, const void* x, moe_dtype x_dtype, int T, void* out,
                                    moe_dtype out_dtype, uint16_t* latent_out, void* ws, size_t ws_bytes,
                                    cudaStream_t stream) {
  moe_status st = ctx_ok(ctx);
  if (st != MOE_OK) return st;
  ProfScope prof_scope(ctx);
  if ((st = check_layer(L)) != MOE_OK) return st;
  if ((st = check_route_shape(T, L->d, layer_experts(L), layer_pairs_per_token(L))) != MOE_OK) return st;
  if (D <= 0 || D % 32) return MOE_ERR_INVALID_ARG;
  if (D > 65536) return MOE_ERR_UNSUPPORTED;
  if (!dtype_ok(x_dtype) || !dtype_ok(out_dtype) || !dtype_ok(w_dtype)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !out || x == out || !w_in || !w_out) return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(out) || !al16(w_in) || !al16(w_out) || !al16(L->router_w)) return MOE_ERR_INVALID_ARG;
  if ((st = ws_check(ws, ws_bytes, moe_latent_layer_forward_ws_bytes(L, D, T))) != MOE_OK) return st;
  const size_t lw = moe_layer_forward_ws_bytes(L, T);
  char* base = static_cast<char*>(ws);
  uint16_t* z = latent_out ? latent_out : reinterpret_cast<uint16_t*>(base + lw);
  float* u = reinterpret_cast<float*>(base + lw + align_up((size_t)T * L->d * sizeof(uint16_t)));
  if (latent_out && !al16(latent_out)) return MOE_ERR_INVALID_ARG;
  // z = bf16(W_in x): the latent input of the experts
  st = cuda_status(moe::launch_project(x, x_dtype, w_in, w_dtype, nullptr, 0, z, MOE_BF16, T, D, L->d, false, stream));
  if (st != MOE_OK) return st;
  // u = the MoE delta of z (no residual)
  Carver c(ws);
  LayerWs w = carve_layer(c, L, T);
  st = layer_forward_impl(ctx, L, z, MOE_BF16, T, u, MOE_F32, nullptr, nullptr, nullptr, w, stream, false);
  if (st != MOE_OK) return st;
  // out = x + W_out u
  return cuda_status(moe::launch_project(u, MOE_F32, w_out, w_dtype, x, x_dtype, out, out_dtype, T, L->d, D, true,
                                         stream));
}

}  // extern "C"

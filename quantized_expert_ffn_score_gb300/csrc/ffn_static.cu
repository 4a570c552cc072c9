// ffn_static.cu -- moe_expert_ffn_mxfp4_static: the MXFP4 expert FFN with its
// scratch memory in this library's own static device array, for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs where the allocator is
// owned by someone else (a host framework with its own memory pool, an
// inference server that forbids allocations on its request path) or that must
// not allocate at all after start-up.  They still pass their inputs and
// outputs; the scratch the kernels need between their launches (the list of
// experts with tokens, a per-token scale, and the hidden activations h) lives
// in g_ffn_scratch below.  Every GPU that loads the library reserves it until
// the process exits.
#include <cstring>
#include <mutex>
#include <utility>

#include "moe_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_ffn_scratch[kStaticScratchBytes];

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// Bytes of scratch one call needs: active list [E+1], max|x| [T], h [T*k][ff].
size_t scratch_bytes(int T, int k, int ff, int E) {
  return align256(((size_t)E + 1) * sizeof(int32_t)) + align256((size_t)T * sizeof(float)) +
         align256((size_t)T * k * ff * sizeof(float));
}

// Device address of g_ffn_scratch on the current device, looked up once per
// device (host code cannot use the symbol itself as a device address).
cudaError_t scratch_address(int device, void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[device] == nullptr) {
    void* p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_ffn_scratch);
    if (err != cudaSuccess) return err;
    addr[device] = p;
  }
  *out = addr[device];
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t moe_expert_ffn_mxfp4_static_max_bytes(void) { return kStaticScratchBytes; }

moe_status moe_expert_ffn_mxfp4_static(moe_ctx* ctx, const void* x, moe_dtype x_dtype, int T, int k,
                                       const moe_mxfp4_experts* experts, moe_act act, const int32_t* offsets,
                                       const int32_t* pair_ids, float* y_pairs, cudaStream_t stream) {
  if (experts == nullptr || experts->records == nullptr) return MOE_ERR_INVALID_ARG;
  const int d = experts->d, ff = experts->ff, E = experts->E;
  moe_status st =
      moe::check_expert_ffn_call(ctx, x, x_dtype, T, k, d, ff, E, act, offsets, pair_ids, y_pairs);
  if (st != MOE_OK || T == 0) return st;
  if (scratch_bytes(T, k, ff, E) > kStaticScratchBytes) return MOE_ERR_UNSUPPORTED;
  moe::ProfScope prof_scope(ctx);  // the launches below show in the context's per-launch profile
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return MOE_ERR_CUDA;
  void* base = nullptr;
  if (scratch_address(device, &base) != cudaSuccess) return MOE_ERR_CUDA;

  // Carve the scratch.  Nothing in it needs to start at zero: each call's
  // kernels write the active list, the scales and h before reading them.
  unsigned char* p = static_cast<unsigned char*>(base);
  int32_t* active = reinterpret_cast<int32_t*>(p);
  p += align256(((size_t)E + 1) * sizeof(int32_t));
  float* max_x = reinterpret_cast<float*>(p);
  p += align256((size_t)T * sizeof(float));
  float* h = reinterpret_cast<float*>(p);

  moe::FfnArgs a;
  std::memset(&a, 0, sizeof a);
  a.records = experts->records;
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
  a.active = active;
  a.max_x = max_x;
  a.h = h;
  a.y_pairs = y_pairs;
  a.err = moe::ctx_error_word(ctx);
  if (moe::launch_active_from_offsets(offsets, E, active, false, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::launch_token_absmax(x, x_dtype, T, d, max_x, true, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::launch_mxfp4_ffn(a, moe_ctx_num_sms(ctx), true, stream) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // extern "C"

// project.cu -- the latent projections either side of the routed experts
// (LazyLoRA README, "The engine": the experts work in a 3584-wide latent
// space entered by a projection from the model's hidden width and left by a
// projection back; the hidden width is a parameter).
//
//   y[t][n] = resid[t][n] + sum_k W[n][k] * x[t][k]      (resid optional)
//
// W row-major [N][K] (bf16 or fp32), x [T][K], y [T][N] (fp32, or bf16
// rounded to nearest even).  The projection streams W once per pass of up to
// 8 tokens: each warp owns two rows and walks K in 16-byte pieces per lane,
// four pieces of each row in flight, multiplying by the pass's tokens (read
// through L1, where every warp of the CTA finds them) with fp32 fused
// multiply-adds; bf16 x bf16 products are exact in fp32.  A reduce-scatter
// over the lanes ends with one (row, token) sum per lane.
#include <cuda_bf16.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = 2;
constexpr int kTok = 8;     // tokens per pass
constexpr int kUnroll = 4;  // 16-byte pieces of each row in flight per lane

template <typename T>
struct Piece;  // one 16-byte piece of a row: its element count and loads as fp32
template <>
struct Piece<uint16_t> {  // bf16
  static constexpr int N = 8;
  static __device__ __forceinline__ void unpack(const uint4& q, float (&f)[8]) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};
template <>
struct Piece<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void unpack(const uint4& q, float (&f)[4]) {
    f[0] = __uint_as_float(q.x);
    f[1] = __uint_as_float(q.y);
    f[2] = __uint_as_float(q.z);
    f[3] = __uint_as_float(q.w);
  }
};

// Sum of v[i] over the 32 lanes for 16 values: lane l ends with value l & 15.
__device__ __forceinline__ float reduce_scatter16(float (&v)[16], int lane) {
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], 16);
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < m; ++i) {
      const float send = upper ? v[i] : v[i + m];
      const float keep = upper ? v[i + m] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  }
  return v[0];
}

// PN consecutive activations from element offset o (a multiple of PN) as fp32.
template <int PN>
__device__ __forceinline__ void load_x(const void* x, int dtype, size_t o, float (&f)[PN]) {
  if (dtype == MOE_BF16) {
    const uint16_t* xb = static_cast<const uint16_t*>(x) + o;
    if constexpr (PN == 8) {
      Piece<uint16_t>::unpack(__ldg(reinterpret_cast<const uint4*>(xb)), reinterpret_cast<float(&)[8]>(f));
    } else {
      const uint2 q = __ldg(reinterpret_cast<const uint2*>(xb));
      f[0] = __uint_as_float(q.x << 16);
      f[1] = __uint_as_float(q.x & 0xFFFF0000u);
      f[2] = __uint_as_float(q.y << 16);
      f[3] = __uint_as_float(q.y & 0xFFFF0000u);
    }
  } else {
    const float4* xf = reinterpret_cast<const float4*>(static_cast<const float*>(x) + o);
#pragma unroll
    for (int i = 0; i < PN / 4; ++i) {
      const float4 v = __ldg(xf + i);
      f[4 * i] = v.x;
      f[4 * i + 1] = v.y;
      f[4 * i + 2] = v.z;
      f[4 * i + 3] = v.w;
    }
  }
}

struct ProjArgs {
  const void* x;
  int x_dtype;
  const void* w;
  const void* resid;  // [T][N] or null
  int resid_dtype;
  void* y;
  int y_dtype;
  int T, K, N;
};

template <typename WT>
__global__ void __launch_bounds__(kThreads) project_kernel(const ProjArgs a) {
  constexpr int PN = Piece<WT>::N;  // elements per 16-byte piece of W
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = (blockIdx.x * kWarps + warp) * kRowsPerWarp;
  if (row0 >= a.N) return;
  const int nrows = min(kRowsPerWarp, a.N - row0);
  const WT* w = static_cast<const WT*>(a.w);
  const int pieces = a.K / PN;  // K is a multiple of 32
  for (int t0 = 0; t0 < a.T; t0 += kTok) {
    const int nt = min(kTok, a.T - t0);
    float acc[kRowsPerWarp][kTok];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
      for (int t = 0; t < kTok; ++t) acc[r][t] = 0.f;
    for (int p0 = lane; p0 < pieces; p0 += 32 * kUnroll) {
      uint4 q[kUnroll][kRowsPerWarp];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int p = p0 + 32 * u;
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
          q[u][r] = (p < pieces && r < nrows)
                        ? __ldg(reinterpret_cast<const uint4*>(w + (size_t)(row0 + r) * a.K) + p)
                        : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int p = p0 + 32 * u;
        if (p >= pieces) break;
        float wf[kRowsPerWarp][PN];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) Piece<WT>::unpack(q[u][r], wf[r]);
        const int k0 = p * PN;
#pragma unroll
        for (int t = 0; t < kTok; ++t) {
          if (t >= nt) break;
          float xf[PN];
          load_x<PN>(a.x, a.x_dtype, (size_t)(t0 + t) * a.K + k0, xf);
#pragma unroll
          for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
            for (int i = 0; i < PN; ++i) acc[r][t] = fmaf(wf[r][i], xf[i], acc[r][t]);
        }
      }
    }
    float v[16];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
      for (int t = 0; t < kTok; ++t) v[r * kTok + t] = acc[r][t];
    const float s = reduce_scatter16(v, lane);
    const int r = (lane & 15) / kTok, t = (lane & 15) % kTok;
    if (lane < 16 && r < nrows && t < nt) {
      const size_t o = (size_t)(t0 + t) * a.N + row0 + r;
      float yv = s;
      if (a.resid) yv += load_act(a.resid, a.resid_dtype, o);
      if (a.y_dtype == MOE_BF16)
        static_cast<__nv_bfloat16*>(a.y)[o] = __float2bfloat16_rn(yv);
      else
        static_cast<float*>(a.y)[o] = yv;
    }
  }
}

}  // namespace

cudaError_t launch_project(const void* x, int x_dtype, const void* w, int w_dtype, const void* resid, int resid_dtype,
                           void* y, int y_dtype, int T, int K, int N, bool pdl, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  ProjArgs a{x, x_dtype, w, resid, resid_dtype, y, y_dtype, T, K, N};
  const dim3 grid((N + kWarps * kRowsPerWarp - 1) / (kWarps * kRowsPerWarp));
  if (w_dtype == MOE_BF16) return launch("project", project_kernel<uint16_t>, grid, dim3(kThreads), 0, s, pdl, a);
  return launch("project", project_kernel<float>, grid, dim3(kThreads), 0, s, pdl, a);
}

}  // namespace moe

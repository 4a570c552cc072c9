// combine.cu -- gate-weighted sum of the selected experts' outputs added to the
// residual ("Running a 2.78-Trillion-Parameter Model Across Two Desks", Act II:
// the layer hands back the weighted sum of the experts it ran).
//   out[t][i] = x[t][i] + sum over j ascending, gates[t][j] != 0, of
//               gates[t][j] * y_pairs[t*k + j][i]      (fp32 fma chain)
// A pair with gate 0 is never read.  bf16 output is the fp32 result rounded to
// nearest even.
#include <cuda_bf16.h>

#include <utility>

#include "moe_internal.cuh"

namespace moe {
namespace {

__global__ void combine_kernel(const CombineArgs a) {
  pdl_wait();
  const int t = blockIdx.y;
  const int i4 = blockIdx.x * blockDim.x + threadIdx.x;
  if (4 * i4 >= a.d) return;
  // groups of 16 slots: the gates, then all 16 y loads (independent of each
  // other), then the fma chain in ascending j
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < a.k; j0 += 16) {
    float g[16];
    float4 y[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) g[u] = j0 + u < a.k ? a.gates[(size_t)t * a.k + j0 + u] : 0.f;
#pragma unroll
    for (int u = 0; u < 16; ++u)
      if (g[u] != 0.f) y[u] = reinterpret_cast<const float4*>(a.y_pairs + ((size_t)t * a.k + j0 + u) * a.d)[i4];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      if (g[u] == 0.f) continue;
      acc.x = fmaf(g[u], y[u].x, acc.x);
      acc.y = fmaf(g[u], y[u].y, acc.y);
      acc.z = fmaf(g[u], y[u].z, acc.z);
      acc.w = fmaf(g[u], y[u].w, acc.w);
    }
  }
  const size_t o = (size_t)t * a.d + 4 * (size_t)i4;
  if (a.x) {
    acc.x += load_act(a.x, a.x_dtype, o);
    acc.y += load_act(a.x, a.x_dtype, o + 1);
    acc.z += load_act(a.x, a.x_dtype, o + 2);
    acc.w += load_act(a.x, a.x_dtype, o + 3);
  }
  if (a.out_dtype == MOE_BF16) {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + o;
    out[0] = __float2bfloat16_rn(acc.x);
    out[1] = __float2bfloat16_rn(acc.y);
    out[2] = __float2bfloat16_rn(acc.z);
    out[3] = __float2bfloat16_rn(acc.w);
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(a.out) + o) = acc;
  }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, bool pdl, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  const int n4 = a.d / 4;
  const int threads = n4 < 256 ? ((n4 + 31) / 32) * 32 : 256;
  const dim3 grid((n4 + threads - 1) / threads, a.T);
  return launch("combine", combine_kernel, grid, dim3(threads), 0, s, pdl, a);
}

}  // namespace moe

// combine.cu -- gate-weighted sum of the selected experts' outputs added to the
// residual ("Running a 2.78-Trillion-Parameter Model Across Two Desks", Act II:
// the layer hands back the weighted sum of the experts it ran).
//   out[t][i] = x[t][i] + sum over j ascending, gates[t][j] != 0, of
//               gates[t][j] * y_pairs[t*k + j][i]      (fp32 fma chain)
// where a pair's y may arrive as partial sums over K slices, added first.
// A pair with gate 0 never enters the sum.  bf16 output is the fp32 result
// rounded to nearest even.
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
  const size_t o = (size_t)t * a.d + 4 * (size_t)i4;
  // The residual, the gates and the pairs' outputs are loaded together (none of
  // these loads waits for a gate): one memory round trip instead of three.  A
  // pair whose gate is 0 may be loaded but never enters the sum.
  float4 xr = make_float4(0.f, 0.f, 0.f, 0.f);
  if (a.x) {
    xr.x = load_act(a.x, a.x_dtype, o);
    xr.y = load_act(a.x, a.x_dtype, o + 1);
    xr.z = load_act(a.x, a.x_dtype, o + 2);
    xr.w = load_act(a.x, a.x_dtype, o + 3);
  }
  // groups of 16 slots: the gates and the y loads, then the fma chain in ascending j
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < a.k; j0 += 16) {
    float g[16];
    float4 y[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      g[u] = 0.f;
      if (j0 + u < a.k) {
        g[u] = a.gates[(size_t)t * a.k + j0 + u];
        y[u] = reinterpret_cast<const float4*>(a.y_pairs + ((size_t)t * a.k + j0 + u) * a.d)[i4];
      }
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      if (g[u] == 0.f) continue;
      acc.x = fmaf(g[u], y[u].x, acc.x);
      acc.y = fmaf(g[u], y[u].y, acc.y);
      acc.z = fmaf(g[u], y[u].z, acc.z);
      acc.w = fmaf(g[u], y[u].w, acc.w);
    }
  }
  if (a.x) {
    acc.x += xr.x;
    acc.y += xr.y;
    acc.z += xr.z;
    acc.w += xr.w;
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

// Pairs whose outputs arrive as nparts partial sums: a CTA owns 128 columns
// of one token and its 8 warps split the token's pairs, each lane loading all
// the partials of its 4 columns at once and adding them in ascending order;
// the per-pair sums meet in shared memory, where warp 0 runs the ascending
// gate chain.  Same order of operations as combine_kernel, so the same bits.
constexpr int kPartsWarps = 8;
constexpr int kPartsInFlight = 16;

__global__ void __launch_bounds__(32 * kPartsWarps) combine_parts_kernel(const CombineArgs a) {
  extern __shared__ float4 ysum[];  // [k][32]
  pdl_wait();
  const int t = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n4 = a.d / 4;
  const int i4 = blockIdx.x * 32 + lane;
  const bool col = i4 < n4;
  for (int j = warp; j < a.k; j += kPartsWarps) {
    const float g = a.gates[(size_t)t * a.k + j];
    if (g == 0.f || !col) continue;
    const float4* src = reinterpret_cast<const float4*>(a.y_pairs + ((size_t)t * a.k + j) * a.nparts * a.d) + i4;
    float4 s;
    if (a.nparts <= kPartsInFlight) {
      float4 v[kPartsInFlight];
#pragma unroll
      for (int q = 0; q < kPartsInFlight; ++q)
        if (q < a.nparts) v[q] = src[(size_t)q * n4];
      s = v[0];
#pragma unroll
      for (int q = 1; q < kPartsInFlight; ++q) {
        if (q >= a.nparts) break;
        s.x += v[q].x;
        s.y += v[q].y;
        s.z += v[q].z;
        s.w += v[q].w;
      }
    } else {
      s = src[0];
      for (int q = 1; q < a.nparts; ++q) {
        const float4 v = src[(size_t)q * n4];
        s.x += v.x;
        s.y += v.y;
        s.z += v.z;
        s.w += v.w;
      }
    }
    ysum[j * 32 + lane] = s;
  }
  __syncthreads();
  if (warp != 0 || !col) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < a.k; ++j) {
    const float g = a.gates[(size_t)t * a.k + j];
    if (g == 0.f) continue;
    const float4 y = ysum[j * 32 + lane];
    acc.x = fmaf(g, y.x, acc.x);
    acc.y = fmaf(g, y.y, acc.y);
    acc.z = fmaf(g, y.z, acc.z);
    acc.w = fmaf(g, y.w, acc.w);
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
  if (a.nparts > 1) {
    const size_t smem = (size_t)a.k * 32 * sizeof(float4);
    if (smem > 48 * 1024) return cudaErrorInvalidValue;  // k <= 96
    const dim3 grid((a.d / 4 + 31) / 32, a.T);
    return launch("combine", combine_parts_kernel, grid, dim3(32 * kPartsWarps), smem, s, pdl, a);
  }
  const int n4 = a.d / 4;
  // few tokens: small blocks, so that the gathers of one token spread over many SMs
  const int tmax = a.T <= 4 ? 64 : 256;
  const int threads = n4 < tmax ? ((n4 + 31) / 32) * 32 : tmax;
  const dim3 grid((n4 + threads - 1) / threads, a.T);
  return launch("combine", combine_kernel, grid, dim3(threads), 0, s, pdl, a);
}

}  // namespace moe

// router.cu -- router logits and certified top-k (LazyLoRA README, "File map":
// top-16 gating over the 896 routed experts with an additive score-correction
// bias; "Running a 2.78-Trillion-Parameter Model Across Two Desks", Act II).
//
// Logits are fp32 sums with a rigorous error bound per logit
//   |l32 - l_ref| <= gamma * ||W_e||_2 * ||x_t||_2 + 2^-23 |l32|,
// where l_ref is the logit summed in fp64 in ascending i.  The top-k kernel
// accepts the fp32 selection only when the bounds prove both the membership
// and the order of the selected experts; otherwise the undecided candidates are
// recomputed in fp64 (parallel, with its own bound) and, if still undecided,
// by one thread with a sequential fp64 sum in ascending i, which reproduces
// l_ref exactly (bf16 x bf16 and fp32 x fp32 products are exact in fp64).
#include <utility>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kLogitWarps = 8;
constexpr int kTokTile = 4;

template <typename T>
struct Vec16;  // 16 bytes of weights as floats
template <>
struct Vec16<uint16_t> {
  static constexpr int N = 8;
  __device__ static void load(const void* base, size_t elem, float* out) {
    uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + elem));
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out[2 * i] = __uint_as_float(w[i] << 16);
      out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ static void load(const void* base, size_t elem, float* out) {
    float4 v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem));
    out[0] = v.x;
    out[1] = v.y;
    out[2] = v.z;
    out[3] = v.w;
  }
};

// One warp per expert row, up to kTokTile tokens per CTA (x staged in shared
// memory as fp32).  Each lane keeps one accumulator per element position of
// its 16-byte chunk; the depth of the summation tree is d/(32N) + log2(N) + 5.
template <typename WT>
__global__ void __launch_bounds__(kLogitWarps * 32) router_logits_kernel(RouteArgs a) {
  extern __shared__ float xs[];  // [kTokTile][d]
  constexpr int N = Vec16<WT>::N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.y * kTokTile;
  const int nt = min(kTokTile, a.T - t0);
  const int d = a.d;
  pdl_wait();
  for (int i = threadIdx.x; i < nt * d; i += blockDim.x)
    xs[i] = load_act(a.x, a.x_dtype, (size_t)t0 * d + i);
  __syncthreads();
  if (blockIdx.x == 0 && warp < nt) {  // ||x_t||_2
    float s = 0.f;
    for (int i = lane; i < d; i += 32) s = fmaf(xs[warp * d + i], xs[warp * d + i], s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) a.nrm_x[t0 + warp] = sqrtf(s);
  }
  const int e = blockIdx.x * kLogitWarps + warp;
  if (e >= a.E) return;
  float acc[kTokTile][N];
#pragma unroll
  for (int t = 0; t < kTokTile; ++t)
#pragma unroll
    for (int m = 0; m < N; ++m) acc[t][m] = 0.f;
  float sq = 0.f;
  const size_t row = (size_t)e * d;
  for (int c = lane * N; c < d; c += 32 * N) {
    float w[N];
    Vec16<WT>::load(a.w, row + c, w);
#pragma unroll
    for (int m = 0; m < N; ++m) sq = fmaf(w[m], w[m], sq);
#pragma unroll
    for (int t = 0; t < kTokTile; ++t) {
      if (t < nt) {
        const float4* xv = reinterpret_cast<const float4*>(xs + t * d + c);  // d, c multiples of 4
#pragma unroll
        for (int q = 0; q < N / 4; ++q) {
          float4 x4 = xv[q];
          acc[t][4 * q + 0] = fmaf(w[4 * q + 0], x4.x, acc[t][4 * q + 0]);
          acc[t][4 * q + 1] = fmaf(w[4 * q + 1], x4.y, acc[t][4 * q + 1]);
          acc[t][4 * q + 2] = fmaf(w[4 * q + 2], x4.z, acc[t][4 * q + 2]);
          acc[t][4 * q + 3] = fmaf(w[4 * q + 3], x4.w, acc[t][4 * q + 3]);
        }
      }
    }
  }
  if (blockIdx.y == 0) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if (lane == 0) a.nrm_w[e] = sqrtf(sq);
  }
  const float b = a.bias ? a.bias[e] : 0.f;
#pragma unroll
  for (int t = 0; t < kTokTile; ++t) {
    if (t >= nt) break;
#pragma unroll
    for (int w = N / 2; w > 0; w >>= 1)
#pragma unroll
      for (int m = 0; m < w; ++m) acc[t][m] += acc[t][m + w];
    float s = acc[t][0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) a.logits[(size_t)(t0 + t) * a.E + e] = s + b;
  }
}

// ---------------------------------------------------------------- top-k
constexpr int kTopkThreads = 128;

struct Key {  // ordering (value descending, index ascending)
  double v;
  int e;
};
__device__ __forceinline__ bool better(double v1, int e1, double v2, int e2) {
  return v1 > v2 || (v1 == v2 && e1 < e2);
}

__device__ __forceinline__ double load_d(const void* p, int dtype, size_t i) {
  if (dtype == MOE_BF16) return (double)bf16_bits_to_f32(static_cast<const uint16_t*>(p)[i]);
  return (double)static_cast<const float*>(p)[i];
}

// fp64 logit by one warp: lanes take i = lane, lane+32, ... sequentially, then
// a shuffle tree.  Returns the value and sum |w_i x_i| (both on every lane).
__device__ void logit_fp64_warp(const RouteArgs& a, int t, int e, double* val, double* abs_sum) {
  const int lane = threadIdx.x & 31;
  double s = 0.0, sa = 0.0;
  const size_t xr = (size_t)t * a.d, wr = (size_t)e * a.d;
  for (int i = lane; i < a.d; i += 32) {
    double p = load_d(a.w, a.w_dtype, wr + i) * load_d(a.x, a.x_dtype, xr + i);
    s += p;
    sa += fabs(p);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    sa += __shfl_xor_sync(0xffffffffu, sa, o);
  }
  *val = s + (a.bias ? (double)a.bias[e] : 0.0);
  *abs_sum = sa;
}

// The reference arithmetic itself: sequential fp64 sum in ascending i, then the
// bias.  Every product is exact in fp64, so fma equals multiply-then-add.
__device__ double logit_fp64_sequential(const RouteArgs& a, int t, int e) {
  double s = 0.0;
  const size_t xr = (size_t)t * a.d, wr = (size_t)e * a.d;
  for (int i = 0; i < a.d; ++i) s = fma(load_d(a.w, a.w_dtype, wr + i), load_d(a.x, a.x_dtype, xr + i), s);
  if (a.bias) s += (double)a.bias[e];
  return s;
}

__device__ __forceinline__ double gamma64(int n) {
  const double u = 1.1102230246251565e-16;  // 2^-53
  return n * u / (1.0 - n * u);
}

// One CTA per token.
// Dynamic shared memory layout for E experts (topk_smem_bytes).
__host__ __device__ inline size_t topk_smem_bytes(int E) {
  size_t e8 = ((size_t)E + 7) / 8 * 8;
  return e8 * (2 * sizeof(double) + 3 * sizeof(float) + 2);
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(RouteArgs a) {
  extern __shared__ double dsm[];
  const size_t e8 = ((size_t)a.E + 7) / 8 * 8;
  double* clo = dsm;                                              // rare path: candidate bounds
  double* chi = clo + e8;
  float* sv = reinterpret_cast<float*>(chi + e8);                 // fp32 logits
  float* sb = sv + e8;                                            // their error bounds
  int* cand = reinterpret_cast<int*>(sb + e8);                    // rare path: candidate experts
  unsigned char* taken = reinterpret_cast<unsigned char*>(cand + e8);
  unsigned char* cflag = taken + e8;
  __shared__ int sel[kMaxK + 1];
  __shared__ int n_cand, certified;
  __shared__ int order[kMaxK];
  __shared__ double oval[kMaxK];

  const int t = blockIdx.x;
  const int E = a.E, k = a.k;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  const float nx = a.nrm_x[t];
  for (int e = tid; e < E; e += blockDim.x) {
    float v = a.logits[(size_t)t * E + e];
    sv[e] = v;
    sb[e] = a.gamma * a.nrm_w[e] * nx + 1.2e-7f * fabsf(v) + 1e-30f;
    taken[e] = 0;
  }
  __syncthreads();
  pdl_launch_dependents();
  const int nsel = min(k + 1, E);
  if (warp == 0) {
    for (int j = 0; j < nsel; ++j) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
      for (int e = lane; e < E; e += 32)
        if (!taken[e] && (sv[e] > bv || (sv[e] == bv && e < be))) {
          bv = sv[e];
          be = e;
        }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if (lane == 0) {
        sel[j] = be;
        taken[be] = 1;
      }
      __syncwarp();
    }
    // certification: strict separation of consecutive selected experts, and
    // every outsider's upper bound below the lowest selected lower bound
    int ok = 1;
    float m = INFINITY;
    for (int j = 0; j < k; ++j) {
      float lo = sv[sel[j]] - sb[sel[j]];
      m = fminf(m, lo);
      if (j + 1 < k && !(lo > sv[sel[j + 1]] + sb[sel[j + 1]])) ok = 0;
    }
    float hi_out = -INFINITY;
    for (int e = lane; e < E; e += 32) {
      bool in = false;
      for (int j = 0; j < k; ++j) in |= (sel[j] == e);
      if (!in) hi_out = fmaxf(hi_out, sv[e] + sb[e]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) hi_out = fmaxf(hi_out, __shfl_xor_sync(0xffffffffu, hi_out, o));
    if (!(hi_out < m)) ok = 0;
    if (lane == 0) {
      certified = ok;
      for (int j = 0; j < k; ++j) {
        order[j] = sel[j];
        oval[j] = (double)sv[sel[j]];
      }
    }
  }
  __syncthreads();

  if (!certified) {
    // ---- rare path: candidates that could be in the top-k ----------------
    if (tid == 0) {
      float m = INFINITY;
      for (int j = 0; j < k; ++j) m = fminf(m, sv[sel[j]] - sb[sel[j]]);
      int n = 0;
      for (int e = 0; e < E; ++e) {
        bool in = false;
        for (int j = 0; j < k; ++j) in |= (sel[j] == e);
        if (in || sv[e] + sb[e] >= m) {
          cand[n] = e;
          clo[n] = (double)sv[e] - (double)sb[e];
          chi[n] = (double)sv[e] + (double)sb[e];
          ++n;
        }
      }
      n_cand = n;
    }
    __syncthreads();
    const int n = n_cand;
    // pass 1: candidates whose interval meets another one's get an fp64 value
    for (int c = tid; c < n; c += blockDim.x) {
      unsigned char f = 0;
      for (int c2 = 0; c2 < n; ++c2)
        if (c2 != c && !(clo[c] > chi[c2] || chi[c] < clo[c2])) f = 1;
      cflag[c] = f;
    }
    __syncthreads();
    const double bound_scale = (gamma64(a.d / 32 + 6) + gamma64(a.d + 1)) * 1.001;
    for (int c = warp; c < n; c += kTopkThreads / 32) {
      if (!cflag[c]) continue;
      double v, sa;
      logit_fp64_warp(a, t, cand[c], &v, &sa);
      if (lane == 0) {
        double bd = bound_scale * sa + 4.5e-16 * fabs(v) + 1e-300;
        clo[c] = v - bd;
        chi[c] = v + bd;
      }
    }
    __syncthreads();
    // pass 2: still undecided -> the reference's own sequential fp64 sum
    for (int c = tid; c < n; c += blockDim.x) {
      unsigned char f = 0;
      for (int c2 = 0; c2 < n; ++c2)
        if (c2 != c && !(clo[c] > chi[c2] || chi[c] < clo[c2])) f = 1;
      cflag[c] = f;
    }
    __syncthreads();
    for (int c = tid; c < n; c += blockDim.x) {
      if (!cflag[c]) continue;
      double v = logit_fp64_sequential(a, t, cand[c]);
      clo[c] = v;
      chi[c] = v;
    }
    __syncthreads();
    // order the candidates: disjoint intervals order by midpoint; overlapping
    // ones are now exact and order by value, ties by expert index
    if (warp == 0) {
      for (int j = 0; j < k; ++j) {
        double bv = -INFINITY;
        int be = 0x7fffffff, bc = -1;
        for (int c = lane; c < n; c += 32) {
          if (cflag[c] == 2) continue;
          double mid = 0.5 * (clo[c] + chi[c]);
          if (bc < 0 || better(mid, cand[c], bv, be)) {
            bv = mid;
            be = cand[c];
            bc = c;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          double ov = __shfl_xor_sync(0xffffffffu, bv, o);
          int oe = __shfl_xor_sync(0xffffffffu, be, o);
          int oc = __shfl_xor_sync(0xffffffffu, bc, o);
          if (oc >= 0 && (bc < 0 || better(ov, oe, bv, be))) {
            bv = ov;
            be = oe;
            bc = oc;
          }
        }
        if (lane == 0) {
          order[j] = be;
          oval[j] = bv;
          cflag[bc] = 2;
        }
        __syncwarp();
      }
    }
    __syncthreads();
  }

  if (tid == 0) {
    double den = 0.0;
    for (int j = 0; j < k; ++j) den += exp(oval[j] - oval[0]);
    for (int j = 0; j < k; ++j) {
      a.topk_idx[(size_t)t * k + j] = order[j];
      a.gates[(size_t)t * k + j] = (float)(exp(oval[j] - oval[0]) / den);
    }
  }
}

}  // namespace

cudaError_t launch_route_topk(const RouteArgs& a, int num_sms, cudaStream_t s) {
  (void)num_sms;
  if (a.T == 0) return cudaSuccess;
  dim3 grid((a.E + kLogitWarps - 1) / kLogitWarps, (a.T + kTokTile - 1) / kTokTile);
  size_t smem = (size_t)kTokTile * a.d * sizeof(float);
  cudaError_t err;
  if (a.w_dtype == MOE_BF16) {
    cudaFuncSetAttribute(router_logits_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    err = launch("router_logits", router_logits_kernel<uint16_t>, grid, dim3(kLogitWarps * 32), smem, s, false, a);
  } else {
    cudaFuncSetAttribute(router_logits_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    err = launch("router_logits", router_logits_kernel<float>, grid, dim3(kLogitWarps * 32), smem, s, false, a);
  }
  if (err != cudaSuccess) return err;
  size_t tsm = topk_smem_bytes(a.E);
  cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tsm);
  return launch("topk", topk_kernel, dim3(a.T), dim3(kTopkThreads), tsm, s, true, a);
}

}  // namespace moe

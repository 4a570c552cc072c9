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
//
// The score-correction bias either joins the logits (selection and gates), or
// steers the selection only: the top-k then ranks fl(l32 + bias) (one more
// rounding in the bound) and takes the gates from l32 itself.  A layer's
// shared experts (LazyLoRA README, "The engine": 2 per MoE layer) close every
// token's row of the routing with gate 1, so that the bucketing, the expert
// FFN and the combine treat them as ordinary pairs.
#include <utility>

#include "bucket_body.cuh"

namespace moe {
namespace {

constexpr int kLogitWarps = 8;
constexpr int kTokTile = 4;
constexpr int kLoadBatch = 16;  // 16-byte chunks each lane has in flight

template <typename T>
struct Vec16;  // 16 bytes of router weights as floats
template <>
struct Vec16<uint16_t> {
  static constexpr int N = 8;
  __device__ static void unpack(const uint4 v, float* out) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
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
  __device__ static void unpack(const uint4 v, float* out) {
    out[0] = __uint_as_float(v.x);
    out[1] = __uint_as_float(v.y);
    out[2] = __uint_as_float(v.z);
    out[3] = __uint_as_float(v.w);
  }
};

// Stages x[t0 .. t0+nt) into shared memory as fp32, 8 (bf16) or 4 (fp32)
// elements per 16-byte load.
__device__ __forceinline__ void stage_x(const RouteArgs& a, int t0, int nt, float* xs) {
  const int d = a.d;
  if (a.x_dtype == MOE_BF16) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + (size_t)t0 * d);
    for (int i = threadIdx.x; i < nt * d / 8; i += blockDim.x) {
      const uint4 v = src[i];
      float4* dst = reinterpret_cast<float4*>(xs + 8 * i);
      dst[0] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                           __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
      dst[1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u),
                           __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u));
    }
  } else {
    const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + (size_t)t0 * d);
    for (int i = threadIdx.x; i < nt * d / 4; i += blockDim.x) reinterpret_cast<float4*>(xs)[i] = src[i];
  }
}

// ||x_t||_2 and max_i |x_t[i]| of one staged token, by one warp.
__device__ __forceinline__ void token_stats(const RouteArgs& a, const float* xt, int t) {
  const int lane = threadIdx.x & 31;
  float s = 0.f, m = 0.f;
  for (int i = lane; i < a.d; i += 32) {
    s = fmaf(xt[i], xt[i], s);
    m = fmaxf(m, fabsf(xt[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  }
  if (lane == 0) {
    a.nrm_x[t] = sqrtf(s);
    a.max_x[t] = m;
  }
}

// Error-free transformation (Knuth's TwoSum): s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// kRowsPerWarp expert rows per warp, taken one after the other, up to
// kTokTile tokens per CTA (x staged in shared memory as fp32 once for the
// CTA's kLogitWarps * kRowsPerWarp rows).  Lane chunk c covers columns
// (32c + lane) * N .. + N, and the lane keeps one accumulator per element
// position of its chunk, so the depth of the summation tree is
// ceil(d/(32N)) + log2(N) + 5.  The weights do not depend on the previous
// kernel, so a lane issues the loads of its first row's first kLoadBatch
// chunks before waiting for it.
constexpr int kRowsPerWarp = 4;
template <typename WT>
__global__ void __launch_bounds__(kLogitWarps * 32) router_logits_kernel(RouteArgs a) {
  extern __shared__ float xs[];  // [kTokTile][d]
  constexpr int N = Vec16<WT>::N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.y * kTokTile;
  const int nt = min(kTokTile, a.T - t0);
  const int d = a.d;
  const int nch = d / (32 * N);        // whole warp-wide chunk rows
  const int rem = d - nch * 32 * N;    // columns left over (a multiple of N)
  const int e_first = (blockIdx.x * kLogitWarps + warp) * kRowsPerWarp;
  uint4 wv[kLoadBatch];
  {
    const uint4* wrow =
        reinterpret_cast<const uint4*>(static_cast<const WT*>(a.w) + (size_t)(e_first < a.E ? e_first : 0) * d);
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u)
      if (e_first < a.E && u < nch) wv[u] = __ldg(wrow + u * 32 + lane);
  }
  pdl_wait();
  stage_x(a, t0, nt, xs);
  __syncthreads();
  if (blockIdx.x == 0 && warp < nt) token_stats(a, xs + warp * d, t0 + warp);
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int e = e_first + r;
    if (e >= a.E) break;
    const uint4* wrow = reinterpret_cast<const uint4*>(static_cast<const WT*>(a.w) + (size_t)e * d);
    if (r > 0) {
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u)
        if (u < nch) wv[u] = __ldg(wrow + u * 32 + lane);
    }
    float acc[kTokTile][N];
#pragma unroll
    for (int t = 0; t < kTokTile; ++t)
#pragma unroll
      for (int m = 0; m < N; ++m) acc[t][m] = 0.f;
    float sq = 0.f;
    auto consume = [&](const uint4 raw, int c) {
      float w[N];
      Vec16<WT>::unpack(raw, w);
#pragma unroll
      for (int m = 0; m < N; ++m) sq = fmaf(w[m], w[m], sq);
#pragma unroll
      for (int t = 0; t < kTokTile; ++t) {
        if (t < nt) {
          const float4* xv = reinterpret_cast<const float4*>(xs + t * d + c);  // d, c multiples of 4
#pragma unroll
          for (int q = 0; q < N / 4; ++q) {
            const float4 x4 = xv[q];
            acc[t][4 * q + 0] = fmaf(w[4 * q + 0], x4.x, acc[t][4 * q + 0]);
            acc[t][4 * q + 1] = fmaf(w[4 * q + 1], x4.y, acc[t][4 * q + 1]);
            acc[t][4 * q + 2] = fmaf(w[4 * q + 2], x4.z, acc[t][4 * q + 2]);
            acc[t][4 * q + 3] = fmaf(w[4 * q + 3], x4.w, acc[t][4 * q + 3]);
          }
        }
      }
    };
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u)
      if (u < nch) consume(wv[u], (u * 32 + lane) * N);
    for (int cb = kLoadBatch; cb < nch; cb += kLoadBatch) {
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u)
        if (cb + u < nch) wv[u] = __ldg(wrow + (cb + u) * 32 + lane);
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u)
        if (cb + u < nch) consume(wv[u], ((cb + u) * 32 + lane) * N);
    }
    if (lane * N < rem) consume(__ldg(wrow + nch * 32 + lane), (nch * 32 + lane) * N);
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
  pdl_launch_dependents();
}

// Tiled form for bf16 x and W with d a multiple of 256 (the prefill router):
// 8 tokens staged per CTA as fp32 with the two halves of every 8-element chunk
// stored apart (xs[(2t + h) * d/8 + c] holds elements 8c + 4h .. 8c + 4h + 3
// of token t), so that lane l's loads of chunk c = 32u + l are conflict-free;
// each warp takes 4 expert rows against all 8 tokens, one accumulator per
// (row, token) and lane, so that a staged token feeds 4 rows and a loaded
// weight chunk 8 tokens.  Per chunk the lane sums each half's 4 products as an
// fma chain started by an exact product (bf16 x bf16 fits fp32) and adds the
// two halves, then adds the chunk sum to its accumulator in ascending chunk
// order; the lanes join in a 5-level tree.  A product thus passes through at
// most 3 + 1 + (d/256 - 1) + 5 = d/256 + 8 roundings, the depth of
// router_logits_kernel's tree that the error bound assumes.
constexpr int kTiledTok = 8;   // tokens staged per CTA
constexpr int kTiledRows = 4;  // expert rows per warp
constexpr int kTiledExperts = kLogitWarps * kTiledRows;

__host__ __device__ inline size_t tiled_smem_bytes(int d) { return (size_t)kTiledTok * d * sizeof(float); }

// Sum over the 32 lanes of each of v[0..31]: lane l ends with the sum of v[l]
// (a 5-level tree per value, one shuffle per value and level halved each time).
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
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

__global__ void __launch_bounds__(kLogitWarps * 32, 2) router_logits_tiled_kernel(RouteArgs a) {
  extern __shared__ float4 xs4[];  // [kTiledTok][2][d/8]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, nc = d / 8, nch = d / 256;
  const int t0 = blockIdx.y * kTiledTok;
  const int nt = min(kTiledTok, a.T - t0);
  // the warp's rows (clamped to the last expert; those sums are not written)
  const int e_first = blockIdx.x * kTiledExperts + warp * kTiledRows;
  const uint4* wrow[kTiledRows];
#pragma unroll
  for (int r = 0; r < kTiledRows; ++r)
    wrow[r] = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.w) +
                                             (size_t)min(e_first + r, a.E - 1) * d);
  // the first chunk's weights do not depend on the previous kernel
  uint4 wq[kTiledRows];
#pragma unroll
  for (int r = 0; r < kTiledRows; ++r) wq[r] = __ldg(wrow[r] + lane);
  pdl_wait();
  {  // stage the tokens (zeros past T)
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + (size_t)t0 * d);
    for (int i = threadIdx.x; i < kTiledTok * nc; i += blockDim.x) {
      const int t = i / nc, c = i % nc;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (t < nt) v = src[(size_t)t * nc + c];
      xs4[(2 * t) * nc + c] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                                          __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
      xs4[(2 * t + 1) * nc + c] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u),
                                              __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u));
    }
  }
  __syncthreads();
  if (blockIdx.x == 0 && warp < nt) {  // ||x_t|| and max|x_t|, in the order of token_stats
    const float* xf = reinterpret_cast<const float*>(xs4);
    float s = 0.f, m = 0.f;
    for (int i = lane; i < d; i += 32) {
      const int c = i >> 3, p = i & 7;
      const float v = xf[((2 * warp + (p >> 2)) * nc + c) * 4 + (p & 3)];
      s = fmaf(v, v, s);
      m = fmaxf(m, fabsf(v));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s += __shfl_xor_sync(0xffffffffu, s, o);
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    }
    if (lane == 0) {
      a.nrm_x[t0 + warp] = sqrtf(s);
      a.max_x[t0 + warp] = m;
    }
  }
  if (e_first >= a.E) {
    pdl_launch_dependents();
    return;
  }
  const bool norms = blockIdx.y == 0;
  float acc[kTiledRows * kTiledTok];  // [row][token]
  float sq[kTiledRows];
#pragma unroll
  for (int i = 0; i < kTiledRows * kTiledTok; ++i) acc[i] = 0.f;
#pragma unroll
  for (int r = 0; r < kTiledRows; ++r) sq[r] = 0.f;
  for (int u = 0; u < nch; ++u) {
    const int c = u * 32 + lane;
    float w[kTiledRows][8];
#pragma unroll
    for (int r = 0; r < kTiledRows; ++r) Vec16<uint16_t>::unpack(wq[r], w[r]);
    if (u + 1 < nch) {  // the next chunk's weights, in flight during this one
#pragma unroll
      for (int r = 0; r < kTiledRows; ++r) wq[r] = __ldg(wrow[r] + c + 32);
    }
    if (norms) {
#pragma unroll
      for (int r = 0; r < kTiledRows; ++r)
#pragma unroll
        for (int m = 0; m < 8; ++m) sq[r] = fmaf(w[r][m], w[r][m], sq[r]);
    }
#pragma unroll
    for (int t = 0; t < kTiledTok; ++t) {
      const float4 x0 = xs4[(2 * t) * nc + c], x1 = xs4[(2 * t + 1) * nc + c];
#pragma unroll
      for (int r = 0; r < kTiledRows; ++r) {
        float h0 = __fmul_rn(w[r][0], x0.x);
        h0 = __fmaf_rn(w[r][1], x0.y, h0);
        h0 = __fmaf_rn(w[r][2], x0.z, h0);
        h0 = __fmaf_rn(w[r][3], x0.w, h0);
        float h1 = __fmul_rn(w[r][4], x1.x);
        h1 = __fmaf_rn(w[r][5], x1.y, h1);
        h1 = __fmaf_rn(w[r][6], x1.z, h1);
        h1 = __fmaf_rn(w[r][7], x1.w, h1);
        acc[r * kTiledTok + t] = __fadd_rn(acc[r * kTiledTok + t], __fadd_rn(h0, h1));  // first add exact (acc = 0)
      }
    }
  }
  pdl_launch_dependents();
  const float s = reduce_scatter32(acc, lane);
  {
    const int r = lane / kTiledTok, t = lane % kTiledTok, e = e_first + r;
    if (t < nt && e < a.E) a.logits[(size_t)(t0 + t) * a.E + e] = s + (a.bias ? a.bias[e] : 0.f);
  }
  if (norms) {
#pragma unroll
    for (int r = 0; r < kTiledRows; ++r) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sq[r] += __shfl_xor_sync(0xffffffffu, sq[r], o);
      if (lane == 0 && e_first + r < a.E) a.nrm_w[e_first + r] = sqrtf(sq[r]);
    }
  }
}

// Compensated variant (used for small T; TT tokens per CTA, 1 when T = 1 so
// that the unrolled code stays small): per lane and token a running sum s,
// the exact rounding errors of the products and of the sums accumulated in c
// (Dot2 of Ogita, Rump and Oishi), and sum|p|; lanes merge with TwoSum.  Writes
// logits = fl(fl(s + c) + bias) and absdot = sum|p|.
template <typename WT, int TT>
__global__ void __launch_bounds__(kLogitWarps * 32) router_logits_comp_kernel(RouteArgs a) {
  extern __shared__ float xs[];  // [TT][d]
  constexpr int N = Vec16<WT>::N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.y * TT;
  const int nt = min(TT, a.T - t0);
  const int d = a.d;
  const int e = blockIdx.x * kLogitWarps + warp;
  const int nch = d / (32 * N);
  const int rem = d - nch * 32 * N;
  uint4 wv[kLoadBatch];
  const uint4* wrow = reinterpret_cast<const uint4*>(static_cast<const WT*>(a.w) + (size_t)(e < a.E ? e : 0) * d);
#pragma unroll
  for (int u = 0; u < kLoadBatch; ++u)
    if (e < a.E && u < nch) wv[u] = __ldg(wrow + u * 32 + lane);
  pdl_wait();
  stage_x(a, t0, nt, xs);
  __syncthreads();
  if (blockIdx.x == 0 && warp < nt) token_stats(a, xs + warp * d, t0 + warp);
  if (e >= a.E) return;
  // two independent compensated chains per token (even / odd element of each
  // chunk) for instruction-level parallelism; merged with TwoSum below
  float s[TT][2], c[TT][2], sa[TT];
#pragma unroll
  for (int t = 0; t < TT; ++t) {
    s[t][0] = s[t][1] = c[t][0] = c[t][1] = sa[t] = 0.f;
  }
  auto consume = [&](const uint4 raw, int col) {
    float w[N];
    Vec16<WT>::unpack(raw, w);
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      if (t < nt) {
        const float4* xv = reinterpret_cast<const float4*>(xs + t * d + col);  // d, col multiples of 4
        float xr[N];
#pragma unroll
        for (int q = 0; q < N / 4; ++q) {
          const float4 x4 = xv[q];
          xr[4 * q] = x4.x;
          xr[4 * q + 1] = x4.y;
          xr[4 * q + 2] = x4.z;
          xr[4 * q + 3] = x4.w;
        }
#pragma unroll
        for (int m = 0; m < N; ++m) {
          const int ch = m & 1;
          const float p = __fmul_rn(w[m], xr[m]);
          const float ep = __fmaf_rn(w[m], xr[m], -p);
          float t2, es;
          two_sum(s[t][ch], p, t2, es);
          s[t][ch] = t2;
          c[t][ch] = __fadd_rn(c[t][ch], __fadd_rn(es, ep));
          sa[t] = __fadd_rn(sa[t], fabsf(p));
        }
      }
    }
  };
#pragma unroll
  for (int u = 0; u < kLoadBatch; ++u)
    if (u < nch) consume(wv[u], (u * 32 + lane) * N);
  for (int cb = kLoadBatch; cb < nch; cb += kLoadBatch) {
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u)
      if (cb + u < nch) wv[u] = __ldg(wrow + (cb + u) * 32 + lane);
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u)
      if (cb + u < nch) consume(wv[u], ((cb + u) * 32 + lane) * N);
  }
  if (lane * N < rem) consume(__ldg(wrow + nch * 32 + lane), (nch * 32 + lane) * N);
  pdl_launch_dependents();
  const float b = a.bias ? a.bias[e] : 0.f;
#pragma unroll
  for (int t = 0; t < TT; ++t) {
    if (t >= nt) break;
    float st, ct, at = sa[t];
    {
      float es;
      two_sum(s[t][0], s[t][1], st, es);
      ct = __fadd_rn(__fadd_rn(c[t][0], c[t][1]), es);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float s2 = __shfl_xor_sync(0xffffffffu, st, o);
      const float c2 = __shfl_xor_sync(0xffffffffu, ct, o);
      at = __fadd_rn(at, __shfl_xor_sync(0xffffffffu, at, o));
      float t2, es;
      two_sum(st, s2, t2, es);
      st = t2;
      ct = __fadd_rn(__fadd_rn(ct, c2), es);
    }
    if (lane == 0) {
      a.logits[(size_t)(t0 + t) * a.E + e] = __fadd_rn(__fadd_rn(st, ct), b);
      a.absdot[(size_t)(t0 + t) * a.E + e] = at;
    }
  }
}

// ---------------------------------------------------------------- top-k
constexpr int kTopkThreads = 256;

// Eight consecutive elements i0 .. i0+7 (i0 a multiple of 8) of a bf16 or fp32
// row as doubles, with one or two 16-byte loads.
__device__ __forceinline__ void load8_d(const void* p, int dtype, size_t i0, double (&v)[8]) {
  if (dtype == MOE_BF16) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p) + i0));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = (double)__uint_as_float(w[j] << 16);
      v[2 * j + 1] = (double)__uint_as_float(w[j] & 0xFFFF0000u);
    }
  } else {
    const float4* q = reinterpret_cast<const float4*>(static_cast<const float*>(p) + i0);
    const float4 f0 = __ldg(q), f1 = __ldg(q + 1);
    v[0] = f0.x, v[1] = f0.y, v[2] = f0.z, v[3] = f0.w;
    v[4] = f1.x, v[5] = f1.y, v[6] = f1.z, v[7] = f1.w;
  }
}

constexpr int kGroupsInFlight = 4;  // 8-element groups a lane loads before summing them


// The reference arithmetic itself: sequential fp64 sum in ascending i, then the
// bias.  Every product is exact in fp64, so fma equals multiply-then-add.  The
// loads run ahead of the sum in 8-element groups.
__device__ double logit_fp64_sequential(const RouteArgs& a, int t, int e) {
  double s = 0.0;
  const size_t xr = (size_t)t * a.d, wr = (size_t)e * a.d;
  const int ng = a.d / 8;
  for (int g0 = 0; g0 < ng; g0 += kGroupsInFlight) {
    double w[kGroupsInFlight][8], x[kGroupsInFlight][8];
#pragma unroll
    for (int u = 0; u < kGroupsInFlight; ++u) {
      if (g0 + u < ng) {
        load8_d(a.w, a.w_dtype, wr + 8 * (size_t)(g0 + u), w[u]);
        load8_d(a.x, a.x_dtype, xr + 8 * (size_t)(g0 + u), x[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < kGroupsInFlight; ++u) {
      if (g0 + u >= ng) break;
#pragma unroll
      for (int j = 0; j < 8; ++j) s = fma(w[u][j], x[u][j], s);
    }
  }
  const float* kb = a.bias ? a.bias : a.sel_bias;  // the selection key's bias (at most one is set)
  if (kb) s += (double)kb[e];
  return s;
}

// Warp-parallel fp64 logit: bf16 x bf16 and fp32 x fp32 products are exact in
// fp64; lane l sums the products of groups l, l+32, ... in order, then a
// 5-level butterfly adds the lanes, and the bias comes last.  Against the
// exact value the error is at most gamma64(d/32 + 6) * sum|p| + u |val|; the
// reference's sequential sum is within gamma64(d) * sum|p| of it.
__device__ void logit_fp64_warp(const RouteArgs& a, int t, int e, double* val, double* abs_sum) {
  const int lane = threadIdx.x & 31;
  double s = 0.0, sa = 0.0;
  const size_t xr = (size_t)t * a.d, wr = (size_t)e * a.d;
  const int ng = a.d / 8;
  for (int g0 = lane; g0 < ng; g0 += 32 * kGroupsInFlight) {
    double w[kGroupsInFlight][8], x[kGroupsInFlight][8];
#pragma unroll
    for (int u = 0; u < kGroupsInFlight; ++u) {
      const int g = g0 + 32 * u;
      if (g < ng) {
        load8_d(a.w, a.w_dtype, wr + 8 * (size_t)g, w[u]);
        load8_d(a.x, a.x_dtype, xr + 8 * (size_t)g, x[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < kGroupsInFlight; ++u) {
      if (g0 + 32 * u >= ng) break;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const double pr = w[u][j] * x[u][j];
        s += pr;
        sa += fabs(pr);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    sa += __shfl_xor_sync(0xffffffffu, sa, o);
  }
  const float* kb = a.bias ? a.bias : a.sel_bias;
  if (kb) s += (double)kb[e];
  *val = s;
  *abs_sum = sa;
}

// Warp-parallel compensated fp32 logit, summed exactly as router_logits_comp_kernel
// sums one token (lane chunks of N elements, two Dot2 chains per lane merged
// by TwoSum, then a TwoSum butterfly over the lanes), so the same coefficient
// bounds it: |val - l_ref| <= gamma_comp * sum|p|, where val = s + c is kept
// unrounded in fp64 (its last addition and the bias add at most 2^-52 |val|).
// fp32 arithmetic at the full rate, where the fp64 form runs at the GPU's far
// lower fp64 rate.
template <typename WT>
__device__ void logit_dot2_warp(const RouteArgs& a, int t, int e, double* val, double* abs_sum) {
  constexpr int N = Vec16<WT>::N;
  constexpr int B = 4;  // chunks whose loads are in flight together (the sums still run in chunk order)
  const int lane = threadIdx.x & 31;
  const int d = a.d, nch = d / (32 * N), rem = d - nch * 32 * N;
  const uint4* wrow = reinterpret_cast<const uint4*>(static_cast<const WT*>(a.w) + (size_t)e * d);
  float s[2] = {0.f, 0.f}, c[2] = {0.f, 0.f}, sa = 0.f;
  // the N activations of the chunk at column col (16-byte aligned)
  auto load_x = [&](int col, float (&xr)[N]) {
    const size_t xo = (size_t)t * d + col;
    if (a.x_dtype == MOE_BF16) {
      const uint16_t* xb = static_cast<const uint16_t*>(a.x) + xo;
#pragma unroll
      for (int q = 0; q < N / 8; ++q) Vec16<uint16_t>::unpack(__ldg(reinterpret_cast<const uint4*>(xb) + q), xr + 8 * q);
      if (N == 4) {
        const uint2 h = __ldg(reinterpret_cast<const uint2*>(xb));
        xr[0] = __uint_as_float(h.x << 16);
        xr[1] = __uint_as_float(h.x & 0xFFFF0000u);
        xr[2] = __uint_as_float(h.y << 16);
        xr[3] = __uint_as_float(h.y & 0xFFFF0000u);
      }
    } else {
      const float4* xf = reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + xo);
#pragma unroll
      for (int q = 0; q < N / 4; ++q) {
        const float4 v = __ldg(xf + q);
        xr[4 * q] = v.x;
        xr[4 * q + 1] = v.y;
        xr[4 * q + 2] = v.z;
        xr[4 * q + 3] = v.w;
      }
    }
  };
  auto consume = [&](const uint4 raw, const float (&xr)[N]) {
    float w[N];
    Vec16<WT>::unpack(raw, w);
#pragma unroll
    for (int m = 0; m < N; ++m) {
      const float xv = xr[m];
      const int ch = m & 1;
      const float p = __fmul_rn(w[m], xv);
      const float ep = __fmaf_rn(w[m], xv, -p);
      float t2, es;
      two_sum(s[ch], p, t2, es);
      s[ch] = t2;
      c[ch] = __fadd_rn(c[ch], __fadd_rn(es, ep));
      sa = __fadd_rn(sa, fabsf(p));
    }
  };
  for (int u0 = 0; u0 < nch; u0 += B) {
    uint4 wq[B];
    float xr[B][N];
#pragma unroll
    for (int j = 0; j < B; ++j) {
      if (u0 + j < nch) {
        wq[j] = __ldg(wrow + (u0 + j) * 32 + lane);
        load_x(((u0 + j) * 32 + lane) * N, xr[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < B; ++j)
      if (u0 + j < nch) consume(wq[j], xr[j]);
  }
  if (lane * N < rem) {
    float xr[N];
    load_x((nch * 32 + lane) * N, xr);
    consume(__ldg(wrow + nch * 32 + lane), xr);
  }
  float st, ct;
  {
    float es;
    two_sum(s[0], s[1], st, es);
    ct = __fadd_rn(__fadd_rn(c[0], c[1]), es);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float s2 = __shfl_xor_sync(0xffffffffu, st, o);
    const float c2 = __shfl_xor_sync(0xffffffffu, ct, o);
    sa = __fadd_rn(sa, __shfl_xor_sync(0xffffffffu, sa, o));
    float t2, es;
    two_sum(st, s2, t2, es);
    st = t2;
    ct = __fadd_rn(__fadd_rn(ct, c2), es);
  }
  double v = (double)st + (double)ct;
  const float* kb = a.bias ? a.bias : a.sel_bias;
  if (kb) v += (double)kb[e];
  *val = v;
  *abs_sum = (double)sa;
}

// Order-preserving integer image of a double that is not NaN (-0 maps with
// +0): the recheck path compares and orders its fp64 interval ends on the
// integer units, since fp64 arithmetic runs at a small fraction of the fp32
// rate on this GPU.
__device__ __forceinline__ long long ord64(double v) {
  long long b = __double_as_longlong(v);
  if (b == (long long)0x8000000000000000ull) b = 0;
  return b < 0 ? (b ^ 0x7fffffffffffffffll) : b;
}

// Whether candidate c's interval [lo, hi] meets candidate c2's.
__device__ __forceinline__ bool meets(const double* lo, const double* hi, int c, int c2) {
  return !(ord64(lo[c]) > ord64(hi[c2]) || ord64(hi[c]) < ord64(lo[c2]));
}

// The recheck path runs in few CTAs, so its code is rarely in the instruction
// caches: it is kept small, and the steps it repeats are out-of-line functions
// fetched once.

// flag[c] = whether candidate c's interval meets another candidate's (the
// whole CTA; followed by a barrier).
__device__ __noinline__ void mark_meeting(const double* lo, const double* hi, unsigned char* flag, int n) {
  for (int c = threadIdx.x; c < n; c += blockDim.x) {
    unsigned char f = 0;
    for (int c2 = 0; c2 < n && !f; ++c2)
      if (c2 != c && meets(lo, hi, c, c2)) f = 1;
    flag[c] = f;
  }
  __syncthreads();
}

// One warp: the gates of a token's k selected experts, lane j < k holding
// expert e and its gate logit lj (others lj = -inf): exp(lj - max) over their
// sum, written with the indices to the routing rows and to out_sel.  lj - max
// is formed exactly in fp64 and rounded once to fp32.
__device__ __noinline__ void write_gates(const RouteArgs& a, int t, double lj, int e, int* out_sel) {
  const int lane = threadIdx.x & 31, k = a.k;
  double lm = lj;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {  // the largest, compared on the integer units
    const double ov = __shfl_xor_sync(0xffffffffu, lm, o);
    if (ord64(ov) > ord64(lm)) lm = ov;
  }
  const float g = lane < k ? expf((float)(lj - lm)) : 0.f;
  float den = g;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  if (lane < k) {
    const size_t r = (size_t)t * (k + a.n_shared) + lane;
    a.topk_idx[r] = e;
    a.gates[r] = g / den;
    out_sel[lane] = e;
  }
}

constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kSlicePerLane = (kMaxE + kTopkThreads - 1) / kTopkThreads;  // logits per thread

// Dynamic shared memory for E experts.
__host__ __device__ inline size_t topk_smem_bytes(int E) {
  const size_t e8 = ((size_t)E + 7) / 8 * 8;
  return e8 * (2 * sizeof(double) + 2 * sizeof(float) + sizeof(int) + 2);
}

// (v1, e1) before (v2, e2): larger value first, then lower index.
__device__ __forceinline__ bool before(float v1, int e1, float v2, int e2) {
  return v1 > v2 || (v1 == v2 && e1 < e2);
}

// Order-preserving unsigned image of an fp32 value (larger value, larger key).
__device__ __forceinline__ uint32_t ord_bits(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ float block_max(float v, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float m = -INFINITY;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, scratch[w]);
  __syncthreads();
  return m;
}

// Recheck path of one token's top-k (the fp32 bounds did not certify the
// selection): every expert that could be in the top k (selected, or upper
// bound at least m, the lowest selected lower bound) gets an interval; those
// meeting another one's are recomputed with compensated fp32 sums (warp-
// parallel, about u^2 relative), those still undecided in fp64 (warp-parallel,
// with its own bound) and, if still undecided, by the reference's sequential
// fp64 sum.
__device__ __noinline__ void topk_recheck(const RouteArgs& a, int t, const float* sv, const float* sb,
                                          const unsigned char* insel, float m, double* clo, double* chi, int* cand,
                                          unsigned char* cflag, int* out_sel) {
  __shared__ int n_cand;
  __shared__ int order[kMaxK];
  __shared__ int order_c[kMaxK];
  const int E = a.E, k = a.k;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    atomicAdd(a.err + 2, 1);
    n_cand = 0;
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    if (insel[e] || sv[e] + sb[e] >= m) {
      const int c = atomicAdd(&n_cand, 1);  // list order is irrelevant: the ordering below is total
      cand[c] = e;
      clo[c] = (double)sv[e] - (double)sb[e];
      chi[c] = (double)sv[e] + (double)sb[e];
    }
  }
  __syncthreads();
  const int n = n_cand;
  // candidates whose interval meets another one's get a tighter value below
  mark_meeting(clo, chi, cflag, n);
  // pass 1: compensated fp32 sums, the bound of the compensated router kernel
  for (int c = warp; c < n; c += kTopkThreads / 32) {
    if (!cflag[c]) continue;
    double val, sa;
    if (a.w_dtype == MOE_BF16)
      logit_dot2_warp<uint16_t>(a, t, cand[c], &val, &sa);
    else
      logit_dot2_warp<float>(a, t, cand[c], &val, &sa);
    if (lane == 0) {
      const double bd = (double)a.gamma_comp * sa * 1.0001 + 2.3e-16 * fabs(val) + 1e-300;
      clo[c] = val - bd;
      chi[c] = val + bd;
    }
  }
  __syncthreads();
  mark_meeting(clo, chi, cflag, n);
  // bound of the warp-parallel fp64 sum against the reference's sequential one
  // (a.gamma_fp64, host computed): its own error gamma64(d/32 + 6) * sum|p|
  // (sum|p| itself within gamma64(d/32 + 5), absorbed by the factor), the
  // reference's gamma64(d + 1) * sum|p|, and the rounding of the bias additions
  const double bound_scale = a.gamma_fp64;
  for (int c = warp; c < n; c += kTopkThreads / 32) {
    if (!cflag[c]) continue;
    double val, sa;
    logit_fp64_warp(a, t, cand[c], &val, &sa);
    if (lane == 0) {
      const double bd = bound_scale * sa + 4.5e-16 * fabs(val) + 1e-300;
      clo[c] = val - bd;
      chi[c] = val + bd;
    }
  }
  __syncthreads();
  // pass 3: still undecided -> the reference's own sequential fp64 sum
  mark_meeting(clo, chi, cflag, n);
  for (int c = tid; c < n; c += blockDim.x) {
    if (!cflag[c]) continue;
    atomicAdd(a.err + 3, 1);
    const double val = logit_fp64_sequential(a, t, cand[c]);
    clo[c] = val;
    chi[c] = val;
  }
  __syncthreads();
  // order the candidates: every two intervals are now disjoint or both exact
  // (any two that met were both recomputed exactly), so the lower ends order
  // them as their values do; equal values (exact) order by expert index.  Rank
  // by counting; the midpoint of a chosen interval is its gate logit.
  for (int c = tid; c < n; c += blockDim.x) {
    const long long kc = ord64(clo[c]);
    const int ec = cand[c];
    int r = 0;
    for (int c2 = 0; c2 < n && r < k; ++c2) {
      const long long k2 = ord64(clo[c2]);
      r += k2 > kc || (k2 == kc && cand[c2] < ec);
    }
    if (r < k) {
      order[r] = ec;
      order_c[r] = c;
    }
  }
  __syncthreads();
  if (warp == 0) {
    // gate logits: the midpoints, or (selection-only bias) the router's fp32
    // logits without the bias, as on the certified path (a key that was not
    // recomputed is an fp32 sum rounded once more by the bias addition)
    double lj = -INFINITY;
    int e = 0;
    if (lane < k) {
      e = order[lane];
      lj = a.sel_bias ? (double)a.logits[(size_t)t * E + e] : 0.5 * (clo[order_c[lane]] + chi[order_c[lane]]);
    }
    write_gates(a, t, lj, e, out_sel);
  }
}

// One CTA per token (the body of the top-k kernel): a radix select finds the (k+1)-th largest fp32 logit,
// the k+1 experts at or above it are ordered by counting, and the bounds then
// certify the selection or send the CTA down the recheck path.
// The selection also lands in out_sel[0 .. k-1] (shared memory of the CTA),
// the shared experts in out_sel[k .. k + n_shared - 1].
__device__ __forceinline__ void topk_token(const RouteArgs& a, int* out_sel) {
  extern __shared__ double tsm[];
  const int E = a.E, k = a.k;
  const size_t e8 = ((size_t)E + 7) / 8 * 8;
  double* clo = tsm;  // recheck path: candidate bounds
  double* chi = clo + e8;
  float* sv = reinterpret_cast<float*>(chi + e8);  // fp32 logits
  float* sb = sv + e8;                             // their error bounds
  int* cand = reinterpret_cast<int*>(sb + e8);     // recheck path: candidate experts
  unsigned char* insel = reinterpret_cast<unsigned char*>(cand + e8);
  unsigned char* cflag = insel + e8;
  __shared__ int sel[kMaxK + 1];
  __shared__ int candA[kMaxK + 1];
  __shared__ int hist[256];
  __shared__ int s_digit, s_need, s_full, s_na, s_nb;
  __shared__ int certified;
  __shared__ float scratch[kTopkWarps];

  const int t = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  const float nx = a.comp ? 0.f : a.nrm_x[t];
  // load: thread tid holds experts e = tid + 256 i as order-preserving keys
  uint32_t key[kSlicePerLane];
#pragma unroll
  for (int i = 0; i < kSlicePerLane; ++i) {
    const int e = tid + kTopkThreads * i;
    key[i] = 0u;
    if (e < E) {
      // v: the router's logit (with the additive bias b, if any); the key adds
      // the selection-only bias.  The compensated sum is rounded before b is
      // added, and that rounding is relative to |v - b|, hence |v| + |b|.
      const float v = a.logits[(size_t)t * E + e];
      const float b = a.bias ? a.bias[e] : 0.f;
      const float kv = a.sel_bias ? v + a.sel_bias[e] : v;
      sv[e] = kv;
      sb[e] = (a.comp ? a.gamma * a.absdot[(size_t)t * E + e] + 2.4e-7f * (fabsf(v) + fabsf(b))
                      : a.gamma * a.nrm_w[e] * nx + 1.2e-7f * fabsf(v)) +
              (a.sel_bias ? 1.2e-7f * fabsf(kv) : 0.f) + 1e-30f;
      insel[e] = 0;
      key[i] = ord_bits(kv);
    }
  }
  if (tid < a.n_shared) {  // the shared experts close every token's row with gate 1
    const int j = k + tid;
    a.topk_idx[(size_t)t * (k + a.n_shared) + j] = E + tid;
    a.gates[(size_t)t * (k + a.n_shared) + j] = 1.f;
    out_sel[j] = E + tid;
  }
  pdl_launch_dependents();
  const int nsel = min(k + 1, E);
  // radix select of the nsel-th largest key, 8 bits per pass from the top
  uint32_t prefix = 0u, mask = 0u;
  int need = nsel;  // how many keys >= the threshold still to account for at this digit
  // A pass whose chosen digit bucket holds exactly the keys still needed ends
  // the search: the selection is then every key whose masked value is at or
  // above the prefix (usually after two of the four passes).
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kSlicePerLane; ++i)
      if (tid + kTopkThreads * i < E && (key[i] & mask) == prefix) atomicAdd(&hist[(key[i] >> shift) & 255u], 1);
    __syncthreads();
    if (warp == 0) {  // lane l scans bins 255-8l .. 248-8l, top down
      int c[8], lsum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * lane - j];
        lsum += c[j];
      }
      int incl = lsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - lsum;
      if (excl < need && need <= incl) {
        int run = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (run + c[j] >= need) {
            s_digit = 255 - 8 * lane - j;
            s_need = need - run;
            s_full = (need - run) == c[j];
            break;
          }
          run += c[j];
        }
      }
    }
    __syncthreads();
    prefix |= (uint32_t)s_digit << shift;
    mask |= 255u << shift;
    need = s_need;
    if (s_full) break;
  }
  // the selection: every key above the threshold, then the `need` lowest-index
  // experts whose key equals it
  if (tid == 0) {
    s_na = 0;
    s_nb = 0;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kSlicePerLane; ++i) {
    const int e = tid + kTopkThreads * i;
    if (e < E) {
      if ((key[i] & mask) > prefix) candA[atomicAdd(&s_na, 1)] = e;
      else if ((key[i] & mask) == prefix) cand[atomicAdd(&s_nb, 1)] = e;
    }
  }
  __syncthreads();
  const int na = s_na, nb = s_nb;
  for (int c = tid; c < nb; c += blockDim.x) {
    int r = 0;
    for (int c2 = 0; c2 < nb; ++c2) r += cand[c2] < cand[c];
    if (r < need) candA[na + r] = cand[c];
  }
  __syncthreads();
  if (tid < nsel) {  // order by (logit descending, index ascending): rank by counting
    const int e = candA[tid];
    const float v = sv[e];
    int r = 0;
    for (int c2 = 0; c2 < nsel; ++c2) {
      const int e2 = candA[c2];
      r += before(sv[e2], e2, v, e);
    }
    sel[r] = e;
  }
  __syncthreads();
  if (tid < k) insel[sel[tid]] = 1;
  __syncthreads();
  // certification: every outsider's upper bound below the lowest selected lower
  // bound, and strict separation of consecutive selected experts
  float hi_out = -INFINITY;
  for (int e = tid; e < E; e += blockDim.x)
    if (!insel[e]) hi_out = fmaxf(hi_out, sv[e] + sb[e]);
  hi_out = block_max(hi_out, scratch);
  float lo_neg = -INFINITY;  // max of -lo_j: the lowest selected lower bound, negated
  bool bad = false;
  if (tid < k) {
    const int e = sel[tid];
    const float lo = sv[e] - sb[e];
    lo_neg = -lo;
    if (tid + 1 < k) bad = !(lo > sv[sel[tid + 1]] + sb[sel[tid + 1]]);
  }
  const float m = -block_max(lo_neg, scratch);
  const int nbad = __syncthreads_or(bad ? 1 : 0);
  if (tid == 0) certified = (!nbad && hi_out < m) ? 1 : 0;
  __syncthreads();
  if (certified) {
    if (warp == 0) {  // gates from the fp32 logits, fixed-order warp sum (inline: the decode path)
      // gate logits: the keys, or (selection-only bias) the router's logits
      // without the bias; the largest of them is subtracted before exp (the
      // fp32 difference, as write_gates forms it for the recheck path)
      float lj = -INFINITY;
      if (lane < k) lj = a.sel_bias ? a.logits[(size_t)t * E + sel[lane]] : sv[sel[lane]];
      float lm = lj;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lm = fmaxf(lm, __shfl_xor_sync(0xffffffffu, lm, o));
      const float g = lane < k ? expf(lj - lm) : 0.f;
      float den = g;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
      if (lane < k) {
        const size_t r = (size_t)t * (k + a.n_shared) + lane;
        a.topk_idx[r] = sel[lane];
        a.gates[r] = g / den;
        out_sel[lane] = sel[lane];
      }
    }
    return;
  }

  topk_recheck(a, t, sv, sb, insel, m, clo, chi, cand, cflag, out_sel);
}

// MINB CTAs per SM at least: 1 where every token's CTA is resident at once
// anyway; 4 for calls of more tokens than SMs, which then run in one wave
// instead of four (the fp64 recheck path, rarely taken, spills a little
// under the 64-register cap).
template <int MINB>
__global__ void __launch_bounds__(kTopkThreads, MINB) topk_kernel(RouteArgs a) {
  __shared__ int sel_smem[kMaxK];
  topk_token(a, sel_smem);
  if (a.fuse_bucket) {  // one token: bucket its k pairs right here (no further launch)
    __syncthreads();
    bucket_one_token(a.bucket, sel_smem, true);
  }
}

}  // namespace

cudaError_t launch_route_topk(const RouteArgs& a, int num_sms, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  const dim3 grid((a.E + kLogitWarps - 1) / kLogitWarps, (a.T + kTokTile - 1) / kTokTile);
  const size_t smem = (size_t)kTokTile * a.d * sizeof(float);
  cudaError_t err;
  if (a.comp && a.T == 1) {
    const dim3 g1((a.E + kLogitWarps - 1) / kLogitWarps, 1);
    const size_t sm1 = (size_t)a.d * sizeof(float);
    if (a.w_dtype == MOE_BF16) {
      ensure_smem(router_logits_comp_kernel<uint16_t, 1>, sm1);
      err = launch("router_logits", router_logits_comp_kernel<uint16_t, 1>, g1, dim3(kLogitWarps * 32), sm1, s,
                   false, a);
    } else {
      ensure_smem(router_logits_comp_kernel<float, 1>, sm1);
      err = launch("router_logits", router_logits_comp_kernel<float, 1>, g1, dim3(kLogitWarps * 32), sm1, s, false,
                   a);
    }
  } else if (a.comp) {
    if (a.w_dtype == MOE_BF16) {
      ensure_smem(router_logits_comp_kernel<uint16_t, kTokTile>, smem);
      err = launch("router_logits", router_logits_comp_kernel<uint16_t, kTokTile>, grid, dim3(kLogitWarps * 32), smem,
                   s, false, a);
    } else {
      ensure_smem(router_logits_comp_kernel<float, kTokTile>, smem);
      err = launch("router_logits", router_logits_comp_kernel<float, kTokTile>, grid, dim3(kLogitWarps * 32), smem, s,
                   false, a);
    }
  } else if (a.T >= 2 * kTiledTok && a.w_dtype == MOE_BF16 && a.x_dtype == MOE_BF16 && a.d % 256 == 0 &&
             tiled_smem_bytes(a.d) <= 112 * 1024) {
    const dim3 gt((a.E + kTiledExperts - 1) / kTiledExperts, (a.T + kTiledTok - 1) / kTiledTok);
    ensure_smem(router_logits_tiled_kernel, tiled_smem_bytes(a.d));
    err = launch("router_logits", router_logits_tiled_kernel, gt, dim3(kLogitWarps * 32), tiled_smem_bytes(a.d), s,
                 false, a);
  } else {
    const dim3 gp((a.E + kLogitWarps * kRowsPerWarp - 1) / (kLogitWarps * kRowsPerWarp), (a.T + kTokTile - 1) / kTokTile);
    if (a.w_dtype == MOE_BF16) {
      ensure_smem(router_logits_kernel<uint16_t>, smem);
      err = launch("router_logits", router_logits_kernel<uint16_t>, gp, dim3(kLogitWarps * 32), smem, s, false, a);
    } else {
      ensure_smem(router_logits_kernel<float>, smem);
      err = launch("router_logits", router_logits_kernel<float>, gp, dim3(kLogitWarps * 32), smem, s, false, a);
    }
  }
  if (err != cudaSuccess) return err;
  const size_t tsm = topk_smem_bytes(a.E);
  if (a.T > num_sms) {
    ensure_smem(topk_kernel<4>, tsm);
    return launch("topk", topk_kernel<4>, dim3(a.T), dim3(kTopkThreads), tsm, s, true, a);
  }
  ensure_smem(topk_kernel<1>, tsm);
  return launch("topk", topk_kernel<1>, dim3(a.T), dim3(kTopkThreads), tsm, s, true, a);
}

}  // namespace moe

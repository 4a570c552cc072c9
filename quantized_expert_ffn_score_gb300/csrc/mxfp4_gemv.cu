// mxfp4_gemv.cu -- routed-expert FFN on MXFP4 weights for small token counts
// per expert (decode).  The packed weights are consumed as stored and never
// widened in memory (LazyLoRA README, "The engine": fused MXFP4 decode-and-dot
// with fp32 expert sums; "Running a 2.78-Trillion-Parameter Model Across Two
// Desks", Act II: fp32 compute after a bf16 path failed its tolerance gate).
//
// Two launches of one persistent kernel:
//   MODE 0  gate/up: tile = rows [r0, r0+16) of Wg and of Wu; the epilogue
//           applies the activation and writes h[slot][r] (fp32).
//   MODE 1  down:    tile = rows [r0, r0+32) of Wd; writes y_pairs[pair][r].
// Data movement: one producer lane streams each tile (codes and E8M0 scales of
// both halves, 4 contiguous byte ranges of the expert record) into a ring of
// shared-memory stages with 1-D bulk async copies completing on an mbarrier.
// Compute: consumer warp w, lane l owns the 32-column block b = 16w + (l & 15)
// of the contraction axis for half (l >> 4) of the tile, keeps that block of
// the input vector in registers, and for each of the tile's 16 rows decodes its
// 16 code bytes (cvt e2m1x2 -> f16x2 -> f32) and accumulates in fp32; the block
// sum is multiplied by 2^(scale-127).  A 16-lane reduce-scatter leaves row
// (l & 15) on lane l; warps are summed through shared memory.
#include <utility>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kMaxStages = 4;
constexpr int kSmemBudget = 220 * 1024;

struct Geom {
  int K;                // contraction length
  int nblk;             // K / 32
  int warps;            // consumer warps: ceil(nblk / 16)
  int tpe;              // tiles per expert
  uint32_t half_codes;  // bytes of codes per half tile: 16 * K / 2
  uint32_t half_scales; // bytes of scales per half tile: 16 * K / 32
  uint32_t stage_bytes;
  int stages;
  size_t smem;
};

__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

__device__ __forceinline__ float2 h2_to_f2(uint32_t h) {
  __half2 v = *reinterpret_cast<__half2*>(&h);
  return __half22float2(v);
}

// sum over the 32 columns of one block: codes q (low nibble = even column) times x.
__device__ __forceinline__ float dot32(const uint4 q, const float* x) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t h[4];
    e2m1x8_to_f16x2(w[i], h);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = h2_to_f2(h[j]);
      s0 = fmaf(f.x, x[8 * i + 2 * j], s0);
      s1 = fmaf(f.y, x[8 * i + 2 * j + 1], s1);
    }
  }
  return s0 + s1;
}

// 16 rows x NT values per lane -> lane (l & 15) holds the half-warp sum of row (l & 15).
template <int NT>
__device__ __forceinline__ void reduce_scatter16(float (&v)[16][NT], int lane) {
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < m; ++i) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const float send = upper ? v[i][n] : v[i + m][n];
        const float keep = upper ? v[i + m][n] : v[i][n];
        v[i][n] = keep + __shfl_xor_sync(0xffffffffu, send, m);
      }
    }
  }
}

template <int MODE>
__device__ __forceinline__ void tile_sources(const FfnArgs& a, const uint8_t* rec, int rt, const Geom& g,
                                             const uint8_t* (&src)[4]) {
  const size_t d = a.d, ff = a.ff;
  const size_t mat = ff * d / 2 + ff * d / 32;
  if (MODE == 0) {
    const size_t r0 = (size_t)rt * 16;
    const uint8_t* gc = rec;
    const uint8_t* gs = gc + ff * d / 2;
    const uint8_t* uc = rec + mat;
    const uint8_t* us = uc + ff * d / 2;
    src[0] = gc + r0 * (d / 2);
    src[1] = uc + r0 * (d / 2);
    src[2] = gs + r0 * (d / 32);
    src[3] = us + r0 * (d / 32);
  } else {
    const size_t r0 = (size_t)rt * 32;
    const uint8_t* dc = rec + 2 * mat;
    const uint8_t* ds = dc + d * ff / 2;
    src[0] = dc + r0 * (ff / 2);
    src[1] = dc + (r0 + 16) * (ff / 2);
    src[2] = ds + r0 * (ff / 32);
    src[3] = ds + (r0 + 16) * (ff / 32);
  }
}

__device__ __forceinline__ bool record_ok(const uint8_t* rec) {
  return rec != nullptr && ((reinterpret_cast<uintptr_t>(rec) & 15u) == 0);
}

template <int MODE>
__global__ void __launch_bounds__(9 * 32) mxfp4_gemv_kernel(const FfnArgs a, const Geom g) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)g.stages * g.stage_bytes);
  uint64_t* empty = full + kMaxStages;
  float* red = reinterpret_cast<float*>(empty + kMaxStages);  // [warps][2][16][kTokChunk]
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int W = g.warps;
  if (threadIdx.x == 0) {
    for (int s = 0; s < g.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], W);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();

  const int n_act = a.active[0];
  const int total = n_act * g.tpe;

  if (warp == W) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;
      for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        const int e = a.active[1 + tile / g.tpe];
        const uint8_t* rec = a.records[e];
        if (!record_ok(rec)) {
          dev_error(a.err, rec == nullptr ? MOE_ERR_MISSING_EXPERT : MOE_ERR_INVALID_ARG, e);
          continue;
        }
        const int stage = it % g.stages, n = it / g.stages;
        if (n > 0 && !mbar_wait(&empty[stage], (n - 1) & 1, a.err)) break;  // consumers time out too
        if (*(volatile int*)&abort_flag) break;
        const uint8_t* src[4];
        tile_sources<MODE>(a, rec, tile % g.tpe, g, src);
        uint8_t* dst = smem + (size_t)stage * g.stage_bytes;
        mbar_arrive_expect_tx(&full[stage], 2 * (g.half_codes + g.half_scales));
        bulk_g2s(dst, src[0], g.half_codes, &full[stage]);
        bulk_g2s(dst + g.half_codes, src[1], g.half_codes, &full[stage]);
        bulk_g2s(dst + 2 * g.half_codes, src[2], g.half_scales, &full[stage]);
        bulk_g2s(dst + 2 * g.half_codes + g.half_scales, src[3], g.half_scales, &full[stage]);
        ++it;
      }
      // never leave the CTA with copies in flight: wait for the last fills
      for (int j = (it > g.stages ? it - g.stages : 0); j < it; ++j)
        mbar_wait(&full[j % g.stages], (j / g.stages) & 1, a.err);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int half = lane >> 4;
  const int b = warp * 16 + (lane & 15);
  const bool vb = b < g.nblk;
  const int K = g.K;
  const int nthreads = W * 32;
  int it = 0;
  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    const int e = a.active[1 + tile / g.tpe];
    if (!record_ok(a.records[e])) continue;
    const int rt = tile % g.tpe;
    const int stage = it % g.stages, n = it / g.stages;
    ++it;
    // A timed-out wait is recorded before the barrier, so every consumer warp
    // reads the same flag after it and they leave the loop together (the
    // producer never writes this flag).
    if (!mbar_wait(&full[stage], n & 1, a.err)) atomicExch(&abort_flag, 1);
    named_bar_sync(1, nthreads);
    if (*(volatile int*)&abort_flag) break;
    const uint8_t* st = smem + (size_t)stage * g.stage_bytes;
    const uint8_t* codes = st + half * g.half_codes + b * 16;
    const uint8_t* scales = st + 2 * g.half_codes + half * g.half_scales + b;
    const int s0 = a.offsets[e];
    const int ne = a.offsets[e + 1] - s0;
    for (int c0 = 0; c0 < ne; c0 += kTokChunk) {
      const int nt = min(kTokChunk, ne - c0);
      float xin[kTokChunk][32];
#pragma unroll
      for (int q = 0; q < kTokChunk; ++q) {
        if (q < nt && vb) {
          const int slot = s0 + c0 + q;
          if (MODE == 0) {
            const size_t base = (size_t)(a.pair_ids[slot] / a.k) * a.d + (size_t)b * 32;
            if (a.x_dtype == MOE_BF16) {
              const uint4* px = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + base);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const uint4 u = px[v];
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  xin[q][8 * v + 2 * j] = __uint_as_float(w4[j] << 16);
                  xin[q][8 * v + 2 * j + 1] = __uint_as_float(w4[j] & 0xFFFF0000u);
                }
              }
            } else {
              const float4* px = reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + base);
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                const float4 f = px[v];
                xin[q][4 * v] = f.x;
                xin[q][4 * v + 1] = f.y;
                xin[q][4 * v + 2] = f.z;
                xin[q][4 * v + 3] = f.w;
              }
            }
          } else {
            const float4* ph = reinterpret_cast<const float4*>(a.h + (size_t)slot * a.ff + (size_t)b * 32);
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              const float4 f = ph[v];
              xin[q][4 * v] = f.x;
              xin[q][4 * v + 1] = f.y;
              xin[q][4 * v + 2] = f.z;
              xin[q][4 * v + 3] = f.w;
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) xin[q][j] = 0.f;
        }
      }
      float acc[16][kTokChunk];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        if (vb) {
          const uint4 q4 = *reinterpret_cast<const uint4*>(codes + (size_t)r * (K / 2));
          const float sc = e8m0_to_f32(scales[(size_t)r * (K / 32)]);
#pragma unroll
          for (int q = 0; q < kTokChunk; ++q) acc[r][q] = dot32(q4, xin[q]) * sc;
        } else {
#pragma unroll
          for (int q = 0; q < kTokChunk; ++q) acc[r][q] = 0.f;
        }
      }
      reduce_scatter16<kTokChunk>(acc, lane);
#pragma unroll
      for (int q = 0; q < kTokChunk; ++q) red[(((warp * 2 + half) * 16) + (lane & 15)) * kTokChunk + q] = acc[0][q];
      named_bar_sync(1, nthreads);
      const int tid = threadIdx.x;
      if (MODE == 0) {
        for (int idx = tid; idx < 16 * nt; idx += nthreads) {
          const int r = idx & 15, q = idx >> 4;
          float gsum = 0.f, usum = 0.f;
          for (int w = 0; w < W; ++w) {
            gsum += red[(((w * 2 + 0) * 16) + r) * kTokChunk + q];
            usum += red[(((w * 2 + 1) * 16) + r) * kTokChunk + q];
          }
          a.h[(size_t)(s0 + c0 + q) * a.ff + (size_t)rt * 16 + r] = act_fn(gsum, usum, a.act);
        }
      } else {
        for (int idx = tid; idx < 32 * nt; idx += nthreads) {
          const int r = idx & 15, hf = (idx >> 4) & 1, q = idx >> 5;
          float ysum = 0.f;
          for (int w = 0; w < W; ++w) ysum += red[(((w * 2 + hf) * 16) + r) * kTokChunk + q];
          const int pair = a.pair_ids[s0 + c0 + q];
          a.y_pairs[(size_t)pair * a.d + (size_t)rt * 32 + hf * 16 + r] = ysum;
        }
      }
      named_bar_sync(1, nthreads);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }
}

Geom make_geom(int mode, int d, int ff) {
  Geom g;
  g.K = mode == 0 ? d : ff;
  g.nblk = g.K / 32;
  g.warps = (g.nblk + 15) / 16;
  g.tpe = mode == 0 ? ff / 16 : d / 32;
  g.half_codes = 16u * (uint32_t)g.K / 2u;
  g.half_scales = 16u * (uint32_t)g.K / 32u;
  g.stage_bytes = 2u * (g.half_codes + g.half_scales);
  const size_t fixed = 2 * kMaxStages * sizeof(uint64_t) + (size_t)g.warps * 2 * 16 * kTokChunk * sizeof(float);
  g.stages = (int)((kSmemBudget - fixed) / g.stage_bytes);
  if (g.stages > kMaxStages) g.stages = kMaxStages;
  g.smem = (size_t)g.stages * g.stage_bytes + fixed;
  return g;
}

}  // namespace

cudaError_t launch_mxfp4_ffn(const FfnArgs& a, int num_sms, bool pdl, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  const Geom g0 = make_geom(0, a.d, a.ff), g1 = make_geom(1, a.d, a.ff);
  if (g0.stages < 2 || g1.stages < 2) return cudaErrorInvalidValue;
  cudaFuncSetAttribute(mxfp4_gemv_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)g0.smem);
  cudaFuncSetAttribute(mxfp4_gemv_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)g1.smem);
  cudaError_t err = launch("mxfp4_gate_up", mxfp4_gemv_kernel<0>, dim3(num_sms), dim3((g0.warps + 1) * 32), g0.smem, s, pdl, a, g0);
  if (err != cudaSuccess) return err;
  return launch("mxfp4_down", mxfp4_gemv_kernel<1>, dim3(num_sms), dim3((g1.warps + 1) * 32), g1.smem, s, true, a, g1);
}

}  // namespace moe

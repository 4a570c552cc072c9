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
// Each CTA owns a contiguous range of the (expert, row tile) list, so it meets
// at most a few experts and keeps an expert's input vectors in registers
// across that expert's tiles.
// Data movement: one producer lane streams each tile (codes and E8M0 scales of
// both halves, 4 contiguous byte ranges of the expert record) into a ring of
// shared-memory stages with 1-D bulk async copies completing on an mbarrier.
// Compute: two groups of consumer warps split each half tile's 16 rows (8
// each); in a group, warp w, lane l owns the 32-column block b = 16w + (l & 15)
// of the contraction axis for half (l >> 4) of the tile.  For each of its 8
// rows it converts its 16 code bytes with cvt.e2m1x2 (two E2M1 codes -> f16x2,
// exact) and accumulates the block in fp32:
//   * bf16 activations: converted once to f16 after an exact power-of-two
//     rescale (x * 2^-s with max|x| * 2^-s < 2^15), then fma.f32.f16 -- the
//     product of two f16 values is exact in fp32 and the sum is fp32;
//   * fp32 inputs (fp32 x, and h for the down projection): the f16 weights are
//     widened to fp32 and multiplied in fp32.
// The block sum is multiplied by 2^(scale-127) (and 2^s).  A reduce-scatter
// over the 16 lanes of a half leaves each row on one lane; warps are summed
// through a double-buffered shared-memory array, one named barrier per tile.
#include <utility>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kMaxStages = 4;
constexpr int kSmemBudget = 220 * 1024;
constexpr int kNT = kTokChunk;  // tokens per pass over a tile (and cached per expert)

struct Geom {
  int K;                 // contraction length
  int nblk;              // K / 32
  int warps;             // consumer warps: ceil(nblk / 16)
  int tpe;               // tiles per expert
  uint32_t half_codes;   // bytes of codes per half tile: 16 * K / 2
  uint32_t half_scales;  // bytes of scales per half tile: 16 * K / 32
  uint32_t stage_bytes;
  int stages;
  size_t smem;
};

// Block dot products: 32 codes q (low nibble = even column) against the lane's
// 32 input values.  f16 inputs: fma.f32.f16 on each half of the converted code
// pair (exact products, fp32 sums); fp32 inputs: the f16 pair widened to fp32.
__device__ __forceinline__ float dot32_f16(const uint4 q, const unsigned short* x) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t h[4];
    e2m1x8_to_f16x2(w[i], h);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2;\n"
          " fma.rn.f32.f16 %0, lo, %3, %0;\n fma.rn.f32.f16 %1, hi, %4, %1; }"
          : "+f"(s[2 * (j & 1)]), "+f"(s[2 * (j & 1) + 1])
          : "r"(h[j]), "h"(x[8 * i + 2 * j]), "h"(x[8 * i + 2 * j + 1]));
  }
  return (s[0] + s[1]) + (s[2] + s[3]);
}

__device__ __forceinline__ float dot32_f32(const uint4 q, const float* x) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t h[4];
    e2m1x8_to_f16x2(w[i], h);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[j]));
      s[2 * (j & 1)] = fmaf(f.x, x[8 * i + 2 * j], s[2 * (j & 1)]);
      s[2 * (j & 1) + 1] = fmaf(f.y, x[8 * i + 2 * j + 1], s[2 * (j & 1) + 1]);
    }
  }
  return (s[0] + s[1]) + (s[2] + s[3]);
}

// RPG (8 or 16) rows x NT values per lane -> the half-warp sum of row
// (l & (RPG-1)) ends on lane l (for RPG = 8 on the lanes with (l & 8) == 0).
template <int RPG, int NT>
__device__ __forceinline__ void reduce_rows(float (&v)[RPG][NT], int lane) {
#pragma unroll
  for (int m = RPG / 2; m >= 1; m >>= 1) {
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
  if (RPG == 8) {
#pragma unroll
    for (int n = 0; n < NT; ++n) v[0][n] += __shfl_xor_sync(0xffffffffu, v[0][n], 8);
  }
}

template <int MODE>
__device__ __forceinline__ void tile_sources(const FfnArgs& a, const uint8_t* rec, int rt,
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

// 2^s as fp32 for |s| <= 126.
__device__ __forceinline__ float pow2f(int s) { return __uint_as_float((uint32_t)(s + 127) << 23); }

// The lane's inputs (its 32-column block) for up to kNT tokens (slots s_begin ..):
// f16 values after a per-token power-of-two rescale (XF16), or fp32.
template <int MODE, bool XF16>
struct Inputs {
  unsigned short xh[XF16 ? kNT : 1][32];
  float xf[XF16 ? 1 : kNT][32];
  float pw[kNT];  // 2^s per token (XF16), else 1

  __device__ void load(const FfnArgs& a, int s_begin, int count, int b, bool vb) {
#pragma unroll
    for (int q = 0; q < kNT; ++q) {
      pw[q] = 1.f;
      float v[32];
      if (q < count && vb) {
        const int slot = s_begin + q;
        if (MODE == 0) {
          const size_t base = (size_t)(a.pair_ids[slot] / a.k) * a.d + (size_t)b * 32;
          if (a.x_dtype == MOE_BF16) {
            const uint4* px = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + base);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint4 w = px[u];
              const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                v[8 * u + 2 * j] = __uint_as_float(w4[j] << 16);
                v[8 * u + 2 * j + 1] = __uint_as_float(w4[j] & 0xFFFF0000u);
              }
            }
          } else {
            const float4* px = reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + base);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float4 f = px[u];
              v[4 * u] = f.x;
              v[4 * u + 1] = f.y;
              v[4 * u + 2] = f.z;
              v[4 * u + 3] = f.w;
            }
          }
        } else {
          const float4* ph = reinterpret_cast<const float4*>(a.h + (size_t)slot * a.ff + (size_t)b * 32);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float4 f = ph[u];
            v[4 * u] = f.x;
            v[4 * u + 1] = f.y;
            v[4 * u + 2] = f.z;
            v[4 * u + 3] = f.w;
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.f;
      }
      if (XF16) {
        // exact power-of-two rescale from the token's max |x| (router kernel)
        float mx = 0.f;
        if (q < count) mx = a.max_x[a.pair_ids[s_begin + q] / a.k];
        int s = 0;
        if (mx > 0.f && mx < INFINITY) s = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127 - 14;
        s = max(-100, min(100, s));
        pw[q] = pow2f(s);
        const float inv = pow2f(-s);
#pragma unroll
        for (int j = 0; j < 32; ++j) xh[XF16 ? q : 0][j] = __half_as_ushort(__float2half_rn(v[j] * inv));
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) xf[XF16 ? 0 : q][j] = v[j];
      }
    }
  }
};

// One pass over the RPG rows of one warp group of a staged half tile for NT
// tokens: block partial sums scaled by the rows' E8M0 scales (and 2^s),
// reduced over the half-warp, written to the pass's reduction buffer rb.
template <int RPG, int NT, bool XF16, int MODE>
__device__ __forceinline__ void pass_rows(const uint8_t* codes, const uint8_t* scales, int K,
                                          const Inputs<MODE, XF16>& in, bool vb, float* rb, int wk, int half, int grp,
                                          int lane) {
  float acc[RPG][NT];
#pragma unroll
  for (int r = 0; r < RPG; ++r) {
#pragma unroll
    for (int q = 0; q < NT; ++q) acc[r][q] = 0.f;
    if (vb) {
      const uint4 q4 = *reinterpret_cast<const uint4*>(codes + (size_t)r * (K / 2));
      const float sc = e8m0_to_f32(scales[(size_t)r * (K / 32)]);
#pragma unroll
      for (int q = 0; q < NT; ++q) {
        if (XF16)
          acc[r][q] = dot32_f16(q4, in.xh[XF16 ? q : 0]) * (sc * in.pw[q]);
        else
          acc[r][q] = dot32_f32(q4, in.xf[XF16 ? 0 : q]) * sc;
      }
    }
  }
  reduce_rows<RPG, NT>(acc, lane);
  if (RPG == 16 || (lane & 8) == 0) {
#pragma unroll
    for (int q = 0; q < NT; ++q) rb[(((wk * 2 + half) * 16) + RPG * grp + (lane & (RPG - 1))) * kNT + q] = acc[0][q];
  }
}

// Warps: G*W consumers (group grp = cw / W takes rows RPG*grp .. of each half
// tile, RPG = 16 / G; wk = cw % W is the lane blocks' K group), then one
// producer warp.  At most 16 warps, so every thread may hold 128 registers.
// Consumers never meet at a CTA-wide barrier: each pass's partial sums go to a
// double-buffered shared array whose fill is counted by an mbarrier, and
// consumer warp 0 alone waits for it and writes the pass's outputs.  Every wait
// is bounded; a warp whose wait runs out records MOE_ERR_TIMEOUT and leaves,
// and the others then run out of their own waits and leave too.
template <int MODE, bool XF16, int G>
__global__ void __launch_bounds__(16 * 32, 1) mxfp4_gemv_kernel(const FfnArgs a, const Geom g) {
  constexpr int RPG = 16 / G;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)g.stages * g.stage_bytes);
  uint64_t* empty = full + kMaxStages;
  uint64_t* red_full = empty + kMaxStages;  // [2]
  uint64_t* red_empty = red_full + 2;       // [2]
  float* red = reinterpret_cast<float*>(red_empty + 2);  // [2][W][2][16][kNT]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int W = g.warps;
  const int NC = G * W;  // consumer warps
  if (threadIdx.x == 0) {
    for (int s = 0; s < g.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NC);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&red_full[b], NC);
      mbar_init(&red_empty[b], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();

  const long long total = (long long)a.active[0] * g.tpe;
  const int t_begin = (int)(total * blockIdx.x / gridDim.x);
  const int t_end = (int)(total * (blockIdx.x + 1) / gridDim.x);

  if (warp == NC) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0, cur_a = -1, e = -1;
      const uint8_t* rec = nullptr;
      for (int tile = t_begin; tile < t_end; ++tile) {
        const int ai = tile / g.tpe;
        if (ai != cur_a) {
          cur_a = ai;
          e = a.active[1 + ai];
          rec = a.records[e];
          if (!record_ok(rec)) dev_error(a.err, rec == nullptr ? MOE_ERR_MISSING_EXPERT : MOE_ERR_INVALID_ARG, e);
        }
        if (!record_ok(rec)) continue;
        const int stage = it % g.stages, n = it / g.stages;
        if (n > 0 && !mbar_wait(&empty[stage], (n - 1) & 1, a.err)) break;
        const uint8_t* src[4];
        tile_sources<MODE>(a, rec, tile % g.tpe, src);
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
        mbar_wait_drain(&full[j % g.stages], (j / g.stages) & 1, a.err);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int cw = warp, grp = cw / W, wk = cw % W;
  const int half = lane >> 4;
  const int b = wk * 16 + (lane & 15);
  const bool vb = b < g.nblk;
  const int K = g.K;
  Inputs<MODE, XF16> in;
  int it = 0, pc = 0, cur_a = -1, s0 = 0, ne = 0;
  bool rec_good = false;
  for (int tile = t_begin; tile < t_end; ++tile) {
    const int ai = tile / g.tpe;
    if (ai != cur_a) {  // a new expert: its slots, and its inputs if they fit the register cache
      cur_a = ai;
      const int e = a.active[1 + ai];
      rec_good = record_ok(a.records[e]);
      s0 = a.offsets[e];
      ne = a.offsets[e + 1] - s0;
      if (rec_good && ne <= kNT) in.load(a, s0, ne, b, vb);
    }
    if (!rec_good) continue;
    const int rt = tile % g.tpe;
    const int stage = it % g.stages;
    if (!mbar_wait(&full[stage], (it / g.stages) & 1, a.err)) return;
    ++it;
    const uint8_t* st = smem + (size_t)stage * g.stage_bytes;
    const uint8_t* codes = st + half * g.half_codes + (size_t)(RPG * grp) * (K / 2) + b * 16;
    const uint8_t* scales = st + 2 * g.half_codes + half * g.half_scales + (size_t)(RPG * grp) * (K / 32) + b;
    for (int c0 = 0; c0 < ne; c0 += kNT) {
      const int nt = min(kNT, ne - c0);
      if (ne > kNT) in.load(a, s0 + c0, nt, b, vb);
      const int bi = pc & 1, use = pc >> 1;
      ++pc;
      if (use > 0 && !mbar_wait(&red_empty[bi], (use - 1) & 1, a.err)) return;
      float* rb = red + bi * (W * 2 * 16 * kNT);
      if (nt == 1)
        pass_rows<RPG, 1, XF16, MODE>(codes, scales, K, in, vb, rb, wk, half, grp, lane);
      else
        pass_rows<RPG, kNT, XF16, MODE>(codes, scales, K, in, vb, rb, wk, half, grp, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_full[bi]);
      if (cw == 0) {  // the pass's outputs, once every consumer warp has published
        if (!mbar_wait(&red_full[bi], use & 1, a.err)) return;
        if (MODE == 0) {
          for (int idx = lane; idx < 16 * nt; idx += 32) {
            const int r = idx & 15, q = idx >> 4;
            float gsum = 0.f, usum = 0.f;
            for (int w = 0; w < W; ++w) {
              gsum += rb[(((w * 2 + 0) * 16) + r) * kNT + q];
              usum += rb[(((w * 2 + 1) * 16) + r) * kNT + q];
            }
            a.h[(size_t)(s0 + c0 + q) * a.ff + (size_t)rt * 16 + r] = act_fn(gsum, usum, a.act);
          }
        } else {
          for (int idx = lane; idx < 32 * nt; idx += 32) {
            const int r = idx & 15, hf = (idx >> 4) & 1, q = idx >> 5;
            float ysum = 0.f;
            for (int w = 0; w < W; ++w) ysum += rb[(((w * 2 + hf) * 16) + r) * kNT + q];
            const int pair = a.pair_ids[s0 + c0 + q];
            a.y_pairs[(size_t)pair * a.d + (size_t)rt * 32 + hf * 16 + r] = ysum;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&red_empty[bi]);
      }
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
  const size_t fixed = (2 * kMaxStages + 4) * sizeof(uint64_t) + (size_t)2 * g.warps * 2 * 16 * kNT * sizeof(float);
  g.stages = (int)((kSmemBudget - fixed) / g.stage_bytes);
  if (g.stages > kMaxStages) g.stages = kMaxStages;
  g.smem = (size_t)g.stages * g.stage_bytes + fixed;
  return g;
}

template <int MODE, bool XF16>
cudaError_t launch_one(const FfnArgs& a, const Geom& g, int num_sms, bool pdl, cudaStream_t s, const char* name) {
  if (2 * g.warps + 1 <= 16) {  // two row groups (K <= 3584)
    ensure_smem(mxfp4_gemv_kernel<MODE, XF16, 2>, g.smem);
    return launch(name, mxfp4_gemv_kernel<MODE, XF16, 2>, dim3(num_sms), dim3((2 * g.warps + 1) * 32), g.smem, s,
                  pdl, a, g);
  }
  ensure_smem(mxfp4_gemv_kernel<MODE, XF16, 1>, g.smem);
  return launch(name, mxfp4_gemv_kernel<MODE, XF16, 1>, dim3(num_sms), dim3((g.warps + 1) * 32), g.smem, s, pdl, a,
                g);
}

// max_i |x_t[i]| per token, one CTA per token (for the standalone expert call).
__global__ void token_absmax_kernel(const void* x, int x_dtype, int d, float* max_x) {
  __shared__ float part[32];
  pdl_wait();
  const int t = blockIdx.x;
  float m = 0.f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) m = fmaxf(m, fabsf(load_act(x, x_dtype, (size_t)t * d + i)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, part[w]);
    max_x[t] = m;
  }
}

}  // namespace

cudaError_t launch_token_absmax(const void* x, int x_dtype, int T, int d, float* max_x, bool pdl, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  return launch("token_absmax", token_absmax_kernel, dim3(T), dim3(256), 0, s, pdl, x, x_dtype, d, max_x);
}

cudaError_t launch_mxfp4_ffn(const FfnArgs& a, int num_sms, bool pdl, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  if (mxfp4_mma_gemv_supported(a.d, a.ff, a.x_dtype)) return launch_mxfp4_ffn_mma(a, num_sms, pdl, s);
  const Geom g0 = make_geom(0, a.d, a.ff), g1 = make_geom(1, a.d, a.ff);
  if (g0.stages < 2 || g1.stages < 2) return cudaErrorInvalidValue;
  cudaError_t err = a.x_dtype == MOE_BF16 ? launch_one<0, true>(a, g0, num_sms, pdl, s, "mxfp4_gate_up")
                                          : launch_one<0, false>(a, g0, num_sms, pdl, s, "mxfp4_gate_up");
  if (err != cudaSuccess) return err;
  return launch_one<1, false>(a, g1, num_sms, true, s, "mxfp4_down");
}

}  // namespace moe

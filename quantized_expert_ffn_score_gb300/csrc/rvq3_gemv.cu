// rvq3_gemv.cu -- routed-expert FFN on 3-stage residual-vector-quantised weights
// (WASTE README, "3 bits per expert weight": 3 stages of 256-entry codebooks
// over 8-dim vectors, 3.00 bits per weight; a weight is the sum of its three
// stage codewords).
//
// The weights are never materialised.  For one input vector x and one K-slice
// of 32 vector positions (256 columns) the kernel builds, in shared memory,
//   LUT[s][c][v] = <codebook_s[c], x[8v .. 8v+8)>      (fp32, 3 x 256 x 32)
// so that a row's partial dot product over the slice is
//   sum_v  LUT[0][code0[v][r]][v] + LUT[1][code1[v][r]][v] + LUT[2][code2[v][r]][v].
// Lane l of every warp owns vector position v = l, so the 32 lanes of a lookup
// hit 32 different banks whatever the codes are.  Codes are stored
// position-major (rows contiguous for a fixed position), so lane l reads 32
// consecutive rows' codes of its position with two 16-byte loads per stage.
// A 32-lane reduce-scatter leaves row r0 + l's slice partial on lane l; the
// slice partials go to a workspace buffer and a finalize kernel sums them in
// ascending slice order (then applies the activation, or scatters y).
#include <utility>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kRvqThreads = 256;
constexpr int kRvqWarps = kRvqThreads / 32;
constexpr int kSlicePos = 32;       // vector positions per K-slice
constexpr int kChunkRowsMax = 1536; // rows per work unit

struct RGeom {
  int K, rows, kinds, ns, nchunks, chunk_rows, upe;
  size_t mat_bytes;   // one matrix: 3 * rows * K / 8
};

RGeom make_rgeom(int mode, int d, int ff) {
  RGeom g;
  g.K = mode == 0 ? d : ff;
  g.rows = mode == 0 ? ff : d;
  g.kinds = mode == 0 ? 2 : 1;
  g.ns = (g.K / 8 + kSlicePos - 1) / kSlicePos;
  g.chunk_rows = g.rows < kChunkRowsMax ? g.rows : kChunkRowsMax;
  g.nchunks = (g.rows + g.chunk_rows - 1) / g.chunk_rows;
  g.upe = g.kinds * g.ns * g.nchunks;
  g.mat_bytes = (size_t)3 * ff * d / 8;
  return g;
}

constexpr size_t kRvqSmem = (size_t)3 * 256 * kSlicePos * sizeof(float)  // LUT
                            + 256 * sizeof(float)                        // x slice
                            + 3 * 256 * sizeof(uint4);                   // codebooks

template <int NV>
__device__ __forceinline__ void reduce_scatter32(float (&v)[NV], int lane) {
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
}

__device__ __forceinline__ uint32_t byte_of(const uint4& q, int r) {  // r static after unrolling
  const uint32_t w = (r >> 2) == 0 ? q.x : (r >> 2) == 1 ? q.y : (r >> 2) == 2 ? q.z : q.w;
  return (w >> (8 * (r & 3))) & 0xFFu;
}

template <int MODE>
__global__ void __launch_bounds__(kRvqThreads, 2) rvq3_unit_kernel(const FfnArgs a, const RGeom g) {
  extern __shared__ __align__(16) float rsm[];
  float* lut = rsm;                                         // [3][256][32]
  float* xs = lut + 3 * 256 * kSlicePos;                    // [256]
  uint4* cbs = reinterpret_cast<uint4*>(xs + 256);          // [3][256]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  pdl_launch_dependents();
  const int n_act = a.active[0];
  const int total = n_act * g.upe;
  for (int unit = blockIdx.x; unit < total; unit += gridDim.x) {
    const int e = a.active[1 + unit / g.upe];
    const uint8_t* rec = a.records[e];
    if (rec == nullptr || (reinterpret_cast<uintptr_t>(rec) & 15u)) {
      if (tid == 0) dev_error(a.err, rec == nullptr ? MOE_ERR_MISSING_EXPERT : MOE_ERR_INVALID_ARG, e);
      continue;
    }
    int u = unit % g.upe;
    const int kind = u / (g.ns * g.nchunks);
    u %= g.ns * g.nchunks;
    const int slice = u / g.nchunks, chunk = u % g.nchunks;
    const uint16_t* cb = a.cb[MODE == 0 ? kind : 2];
    const uint8_t* mat = rec + (size_t)(MODE == 0 ? kind : 2) * g.mat_bytes;
    const int v0 = slice * kSlicePos;
    const int nv = min(kSlicePos, g.K / 8 - v0);
    const int r_begin = chunk * g.chunk_rows, r_end = min(g.rows, r_begin + g.chunk_rows);
    const int s0 = a.offsets[e], ne = a.offsets[e + 1] - s0;
    __syncthreads();  // previous unit's readers of cbs / lut are done
    for (int i = tid; i < 3 * 256; i += kRvqThreads) cbs[i] = reinterpret_cast<const uint4*>(cb)[i];
    for (int q = 0; q < ne; ++q) {
      const int slot = s0 + q;
      __syncthreads();
      for (int i = tid; i < 256; i += kRvqThreads) {
        float v = 0.f;
        if (i < 8 * nv) {
          const int col = 8 * v0 + i;
          v = MODE == 0 ? load_act(a.x, a.x_dtype, (size_t)(a.pair_ids[slot] / a.k) * a.d + col)
                        : a.h[(size_t)slot * a.ff + col];
        }
        xs[i] = v;
      }
      __syncthreads();
      {  // LUT build: warp w takes entries (s, c) = w, w + 8, ...; lane = position
        float xv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) xv[i] = xs[8 * lane + i];
        for (int p = warp; p < 3 * 256; p += kRvqWarps) {
          const uint4 c8 = cbs[p];
          const uint32_t hw[4] = {c8.x, c8.y, c8.z, c8.w};
          float acc = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hw[j]));
            acc = fmaf(f.x, xv[2 * j], acc);
            acc = fmaf(f.y, xv[2 * j + 1], acc);
          }
          lut[p * kSlicePos + lane] = acc;
        }
      }
      __syncthreads();
      const bool vl = lane < nv;
      const float* l0 = lut + lane;
      const float* l1 = lut + 256 * kSlicePos + lane;
      const float* l2 = lut + 2 * 256 * kSlicePos + lane;
      for (int rg = r_begin + 32 * warp; rg < r_end; rg += 32 * kRvqWarps) {
        float acc[32];
        if (vl) {
          uint4 c[3][2];
#pragma unroll
          for (int s = 0; s < 3; ++s) {
            const uint4* p = reinterpret_cast<const uint4*>(mat + ((size_t)s * (g.K / 8) + v0 + lane) * g.rows + rg);
            c[s][0] = __ldg(p);
            c[s][1] = __ldg(p + 1);
          }
#pragma unroll
          for (int r = 0; r < 32; ++r) {
            const uint32_t k0 = byte_of(c[0][r >> 4], r & 15);
            const uint32_t k1 = byte_of(c[1][r >> 4], r & 15);
            const uint32_t k2 = byte_of(c[2][r >> 4], r & 15);
            acc[r] = l0[k0 * kSlicePos] + l1[k1 * kSlicePos] + l2[k2 * kSlicePos];
          }
        } else {
#pragma unroll
          for (int r = 0; r < 32; ++r) acc[r] = 0.f;
        }
        reduce_scatter32<32>(acc, lane);
        a.partial[(((size_t)slot * g.kinds + kind) * g.ns + slice) * g.rows + rg + lane] = acc[0];
      }
    }
  }
}

// The same lookups with the table shared by every expert of a token (gate/up:
// the codebooks are per layer and the experts of a token see the same x) or
// of a slot (down: h is per slot).  Work units, in this order:
//   (group g, kind, slice, slot of the group, 1536-row chunk)
// with g = token (MODE 0, the token's k slots) or slot (MODE 1, one slot);
// each unit streams one expert's rows of the slice (long contiguous runs per
// vector position), persistent CTAs take contiguous unit ranges and rebuild
// the table only when (g, kind, slice) changes.  For at most kLutMaxPairs pairs.
constexpr int kLutChunk = 1536;
constexpr int kLutMaxPairs = 512;
constexpr size_t kLutSmem = kRvqSmem + 2 * kLutMaxPairs * sizeof(uint16_t);  // two CTAs per SM

template <int MODE>
__global__ void __launch_bounds__(kRvqThreads, 2) rvq3_lut_kernel(const FfnArgs a, const RGeom g) {
  extern __shared__ __align__(16) float rsm[];
  float* lut = rsm;                                         // [3][256][32]
  float* xs = lut + 3 * 256 * kSlicePos;                    // [256]
  uint4* cbs = reinterpret_cast<uint4*>(xs + 256);          // [3][256]
  uint16_t* slot_of_pair = reinterpret_cast<uint16_t*>(cbs + 3 * 256);  // [P]
  uint16_t* expert_of_slot = slot_of_pair + kLutMaxPairs;                // [P]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  pdl_launch_dependents();
  const int P = a.T * a.k;
  for (int i = tid; i < P; i += kRvqThreads) slot_of_pair[a.pair_ids[i]] = (uint16_t)i;
  const int n_act = a.active[0];
  for (int ai = warp; ai < n_act; ai += kRvqWarps) {
    const int e = a.active[1 + ai];
    for (int sl = a.offsets[e] + lane; sl < a.offsets[e + 1]; sl += 32) expert_of_slot[sl] = (uint16_t)e;
  }
  const int ngroups = MODE == 0 ? a.T : P;
  const int nchunks = (g.rows + kLutChunk - 1) / kLutChunk;
  const int nslots = MODE == 0 ? a.k : 1;
  const long long total = (long long)ngroups * g.kinds * g.ns * nslots * nchunks;
  const int ub = (int)(total * blockIdx.x / gridDim.x), ue = (int)(total * (blockIdx.x + 1) / gridDim.x);
  int cur_key = -1, cur_kind = -1;
  for (int unit = ub; unit < ue; ++unit) {
    int u = unit;
    const int chunk = u % nchunks;
    u /= nchunks;
    const int j = u % nslots;
    u /= nslots;
    const int slice = u % g.ns;
    u /= g.ns;
    const int kind = u % g.kinds;
    const int grp = u / g.kinds;
    const int key = (grp * g.kinds + kind) * g.ns + slice;
    const int v0 = slice * kSlicePos;
    const int nv = min(kSlicePos, g.K / 8 - v0);
    __syncthreads();  // the prologue's tables; the previous unit's readers of lut / cbs / xs
    if (key != cur_key) {
      if (kind != cur_kind) {
        const uint16_t* cb = a.cb[MODE == 0 ? kind : 2];
        for (int i = tid; i < 3 * 256; i += kRvqThreads) cbs[i] = reinterpret_cast<const uint4*>(cb)[i];
        cur_kind = kind;
      }
      for (int i = tid; i < 256; i += kRvqThreads) {
        float v = 0.f;
        if (i < 8 * nv) {
          const int col = 8 * v0 + i;
          v = MODE == 0 ? load_act(a.x, a.x_dtype, (size_t)grp * a.d + col) : a.h[(size_t)grp * a.ff + col];
        }
        xs[i] = v;
      }
      __syncthreads();
      float xv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) xv[i] = xs[8 * lane + i];
      for (int p = warp; p < 3 * 256; p += kRvqWarps) {
        const uint4 c8 = cbs[p];
        const uint32_t hw[4] = {c8.x, c8.y, c8.z, c8.w};
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hw[j]));
          acc = fmaf(f.x, xv[2 * j], acc);
          acc = fmaf(f.y, xv[2 * j + 1], acc);
        }
        lut[p * kSlicePos + lane] = acc;
      }
      cur_key = key;
      __syncthreads();
    }
    const bool vl = lane < nv;
    const float* l0 = lut + lane;
    const float* l1 = lut + 256 * kSlicePos + lane;
    const float* l2 = lut + 2 * 256 * kSlicePos + lane;
    const int r_begin = chunk * kLutChunk, r_end = min(g.rows, r_begin + kLutChunk);
    const int ngrp = (r_end - r_begin + 31) / 32;
    // 32-row groups of the unit's expert rows; warp w takes groups w, w + 8, ...
    const int slot = MODE == 0 ? slot_of_pair[grp * a.k + j] : grp;
    for (int task = warp; task < ngrp; task += kRvqWarps) {
      const int rg = r_begin + 32 * task;
      const int e = expert_of_slot[slot];
      const uint8_t* rec = a.records[e];
      if (rec == nullptr || (reinterpret_cast<uintptr_t>(rec) & 15u)) {
        if (lane == 0) dev_error(a.err, rec == nullptr ? MOE_ERR_MISSING_EXPERT : MOE_ERR_INVALID_ARG, e);
        continue;
      }
      const uint8_t* mat = rec + (size_t)(MODE == 0 ? kind : 2) * g.mat_bytes;
      float acc[32];
      if (vl) {
        uint4 c[3][2];
#pragma unroll
        for (int st = 0; st < 3; ++st) {
          const uint4* q = reinterpret_cast<const uint4*>(mat + ((size_t)st * (g.K / 8) + v0 + lane) * g.rows + rg);
          c[st][0] = __ldg(q);
          c[st][1] = __ldg(q + 1);
        }
#pragma unroll
        for (int r = 0; r < 32; ++r) {
          const uint32_t k0 = byte_of(c[0][r >> 4], r & 15);
          const uint32_t k1 = byte_of(c[1][r >> 4], r & 15);
          const uint32_t k2 = byte_of(c[2][r >> 4], r & 15);
          acc[r] = l0[k0 * kSlicePos] + l1[k1 * kSlicePos] + l2[k2 * kSlicePos];
        }
      } else {
#pragma unroll
        for (int r = 0; r < 32; ++r) acc[r] = 0.f;
      }
      reduce_scatter32<32>(acc, lane);
      a.partial[(((size_t)slot * g.kinds + kind) * g.ns + slice) * g.rows + rg + lane] = acc[0];
    }
  }
}

// Sums the slice partials in ascending slice order.
template <int MODE>
__global__ void rvq3_finalize_kernel(const FfnArgs a, const RGeom g, int P) {
  pdl_wait();
  pdl_launch_dependents();
  const size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (idx >= (size_t)P * g.rows) return;
  const int slot = (int)(idx / g.rows), r = (int)(idx % g.rows);
  const float* base = a.partial + (size_t)slot * g.kinds * g.ns * g.rows + r;
  float s0 = 0.f;
  for (int s = 0; s < g.ns; ++s) s0 += base[(size_t)s * g.rows];
  if (MODE == 0) {
    float s1 = 0.f;
    for (int s = 0; s < g.ns; ++s) s1 += base[(size_t)(g.ns + s) * g.rows];
    a.h[(size_t)slot * a.ff + r] = act_fn(s0, s1, a.act);
  } else {
    a.y_pairs[(size_t)a.pair_ids[slot] * a.d + r] = s0;
  }
}

}  // namespace

size_t rvq3_partial_floats(int T, int k, int d, int ff) {
  const RGeom g0 = make_rgeom(0, d, ff), g1 = make_rgeom(1, d, ff);
  const size_t per0 = (size_t)g0.kinds * g0.ns * g0.rows, per1 = (size_t)g1.kinds * g1.ns * g1.rows;
  return (size_t)T * k * (per0 > per1 ? per0 : per1);
}

cudaError_t launch_rvq3_ffn(const FfnArgs& a, int num_sms, bool pdl, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  const int P = a.T * a.k;
  const RGeom g0 = make_rgeom(0, a.d, a.ff), g1 = make_rgeom(1, a.d, a.ff);
  const dim3 grid(2 * num_sms);
  const bool lut_shared = P <= kLutMaxPairs && a.E <= 65536 && g0.rows % 32 == 0 && g1.rows % 32 == 0;
  // down tables are per slot: sharing saves nothing at one token, where the per-expert units are faster
  // (K3 shape: 59 against 64 us); gate/up tables are shared by the token's experts (93 -> 90 us)
  const bool lut_down = lut_shared && a.T >= 2;
  cudaError_t err;
  if (lut_shared) {
    ensure_smem(rvq3_lut_kernel<0>, kLutSmem);
    err = launch("rvq3_gate_up", rvq3_lut_kernel<0>, grid, dim3(kRvqThreads), kLutSmem, s, pdl, a, g0);
  } else {
    ensure_smem(rvq3_unit_kernel<0>, kRvqSmem);
    err = launch("rvq3_gate_up", rvq3_unit_kernel<0>, grid, dim3(kRvqThreads), kRvqSmem, s, pdl, a, g0);
  }
  if (err != cudaSuccess) return err;
  const size_t n0 = (size_t)P * g0.rows, n1 = (size_t)P * g1.rows;
  err = launch("rvq3_gate_up_sum", rvq3_finalize_kernel<0>, dim3((unsigned)((n0 + 255) / 256)), dim3(256), 0, s, true, a, g0, P);
  if (err != cudaSuccess) return err;
  if (lut_down) {
    ensure_smem(rvq3_lut_kernel<1>, kLutSmem);
    err = launch("rvq3_down", rvq3_lut_kernel<1>, grid, dim3(kRvqThreads), kLutSmem, s, true, a, g1);
  } else {
    ensure_smem(rvq3_unit_kernel<1>, kRvqSmem);
    err = launch("rvq3_down", rvq3_unit_kernel<1>, grid, dim3(kRvqThreads), kRvqSmem, s, true, a, g1);
  }
  if (err != cudaSuccess) return err;
  return launch("rvq3_down_sum", rvq3_finalize_kernel<1>, dim3((unsigned)((n1 + 255) / 256)), dim3(256), 0, s, true, a, g1, P);
}

}  // namespace moe

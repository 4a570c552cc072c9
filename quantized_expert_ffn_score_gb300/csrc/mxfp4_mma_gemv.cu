// mxfp4_mma_gemv.cu -- routed-expert FFN on MXFP4 weights for experts with a
// few tokens (decode), the inner products on the warp-level tensor
// instruction mma.sync.m16n8k16 (f16 operands, fp32 accumulation).  The packed
// weights are consumed as stored and never widened in memory (LazyLoRA README,
// "The engine": fused MXFP4 decode-and-dot with fp32 expert sums).
//
// Per 32-column block of a weight row (one E8M0 scale) the block's partial
// sums are formed exactly: an E2M1 code is an f16 (cvt.e2m1x2), the
// activation is an exact f16 (bf16 x after a power-of-two rescale per token;
// h as an f16 pair hi + lo after a power-of-two rescale per warp and token),
// the products are exact in fp32 and summed in fp32 by the tensor core.  The
// block scale 2^(B-127) then multiplies the block's partial sum in fp32.
//
// The block's 32 columns are assigned to the MMA's K positions in the order
// that lets each thread use whole bytes of the stored codes: thread (g, t) of
// the warp (g = lane / 4, t = lane % 4) takes the 8 codes of bytes 4t..4t+3 of
// its rows' block, i.e. columns 8t..8t+7, which fill its A fragment of two
// m16n8k16 instructions; its B fragment holds the activations of the same
// columns for token g.  A dot product is a sum, so the order does not matter.
//
// Two launches of one persistent kernel (as the FMA-based kernel in
// mxfp4_gemv.cu, whose tiling this follows):
//   MODE 0  gate/up: tile = rows [r0, r0+16) of Wg and of Wu (two M tiles);
//           the epilogue applies the activation and writes h[slot][r] (fp32).
//   MODE 1  down: tile = rows [r0, r0+32) of Wd (two M tiles); writes
//           y_pairs[pair][r].
// Consumer warps split K in ranges of 8 blocks (up to 15 warps).
// Up to 8 tokens of an expert per pass (the MMA's N); more tokens take more
// passes over each staged tile.
// The producer warp copies each tile row by row (bulk async copies, one per
// lane) into shared memory rows padded by 16 bytes, so that the fragment
// loads (32-bit words of 8 rows at the same column) hit distinct banks.
//
// One-token launches (T = 1) keep the B fragments in shared memory instead of
// registers: only the lanes of the token's column (gate/up: lanes 0-3; down,
// whose hi and lo parts fill two columns: lanes 0-7) hold non-zero values, so
// a block's fragments are 64 or 128 bytes, read back once per block with one
// 16-byte load (the other lanes read a zeroed slot), and the warps' partial
// sums keep one token column.  Measured against the register form on one
// GB300: gate/up 49.2 -> 47.7 us, decode step 91.9 -> 90.7 us; with the
// registers freed, 4 blocks per warp and 28 compute warps were slower (57 us).
#include <type_traits>
#include <utility>

#include "moe_internal.cuh"
#include "tc_ops.cuh"

namespace moe {
namespace {

constexpr int kTok = 8;  // tokens per pass (MMA N)
constexpr int kRows = 32;  // weight rows per tile (two 16-row M tiles)
constexpr int kMaxStagesM = 4;
constexpr int kSmemBudgetM = 224 * 1024;
constexpr int kMaxConsumerWarps = 14;  // compute warps of 8 blocks (plus one reducer and one producer warp)
constexpr int kMaxBlocks = kMaxConsumerWarps * 8;  // K / 32 at most (d, ff <= 3584)

struct GeomM {
  int K;            // contraction length
  uint32_t sb_lane_bytes;  // one-token launches: bytes of B fragments per block (0: fragments in registers)
  uint32_t sb_off;         // their offset in shared memory (then a zeroed 16-byte slot)
  int nblk;         // K / 32
  int bpw;          // blocks per consumer warp
  int warps;        // consumer warps
  int tpe;          // tiles per expert
  uint32_t pitch;   // shared-memory bytes per staged row: K / 2 + 16
  uint32_t scales;  // bytes of scales per stage: 32 rows x K / 32
  uint32_t stage_bytes;
  int stages;
  size_t red_floats;  // one reduction buffer: warps x 32 rows x 8 tokens (1 token for one-token launches)
  size_t smem;
};

GeomM make_geom_m(int mode, int d, int ff, int bpw, bool staged_b) {
  GeomM g;
  g.K = mode == 0 ? d : ff;
  g.sb_lane_bytes = staged_b ? (mode == 0 ? 64u : 128u) : 0u;
  g.nblk = g.K / 32;
  g.bpw = bpw;
  g.warps = (g.nblk + g.bpw - 1) / g.bpw;
  g.tpe = mode == 0 ? ff / 16 : d / 32;
  g.pitch = (uint32_t)g.K / 2 + 16;
  g.scales = (uint32_t)kRows * (uint32_t)g.K / 32;
  g.stage_bytes = (uint32_t)kRows * g.pitch + ((g.scales + 15) & ~15u);
  g.red_floats = (size_t)g.warps * kRows * (staged_b ? 1 : kTok);
  const size_t sb = staged_b ? (size_t)g.nblk * g.sb_lane_bytes + 16 : 0;
  const size_t fixed = (2 * kMaxStagesM + 4) * sizeof(uint64_t) + (2 * g.red_floats + 2 * kTok) * sizeof(float) + sb;
  g.stages = (int)((kSmemBudgetM - fixed) / g.stage_bytes);
  if (g.stages > kMaxStagesM) g.stages = kMaxStagesM;
  g.smem = (size_t)g.stages * g.stage_bytes + fixed;
  g.sb_off = (uint32_t)(g.smem - sb);
  return g;
}

__device__ __forceinline__ bool rec_ok(const uint8_t* rec) {
  return rec != nullptr && ((reinterpret_cast<uintptr_t>(rec) & 15u) == 0);
}

// D += A * B for one m16n8k16 (row-major A, column-major B), f16 in, f32 out.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Two E8M0 scale bytes (lo: first) -> their fp32 values 2^(B-127), with
// 0 -> 2^-127 and 255 -> NaN, through the bf16 pair conversion.
__device__ __forceinline__ void e8m0x2_to_f32(uint32_t two, float& f0, float& f1) {
  uint32_t r;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.bf16x2.ue8m0x2 %0, t; }" : "=r"(r) : "r"(two));
  f0 = __uint_as_float(r << 16);
  f1 = __uint_as_float(r & 0xFFFF0000u);
}

// fp32 2^e for -126 <= e <= 127.
__device__ __forceinline__ float pow2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// Power-of-two shift s with max * 2^-s in [2^14, 2^15) (0 for max 0 or not finite).
__device__ __forceinline__ int shift_for(float mx) {
  int s = 0;
  if (mx > 0.f && mx < INFINITY) s = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127 - 14;
  return max(-100, min(100, s));
}

// The activations of one pass as B fragments: for each of the warp's blocks,
// token g's columns 8t..8t+7 as four f16 pairs (MODE 1: hi and lo).  PAIR
// (MODE 1, at most 4 tokens per pass): column 2n holds token n's hi part and
// column 2n + 1 its lo part, so one MMA forms both partial sums (lane group g
// holds token g / 2, part g % 2) and the lo array is not needed.
template <int MODE, int BPW, bool PAIR, bool SB>
struct Frags {
  uint32_t hi[SB ? 1 : BPW][4];
  uint32_t lo[(MODE == 1 && !PAIR && !SB) ? BPW : 1][4];
  float unscale;  // MODE 1: 2^s of this warp's rescale for the lane's token (MODE 0: unused)
  uint8_t* sb;    // SB: the blocks' fragments in shared memory, lane_bytes per block
  uint32_t lane_bytes;

  // SB: lanes below lane_bytes / 16 keep block b's fragment at sb + b * lane_bytes + 16 lane
  __device__ __forceinline__ void put(int j, int b, int i, uint32_t v, int lane) {
    if (SB) {
      if ((uint32_t)lane * 16u < lane_bytes) reinterpret_cast<uint32_t*>(sb + (size_t)b * lane_bytes + 16 * lane)[i] = v;
    } else {
      hi[j][i] = v;
    }
  }

  // tok_fixed >= 0: the pass's one token is that token (no routing read)
  __device__ void load(const FfnArgs& a, int slot0, int nt, int b0, int nblk, int lane, int tok_fixed = -1) {
    const int g0 = lane >> 2, t = lane & 3;
    const int g = PAIR ? g0 >> 1 : g0;  // the lane's token in the pass
    const bool live = g < nt;
    unscale = 1.f;
    if (MODE == 0) {
      float inv = 1.f;
      const uint16_t* xrow = nullptr;
      if (live) {
        const int tok = tok_fixed >= 0 ? tok_fixed : a.pair_ids[slot0 + g] / a.k;
        inv = pow2i(-shift_for(a.max_x[tok]));
        xrow = static_cast<const uint16_t*>(a.x) + (size_t)tok * a.d;
      }
#pragma unroll
      for (int j = 0; j < BPW; ++j) {
        const int b = b0 + j;
        uint4 w = make_uint4(0, 0, 0, 0);
        if (live && b < nblk) w = *reinterpret_cast<const uint4*>(xrow + 32 * b + 8 * t);
        const uint32_t v[4] = {w.x, w.y, w.z, w.w};
        if (SB && b >= nblk) continue;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          put(j, b, i, pack_f16x2(__uint_as_float(v[i] << 16) * inv, __uint_as_float(v[i] & 0xFFFF0000u) * inv), lane);
      }
    } else {
      // two passes over the (cached) rows: the token's max over this warp's
      // columns first, then the rescaled hi/lo pairs
      const float* hrow = live ? a.h + (size_t)(slot0 + g) * a.ff : nullptr;
      float m = 0.f;
#pragma unroll
      for (int j = 0; j < BPW; ++j) {
        const int b = b0 + j;
        if (live && b < nblk) {
          const float4 p = *reinterpret_cast<const float4*>(hrow + 32 * b + 8 * t);
          const float4 q = *reinterpret_cast<const float4*>(hrow + 32 * b + 8 * t + 4);
          m = fmaxf(m, fmaxf(fmaxf(fabsf(p.x), fabsf(p.y)), fmaxf(fabsf(p.z), fabsf(p.w))));
          m = fmaxf(m, fmaxf(fmaxf(fabsf(q.x), fabsf(q.y)), fmaxf(fabsf(q.z), fabsf(q.w))));
        }
      }
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));  // the 4 lanes of group g
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      const int s = shift_for(m);
      const float inv = pow2i(-s);
      unscale = pow2i(s);
#pragma unroll
      for (int j = 0; j < BPW; ++j) {
        const int b = b0 + j;
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (live && b < nblk) {
          const float4 p = *reinterpret_cast<const float4*>(hrow + 32 * b + 8 * t);
          const float4 q = *reinterpret_cast<const float4*>(hrow + 32 * b + 8 * t + 4);
          v[0] = p.x; v[1] = p.y; v[2] = p.z; v[3] = p.w;
          v[4] = q.x; v[5] = q.y; v[6] = q.z; v[7] = q.w;
        }
        if (SB && b >= nblk) continue;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float x0 = v[2 * i] * inv, x1 = v[2 * i + 1] * inv;
          const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
          const uint32_t hv = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
          const uint32_t lv = pack_f16x2(x0 - __half2float(h0), x1 - __half2float(h1));
          if (PAIR) {
            put(j, b, i, (g0 & 1) ? lv : hv, lane);
          } else {
            hi[SB ? 0 : j][i] = hv;
            lo[(MODE == 1 && !PAIR && !SB) ? j : 0][i] = lv;
          }
        }
      }
    }
    if (SB) __syncwarp();
  }
};

// Per token of a pass, for the epilogue (consumer warp 0 only, which alone
// reads them): MODE 0 the activation rescale 2^s_t and the slot, MODE 1 the
// pair id.
template <int MODE>
__device__ __forceinline__ void note_tokens(const FfnArgs& a, int slot0, int nt, int lane, float* tok_f, int* tok_i) {
  if (lane < nt) {
    const int slot = slot0 + lane;
    if (MODE == 0) {
      tok_f[lane] = pow2i(shift_for(a.max_x[a.T == 1 ? 0 : a.pair_ids[slot] / a.k]));
      tok_i[lane] = slot;
    } else {
      tok_i[lane] = a.pair_ids[slot];
    }
  }
  __syncwarp();
}

// Consumers: `warps` warps (warp w owns blocks [BPW w, BPW w + BPW)), then one
// producer warp.  Consumers never meet at a CTA-wide barrier: each pass's
// partial sums go to a double-buffered shared array whose fill is counted by an
// mbarrier, and a reducer warp (warp 0, which computes nothing else) adds them
// and writes the pass's outputs.  Every wait is bounded.
template <int MODE, int BPW, bool PAIR, bool SB>
__global__ void __launch_bounds__((kMaxBlocks / BPW + 2) * 32, 1) mxfp4_mma_gemv_kernel(const FfnArgs a, const GeomM g) {
  static_assert(!SB || MODE == 0 || PAIR, "one-token fragments in shared memory: gate/up, or down with paired columns");
  constexpr int kRedTok = SB ? 1 : kTok;  // token columns of a reduction buffer row
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)g.stages * g.stage_bytes);
  uint64_t* empty = full + kMaxStagesM;
  uint64_t* red_full = empty + kMaxStagesM;  // [2]
  uint64_t* red_empty = red_full + 2;        // [2]
  float* red = reinterpret_cast<float*>(red_empty + 2);  // [2][warps][32 rows][8 tokens]
  float* tok_f = red + 2 * g.red_floats;                  // [8] per token of the pass: 2^s (MODE 0)
  int* tok_i = reinterpret_cast<int*>(tok_f + kTok);      // [8] per token: slot (MODE 0) or pair id (MODE 1)

  // warp 0 reduces, warps 1 .. W compute (warp w owns blocks [BPW (w-1), BPW w)), warp W + 1 loads
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < g.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], g.warps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&red_full[b], g.warps);
      mbar_init(&red_empty[b], 1);
    }
    fence_mbar_init();
  }
  if (SB && threadIdx.x < 4)  // the zeroed slot after the fragments
    reinterpret_cast<uint32_t*>(smem + g.sb_off + (size_t)g.nblk * g.sb_lane_bytes)[threadIdx.x] = 0u;
  __syncthreads();
  // The down pass's producer stages weights only, and the routing it follows
  // was written two launches earlier (complete before the gate/up pass passed
  // its own wait, which precedes this launch): it starts streaming while the
  // gate/up pass finishes.  Everything that reads h or writes outputs waits.
  // One-token gate/up: when x and max |x| were complete before the kernel just
  // ahead of this one (a.x_early: the layer path, where the router wrote max |x|
  // two launches earlier), the compute warps stage the token's B fragments
  // before the wait; the producer pulls the record table into L2 while the
  // routing is made.  Dependents are released only after the wait: the down
  // pass's producer reads the routing without waiting, which is safe only
  // because this pass's wait has returned before that launch.
  const int W = g.warps;
  const bool x_staged = SB && MODE == 0 && a.x_early;
  if (x_staged && warp >= 1 && warp <= W) {
    Frags<MODE, BPW, PAIR, SB> f0;
    f0.sb = smem + g.sb_off;
    f0.lane_bytes = g.sb_lane_bytes;
    f0.load(a, 0, 1, (warp - 1) * BPW, g.nblk, lane, 0);
  }
  if (MODE == 0 && warp == W + 1)
    for (int i = 16 * lane; i < a.E; i += 16 * 32) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.records + i));
  if (MODE == 0 || warp != W + 1) pdl_wait();
  pdl_launch_dependents();

  const long long total = (long long)a.active[0] * g.tpe;
  const int t_begin = (int)(total * blockIdx.x / gridDim.x);
  const int t_end = (int)(total * (blockIdx.x + 1) / gridDim.x);
  const size_t mat = (size_t)a.ff * a.d / 2 + (size_t)a.ff * a.d / 32;
  const int K = g.K;

  if (warp == W + 1) {
    // ------------------------------------------------------------ producer (whole warp: one row copy per lane)
    int it = 0, cur_a = -1;
    const uint8_t* rec = nullptr;
    bool alive = true;
    // tile = ai * tpe + rt and the ring position advance without divisions
    int ai = t_begin / g.tpe, rt = t_begin - ai * g.tpe - 1, stage = -1;
    uint32_t rph = 1;  // parity of the current round over the stage ring
    for (int tile = t_begin; tile < t_end && alive; ++tile) {
      if (++rt == g.tpe) {
        rt = 0;
        ++ai;
      }
      if (ai != cur_a) {
        cur_a = ai;
        const int e = a.active[1 + ai];
        rec = a.records[e];
        if (lane == 0 && !rec_ok(rec))
          dev_error(a.err, rec == nullptr ? MOE_ERR_MISSING_EXPERT : MOE_ERR_INVALID_ARG, e);
      }
      if (!rec_ok(rec)) continue;
      if (++stage == g.stages) stage = 0;
      if (stage == 0) rph ^= 1u;
      int ok = 1;
      if (lane == 0) {
        if (it >= g.stages && !mbar_wait(&empty[stage], rph ^ 1u, a.err)) ok = 0;
        if (ok) mbar_arrive_expect_tx(&full[stage], (uint32_t)kRows * (uint32_t)(K / 2) + g.scales);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        alive = false;
        break;
      }
      uint8_t* dst = smem + (size_t)stage * g.stage_bytes;
      // lane l copies staged row l: MODE 0 rows 0..15 = Wg rows, 16..31 = Wu rows
      const uint8_t* src;
      if (MODE == 0) {
        const size_t r = (size_t)rt * 16 + (lane & 15);
        src = rec + (lane < 16 ? 0 : mat) + r * (K / 2);
      } else {
        src = rec + 2 * mat + ((size_t)rt * kRows + lane) * (K / 2);
      }
      bulk_g2s(dst + (size_t)lane * g.pitch, src, (uint32_t)(K / 2), &full[stage]);
      uint8_t* sdst = dst + (size_t)kRows * g.pitch;
      if (MODE == 0) {
        if (lane < 2) {
          const size_t off = (lane == 0 ? 0 : mat) + (size_t)a.ff * (K / 2) + (size_t)rt * 16 * (K / 32);
          bulk_g2s(sdst + (size_t)lane * 16 * (K / 32), rec + off, (uint32_t)(16 * (K / 32)), &full[stage]);
        }
      } else if (lane == 0) {
        const size_t off = 2 * mat + (size_t)a.d * (K / 2) + (size_t)rt * kRows * (K / 32);
        bulk_g2s(sdst, rec + off, (uint32_t)(kRows * (K / 32)), &full[stage]);
      }
      ++it;
    }
    // never leave with copies in flight
    if (lane == 0)
      for (int j = (it > g.stages ? it - g.stages : 0); j < it; ++j)
        mbar_wait_drain(&full[j % g.stages], (j / g.stages) & 1, a.err);
    return;
  }

  if (warp == 0) {
    // -------------------------------------------------------------- reducer
    int pc = 0, cur_a = -1, s0 = 0, ne = 0, noted = -1;
    bool rec_good = false;
    int ai = t_begin / g.tpe, rt = t_begin - ai * g.tpe - 1;
    for (int tile = t_begin; tile < t_end; ++tile) {
      if (++rt == g.tpe) {
        rt = 0;
        ++ai;
      }
      if (ai != cur_a) {
        cur_a = ai;
        const int e = a.active[1 + ai];
        rec_good = rec_ok(a.records[e]);
        s0 = a.offsets[e];
        ne = a.offsets[e + 1] - s0;
      }
      if (!rec_good) continue;
      for (int c0 = 0; c0 < ne; c0 += kTok) {
        const int nt = min(kTok, ne - c0);
        const int bi = pc & 1, use = pc >> 1;
        ++pc;
        if (ne > kTok || noted != cur_a) {  // a one-pass expert's tokens are noted once
          note_tokens<MODE>(a, s0 + c0, nt, lane, tok_f, tok_i);
          noted = cur_a;
        }
        if (!mbar_wait(&red_full[bi], use & 1, a.err)) return;
        const float* rbase = red + bi * g.red_floats;
        if (MODE == 0) {  // lane = (half, row): gate rows on lanes 0-15, up rows on lanes 16-31
          for (int n = 0; n < nt; ++n) {
            float sum0 = 0.f, sum1 = 0.f;
            int w = 0;
            for (; w + 1 < W; w += 2) {
              sum0 += rbase[((size_t)w * kRows + lane) * kRedTok + n];
              sum1 += rbase[((size_t)(w + 1) * kRows + lane) * kRedTok + n];
            }
            if (w < W) sum0 += rbase[((size_t)w * kRows + lane) * kRedTok + n];
            const float sum = sum0 + sum1;
            const float us = __shfl_down_sync(0xffffffffu, sum, 16);
            if (lane < 16) {
              const float pw = tok_f[n];
              a.h[(size_t)tok_i[n] * a.ff + (size_t)rt * 16 + lane] = act_fast(sum * pw, us * pw, a.act);
            }
          }
        } else {
          for (int idx = lane; idx < kRows * nt; idx += 32) {
            const int r = idx & 31, n = idx >> 5;
            float ys = 0.f;
            for (int w = 0; w < W; ++w) ys += rbase[((size_t)w * kRows + r) * kRedTok + n];
            a.y_pairs[(size_t)tok_i[n] * a.d + (size_t)rt * kRows + r] = ys;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&red_empty[bi]);
      }
    }
    return;
  }

  // -------------------------------------------------------------- compute warps
  const int cw = warp - 1;
  const int gq = lane >> 2, tq = lane & 3;
  const int b0 = cw * BPW;
  Frags<MODE, BPW, PAIR, SB> fr;
  fr.sb = smem + g.sb_off;
  fr.lane_bytes = g.sb_lane_bytes;
  // SB: this lane's fragment of block b at sb_lane + b * lane_bytes, or the zeroed slot
  const uint32_t sb_zero = tc::saddr(smem + g.sb_off + (size_t)g.nblk * g.sb_lane_bytes);
  const bool sb_live = (uint32_t)lane * 16u < g.sb_lane_bytes;
  const uint32_t sb_lane = tc::saddr(smem + g.sb_off) + 16u * (uint32_t)lane;
  int it = 0, pc = 0, cur_a = -1, s0 = 0, ne = 0;
  bool rec_good = false;
  int ai = t_begin / g.tpe, rt_ = t_begin - ai * g.tpe - 1, stage = -1;
  uint32_t cph = 1;  // parity of the current round over the stage ring
  for (int tile = t_begin; tile < t_end; ++tile) {
    if (++rt_ == g.tpe) {
      rt_ = 0;
      ++ai;
    }
    if (ai != cur_a) {  // a new expert: its slots, and its activations if one pass holds them
      cur_a = ai;
      const int e = a.active[1 + ai];
      rec_good = rec_ok(a.records[e]);
      s0 = a.offsets[e];
      ne = a.offsets[e + 1] - s0;
      // (one-token gate/up of the layer path: staged before the wait)
      if (rec_good && ne <= kTok && !x_staged) fr.load(a, s0, ne, b0, g.nblk, lane);
    }
    if (!rec_good) continue;
    if (++stage == g.stages) stage = 0;
    if (stage == 0) cph ^= 1u;
    if (!mbar_wait(&full[stage], cph, a.err)) return;
    ++it;
    const uint8_t* st = smem + (size_t)stage * g.stage_bytes;
    const uint8_t* sc = st + (size_t)kRows * g.pitch;
    for (int c0 = 0; c0 < ne; c0 += kTok) {
      const int nt = min(kTok, ne - c0);
      if (ne > kTok) fr.load(a, s0 + c0, nt, b0, g.nblk, lane);
      float acc[2][4];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[m][i] = 0.f;
      // the warp's block scales of its rows ra = 16 m + gq and rb = ra + 8: one 8-byte load each when
      // the warp's first scale byte is 8-byte aligned (8 blocks per warp and K / 32 a multiple of 8),
      // else bytes (only blocks < nblk)
      uint2 sra[2], srb[2];
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const uint8_t* pa = sc + (size_t)(16 * m + gq) * (K / 32) + b0;
        const uint8_t* pb = sc + (size_t)(16 * m + gq + 8) * (K / 32) + b0;
        if (BPW == 8 && ((K / 32) & 7) == 0) {
          sra[m] = *reinterpret_cast<const uint2*>(pa);
          srb[m] = *reinterpret_cast<const uint2*>(pb);
        } else {
          uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (b0 + j < g.nblk) {
              w[j >> 2] |= (uint32_t)pa[j] << (8 * (j & 3));
              w[2 + (j >> 2)] |= (uint32_t)pb[j] << (8 * (j & 3));
            }
          }
          sra[m] = make_uint2(w[0], w[1]);
          srb[m] = make_uint2(w[2], w[3]);
        }
      }
      // the block loop, compiled twice: a pass of one token (decode) skips the
      // products of the MMA's second token column, which are zero
      auto blocks = [&](auto one_tag) {
        constexpr bool ONE = decltype(one_tag)::value;
#pragma unroll
        for (int j = 0; j < BPW; ++j) {
          const int b = b0 + j;
          if (b >= g.nblk) continue;  // (fully unrolled: the fragments stay in registers)
          uint4 bj = make_uint4(0u, 0u, 0u, 0u);
          if (SB) {
            const uint32_t ad = sb_live ? sb_lane + (uint32_t)b * g.sb_lane_bytes : sb_zero;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(bj.x), "=r"(bj.y), "=r"(bj.z), "=r"(bj.w) : "r"(ad));
          }
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const int ra = 16 * m + gq, rb = ra + 8;
            const uint32_t wa = *reinterpret_cast<const uint32_t*>(st + (size_t)ra * g.pitch + 16 * b + 4 * tq);
            const uint32_t wb = *reinterpret_cast<const uint32_t*>(st + (size_t)rb * g.pitch + 16 * b + 4 * tq);
            uint32_t pa[4], pb[4];
            e2m1x8_to_f16x2(wa, pa);
            e2m1x8_to_f16x2(wb, pb);
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t A0[4] = {pa[0], pb[0], pa[1], pb[1]};
            const uint32_t A1[4] = {pa[2], pb[2], pa[3], pb[3]};
            if (SB) {
              mma16816(d, A0, bj.x, bj.y);
              mma16816(d, A1, bj.z, bj.w);
            } else {
              mma16816(d, A0, fr.hi[SB ? 0 : j][0], fr.hi[SB ? 0 : j][1]);
              mma16816(d, A1, fr.hi[SB ? 0 : j][2], fr.hi[SB ? 0 : j][3]);
            }
            if (MODE == 1 && !PAIR) {
              constexpr bool kLo = MODE == 1 && !PAIR;
              mma16816(d, A0, fr.lo[kLo ? j : 0][0], fr.lo[kLo ? j : 0][1]);
              mma16816(d, A1, fr.lo[kLo ? j : 0][2], fr.lo[kLo ? j : 0][3]);
            }
            float sa, sb;
            {  // bytes j of rows ra and rb as one 16-bit pair
              const uint32_t wa2 = j < 4 ? sra[m].x : sra[m].y, wb2 = j < 4 ? srb[m].x : srb[m].y;
              e8m0x2_to_f32(__byte_perm(wa2, wb2, (uint32_t)(j & 3) | ((uint32_t)((j & 3) + 4) << 4)), sa, sb);
            }
            if (PAIR) {  // columns 2 tq and 2 tq + 1: token tq's hi and lo sums
              acc[m][0] = fmaf(sa, d[0] + d[1], acc[m][0]);
              acc[m][2] = fmaf(sb, d[2] + d[3], acc[m][2]);
            } else {
              acc[m][0] = fmaf(sa, d[0], acc[m][0]);
              acc[m][2] = fmaf(sb, d[2], acc[m][2]);
              if (!ONE) {  // token columns 2 tq + 1 (all zero when the pass holds one token)
                acc[m][1] = fmaf(sa, d[1], acc[m][1]);
                acc[m][3] = fmaf(sb, d[3], acc[m][3]);
              }
            }
          }
        }
      };
      if (nt == 1) blocks(std::true_type{});
      else blocks(std::false_type{});
      if (MODE == 1 && PAIR) {  // undo this warp's rescale for token t (lane groups 2t, 2t + 1 hold it)
        const float u0 = __shfl_sync(0xffffffffu, fr.unscale, (2 * tq) * 4);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          acc[m][0] *= u0;
          acc[m][2] *= u0;
        }
      } else if (MODE == 1) {  // undo this warp's rescale for tokens 2t, 2t+1
        const float u0 = __shfl_sync(0xffffffffu, fr.unscale, (2 * tq) * 4);
        const float u1 = __shfl_sync(0xffffffffu, fr.unscale, (2 * tq + 1) * 4);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          acc[m][0] *= u0;
          acc[m][1] *= u1;
          acc[m][2] *= u0;
          acc[m][3] *= u1;
        }
      }
      const int bi = pc & 1, use = pc >> 1;
      ++pc;
      if (use > 0 && !mbar_wait(&red_empty[bi], (use - 1) & 1, a.err)) return;
      float* rb = red + bi * g.red_floats + (size_t)cw * kRows * kRedTok;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int ra = 16 * m + gq;
        if (SB) {  // the one token: column 0, held by the lanes with tq = 0
          if (tq == 0) {
            rb[ra] = acc[m][0];
            rb[ra + 8] = acc[m][2];
          }
        } else if (PAIR) {  // token tq (columns >= nt are never read)
          rb[ra * kTok + tq] = acc[m][0];
          rb[(ra + 8) * kTok + tq] = acc[m][2];
        } else {
          rb[ra * kTok + 2 * tq] = acc[m][0];
          rb[ra * kTok + 2 * tq + 1] = acc[m][1];
          rb[(ra + 8) * kTok + 2 * tq] = acc[m][2];
          rb[(ra + 8) * kTok + 2 * tq + 1] = acc[m][3];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_full[bi]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }
}

template <int MODE, int BPW, bool PAIR, bool SB>
cudaError_t launch_m(const FfnArgs& a, const GeomM& g, int num_sms, bool pdl, cudaStream_t s, const char* name) {
  if (g.bpw != BPW || g.warps > kMaxBlocks / BPW || g.stages < 2) return cudaErrorInvalidValue;
  ensure_smem(mxfp4_mma_gemv_kernel<MODE, BPW, PAIR, SB>, g.smem);
  return launch(name, mxfp4_mma_gemv_kernel<MODE, BPW, PAIR, SB>, dim3(num_sms), dim3((g.warps + 2) * 32), g.smem, s,
                pdl, a, g);
}

}  // namespace

// bf16 activations (the gate/up B fragments are their exact f16 rescale);
// at most 14 compute warps of 8 blocks (d, ff <= 3584), so that every thread
// of the 16-warp CTA keeps its fragments in 128 registers.
bool mxfp4_mma_gemv_supported(int d, int ff, int x_dtype) {
  return x_dtype == MOE_BF16 && d <= kMaxConsumerWarps * 8 * 32 && ff <= kMaxConsumerWarps * 8 * 32;
}

cudaError_t launch_mxfp4_ffn_mma(const FfnArgs& a, int num_sms, bool pdl, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  if (a.T == 1) {  // one token: fragments in shared memory, 8 blocks per warp
    const GeomM g0 = make_geom_m(0, a.d, a.ff, 8, true), g1 = make_geom_m(1, a.d, a.ff, 8, true);
    cudaError_t err = launch_m<0, 8, false, true>(a, g0, num_sms, pdl, s, "mxfp4_gate_up");
    if (err != cudaSuccess) return err;
    return launch_m<1, 8, true, true>(a, g1, num_sms, true, s, "mxfp4_down");
  }
  const GeomM g0 = make_geom_m(0, a.d, a.ff, 8, false), g1 = make_geom_m(1, a.d, a.ff, 8, false);
  cudaError_t err = launch_m<0, 8, false, false>(a, g0, num_sms, pdl, s, "mxfp4_gate_up");
  if (err != cudaSuccess) return err;
  // an expert gets at most T tokens, so with T <= 4 every pass fits the paired columns
  if (a.T <= 4) return launch_m<1, 8, true, false>(a, g1, num_sms, true, s, "mxfp4_down");
  return launch_m<1, 8, false, false>(a, g1, num_sms, true, s, "mxfp4_down");
}

}  // namespace moe

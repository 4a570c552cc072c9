// mxfp4_gemm.cu -- routed-expert FFN on MXFP4 weights for experts that many
// tokens share (prefill): per expert, the gate/up and down projections become
// grouped GEMMs on the fifth-generation tensor cores (LazyLoRA README,
// "Batching is the lever": a weight matrix read once serves every token routed
// to it; "Running a 2.78-Trillion-Parameter Model Across Two Desks", Act II:
// fp32 accumulation, since a bf16 path failed its tolerance gate).
//
// Work unit (tile): one expert e, 128 rows of one weight matrix, up to 128 of
// e's tokens; an fp32 accumulator of 128 rows x N tokens in TMEM.
//   gate/up launch: tiles over the rows of Wg and of Wu; the epilogue writes
//                   g and u (fp32) for the tokens;
//   act pass:       h = act(g, u) per hot slot, stored as an f16 pair;
//   down launch:    tiles over the rows of Wd; the epilogue writes y_pairs.
// Persistent CTAs (one per SM) walk the tile list round-robin; tiles of one
// (expert, row block) with different token blocks are adjacent, so CTAs that
// run together share the weight bytes in L2.
//
// Operands are f16, exact:
//   * weights: an E2M1 code is an f16 (cvt.e2m1x2); its block scale 2^(B-127)
//     is split into 2^(B-R+13), applied in f16 (HMUL2, exact: the product has
//     at most two significant bits and stays below 6 * 2^13), and 2^(R-140),
//     applied to the fp32 accumulator, with R the row's largest scale byte.  A
//     block more than 2^36 below its row's largest is rounded to f16
//     subnormals or zero: an absolute error below 2^-37 of the row's largest
//     weight (the only inexact case);
//   * activations: x * 2^-s_t with 2^s_t a power of two from max|x_t| (bf16 ->
//     f16 exact down to 2^-29 of the token's largest value); 2^s_t is applied
//     to the accumulator;
//   * h for the down projection: h * 2^-s as an f16 pair hi + lo (22
//     significant bits) with 2^s from the slot's max|h|, both products summed in
//     the same accumulator.
//
// Roles inside a CTA (14 warps):
//   warp 0       producer: TMA loads of the token operand (B), 64 K-columns per
//                stage, in boxes of 16 rows, into a ring of 128-byte-swizzled
//                shared-memory stages;
//   warp 1       allocates TMEM; one lane issues tcgen05.mma (M = 128,
//                N = token count rounded up to 16, K = 16) with A in TMEM,
//                alternating between two accumulators;
//   warps 2..9   dequantisers.  Warp w owns TMEM lanes 32 (w % 4) .. + 31 (one
//                weight row per thread) and one half (64 K-columns) of every
//                128-column A stage.  A thread streams its row's codes and scale
//                bytes with cp.async into a private shared-memory ring (7 stages
//                ahead), decodes its 64 codes per stage into f16 and stores them
//                into one of four TMEM A stages with a single tcgen05.st;
//   warps 10..13 epilogue, overlapped with the next tile's MMAs: TMEM -> fp32
//                outputs with the row and token factors.
// Every wait is bounded; a role that gives up records MOE_ERR_TIMEOUT and
// leaves its loop, the others then run out of their own waits, and the CTA
// drains its copies and MMAs before it frees TMEM.
#include <cudaTypedefs.h>

#include <mutex>
#include <utility>

#include "moe_internal.cuh"
#include "tc_ops.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;      // weight rows per tile = TMEM lanes
constexpr int kBN = 128;      // tokens per tile (accumulator columns)
constexpr int kAK = 128;      // K-columns per A stage
constexpr int kBK = 64;       // K-columns per B stage (one 128-byte f16 row)
constexpr int kBoxRows = 16;  // TMA box height
constexpr int kDeqWarps = 8;
constexpr int kEpiWarps = 4;
constexpr int kThreads = (2 + kDeqWarps + kEpiWarps) * 32;
constexpr int kAStages = 4;
constexpr int kAColBase = 2 * kBN;           // TMEM: two accumulators, then the A stages
constexpr int kAColsPerStage = kAK / 2;      // f16 pairs per lane
constexpr int kRawBytes = kAK / 2 / 2;       // code bytes per dequantiser thread per A stage (half a row-stage)
constexpr int kRawStages = 8;
constexpr uint32_t kBStageBytes = kBN * kBK * 2;  // 16 KB per operand

template <int MODE>
struct Cfg {
  static constexpr int kBOps = MODE == 0 ? 1 : 2;     // token operands per stage (down: hi, lo)
  static constexpr int kBStages = MODE == 0 ? 8 : 4;  // 128 KB of ring either way
  static constexpr size_t kBRing = (size_t)kBStages * kBOps * kBStageBytes;
  static constexpr size_t kRawCodes = (size_t)kRawStages * kDeqWarps * 32 * kRawBytes;
  static constexpr size_t kRawScales = (size_t)kRawStages * kDeqWarps * 32 * 4;
  static constexpr size_t kRowRef = 2 * kBM * sizeof(int);                       // [accumulator][row]
  static constexpr int kNumBars = 2 * kBStages + 2 * kAStages + 8 + 1;
  static constexpr size_t kSmem = 1024 + kBRing + kRawCodes + kRawScales + kRowRef + kNumBars * 8 + 16;
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

struct Tile {
  int e, mat, r0, s0, cnt;
  const uint8_t* rec;
  bool ok;
};

// Tile t of the list: hot experts in order; for each, its row blocks (gate/up:
// those of Wg, then those of Wu); for each row block, its token blocks.
__device__ __forceinline__ void decode_tile(const GemmArgs& a, int t, int RBm, int RBt, Tile& tl) {
  const int n = a.hot[0];
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (RBt * a.hot_blk[mid] <= t) lo = mid;
    else hi = mid;
  }
  const int nb = a.hot_blk[lo + 1] - a.hot_blk[lo];
  const int local = t - RBt * a.hot_blk[lo];
  const int rb = local / nb;
  const int tb = local - rb * nb;
  tl.mat = rb / RBm;
  tl.r0 = (rb - tl.mat * RBm) * kBM;
  tl.e = a.hot[1 + lo];
  const int off = a.offsets[tl.e], N = a.offsets[tl.e + 1] - off;
  tl.s0 = off + tb * kBN;
  tl.cnt = min(kBN, N - tb * kBN);
  tl.rec = a.records[tl.e];
  tl.ok = tl.rec != nullptr && (reinterpret_cast<uintptr_t>(tl.rec) & 15u) == 0;
}

// f16 bits of 2^e in both halves (0 below the subnormal range); e <= 15.
__device__ __forceinline__ uint32_t f16x2_pow2(int e) {
  uint32_t b = 0;
  if (e >= -14) b = (uint32_t)(e + 15) << 10;
  else if (e >= -24) b = 1u << (e + 24);
  return b | (b << 16);
}

// fp32 2^e for -149 <= e <= 127 (0 below).
__device__ __forceinline__ float f32_pow2(int e) {
  if (e >= -126) return __uint_as_float((uint32_t)(e + 127) << 23);
  if (e >= -149) return __uint_as_float(1u << (e + 149));
  return 0.f;
}

// f16x2 multiplier of a block with scale byte B in a row whose largest is R.
__device__ __forceinline__ uint32_t block_mult(uint32_t B, int R) {
  return B == 255u ? 0x7E007E00u : f16x2_pow2((int)B - R + 13);
}

// 32 codes of one block (16 bytes) times the block multiplier -> 16 f16 pairs.
__device__ __forceinline__ void dequant_block(const uint4 q, uint32_t mult, uint32_t* out) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  const __half2 m = *reinterpret_cast<const __half2*>(&mult);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t h[4];
    e2m1x8_to_f16x2(w[i], h);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&h[j]), m);
      out[4 * i + j] = *reinterpret_cast<const uint32_t*>(&v);
    }
  }
}

// A row's scale bytes in flight: up to kMaxDim / 32 bytes as 4-byte words,
// loaded early and reduced to their largest byte later.
struct RowScales {
  uint32_t w[kMaxDim / 32 / 4];
  __device__ __forceinline__ void load(const uint8_t* src, int nwords) {
#pragma unroll
    for (int i = 0; i < kMaxDim / 32 / 4; ++i)
      w[i] = i < nwords ? __ldg(reinterpret_cast<const uint32_t*>(src) + i) : 0u;
  }
  __device__ __forceinline__ int max_byte() const {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < kMaxDim / 32 / 4; ++i) m = __vmaxu4(m, w[i]);
    return (int)max(m & 0xFFu, max((m >> 8) & 0xFFu, max((m >> 16) & 0xFFu, m >> 24)));
  }
};

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    mxfp4_gemm_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap map0,
                      const __grid_constant__ CUtensorMap map1) {
  using C = Cfg<MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* bring = smem;
  uint8_t* raw_codes = bring + C::kBRing;
  uint8_t* raw_scales = raw_codes + C::kRawCodes;
  int* row_ref = reinterpret_cast<int*>(raw_scales + C::kRawScales);
  uint64_t* bars = reinterpret_cast<uint64_t*>(row_ref + 2 * kBM);
  uint64_t* b_full = bars;
  uint64_t* b_empty = b_full + C::kBStages;
  uint64_t* a_full = b_empty + C::kBStages;
  uint64_t* a_empty = a_full + kAStages;
  uint64_t* acc_full = a_empty + kAStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;       // [2]
  uint64_t* ref_full = acc_empty + 2;       // [2] row factors of the accumulator's tile written
  uint64_t* ref_empty = ref_full + 2;       // [2] ... and read
  uint64_t* mma_done = ref_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = MODE == 0 ? a.d : a.ff;
  const int RBm = (MODE == 0 ? a.ff : a.d) / kBM;  // row blocks per matrix
  const int RBt = MODE == 0 ? 2 * RBm : RBm;       // row blocks per expert
  const int KS = K / kAK;                          // A stages per tile

  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kBStages; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(&a_full[i], kDeqWarps);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarps);
      mbar_init(&ref_full[i], kDeqWarps / 2);
      mbar_init(&ref_empty[i], kEpiWarps);
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&map0);
    if (MODE == 1) tc::tma_prefetch_desc(&map1);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_launch_dependents();

  const int total = RBt * a.hot_blk[a.hot[0]];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;
      bool alive = true;
      for (int t = blockIdx.x; t < total && alive; t += gridDim.x) {
        Tile tl;
        decode_tile(a, t, RBm, RBt, tl);
        if (!tl.ok) {
          dev_error(a.err, tl.rec == nullptr ? MOE_ERR_MISSING_EXPERT : MOE_ERR_INVALID_ARG, tl.e);
          continue;
        }
        const int nbox = (tl.cnt + kBoxRows - 1) / kBoxRows;
        for (int j = 0; j < K / kBK; ++j, ++it) {
          const int slot = it % C::kBStages, use = it / C::kBStages;
          if (use > 0 && !mbar_wait(&b_empty[slot], (use - 1) & 1, a.err)) {
            alive = false;
            break;
          }
          mbar_arrive_expect_tx(&b_full[slot], (uint32_t)(nbox * C::kBOps) * (kBoxRows * kBK * 2));
          uint8_t* dst = bring + (size_t)slot * C::kBOps * kBStageBytes;
          for (int i = 0; i < nbox; ++i) {
            tc::tma_load_2d(dst + i * kBoxRows * kBK * 2, &map0, j * kBK, tl.s0 + i * kBoxRows, &b_full[slot]);
            if (MODE == 1)
              tc::tma_load_2d(dst + kBStageBytes + i * kBoxRows * kBK * 2, &map1, j * kBK, tl.s0 + i * kBoxRows,
                              &b_full[slot]);
          }
        }
      }
      // never leave with copies in flight
      for (int j = (it > C::kBStages ? it - C::kBStages : 0); j < it; ++j)
        mbar_wait(&b_full[j % C::kBStages], (j / C::kBStages) & 1, a.err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int bit = 0, ait = 0, tcount = 0;
      bool alive = true;
      for (int t = blockIdx.x; t < total && alive; t += gridDim.x) {
        Tile tl;
        decode_tile(a, t, RBm, RBt, tl);
        if (!tl.ok) continue;
        const int n_mma = (tl.cnt + 15) & ~15;
        const uint32_t idesc = tc::idesc_f16_f32(kBM, n_mma);
        const int ab = tcount & 1;
        if (tcount >= 2 && !mbar_wait(&acc_empty[ab], ((tcount >> 1) - 1) & 1, a.err)) break;
        tc::fence_after();
        const uint32_t d_tmem = tmem + ab * kBN;
        for (int ks = 0; ks < KS && alive; ++ks, ++ait) {
          const int as = ait % kAStages;
          if (!mbar_wait(&a_full[as], (ait / kAStages) & 1, a.err)) {
            alive = false;
            break;
          }
          tc::fence_after();
          const uint32_t a_col = tmem + kAColBase + (uint32_t)as * kAColsPerStage;
          for (int half = 0; half < 2; ++half, ++bit) {
            const int bs = bit % C::kBStages;
            if (!mbar_wait(&b_full[bs], (bit / C::kBStages) & 1, a.err)) {
              alive = false;
              break;
            }
            tc::fence_after();
            const uint8_t* bst = bring + (size_t)bs * C::kBOps * kBStageBytes;
            const uint64_t bd0 = tc::desc_kmajor_sw128(tc::saddr(bst));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t k16 = half * 4 + kk;
              const uint32_t acc = (ks | half | kk) != 0;
              tc::mma_f16_ts(d_tmem, a_col + 8 * k16, bd0 + 2 * kk, idesc, acc);
              if (MODE == 1) {
                const uint64_t bd1 = tc::desc_kmajor_sw128(tc::saddr(bst + kBStageBytes));
                tc::mma_f16_ts(d_tmem, a_col + 8 * k16, bd1 + 2 * kk, idesc, 1u);
              }
            }
            tc::mma_commit(&b_empty[bs]);
          }
          if (!alive) break;
          tc::mma_commit(&a_empty[as]);
        }
        if (!alive) break;
        tc::mma_commit(&acc_full[ab]);
        ++tcount;
      }
      // drain: every MMA issued has completed before TMEM is freed
      tc::mma_commit(mma_done);
      mbar_wait(mma_done, 0, a.err);
    }
  } else if (warp < 2 + kDeqWarps) {
    // ------------------------------------------------------------ dequantisers
    const int dt = threadIdx.x - 64;   // 0..255
    const int q = warp & 3;            // TMEM lane quarter
    const int half = (warp - 2) >> 2;  // K half of each A stage
    const int rr = 32 * q + lane;      // row inside the tile
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const size_t mat_bytes = (size_t)a.ff * a.d / 2 + (size_t)a.ff * a.d / 32;
    const size_t row_codes = (size_t)K / 2, row_scales_n = (size_t)K / 32;
    const size_t mat_rows = MODE == 0 ? (size_t)a.ff : (size_t)a.d;
    uint8_t* my_codes = raw_codes + (size_t)dt * kRawBytes;
    uint8_t* my_scales = raw_scales + (size_t)dt * 4;
    constexpr size_t kCodeStageStride = (size_t)kDeqWarps * 32 * kRawBytes;
    constexpr size_t kScaleStageStride = (size_t)kDeqWarps * 32 * 4;
    const int swz = (dt >> 2) & 1;  // 32-byte rows: conflict-free 16-byte reads across 8 lanes

    // fetch cursor: the flat (tile, stage) sequence of this CTA, kRawStages - 1
    // stages ahead
    int ft = blockIdx.x, fks = 0;
    Tile ftl;
    if (ft < total) decode_tile(a, ft, RBm, RBt, ftl);
    auto issue = [&](int slot) {
      if (ft < total) {
        if (ftl.ok) {
          const size_t mat_off = MODE == 0 ? (size_t)ftl.mat * mat_bytes : 2 * mat_bytes;
          const size_t row = (size_t)(ftl.r0 + rr);
          const uint8_t* src = ftl.rec + mat_off + row * row_codes + (size_t)fks * (kAK / 2) + half * kRawBytes;
          const uint8_t* ssrc = ftl.rec + mat_off + mat_rows * row_codes + row * row_scales_n;
          tc::cp_async16(my_codes + slot * kCodeStageStride + ((0 ^ swz) << 4), src);
          tc::cp_async16(my_codes + slot * kCodeStageStride + ((1 ^ swz) << 4), src + 16);
          tc::cp_async4(my_scales + slot * kScaleStageStride, ssrc + (size_t)fks * 4);
        }
        if (++fks == KS) {
          fks = 0;
          ft += gridDim.x;
          if (ft < total) decode_tile(a, ft, RBm, RBt, ftl);
        }
      }
      tc::cp_async_commit();
    };
#pragma unroll
    for (int i = 0; i < kRawStages - 1; ++i) issue(i);

    // R of each tile: its row's largest scale byte.  The next tile's scale
    // bytes are loaded at this tile's first stage and reduced half a tile later.
    auto row_scale_src = [&](const Tile& x) {
      const size_t mat_off = MODE == 0 ? (size_t)x.mat * mat_bytes : 2 * mat_bytes;
      return x.rec + mat_off + mat_rows * row_codes + (size_t)(x.r0 + rr) * row_scales_n;
    };
    RowScales nsc;
    int R_next = 0;
    if (blockIdx.x < total) {
      Tile first;
      decode_tile(a, blockIdx.x, RBm, RBt, first);
      if (first.ok) {
        nsc.load(row_scale_src(first), (int)(row_scales_n / 4));
        R_next = nsc.max_byte();
      }
    }
    int sit = 0, ait = 0, tcount = 0;
    bool alive = true;
    for (int t = blockIdx.x; t < total && alive; t += gridDim.x) {
      Tile tl;
      decode_tile(a, t, RBm, RBt, tl);
      const int R = R_next;
      const int tn = t + (int)gridDim.x;
      Tile nxt;
      nxt.ok = false;
      if (tn < total) decode_tile(a, tn, RBm, RBt, nxt);
      for (int ks = 0; ks < KS; ++ks, ++sit) {
        issue((sit + kRawStages - 1) % kRawStages);
        tc::cp_async_wait<kRawStages - 1>();
        if (ks == 0 && nxt.ok) nsc.load(row_scale_src(nxt), (int)(row_scales_n / 4));
        if (ks == KS / 2 && nxt.ok) R_next = nsc.max_byte();
        if (!tl.ok) continue;
        if (ks == 0) {
          if (half == 0) {  // publish R for the epilogue
            const int ab = tcount & 1;
            if (tcount >= 2 && !mbar_wait(&ref_empty[ab], ((tcount >> 1) - 1) & 1, a.err)) {
              alive = false;
              break;
            }
            row_ref[ab * kBM + rr] = R;
            __syncwarp();
            if (lane == 0) mbar_arrive(&ref_full[ab]);
          }
        }
        const int rs = sit % kRawStages;
        const uint4 q0 = *reinterpret_cast<const uint4*>(my_codes + rs * kCodeStageStride + ((0 ^ swz) << 4));
        const uint4 q1 = *reinterpret_cast<const uint4*>(my_codes + rs * kCodeStageStride + ((1 ^ swz) << 4));
        const uint32_t sw = *reinterpret_cast<const uint32_t*>(my_scales + rs * kScaleStageStride);
        uint32_t v[32];
        dequant_block(q0, block_mult((sw >> (16 * half)) & 0xFFu, R), v);
        dequant_block(q1, block_mult((sw >> (16 * half + 8)) & 0xFFu, R), v + 16);
        const int as = ait % kAStages;
        if (ait >= kAStages && !mbar_wait(&a_empty[as], ((ait / kAStages) - 1) & 1, a.err)) {
          alive = false;
          break;
        }
        tc::fence_after();
        tc::tmem_st32(tmem + lane_base + kAColBase + (uint32_t)as * kAColsPerStage + half * (kAColsPerStage / 2), v);
        tc::tmem_wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[as]);
        ++ait;
      }
      if (tl.ok) ++tcount;
    }
    tc::cp_async_wait<0>();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int rr = 32 * q + lane;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    int tcount = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      Tile tl;
      decode_tile(a, t, RBm, RBt, tl);
      if (!tl.ok) continue;
      const int ab = tcount & 1, ph = (tcount >> 1) & 1;
      if (!mbar_wait(&acc_full[ab], ph, a.err)) break;
      tc::fence_after();
      if (!mbar_wait(&ref_full[ab], ph, a.err)) break;
      const int R = row_ref[ab * kBM + rr];
      __syncwarp();
      if (lane == 0) mbar_arrive(&ref_empty[ab]);
      const float fr = f32_pow2(R - 140);
      const int row = tl.r0 + rr;
      float* out = MODE == 0 ? (tl.mat == 0 ? a.h : a.u) : a.y_pairs;
      const size_t pitch = MODE == 0 ? (size_t)a.ff : (size_t)a.d;
      const float* tscale = MODE == 0 ? a.xscale : a.hscale;
      for (int c0 = 0; c0 < tl.cnt; c0 += 16) {
        uint32_t v[16];
        tc::tmem_ld16_sync(tmem + lane_base + ab * kBN + c0, v);
        // lane j < 16 fetches token c0 + j's factor and output row
        float f_j = 0.f;
        int p_j = 0;
        if (lane < 16 && c0 + lane < tl.cnt) {
          const int slot = tl.s0 + c0 + lane;
          f_j = tscale[slot];
          p_j = MODE == 0 ? slot : a.pair_ids[slot];
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float f = __shfl_sync(0xffffffffu, f_j, j);
          const int p = __shfl_sync(0xffffffffu, p_j, j);
          if (c0 + j < tl.cnt) out[(size_t)p * pitch + row] = __uint_as_float(v[j]) * fr * f;
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
      ++tcount;
    }
  }

  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

// Slot of the hot list from a hot block index and a row inside it; false past
// the expert's bucket.
__device__ __forceinline__ bool hot_slot(const GemmArgs& a, int blk, int r, int& slot) {
  const int n = a.hot[0];
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a.hot_blk[mid] <= blk) lo = mid;
    else hi = mid;
  }
  const int e = a.hot[1 + lo];
  slot = a.offsets[e] + (blk - a.hot_blk[lo]) * kBN + r;
  return slot < a.offsets[e + 1];
}

// Power of two 2^s with max * 2^-s in [2^14, 2^15) (s = 0 for max 0 or not finite).
__device__ __forceinline__ int f16_shift(float mx) {
  int s = 0;
  if (mx > 0.f && mx < INFINITY) s = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127 - 14;
  return max(-100, min(100, s));
}

// Hot slots' activations in slot order, as f16 after an exact power-of-two
// rescale per token: xs[slot] = x[t] * 2^-s_t, xscale[slot] = 2^s_t.
__global__ void gather_hot_kernel(const GemmArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  const int nblk = a.hot_blk[a.hot[0]];
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int lane = threadIdx.x & 31;
  for (int idx = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); idx < nblk * kBN; idx += warps) {
    int slot;
    if (!hot_slot(a, idx / kBN, idx % kBN, slot)) continue;
    const int tok = a.pair_ids[slot] / a.k;
    const int sh = f16_shift(a.max_x[tok]);
    const float inv = f32_pow2(-sh);
    if (lane == 0) a.xscale[slot] = f32_pow2(sh);
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + (size_t)tok * a.d);
    uint4* dst = reinterpret_cast<uint4*>(a.xs + (size_t)slot * a.d);
    for (int v = lane; v < a.d / 8; v += 32) {
      const uint4 w = src[v];
      const uint32_t in[4] = {w.x, w.y, w.z, w.w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 hv = __floats2half2_rn(__uint_as_float(in[j] << 16) * inv,
                                             __uint_as_float(in[j] & 0xFFFF0000u) * inv);
        o[j] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// Per hot slot: h = act(g, u) from the gate/up epilogue's fp32 rows, written
// in place over g as the f16 pair hi[ff] | lo[ff] of h * 2^-s, 2^s from the
// row's max |h|.  One CTA of 128 threads per slot; the row stays in registers
// across the rewrite.
constexpr int kActThreads = 128;
__global__ void __launch_bounds__(kActThreads) act_f16_pair_kernel(const GemmArgs a) {
  __shared__ float red[kActThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int nblk = a.hot_blk[a.hot[0]];
  constexpr int kPer = kMaxDim / kActThreads;  // values per thread
  for (int idx = blockIdx.x; idx < nblk * kBN; idx += gridDim.x) {
    int slot;
    if (!hot_slot(a, idx / kBN, idx % kBN, slot)) continue;
    float* row = a.h + (size_t)slot * a.ff;
    const float* urow = a.u + (size_t)slot * a.ff;
    float v[kPer];
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int c = threadIdx.x + i * kActThreads;
      v[i] = c < a.ff ? act_fn(row[c], urow[c], a.act) : 0.f;
      m = fmaxf(m, fabsf(v[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();  // every value of the row is now in registers
    m = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    const int sh = f16_shift(m);
    const float inv = f32_pow2(-sh);
    __half* out = reinterpret_cast<__half*>(row);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int c = threadIdx.x + i * kActThreads;
      if (c < a.ff) {
        const float sv = v[i] * inv;
        const __half hi = __float2half_rn(sv);
        out[c] = hi;
        out[a.ff + c] = __float2half_rn(sv - __half2float(hi));
      }
    }
    if (threadIdx.x == 0) a.hscale[slot] = f32_pow2(sh);
    __syncthreads();  // red[] is reused by the next slot
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// f16 matrix [rows][cols] with a row pitch of `pitch` bytes, read in boxes of
// 64 columns x 16 rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t pitch) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBoxRows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool mxfp4_gemm_supported(int d, int ff, int x_dtype) {
  return x_dtype == MOE_BF16 && d % kAK == 0 && ff % kAK == 0 && d % kBM == 0 && ff % kBM == 0;
}

cudaError_t launch_mxfp4_gemm(const GemmArgs& a, int num_sms, bool pdl, cudaStream_t s) {
  const int P = a.T * a.k;
  CUtensorMap mx, mhi, mlo;
  if (!make_map(&mx, a.xs, (uint64_t)a.d, (uint64_t)P, (uint64_t)a.d * 2) ||
      !make_map(&mhi, a.h, (uint64_t)a.ff, (uint64_t)P, (uint64_t)a.ff * 4) ||
      !make_map(&mlo, reinterpret_cast<const char*>(a.h) + (size_t)a.ff * 2, (uint64_t)a.ff, (uint64_t)P,
                (uint64_t)a.ff * 4))
    return cudaErrorInvalidValue;
  cudaError_t err = launch("gemm_gather", gather_hot_kernel, dim3(2 * num_sms), dim3(256), 0, s, pdl, a);
  if (err != cudaSuccess) return err;
  ensure_smem(mxfp4_gemm_kernel<0>, Cfg<0>::kSmem);
  err = launch("mxfp4_gemm_gate_up", mxfp4_gemm_kernel<0>, dim3(num_sms), dim3(kThreads), Cfg<0>::kSmem, s, true, a,
               mx, mx);
  if (err != cudaSuccess) return err;
  err = launch("gemm_act", act_f16_pair_kernel, dim3(8 * num_sms), dim3(kActThreads), 0, s, true, a);
  if (err != cudaSuccess) return err;
  ensure_smem(mxfp4_gemm_kernel<1>, Cfg<1>::kSmem);
  return launch("mxfp4_gemm_down", mxfp4_gemm_kernel<1>, dim3(num_sms), dim3(kThreads), Cfg<1>::kSmem, s, true, a,
                mhi, mlo);
}

}  // namespace moe

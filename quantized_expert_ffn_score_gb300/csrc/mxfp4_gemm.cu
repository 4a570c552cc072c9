// mxfp4_gemm.cu -- routed-expert FFN on MXFP4 weights for experts that many
// tokens share (prefill): per expert, the gate/up and down projections become
// grouped GEMMs on the fifth-generation tensor cores (LazyLoRA README,
// "Batching is the lever": a weight matrix read once serves every token routed
// to it; "Running a 2.78-Trillion-Parameter Model Across Two Desks", Act II:
// fp32 accumulation, since a bf16 path failed its tolerance gate).
//
// Each tile computes D[tokens][weight rows] = A[tokens][K] * W[weight rows][K]^T
// with tcgen05.mma (M = 128 tokens, N = 256 weight rows, K = 16 per
// instruction), both operands in shared memory and an fp32 accumulator of
// 128 lanes x 256 columns in TMEM (two of them, so that the epilogue of one
// tile overlaps the MMAs of the next):
//   gate/up: 128 ff indices per tile, their Wg rows in columns 0..127 and their
//            Wu rows in columns 128..255, so that a token's g and u meet in
//            one TMEM lane; the epilogue writes h = act(g, u) (fp32);
//   act pass: h rewritten per hot slot as an f16 pair (below);
//   down:    256 rows of Wd per tile; the epilogue writes y_pairs.
// A token tile is up to 128 of one expert's tokens; persistent CTAs (one per
// SM) walk the tile list round-robin, tiles of one (expert, row block) with
// different token blocks adjacent so that CTAs running together share weight
// bytes in L2.
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
// Roles inside a CTA (22 warps):
//   warp 0       producer: TMA loads of the token operand, 64 K-columns per
//                stage, in boxes of 16 rows (only the tile's tokens), into a
//                ring of 128-byte-swizzled stages;
//   warp 1       allocates TMEM; one lane issues the MMAs;
//   warps 2..17  dequantisers: they fetch the packed codes and scale bytes of
//                256 K-columns at a time with coalesced cp.async (8 lanes per
//                128-byte row line) into a two-stage ring, then decode one
//                block of 32 codes per thread and 64-column stage (warps 2..9
//                the first half of every row's 64 columns, warps 10..17 the
//                second) into f16, written into a 128-byte-swizzled weight
//                stage (conflict-free 16-byte stores), fenced for the tensor
//                core;
//   warps 18..21 epilogue, one token per thread: TMEM -> registers, row and
//                token factors, outputs with 16-byte stores.
// R per weight row comes from a pre-pass over the hot experts' scale bytes.
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

constexpr int kTM = 128;      // tokens per tile (MMA M, accumulator lanes)
constexpr int kWN = 256;      // weight rows per tile (MMA N, accumulator columns)
constexpr int kBK = 64;       // K-columns per stage (one 128-byte f16 row)
constexpr int kBoxRows = 16;  // TMA box height
constexpr int kDeqWarps = 2 * kWN / 32;  // two threads per weight row
constexpr int kDeqThreads = kDeqWarps * 32;
constexpr int kEpiWarps = kTM / 32;
constexpr int kThreads = (2 + kDeqWarps + kEpiWarps) * 32;
constexpr int kRawK = 256;                                    // K-columns per raw stage
constexpr int kSub = kRawK / kBK;                             // stages per raw stage
constexpr uint32_t kRawCodeStage = kWN * (kRawK / 2);          // 32 KB of packed codes
constexpr uint32_t kRawScaleStage = kWN * (kRawK / 32);        // 8 scale bytes per row
constexpr uint32_t kTokStageBytes = kTM * kBK * 2;  // 16 KB per token operand
constexpr uint32_t kWStageBytes = kWN * kBK * 2;    // 32 KB

template <int MODE>
struct Cfg {
  static constexpr int kTOps = MODE == 0 ? 1 : 2;     // token operands (down: h hi, lo)
  static constexpr int kTStages = 2;                  // token ring
  static constexpr int kWStages = MODE == 0 ? 3 : 2;  // weight ring
  static constexpr int kRawStages = 2;                // packed-code ring
  static constexpr size_t kTRing = (size_t)kTStages * kTOps * kTokStageBytes;
  static constexpr size_t kWRing = (size_t)kWStages * kWStageBytes;
  static constexpr size_t kRawCodes = (size_t)kRawStages * kRawCodeStage;
  static constexpr size_t kRawScales = (size_t)kRawStages * kRawScaleStage;
  static constexpr size_t kRowF = 2 * kWN * sizeof(float);  // row factors per accumulator
  static constexpr int kNumBars = 2 * kTStages + 2 * kWStages + 2 * kRawStages + 8 + 1;
  static constexpr size_t kSmem = 1024 + kTRing + kWRing + kRawCodes + kRawScales + kRowF + kNumBars * 8 + 16;
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

struct Tile {
  int e, hi, wb, s0, cnt;
  const uint8_t* rec;
  bool ok;
};

// Tile t of the list: hot experts in order; for each, its weight-row blocks;
// for each row block, its token blocks.
__device__ __forceinline__ void decode_tile(const GemmArgs& a, int t, int RB, Tile& tl) {
  const int n = a.hot[0];
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (RB * a.hot_blk[mid] <= t) lo = mid;
    else hi = mid;
  }
  const int nb = a.hot_blk[lo + 1] - a.hot_blk[lo];
  const int local = t - RB * a.hot_blk[lo];
  tl.wb = local / nb;
  const int tb = local - tl.wb * nb;
  tl.e = a.hot[1 + lo];
  tl.hi = lo;
  const int off = a.offsets[tl.e], N = a.offsets[tl.e + 1] - off;
  tl.s0 = off + tb * kTM;
  tl.cnt = min(kTM, N - tb * kTM);
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

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    mxfp4_gemm_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap map0,
                      const __grid_constant__ CUtensorMap map1) {
  using C = Cfg<MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tring = smem;
  uint8_t* wring = tring + C::kTRing;
  uint8_t* raw_codes = wring + C::kWRing;
  uint8_t* raw_scales = raw_codes + C::kRawCodes;
  float* rowf = reinterpret_cast<float*>(raw_scales + C::kRawScales);  // [accumulator][weight row]
  uint64_t* bars = reinterpret_cast<uint64_t*>(rowf + 2 * kWN);
  uint64_t* t_full = bars;
  uint64_t* t_empty = t_full + C::kTStages;
  uint64_t* w_full = t_empty + C::kTStages;
  uint64_t* w_empty = w_full + C::kWStages;
  uint64_t* acc_full = w_empty + C::kWStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;          // [2]
  uint64_t* ref_full = acc_empty + 2;          // [2] row factors of the accumulator's tile written
  uint64_t* ref_empty = ref_full + 2;          // [2] ... and read
  uint64_t* mma_done = ref_empty + 2;
  uint64_t* raw_full = mma_done + 1;              // [kRawStages] packed codes landed (cp.async arrivals)
  uint64_t* raw_empty = raw_full + C::kRawStages;  // [kRawStages] ... and read by every dequantiser warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(raw_empty + C::kRawStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = MODE == 0 ? a.d : a.ff;
  const int RB = MODE == 0 ? a.ff / (kWN / 2) : a.d / kWN;  // weight-row blocks per expert
  const int KS = K / kBK;                                    // stages per tile

  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kTStages; ++i) {
      mbar_init(&t_full[i], 1);
      mbar_init(&t_empty[i], 1);
    }
    for (int i = 0; i < C::kWStages; ++i) {
      mbar_init(&w_full[i], kDeqWarps);
      mbar_init(&w_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarps);
      mbar_init(&ref_full[i], kDeqWarps / 2);  // the first-half warps publish
      mbar_init(&ref_empty[i], kEpiWarps);
    }
    mbar_init(mma_done, 1);
    for (int i = 0; i < C::kRawStages; ++i) {
      mbar_init(&raw_full[i], kDeqThreads);
      mbar_init(&raw_empty[i], kDeqWarps);
    }
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

  const int total = RB * a.hot_blk[a.hot[0]];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;
      bool alive = true;
      for (int t = blockIdx.x; t < total && alive; t += gridDim.x) {
        Tile tl;
        decode_tile(a, t, RB, tl);
        if (!tl.ok) {
          dev_error(a.err, tl.rec == nullptr ? MOE_ERR_MISSING_EXPERT : MOE_ERR_INVALID_ARG, tl.e);
          continue;
        }
        const int nbox = (tl.cnt + kBoxRows - 1) / kBoxRows;
        for (int j = 0; j < KS; ++j, ++it) {
          const int slot = it % C::kTStages, use = it / C::kTStages;
          if (use > 0 && !mbar_wait(&t_empty[slot], (use - 1) & 1, a.err)) {
            alive = false;
            break;
          }
          mbar_arrive_expect_tx(&t_full[slot], (uint32_t)(nbox * C::kTOps) * (kBoxRows * kBK * 2));
          uint8_t* dst = tring + (size_t)slot * C::kTOps * kTokStageBytes;
          for (int i = 0; i < nbox; ++i) {
            tc::tma_load_2d(dst + i * kBoxRows * kBK * 2, &map0, j * kBK, tl.s0 + i * kBoxRows, &t_full[slot]);
            if (MODE == 1)
              tc::tma_load_2d(dst + kTokStageBytes + i * kBoxRows * kBK * 2, &map1, j * kBK, tl.s0 + i * kBoxRows,
                              &t_full[slot]);
          }
        }
      }
      // never leave with copies in flight
      for (int j = (it > C::kTStages ? it - C::kTStages : 0); j < it; ++j)
        mbar_wait(&t_full[j % C::kTStages], (j / C::kTStages) & 1, a.err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_f16_f32(kTM, kWN);
      int tit = 0, wit = 0, tcount = 0;
      bool alive = true;
      for (int t = blockIdx.x; t < total && alive; t += gridDim.x) {
        Tile tl;
        decode_tile(a, t, RB, tl);
        if (!tl.ok) continue;
        const int ab = tcount & 1;
        if (tcount >= 2 && !mbar_wait(&acc_empty[ab], ((tcount >> 1) - 1) & 1, a.err)) break;
        tc::fence_after();
        const uint32_t d_tmem = tmem + ab * kWN;
        for (int ks = 0; ks < KS; ++ks, ++tit, ++wit) {
          const int ts = tit % C::kTStages, ws = wit % C::kWStages;
          if (!mbar_wait(&t_full[ts], (tit / C::kTStages) & 1, a.err) ||
              !mbar_wait(&w_full[ws], (wit / C::kWStages) & 1, a.err)) {
            alive = false;
            break;
          }
          tc::fence_after();
          const uint8_t* tst = tring + (size_t)ts * C::kTOps * kTokStageBytes;
          const uint64_t ad0 = tc::desc_kmajor_sw128(tc::saddr(tst));
          const uint64_t wd = tc::desc_kmajor_sw128(tc::saddr(wring + (size_t)ws * kWStageBytes));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t acc = (ks | kk) != 0;
            tc::mma_f16_ss(d_tmem, ad0 + 2 * kk, wd + 2 * kk, idesc, acc);
            if (MODE == 1) {
              const uint64_t ad1 = tc::desc_kmajor_sw128(tc::saddr(tst + kTokStageBytes));
              tc::mma_f16_ss(d_tmem, ad1 + 2 * kk, wd + 2 * kk, idesc, 1u);
            }
          }
          tc::mma_commit(&t_empty[ts]);
          tc::mma_commit(&w_empty[ws]);
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
    // Packed codes move in raw stages of 256 K-columns: 128 bytes per weight
    // row, fetched with 8 lanes per row (coalesced), into a 128-byte-swizzled
    // ring; each stage completes on raw_full through cp.async arrivals.  Every
    // thread then decodes one block of 32 codes per 64-column stage.
    const int dt = threadIdx.x - 64;  // 0..kDeqThreads-1
    const int wrow = dt & (kWN - 1);  // weight row this thread decodes
    const int half = dt / kWN;        // which 32-column block of each 64-column stage
    const size_t mat_bytes = (size_t)a.ff * a.d / 2 + (size_t)a.ff * a.d / 32;
    const size_t row_codes = (size_t)K / 2, row_scales_n = (size_t)K / 32;
    const size_t mat_rows = MODE == 0 ? (size_t)a.ff : (size_t)a.d;
    const int rows_per_block = MODE == 0 ? kWN / 2 : kWN;
    const size_t ref_pitch = 2 * (size_t)a.ff + (size_t)a.d;  // R bytes per hot expert: Wg, Wu, Wd rows
    // gate/up: tile rows 0..127 are Wg rows, 128..255 the Wu rows of the same ff indices
    auto row_base = [&](const Tile& x, int r) {
      const int mat = MODE == 0 ? (r >> 7) : 2;
      const int rin = MODE == 0 ? (r & 127) : r;
      return x.rec + (size_t)mat * mat_bytes + (size_t)(x.wb * rows_per_block + rin) * row_codes;
    };
    auto scale_base = [&](const Tile& x, int r) {
      const int mat = MODE == 0 ? (r >> 7) : 2;
      const int rin = MODE == 0 ? (r & 127) : r;
      return x.rec + (size_t)mat * mat_bytes + mat_rows * row_codes + (size_t)(x.wb * rows_per_block + rin) * row_scales_n;
    };
    const int KR = KS / kSub;  // raw stages per tile

    // fetch cursor over the flat (tile, raw stage) sequence of this CTA
    int ft = blockIdx.x, fk = 0, rn_fetch = 0;
    Tile ftl;
    if (ft < total) decode_tile(a, ft, RB, ftl);
    auto fetch = [&]() {
      if (ft >= total) return;
      const int slot = rn_fetch % C::kRawStages;
      if (ftl.ok) {
        uint8_t* cst = raw_codes + (size_t)slot * kRawCodeStage;
#pragma unroll
        for (int i = 0; i < (int)(kRawCodeStage / 16) / kDeqThreads; ++i) {
          const int g = dt + i * kDeqThreads;  // 16-byte chunk: row g / 8, chunk g % 8
          const int r = g >> 3, j = g & 7;
          tc::cp_async16(cst + (size_t)r * (kRawK / 2) + ((j ^ (r & 7)) << 4),
                         row_base(ftl, r) + (size_t)fk * (kRawK / 2) + j * 16);
        }
        if (dt < kWN)
          tc::cp_async8(raw_scales + (size_t)slot * kRawScaleStage + (size_t)dt * (kRawK / 32),
                        scale_base(ftl, dt) + (size_t)fk * (kRawK / 32));
      }
      tc::cp_async_arrive_noinc(&raw_full[slot]);
      ++rn_fetch;
      if (++fk == KR) {
        fk = 0;
        ft += gridDim.x;
        if (ft < total) decode_tile(a, ft, RB, ftl);
      }
    };
    for (int i = 0; i < C::kRawStages; ++i) fetch();

    int rn = 0, wit = 0, tcount = 0;
    bool alive = true;
    for (int t = blockIdx.x; t < total && alive; t += gridDim.x) {
      Tile tl;
      decode_tile(a, t, RB, tl);
      const int R = tl.ok ? (int)a.row_ref[(size_t)tl.hi * ref_pitch +
                                          (MODE == 0 ? (size_t)(wrow >> 7) * a.ff : 2 * (size_t)a.ff) +
                                          (size_t)(tl.wb * rows_per_block + (MODE == 0 ? (wrow & 127) : wrow))]
                          : 0;
      for (int ks = 0; ks < KS; ++ks) {
        const int sub = ks % kSub;
        const int rslot = rn % C::kRawStages;
        if (sub == 0) {
          if (rn >= 1) {  // the previous raw stage is free once every warp has read it: refill it
            if (!mbar_wait(&raw_empty[(rn - 1) % C::kRawStages], ((rn - 1) / C::kRawStages) & 1, a.err)) {
              alive = false;
              break;
            }
            fetch();
          }
          if (!mbar_wait(&raw_full[rslot], (rn / C::kRawStages) & 1, a.err)) {
            alive = false;
            break;
          }
        }
        if (tl.ok) {
          if (ks == 0 && half == 0) {  // publish the row factor 2^(R-140) for the epilogue
            const int ab = tcount & 1;
            if (tcount >= 2 && !mbar_wait(&ref_empty[ab], ((tcount >> 1) - 1) & 1, a.err)) {
              alive = false;
              break;
            }
            rowf[ab * kWN + wrow] = f32_pow2(R - 140);
            __syncwarp();
            if (lane == 0) mbar_arrive(&ref_full[ab]);
          }
          const int blk = 2 * sub + half;  // 32-column block inside the raw stage
          const uint4 qv = *reinterpret_cast<const uint4*>(raw_codes + (size_t)rslot * kRawCodeStage +
                                                           (size_t)wrow * (kRawK / 2) + ((blk ^ (wrow & 7)) << 4));
          const uint32_t sb = raw_scales[(size_t)rslot * kRawScaleStage + (size_t)wrow * (kRawK / 32) + blk];
          uint32_t v[16];
          dequant_block(qv, block_mult(sb, R), v);
          const int ws = wit % C::kWStages;
          if (wit >= C::kWStages && !mbar_wait(&w_empty[ws], ((wit / C::kWStages) - 1) & 1, a.err)) {
            alive = false;
            break;
          }
          uint8_t* wr = wring + (size_t)ws * kWStageBytes + (size_t)wrow * (kBK * 2);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            *reinterpret_cast<uint4*>(wr + (((4 * half + c) ^ (wrow & 7)) << 4)) =
                make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
          tc::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&w_full[ws]);
          ++wit;
        }
        if (sub == kSub - 1) {  // this warp is done with the raw stage
          __syncwarp();
          if (lane == 0) mbar_arrive(&raw_empty[rslot]);
          ++rn;
        }
      }
      if (tl.ok) ++tcount;
    }
    tc::cp_async_wait<0>();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int tok = 32 * q + lane;  // token inside the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const float* tscale = MODE == 0 ? a.xscale : a.hscale;
    int tcount = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      Tile tl;
      decode_tile(a, t, RB, tl);
      if (!tl.ok) continue;
      const int ab = tcount & 1, ph = (tcount >> 1) & 1;
      if (!mbar_wait(&acc_full[ab], ph, a.err)) break;
      tc::fence_after();
      if (!mbar_wait(&ref_full[ab], ph, a.err)) break;
      const bool valid = tok < tl.cnt;
      const int slot = tl.s0 + tok;
      const float ft = valid ? tscale[slot] : 0.f;
      const float* rf = rowf + ab * kWN;
      const uint32_t acc = tmem + lane_base + ab * kWN;
      if (MODE == 0) {
        float* hrow = a.h + (size_t)slot * a.ff + tl.wb * (kWN / 2);
        for (int c0 = 0; c0 < kWN / 2; c0 += 16) {
          uint32_t g[16], u[16];
          tc::tmem_ld16_sync(acc + c0, g);
          tc::tmem_ld16_sync(acc + kWN / 2 + c0, u);
          float hv[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            hv[j] = act_fast(__uint_as_float(g[j]) * rf[c0 + j] * ft, __uint_as_float(u[j]) * rf[kWN / 2 + c0 + j] * ft,
                             a.act);
          if (valid) {
#pragma unroll
            for (int j = 0; j < 16; j += 4)
              *reinterpret_cast<float4*>(hrow + c0 + j) = make_float4(hv[j], hv[j + 1], hv[j + 2], hv[j + 3]);
          }
        }
      } else {
        const int pair = valid ? a.pair_ids[slot] : 0;
        float* yrow = a.y_pairs + (size_t)pair * a.d + tl.wb * kWN;
        for (int c0 = 0; c0 < kWN; c0 += 16) {
          uint32_t y[16];
          tc::tmem_ld16_sync(acc + c0, y);
          if (valid) {
#pragma unroll
            for (int j = 0; j < 16; j += 4)
              *reinterpret_cast<float4*>(yrow + c0 + j) =
                  make_float4(__uint_as_float(y[j]) * rf[c0 + j] * ft, __uint_as_float(y[j + 1]) * rf[c0 + j + 1] * ft,
                              __uint_as_float(y[j + 2]) * rf[c0 + j + 2] * ft,
                              __uint_as_float(y[j + 3]) * rf[c0 + j + 3] * ft);
          }
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ref_empty[ab]);
        mbar_arrive(&acc_empty[ab]);
      }
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
  slot = a.offsets[e] + (blk - a.hot_blk[lo]) * kTM + r;
  return slot < a.offsets[e + 1];
}

// R per weight row of every hot expert: the row's largest E8M0 scale byte,
// for Wg, Wu and Wd (row_ref[hot][2 ff + d]).  One thread per row.
__global__ void row_ref_kernel(const GemmArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  const int n = a.hot[0];
  const size_t pitch = 2 * (size_t)a.ff + (size_t)a.d;
  const size_t mat_bytes = (size_t)a.ff * a.d / 2 + (size_t)a.ff * a.d / 32;
  const size_t total = (size_t)n * pitch;
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
    const int i = (int)(idx / pitch);
    const size_t r = idx - (size_t)i * pitch;
    const uint8_t* rec = a.records[a.hot[1 + i]];
    if (rec == nullptr || (reinterpret_cast<uintptr_t>(rec) & 15u)) continue;  // reported by the GEMM
    const int m = r < (size_t)a.ff ? 0 : (r < 2 * (size_t)a.ff ? 1 : 2);
    const size_t row = m == 2 ? r - 2 * (size_t)a.ff : r - (size_t)m * a.ff;
    const int K = m == 2 ? a.ff : a.d;
    const size_t rows = m == 2 ? (size_t)a.d : (size_t)a.ff;
    const uint32_t* w = reinterpret_cast<const uint32_t*>(rec + m * mat_bytes + rows * (size_t)K / 2 + row * (size_t)K / 32);
    uint32_t mx = 0;
    for (int j = 0; j < K / 128; ++j) mx = __vmaxu4(mx, __ldg(w + j));
    a.row_ref[idx] = (uint8_t)max(mx & 0xFFu, max((mx >> 8) & 0xFFu, max((mx >> 16) & 0xFFu, mx >> 24)));
  }
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
  for (int idx = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); idx < nblk * kTM; idx += warps) {
    int slot;
    if (!hot_slot(a, idx / kTM, idx % kTM, slot)) continue;
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

// Hot slots' h rows (fp32, from the gate/up epilogue) rewritten in place as
// the f16 pair hi[ff] | lo[ff] of h * 2^-s, 2^s from the row's max |h|.  One
// CTA of 128 threads per slot; the row stays in registers across the rewrite.
constexpr int kConvThreads = 128;
__global__ void __launch_bounds__(kConvThreads) h_to_f16_pair_kernel(const GemmArgs a) {
  __shared__ float red[kConvThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int nblk = a.hot_blk[a.hot[0]];
  constexpr int kPer = kMaxDim / kConvThreads;  // values per thread
  for (int idx = blockIdx.x; idx < nblk * kTM; idx += gridDim.x) {
    int slot;
    if (!hot_slot(a, idx / kTM, idx % kTM, slot)) continue;
    float* row = a.h + (size_t)slot * a.ff;
    float v[kPer];
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int c = threadIdx.x + i * kConvThreads;
      v[i] = c < a.ff ? row[c] : 0.f;
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
      const int c = threadIdx.x + i * kConvThreads;
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
  // K a multiple of the raw stage (256), gate/up row blocks of 128, down row blocks of 256
  return x_dtype == MOE_BF16 && d % kRawK == 0 && ff % kRawK == 0 && d % kWN == 0;
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
  err = launch("gemm_row_ref", row_ref_kernel, dim3(4 * num_sms), dim3(256), 0, s, true, a);
  if (err != cudaSuccess) return err;
  ensure_smem(mxfp4_gemm_kernel<0>, Cfg<0>::kSmem);
  err = launch("mxfp4_gemm_gate_up", mxfp4_gemm_kernel<0>, dim3(num_sms), dim3(kThreads), Cfg<0>::kSmem, s, true, a,
               mx, mx);
  if (err != cudaSuccess) return err;
  err = launch("gemm_h_to_f16", h_to_f16_pair_kernel, dim3(8 * num_sms), dim3(kConvThreads), 0, s, true, a);
  if (err != cudaSuccess) return err;
  ensure_smem(mxfp4_gemm_kernel<1>, Cfg<1>::kSmem);
  return launch("mxfp4_gemm_down", mxfp4_gemm_kernel<1>, dim3(num_sms), dim3(kThreads), Cfg<1>::kSmem, s, true, a,
                mhi, mlo);
}

}  // namespace moe

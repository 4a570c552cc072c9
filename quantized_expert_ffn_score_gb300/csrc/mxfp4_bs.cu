// mxfp4_bs.cu -- routed-expert FFN on MXFP4 weights with the block-scaled
// tensor-core MMA (tcgen05.mma kind::mxf8f6f4): the E2M1 codes and their E8M0
// block scales (OCP Microscaling Formats v1.0: one scale per 32 elements along
// the contraction axis) go to the tensor core as stored, so no core decodes a
// weight (LazyLoRA README, "The engine": a fused MXFP4 decode-and-dot that
// consumes the packed weights, expert sums in fp32).
//
// Operands of one MMA (M = 128 weight rows, K = 32, N = activation columns):
//   A  128 rows of one weight matrix: the record's code bytes, moved by TMA
//      with the 16 x U4 (16-byte aligned) tensor-map type, which places every
//      8 code bytes in a 16-byte slot of shared memory (the operand layout of
//      4-bit types in this MMA kind); scale factors = the record's E8M0 bytes.
//      One pipeline stage holds one or two K chunks of 128 for both matrices
//      of a tile, brought by a single 4-D box (codes, rows, chunk, matrix):
//      a CTA's copy engine completes about one stage per 0.4 us however few
//      bytes it holds, so stages are made as large as shared memory allows.
//   B  activation terms in E4M3 with their own E8M0 block scales: an
//      activation a is written as a sum of E4M3 terms, t_1 = RN(a / 2^s1),
//      t_2 = RN((a - t_1 2^s1) / 2^s2), ..., each with a per-32-block scale
//      that maps the block's largest remaining magnitude into [128, 256).
//      Two terms reproduce a bf16 x exactly (8 significant bits; E4M3 holds 4),
//      three terms carry about 12 significant bits of the fp32 h.  Term i of
//      token n is row (i * nt + n) of B, so one MMA computes every term and the
//      epilogue adds the columns of a token.  The terms and chunks of a stage
//      also come as one 4-D box (K bytes, tokens, term, chunk).
//   D  fp32 in tensor memory.
// Products and their sum are formed by the tensor core in fp32.
//
// Work units: (active expert, 128-row tile, n-tile of up to nt tokens -- 48
// for gate/up, 40 for down -- K part).  gate/up (MODE 0) keeps the gate and
// up rows of the same 128 ff indices in two accumulators, so the epilogue
// applies the activation; down (MODE 1) writes y_pairs.  Whole-K units are
// dealt round robin over the persistent CTAs.  When there are at most half as
// many tiles as CTAs, each tile's K is split in two halves (parts of 512) for
// two CTAs; consecutive parts in one CTA accumulate in tensor memory, and the
// CTA that arrives last finishes the tile (fp32 partial sums added in memory,
// then the activation), which depends on no timing: two partial sums, and
// fp32 addition of two values is commutative.
//
// Warp roles (320 threads): 0 TMA producer (and the per-expert tensor maps),
// 1 MMA issuer and TMEM owner, 2-5 scale-factor writers (one per TMEM lane
// quarter), 6-9 epilogue (one per lane quarter).  Every wait is bounded.
#include <cudaTypedefs.h>

#include <mutex>

#include "bucket_body.cuh"
#include "moe_internal.cuh"
#include "tc_ops.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;           // weight rows per tile (MMA M)
constexpr int kBK = 128;           // K per chunk (one A box plane, four MMAs)
constexpr int kMaxChunks = 2;      // K chunks per pipeline stage
constexpr int kGroupK = 512;       // K per scale-factor group (4 stages)

constexpr int kMaxStages = 12;
constexpr int kMaxSfSlots = 4;
constexpr int kThreads = 320;
constexpr int kSplitMaxPairs = 128;  // K is split only for at most this many pairs
constexpr int kMaxExperts = 4096;
constexpr int kABytes = kBM * kBK;   // one A box in shared memory: 128 rows x 128 codes in 8-bit slots
constexpr int kTxA = kBM * kBK / 2;  // bytes TMA moves for it
constexpr int kBarBytes = 512;
constexpr int kSmemBudget = 227 * 1024;

template <int MODE>
struct Bs {
  static constexpr int kMats = MODE == 0 ? 2 : 1;   // weight matrices per tile
  static constexpr int kTerms = MODE == 0 ? 2 : 3;  // activation terms
  // Tokens per n-tile at most (more tokens per MMA: an MMA's issue time is
  // nearly flat in N up to 128).  terms x tokens rows of B must fit the 128
  // rows whose scale factors one tensor-memory column group holds (down:
  // 3 x 40 = 120), and gate/up's two double-buffered accumulators (2 x 2 x 96
  // columns) leave room for two scale-factor slots.  Measured on the 512-token
  // layers: Zipf gate/up 930 -> 894 us, uniform 2049 -> 2069 us.
  static constexpr int kNt = MODE == 0 ? 48 : 40;
  static constexpr int kSfACols = kMats * 16;       // per slot: 4 stages x 4 column groups per matrix
  static constexpr int kSlotCols = kSfACols + 16;
};

// Pipeline and tensor-memory geometry of one launch (host computed).
struct BsGeom {
  int n_mma;        // MMA N (activation rows: terms x nt, rounded to 16)
  int chunks;       // K chunks of kBK per stage (1, 2 or 4 stages per scale group)
  int b_chunk;      // shared-memory bytes of one chunk's activation rows (terms x nt x kBK)
  int stages;       // shared-memory pipeline stages
  int stage_bytes;  // kMats x chunks A planes + chunks x the B rows (1 KB multiple)
  int dcols;        // TMEM columns of one accumulator buffer (kMats x n_mma)
  int sf_base;      // first scale-factor column (two accumulator buffers before it)
  int sf_slots;
};

struct BsArgs {
  const uint8_t* const* records;
  int d, ff, E, k, T, P;
  int act;
  int nt[2];          // tokens per n-tile of each kernel (multiple of 8, at most Bs<MODE>::kNt)
  const int32_t* offsets;
  const int32_t* pair_ids;
  const int32_t* active;  // active[0] = count, then every expert with tokens
  int* counters;          // [4 * units] split-tile arrival counts (zeroed by the prep kernel)
  float* gsum;            // [P][ff] split accumulators of the gate and up sums (P <= kSplitMaxPairs)
  float* usum;
  uint8_t* xq;   // [2][P][d]   E4M3 terms of x, slot order
  uint8_t* xsf;  // [2][P][d/32]
  uint8_t* hq;   // [3][P][ff]  E4M3 terms of h, slot order
  uint8_t* hsf;  // [3][P][ff/32]
  float* y_pairs;
  CUtensorMap* gmaps;  // [grid][2 matrices][2 buffers] per-CTA tensor maps of the current expert
  int* err;
  BsGeom g[2];  // per MODE
  int max_units;  // per CTA (bound of the unit table in shared memory)
};

__device__ __forceinline__ bool rec_ok32(const uint8_t* rec) {
  return rec != nullptr && ((reinterpret_cast<uintptr_t>(rec) & 31u) == 0);
}

__device__ __forceinline__ uint4 ldg128(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Round-to-nearest-even E4M3 byte of v (|v| < 448) and its exact value.
__device__ __forceinline__ uint32_t to_e4m3(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(r) : "f"(v));
  return r & 0xFFu;
}
__device__ __forceinline__ float from_e4m3(uint32_t b) {
  uint32_t h2;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h2) : "r"(b | (b << 8)));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// Writes the E4M3 terms of one 32-element block held one value per lane:
// q[i * plane + lane] and the scale bytes sf[i * splane] (lane 0).
template <int TERMS>
__device__ __forceinline__ void emit_terms(float v, uint8_t* q, size_t plane, uint8_t* sf, size_t splane, int lane) {
  float r = v;
#pragma unroll
  for (int i = 0; i < TERMS; ++i) {
    const uint32_t mx = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(r)));
    const int e = (int)((mx >> 23) & 0xFFu);
    // scale 2^(sb - 127) maps the block maximum into [128, 256)
    const int sb = mx == 0u ? 127 : max(1, min(254, e - 7));
    const uint32_t c = to_e4m3(r * pow2f(127 - sb));
    r -= from_e4m3(c) * pow2f(sb - 127);
    q[i * plane] = (uint8_t)c;
    if (lane == 0) sf[i * splane] = (uint8_t)sb;
  }
}

// The TERMS E4M3 terms of one 32-element block held by one thread: codes to
// q[i * plane + j] (16-byte stores), scale bytes to sf[i * splane].
template <int TERMS>
__device__ __forceinline__ void block_terms(float (&r)[32], uint8_t* q, size_t plane, uint8_t* sf, size_t splane) {
#pragma unroll
  for (int i = 0; i < TERMS; ++i) {
    uint32_t mx = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) mx = max(mx, __float_as_uint(fabsf(r[j])));
    const int e = (int)((mx >> 23) & 0xFFu);
    const int sb = mx == 0u ? 127 : max(1, min(254, e - 7));
    const float inv = pow2f(127 - sb), scl = pow2f(sb - 127);
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const uint32_t c = to_e4m3(r[j] * inv);
      r[j] -= from_e4m3(c) * scl;
      w[j >> 2] |= c << (8 * (j & 3));
    }
    uint4* dst = reinterpret_cast<uint4*>(q + i * plane);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    sf[i * splane] = (uint8_t)sb;
  }
}

// x terms per slot (bucket order), one 32-element block per thread, and the
// zeroing of the split accumulators.
__global__ void __launch_bounds__(256) bs_prep_x_kernel(const BsArgs a, const void* x) {
  pdl_wait();
  pdl_launch_dependents();
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x, nth = (long long)gridDim.x * blockDim.x;
  const int nb = a.d / 32;
  const long long tasks = (long long)a.P * nb;
  const size_t plane = (size_t)a.P * a.d, splane = (size_t)a.P * nb;
  for (long long t = tid; t < tasks; t += nth) {
    const int slot = (int)(t / nb), b = (int)(t % nb);
    const int tok = a.pair_ids[slot] / a.k;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + (size_t)tok * a.d + 32 * b);
    float r[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = src[q];
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        r[8 * q + 2 * h] = __uint_as_float(u[h] << 16);
        r[8 * q + 2 * h + 1] = __uint_as_float(u[h] & 0xFFFF0000u);
      }
    }
    block_terms<2>(r, a.xq + (size_t)slot * a.d + 32 * b, plane, a.xsf + (size_t)slot * nb + b, splane);
  }
  if (a.P <= kSplitMaxPairs) {  // the split path accumulates into these
    const long long ng = (long long)a.P * a.ff, ny = (long long)a.P * a.d;
    for (long long i = tid; i < ng; i += nth) {
      a.gsum[i] = 0.f;
      a.usum[i] = 0.f;
    }
    for (long long i = tid; i < ny; i += nth) a.y_pairs[i] = 0.f;
    for (long long i = tid; i < 4LL * 8 * 160 * 2; i += nth) a.counters[i] = 0;
  }
}

struct Unit {
  int e, tile, kpart, s0, ntok;
};
// One entry of a CTA's unit table in shared memory (decoded once, in parallel,
// so that no role waits on the dependent global loads of the decoding).
struct UnitRec {
  const uint8_t* rec;
  int e, tile, kpart, s0, ntok, ok;
};

struct Plan {
  int units, kparts, gpk;  // total units, K parts per tile, scale groups per part
  const int* off;          // [n_active + 1] unit offsets (shared memory)
};

__device__ __forceinline__ Unit decode_unit(const BsArgs& a, const Plan& pl, int u, int nt) {
  const int na = a.active[0];
  int lo = 0, hi = na - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pl.off[mid] <= u) lo = mid;
    else hi = mid - 1;
  }
  Unit t;
  t.e = a.active[1 + lo];
  const int s_beg = a.offsets[t.e], ne = a.offsets[t.e + 1] - s_beg;
  const int ntiles = (ne + nt - 1) / nt;
  int local = u - pl.off[lo];
  t.kpart = local % pl.kparts;
  local /= pl.kparts;
  const int ntile = local % ntiles;
  t.tile = local / ntiles;
  t.s0 = s_beg + ntile * nt;
  t.ntok = min(nt, ne - ntile * nt);
  return t;
}

// Position in a CTA's sequence of scale groups (units in order, each unit's
// groups in order), skipping units whose expert record is unusable.
struct Cursor {
  int u, gi;  // u indexes the CTA's unit table
  UnitRec t;
  bool valid;
  __device__ void seek(const UnitRec* tab, int nu) {
    valid = false;
    for (; u < nu; ++u) {
      t = tab[u];
      if (t.ok) {
        valid = true;
        return;
      }
    }
  }
  __device__ void advance(const UnitRec* tab, int nu, int gpk) {
    if (++gi < gpk) return;
    gi = 0;
    ++u;
    seek(tab, nu);
  }
};

// The scale bytes one lane moves into TMEM for one group: its weight row's
// 16 bytes per matrix (the group's 16 blocks = 4 stages x 4 K steps) and the
// 16 bytes of activation rows 32 j + lane, j < 4.
template <int MODE>
struct SfRegs {
  uint4 a[Bs<MODE>::kMats];
  uint4 b[4];
};

template <int MODE>
__device__ __forceinline__ void sf_load(SfRegs<MODE>& r, const BsArgs& a, const UnitRec& t, int grp, int q, int lane,
                                        int nt) {
  using C = Bs<MODE>;
  const int K = MODE == 0 ? a.d : a.ff, rows = MODE == 0 ? a.ff : a.d, nbk = K / 32;
  const size_t mat = (size_t)a.ff * a.d / 2 + (size_t)a.ff * a.d / 32;
  const uint8_t* rec = t.rec;
#pragma unroll
  for (int m = 0; m < C::kMats; ++m) {
    // the matrix's scale bytes [rows][K/32] follow its codes
    const uint8_t* sc = rec + (MODE == 0 ? m * mat : 2 * mat) + (size_t)rows * (K / 2);
    r.a[m] = ldg128(sc + (size_t)(t.tile * kBM + 32 * q + lane) * nbk + 16 * grp);
  }
  const uint8_t* bsf = MODE == 0 ? a.xsf : a.hsf;
  const size_t bplane = (size_t)a.P * nbk;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int n = 32 * j + lane;
    r.b[j] = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
    if (n < C::kTerms * nt) {
      const int p = n / nt, sl = t.s0 + n % nt;
      if (sl < a.P) r.b[j] = ldg128(bsf + p * bplane + (size_t)sl * nbk + 16 * grp);
    }
  }
}

// One token's activation and its three E4M3 terms, kept out of line: ten
// warps in four roles share the SM's instruction caches, and an epilogue
// unrolled over every token of an n-tile evicted the issuing thread's loop
// (measured: gate/up 974 -> 930 us on the 512-token Zipf layer).
__device__ __noinline__ void finish_token(float g, float u, int act, uint8_t* q, size_t plane, uint8_t* sf,
                                          size_t splane, int lane) {
  emit_terms<3>(act_fast(g, u, act), q, plane, sf, splane, lane);
}

// The MMAs of one stage: CH chunks x 4 K steps x the tile's matrices.  sd is
// the shared-memory descriptor of the stage's first byte; descriptors count
// in 16-byte units, so operand offsets are added to it directly (every
// operand address stays below 2^18, so the 14-bit address field never
// carries).  sfc = scale-factor columns of the stage's first chunk.
template <int MODE, int CH>
__device__ __forceinline__ void issue_stage(uint64_t sd, uint32_t b_off16, uint32_t b_step16, uint32_t d0,
                                            uint32_t n_mma, const uint32_t (&id)[4], uint32_t sfc, bool& fresh) {
  using C = Bs<MODE>;
  // the descriptors' address field is in the low half and never carries (see above)
  const uint32_t lo = (uint32_t)sd, hi = (uint32_t)(sd >> 32);
#pragma unroll
  for (int ch = 0; ch < CH; ++ch) {
    const uint32_t blo = lo + b_off16 + (uint32_t)ch * b_step16;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
      for (int m = 0; m < C::kMats; ++m) {
        const uint32_t alo = lo + (uint32_t)((m * CH + ch) * (kABytes >> 4) + 2 * ks);
        tc::mma_bs_lohi(d0 + m * n_mma, alo, blo + 2 * ks, hi, id[ks], sfc + m * 16 + 4 * ch,
                        sfc + C::kSfACols + 4 * ch, fresh ? 0u : 1u);
      }
      fresh = false;
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    mxfp4_bs_kernel(const __grid_constant__ CUtensorMap tmpl, const __grid_constant__ CUtensorMap bmap, const BsArgs a) {
  using C = Bs<MODE>;
  const BsGeom G = a.g[MODE];
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* smaps = smem + (size_t)G.stages * G.stage_bytes;  // the 128-byte weight tensor map being patched
  uint64_t* full = reinterpret_cast<uint64_t*>(smaps + C::kMats * 128);
  uint64_t* empty = full + kMaxStages;
  uint64_t* sf_full = empty + kMaxStages;
  uint64_t* sf_empty = sf_full + kMaxSfSlots;
  uint64_t* acc_full = sf_empty + kMaxSfSlots;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done = acc_empty + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
  int* scan_scratch = reinterpret_cast<int*>(tslot + 2);  // [kThreads / 32]
  int* unit_off = reinterpret_cast<int*>(smaps + C::kMats * 128 + kBarBytes);  // [n_active]
  UnitRec* table = reinterpret_cast<UnitRec*>(
      (reinterpret_cast<uintptr_t>(unit_off + a.E + 1) + 15) & ~uintptr_t(15));  // [max_units]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 1) {
    tc::tmem_alloc(tslot, 512);
    tc::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < G.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int j = 0; j < G.sf_slots; ++j) {
      mbar_init(&sf_full[j], 4);
      mbar_init(&sf_empty[j], 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(&acc_full[j], 1);
      mbar_init(&acc_empty[j], 4);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == 0) {  // a copy of the weight tensor-map template, patched per expert
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&tmpl);
    reinterpret_cast<uint32_t*>(smaps)[lane] = src[lane];
  }
  pdl_wait();
  pdl_launch_dependents();

  // ---- the unit plan (identical in every CTA)
  const int K = MODE == 0 ? a.d : a.ff;
  const int rows = MODE == 0 ? a.ff : a.d;
  const int ntiles_rows = rows / kBM, ngroups = K / kGroupK;
  const int na = a.active[0];
  int total0 = 0;
  Plan pl;
  {
    const int per = (na + kThreads - 1) / kThreads;
    const int i0 = min(na, (int)threadIdx.x * per), i1 = min(na, i0 + per);
    int local = 0;
    for (int i = i0; i < i1; ++i) {
      const int e = a.active[1 + i], ne = a.offsets[e + 1] - a.offsets[e];
      local += ntiles_rows * ((ne + a.nt[MODE] - 1) / a.nt[MODE]);
    }
    int base = bucket_detail::block_exclusive_scan(local, scan_scratch, &total0);
    // at most half as many tiles as CTAs: every tile's K is split in two halves
    // (parts of one scale group) for two CTAs; whole tiles are kept otherwise
    // (one token's 384 gate/up tiles run 53 us whole against 56 us split in
    // parts spread over all CTAs: the imbalance of 2 or 3 tiles per CTA costs
    // less than the split tiles' partial-sum round trips)
    const bool split = 2 * total0 <= (int)gridDim.x && a.P <= kSplitMaxPairs && ngroups > 1;
    pl.kparts = split ? ngroups : 1;
    pl.gpk = ngroups / pl.kparts;
    pl.units = total0 * pl.kparts;
    pl.off = unit_off;
    for (int i = i0; i < i1; ++i) {
      unit_off[i] = base * pl.kparts;
      const int e = a.active[1 + i], ne = a.offsets[e + 1] - a.offsets[e];
      base += ntiles_rows * ((ne + a.nt[MODE] - 1) / a.nt[MODE]);
    }
  }
  __syncthreads();
  // Whole-K units are dealt round robin: at any time the CTAs work on a window
  // of consecutive units, so the n-tiles of one weight tile are streamed by
  // several CTAs together and all but the first read it from L2.  A split tile
  // goes to CTAs 2 t and 2 t + 1, the first half of its parts to the first:
  // exactly two partial sums meet in memory, and fp32 addition of two values
  // (to a zeroed word) does not depend on their order.
  const bool dealt = pl.kparts == 1;
  int ub, nu;
  if (dealt) {
    ub = (int)blockIdx.x;
    nu = pl.units > (int)blockIdx.x ? (pl.units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  } else {
    const int tile = (int)blockIdx.x >> 1, half = (int)blockIdx.x & 1, h = pl.kparts / 2;
    ub = tile * pl.kparts + (half ? h : 0);
    nu = tile < total0 ? (half ? pl.kparts - h : h) : 0;
  }
  if (nu > a.max_units) {  // cannot happen with the host's bound; leave the rest undone, reported
    if (threadIdx.x == 0) dev_error(a.err, MOE_ERR_UNSUPPORTED, nu);
    nu = a.max_units;
  }
  for (int i = threadIdx.x; i < nu; i += kThreads) {
    const Unit t = decode_unit(a, pl, dealt ? ub + i * (int)gridDim.x : ub + i, a.nt[MODE]);
    UnitRec r;
    r.rec = a.records[t.e];
    r.e = t.e;
    r.tile = t.tile;
    r.kpart = t.kpart;
    r.s0 = t.s0;
    r.ntok = t.ntok;
    r.ok = rec_ok32(r.rec) ? 1 : 0;
    table[i] = r;
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tslot;
  const size_t mat = (size_t)a.ff * a.d / 2 + (size_t)a.ff * a.d / 32;
  const int nt = a.nt[MODE];

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int it = 0, cur_e = -1, mbuf = 0, pstage = 0;
    uint32_t pph = 0;  // phase of the current round over the stage ring
    bool ok = true;
    for (int u = 0; u < nu && ok; ++u) {
      const UnitRec t = table[u];
      const uint8_t* rec = t.rec;
      if (!t.ok) {
        if (lane == 0) dev_error(a.err, rec == nullptr ? MOE_ERR_MISSING_EXPERT : MOE_ERR_INVALID_ARG, t.e);
        continue;
      }
      CUtensorMap* gm = a.gmaps + (size_t)blockIdx.x * 4;
      if (t.e != cur_e) {  // this expert's weight tensor map, in the buffer not used by copies in flight
        cur_e = t.e;
        mbuf ^= 1;
        if (lane == 0) tc::tensormap_set_address(smaps, rec + (MODE == 0 ? 0 : 2 * mat));
        __syncwarp();
        tc::tensormap_publish(gm + mbuf, smaps);
        if (lane == 0) tc::tensormap_acquire(gm + mbuf);
        __syncwarp();
      }
      if (lane == 0) {
        // stage cs covers K chunks cs * chunks .. + chunks - 1; a scale group is 4 chunks
        const int spg = 4 / G.chunks;
        const uint32_t tx = (uint32_t)(G.chunks * (C::kMats * kTxA + C::kTerms * nt * kBK));
        const int c_end = (t.kpart + 1) * pl.gpk * spg;
        for (int cs = t.kpart * pl.gpk * spg; cs < c_end; ++cs, ++it) {
          const int stage = pstage;
          if (it >= G.stages && !mbar_wait(&empty[stage], pph ^ 1u, a.err)) {
            ok = false;
            break;
          }
          if (++pstage == G.stages) {
            pstage = 0;
            pph ^= 1u;
          }
          mbar_arrive_expect_tx(&full[stage], tx);
          uint8_t* st = stages + (size_t)stage * G.stage_bytes;
          // A box (codes, rows, chunk, matrix) -> [matrix][chunk][128 rows][128 slots]
          tc::tma_load_4d(st, gm + mbuf, 0, t.tile * kBM, cs * G.chunks, 0, &full[stage]);
          // B box (K bytes, tokens, term, chunk) -> [chunk][term][nt rows][128 bytes]
          tc::tma_load_4d(st + C::kMats * G.chunks * kABytes, &bmap, 0, t.s0, 0, cs * G.chunks, &full[stage]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0)  // never leave with copies in flight
      for (int j = (it > G.stages ? it - G.stages : 0); j < it; ++j)
        mbar_wait_drain(&full[j % G.stages], (j / G.stages) & 1, a.err);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (one thread: ring positions and descriptors advance incrementally, so
    // the issue loop carries no division and little address arithmetic)
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_e2m1_e4m3_bs(kBM, G.n_mma);
      uint32_t id[4];
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) id[ks] = idesc | tc::idesc_sf_ids((uint32_t)ks, (uint32_t)ks);
      const uint64_t sd0 = tc::desc_kmajor_sw128(tc::saddr(stages));
      const uint32_t step16 = (uint32_t)G.stage_bytes >> 4;
      const uint32_t b_off16 = (uint32_t)(C::kMats * G.chunks * kABytes) >> 4, b_step16 = (uint32_t)G.b_chunk >> 4;
      int stage = 0, slot = 0, seg = 0, buf = 0;
      uint32_t ph = 0, sph = 0;
      bool ok = true, fresh = true;
      for (int u = 0; u < nu && ok; ++u) {
        const UnitRec t = table[u];
        if (!t.ok) continue;
        const bool seg_start = u == 0 || t.kpart == 0;
        const bool seg_end = u + 1 == nu || t.kpart == pl.kparts - 1;
        if (seg_start) {
          buf = seg & 1;
          if (seg >= 2 && !mbar_wait(&acc_empty[buf], ((seg >> 1) - 1) & 1, a.err)) break;
          tc::fence_after();
          fresh = true;
        }
        const uint32_t d0 = tmem + (uint32_t)(buf * G.dcols);
        for (int g = 0; g < pl.gpk && ok; ++g) {
          if (!mbar_wait(&sf_full[slot], sph, a.err)) {
            ok = false;
            break;
          }
          tc::fence_after();
          const uint32_t sfa = tmem + (uint32_t)(G.sf_base + slot * C::kSlotCols);
          for (int c = 0; c < 4; c += G.chunks) {  // the group's 4 chunks, G.chunks per stage
            if (!mbar_wait(&full[stage], ph, a.err)) {
              ok = false;
              break;
            }
            tc::fence_after();
            const uint64_t sd = sd0 + (uint32_t)stage * step16;
            if (G.chunks == 2)
              issue_stage<MODE, 2>(sd, b_off16, b_step16, d0, (uint32_t)G.n_mma, id, sfa + 4 * c, fresh);
            else
              issue_stage<MODE, 1>(sd, b_off16, b_step16, d0, (uint32_t)G.n_mma, id, sfa + 4 * c, fresh);
            tc::mma_commit(&empty[stage]);
            if (++stage == G.stages) {
              stage = 0;
              ph ^= 1u;
            }
          }
          if (!ok) break;
          tc::mma_commit(&sf_empty[slot]);
          if (++slot == G.sf_slots) {
            slot = 0;
            sph ^= 1u;
          }
        }
        if (ok && seg_end) {
          tc::mma_commit(&acc_full[buf]);
          ++seg;
        }
      }
      tc::mma_commit(done);  // every MMA issued above has completed before teardown
      mbar_wait_drain(done, 0, a.err);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ scale factors into TMEM
    // Weight rows: lane quarter q reads row 32 q + r of every 128-row tile from
    // lane 32 q + r, column (4 c + q) of the matrix's slot area for stage c of
    // the group.  Activation rows 32 j + r: every quarter reads column (4 c + j)
    // of its own lanes, so each quarter writes all of them.
    const int q = warp & 3;
    const uint32_t lb = (uint32_t)(32 * q) << 16;
    Cursor cur;
    cur.u = 0;
    cur.gi = 0;
    cur.seek(table, nu);
    SfRegs<MODE> r0, r1;
    if (cur.valid) sf_load<MODE>(r0, a, cur.t, cur.t.kpart * pl.gpk + cur.gi, q, lane, nt);
    int sfi = 0, slot = 0;
    uint32_t sph = 0;  // phase of the current round over the scale-factor slots
    while (cur.valid) {
      Cursor nx = cur;
      nx.advance(table, nu, pl.gpk);
      if (nx.valid) sf_load<MODE>(r1, a, nx.t, nx.t.kpart * pl.gpk + nx.gi, q, lane, nt);  // in flight below
      if (sfi >= G.sf_slots && !mbar_wait(&sf_empty[slot], sph ^ 1u, a.err)) break;
      tc::fence_after();
      const uint32_t col = tmem + lb + (uint32_t)(G.sf_base + slot * C::kSlotCols);
#pragma unroll
      for (int m = 0; m < C::kMats; ++m) {
        const uint32_t w[4] = {r0.a[m].x, r0.a[m].y, r0.a[m].z, r0.a[m].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::tmem_st1(col + m * 16 + 4 * c + q, w[c]);
      }
      {
        uint32_t v[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[j] = r0.b[j].x;
          v[4 + j] = r0.b[j].y;
          v[8 + j] = r0.b[j].z;
          v[12 + j] = r0.b[j].w;
        }
        tc::tmem_st16(col + C::kSfACols, v);
      }
      tc::tmem_wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sf_full[slot]);
      ++sfi;
      if (++slot == G.sf_slots) {
        slot = 0;
        sph ^= 1u;
      }
      cur = nx;
      r0 = r1;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const uint32_t lb = (uint32_t)(32 * q) << 16;
    int seg = 0, kp0 = 0;
    for (int u = 0; u < nu; ++u) {
      const UnitRec t = table[u];
      if (!t.ok) continue;
      if (u == 0 || t.kpart == 0) kp0 = t.kpart;
      if (!(u + 1 == nu || t.kpart == pl.kparts - 1)) continue;
      const int buf = seg & 1;
      if (!mbar_wait(&acc_full[buf], (seg >> 1) & 1, a.err)) break;
      tc::fence_after();
      ++seg;
      const bool whole = kp0 == 0 && t.kpart == pl.kparts - 1;
      const int row = t.tile * kBM + 32 * q + lane;
      const uint32_t dcol = tmem + lb + (uint32_t)(buf * G.dcols);
      float s0[C::kNt], s1[MODE == 0 ? C::kNt : 1];  // MODE 0: gate and up sums; MODE 1: y in s0
#pragma unroll
      for (int n0 = 0; n0 < C::kNt; n0 += 8) {
        if (n0 < t.ntok) {  // this chunk's term columns of every matrix, with one wait
          uint32_t v0[8], v1[8], v2[8], v3[8];
          tc::tmem_ld8(dcol + n0, v0);
          tc::tmem_ld8(dcol + nt + n0, v1);
          if (MODE == 0) {
            tc::tmem_ld8(dcol + G.n_mma + n0, v2);
            tc::tmem_ld8(dcol + G.n_mma + nt + n0, v3);
            tc::tmem_wait_ld_bind(v0, v1, v2, v3);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              s0[n0 + i] = __uint_as_float(v0[i]) + __uint_as_float(v1[i]);
              s1[n0 + i] = __uint_as_float(v2[i]) + __uint_as_float(v3[i]);
            }
          } else {
            tc::tmem_ld8(dcol + 2 * nt + n0, v2);
#pragma unroll
            for (int i = 0; i < 8; ++i) v3[i] = 0u;
            tc::tmem_wait_ld_bind(v0, v1, v2, v3);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              s0[n0 + i] = (__uint_as_float(v0[i]) + __uint_as_float(v1[i])) + __uint_as_float(v2[i]);
          }
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);

      if (MODE == 1) {
#pragma unroll
        for (int n = 0; n < C::kNt; ++n) {
          if (n < t.ntok) {
            float* dst = a.y_pairs + (size_t)a.pair_ids[t.s0 + n] * a.d + row;
            if (whole) *dst = s0[n];
            else atomicAdd(dst, s0[n]);
          }
        }
      } else {
        const size_t hplane = (size_t)a.P * a.ff, hsplane = (size_t)a.P * (a.ff / 32);
        bool finish = whole;
        if (!whole) {  // add this part's sums; the last of the tile's parts to arrive finishes it
#pragma unroll
          for (int n = 0; n < C::kNt; ++n) {
            if (n < t.ntok) {
              atomicAdd(a.gsum + (size_t)(t.s0 + n) * a.ff + row, s0[n]);
              atomicAdd(a.usum + (size_t)(t.s0 + n) * a.ff + row, s1[n]);
            }
          }
          __threadfence();
          __syncwarp();
          int last = 0;
          if (lane == 0) {
            const int id = (ub + u - t.kpart) / pl.kparts;
            const int parts = t.kpart - kp0 + 1;
            last = atomicAdd(a.counters + 4 * id + q, parts) + parts == pl.kparts;
          }
          finish = __shfl_sync(0xffffffffu, last, 0) != 0;
          if (finish) {
            __threadfence();
#pragma unroll
            for (int n = 0; n < C::kNt; ++n) {
              if (n < t.ntok) {
                s0[n] = __ldcg(a.gsum + (size_t)(t.s0 + n) * a.ff + row);
                s1[n] = __ldcg(a.usum + (size_t)(t.s0 + n) * a.ff + row);
              }
            }
          }
        }
        if (finish) {
#pragma unroll
          for (int n = 0; n < C::kNt; ++n) {
            if (n < t.ntok) {
              const int slot = t.s0 + n;
              finish_token(s0[n], s1[n], a.act, a.hq + (size_t)slot * a.ff + row, hplane,
                           a.hsf + (size_t)slot * (a.ff / 32) + row / 32, hsplane, lane);
            }
          }
        }
      }
    }
  }

  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

// Stage and tensor-memory geometry for nt tokens per n-tile, E experts and
// `chunks` K chunks per stage.  The B rows of the last chunk are followed by
// room for the n_mma - terms x nt rows the MMA reads past them (ignored
// accumulator columns).
template <int MODE>
bool make_geom(BsGeom* g, int nt, int E, int max_units, int chunks) {
  using C = Bs<MODE>;
  g->n_mma = (C::kTerms * nt + 15) & ~15;
  g->chunks = chunks;
  g->b_chunk = C::kTerms * nt * kBK;
  const int b_bytes = (chunks * g->b_chunk + (g->n_mma - C::kTerms * nt) * kBK + 1023) & ~1023;
  g->stage_bytes = C::kMats * chunks * kABytes + b_bytes;
  const int avail = kSmemBudget - 1024 - C::kMats * 128 - kBarBytes - (E + 1) * (int)sizeof(int) - 16 -
                    max_units * (int)sizeof(UnitRec);
  g->stages = avail / g->stage_bytes < kMaxStages ? avail / g->stage_bytes : kMaxStages;
  g->dcols = C::kMats * g->n_mma;
  g->sf_base = 2 * g->dcols;
  const int slots = (512 - g->sf_base) / C::kSlotCols;
  g->sf_slots = slots < kMaxSfSlots ? slots : kMaxSfSlots;
  return g->stages >= 2 && g->sf_slots >= 2 && chunks >= 1 && chunks <= kMaxChunks && 4 % chunks == 0;
}
template <int MODE>
size_t smem_bytes(const BsGeom& g, int E, int max_units) {
  return 1024 + (size_t)g.stages * g.stage_bytes + Bs<MODE>::kMats * 128 + kBarBytes + ((size_t)E + 1) * sizeof(int) +
         16 + (size_t)max_units * sizeof(UnitRec);
}

// Bound on the units one CTA gets: every active expert has at most
// ceil(ne / nt) <= ne / nt + 1 n-tiles dealt round robin, and a split tile
// gives a CTA at most the larger half of its K parts.
int max_units_per_cta(int rows, int K, int P, int E, int nt, int grid) {
  const long long ntiles = (long long)(P + nt - 1) / nt + (P < E ? P : E);
  const long long u0 = (long long)(rows / kBM) * ntiles;
  const int whole = (int)((u0 + grid - 1) / grid) + 1;
  const int half = P <= kSplitMaxPairs ? (K / kGroupK + 1) / 2 : 0;
  return whole > half ? whole : half;
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

// The weight matrices of a record as a 4-D tensor (codes within a K chunk,
// row, K chunk, matrix): strides K / 2 bytes (row), 64 bytes (chunk of 128
// codes) and `mat_bytes` (matrix); one box = `chunks` chunks of 128 rows of
// `mats` matrices.  The address is replaced per expert on the device.
bool make_weight_map(CUtensorMap* m, const void* any_base, int K, int rows, int mats, size_t mat_bytes, int chunks) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {(cuuint64_t)kBK, (cuuint64_t)rows, (cuuint64_t)(K / kBK), (cuuint64_t)mats};
  cuuint64_t strides[3] = {(cuuint64_t)K / 2, (cuuint64_t)kBK / 2, (cuuint64_t)mat_bytes};
  cuuint32_t box[4] = {kBK, kBM, (cuuint32_t)chunks, (cuuint32_t)mats};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 4, const_cast<void*>(any_base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// The E4M3 activation terms [terms][P][K] as a 4-D tensor (K byte within a
// chunk, slot, term, K chunk); one box = nt slots x all terms x `chunks`
// chunks, landing as [chunk][term][slot][128 bytes].
bool make_term_map(CUtensorMap* m, const void* base, int K, int P, int nt, int terms, int chunks) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {(cuuint64_t)kBK, (cuuint64_t)P, (cuuint64_t)terms, (cuuint64_t)(K / kBK)};
  cuuint64_t strides[3] = {(cuuint64_t)K, (cuuint64_t)P * K, (cuuint64_t)kBK};
  cuuint32_t box[4] = {kBK, (cuuint32_t)nt, (cuuint32_t)terms, (cuuint32_t)chunks};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K chunks per stage: two where two stages of that size fit, else one.
constexpr int kChunksGateUp = 2;
constexpr int kChunksDown = 2;

}  // namespace

bool mxfp4_bs_supported(int d, int ff, int E, int x_dtype) {
  return x_dtype == MOE_BF16 && d % kGroupK == 0 && ff % kGroupK == 0 && E <= kMaxExperts;
}

size_t mxfp4_bs_ws_bytes(int T, int k, int d, int ff, int max_sms) {
  const size_t P = (size_t)T * k, Ps = P <= (size_t)kSplitMaxPairs ? P : 1;
  return 2 * P * (d + d / 32) + 3 * P * (ff + ff / 32) + 2 * Ps * ff * sizeof(float) +
         (size_t)4 * 8 * 160 * 2 * sizeof(int) + (size_t)max_sms * 4 * sizeof(CUtensorMap) + 8 * 256;
}

cudaError_t launch_mxfp4_bs(const BsLaunch& L, int num_sms, bool pdl, cudaStream_t s) {
  if (L.T == 0) return cudaSuccess;
  BsArgs a;
  a.records = L.records;
  a.d = L.d;
  a.ff = L.ff;
  a.E = L.E;
  a.k = L.k;
  a.T = L.T;
  a.P = L.T * L.k;
  a.act = L.act;
  a.nt[0] = L.T >= Bs<0>::kNt ? Bs<0>::kNt : ((L.T + 7) & ~7);
  a.nt[1] = L.T >= Bs<1>::kNt ? Bs<1>::kNt : ((L.T + 7) & ~7);
  a.offsets = L.offsets;
  a.pair_ids = L.pair_ids;
  a.active = L.active;
  // carve the workspace
  uint8_t* p = static_cast<uint8_t*>(L.ws);
  auto take = [&](size_t bytes) {
    uint8_t* r = p;
    p += (bytes + 255) & ~size_t(255);
    return r;
  };
  const size_t P = (size_t)a.P, Ps = P <= (size_t)kSplitMaxPairs ? P : 1;
  a.gmaps = reinterpret_cast<CUtensorMap*>(take((size_t)num_sms * 4 * sizeof(CUtensorMap)));
  a.xq = take(2 * P * a.d);
  a.xsf = take(2 * P * (a.d / 32));
  a.hq = take(3 * P * a.ff);
  a.hsf = take(3 * P * (a.ff / 32));
  a.gsum = reinterpret_cast<float*>(take(Ps * a.ff * sizeof(float)));
  a.usum = reinterpret_cast<float*>(take(Ps * a.ff * sizeof(float)));
  a.counters = reinterpret_cast<int*>(take((size_t)4 * 8 * 160 * 2 * sizeof(int)));
  a.y_pairs = L.y_pairs;
  a.err = L.err;
  if (num_sms > 160) return cudaErrorInvalidValue;  // the split counters are sized for 8 units per SM
  const int mu0 = max_units_per_cta(a.ff, a.d, a.P, a.E, a.nt[0], num_sms);
  const int mu1 = max_units_per_cta(a.d, a.ff, a.P, a.E, a.nt[1], num_sms);
  a.max_units = mu0 > mu1 ? mu0 : mu1;
  if (!make_geom<0>(&a.g[0], a.nt[0], a.E, a.max_units, kChunksGateUp) &&
      !make_geom<0>(&a.g[0], a.nt[0], a.E, a.max_units, 1))
    return cudaErrorInvalidValue;
  if (!make_geom<1>(&a.g[1], a.nt[1], a.E, a.max_units, kChunksDown) &&
      !make_geom<1>(&a.g[1], a.nt[1], a.E, a.max_units, 1))
    return cudaErrorInvalidValue;
  const size_t mat = (size_t)a.ff * a.d / 2 + (size_t)a.ff * a.d / 32;  // bytes of one matrix in a record
  CUtensorMap w0, w1, xm, hm;
  if (!make_weight_map(&w0, a.xq, a.d, a.ff, 2, mat, a.g[0].chunks) ||
      !make_weight_map(&w1, a.xq, a.ff, a.d, 1, mat, a.g[1].chunks) ||
      !make_term_map(&xm, a.xq, a.d, a.P, a.nt[0], 2, a.g[0].chunks) ||
      !make_term_map(&hm, a.hq, a.ff, a.P, a.nt[1], 3, a.g[1].chunks))
    return cudaErrorInvalidValue;
  cudaError_t err = launch("bs_prep_x", bs_prep_x_kernel, dim3(4 * num_sms), dim3(256), 0, s, pdl, a, L.x);
  if (err != cudaSuccess) return err;
  const size_t smem0 = smem_bytes<0>(a.g[0], a.E, a.max_units), smem1 = smem_bytes<1>(a.g[1], a.E, a.max_units);
  ensure_smem(mxfp4_bs_kernel<0>, smem0);
  err = launch("mxfp4_bs_gate_up", mxfp4_bs_kernel<0>, dim3(num_sms), dim3(kThreads), smem0, s, true, w0, xm, a);
  if (err != cudaSuccess) return err;
  ensure_smem(mxfp4_bs_kernel<1>, smem1);
  return launch("mxfp4_bs_down", mxfp4_bs_kernel<1>, dim3(num_sms), dim3(kThreads), smem1, s, true, w1, hm, a);
}

}  // namespace moe

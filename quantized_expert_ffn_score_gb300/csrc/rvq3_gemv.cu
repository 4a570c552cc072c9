// rvq3_gemv.cu -- routed-expert FFN on 3-stage residual-vector-quantised weights
// (WASTE README, "3 bits per expert weight": 3 stages of 256-entry codebooks
// over 8-dim vectors, 3.00 bits per weight; a weight is the sum of its three
// stage codewords).
//
// The weights are never materialised.  For one input vector a (a token's x for
// gate/up, a pair's h for down) and one K-slice of 32 vector positions (256
// columns) the kernel builds, in shared memory,
//   LUT[s][c][v] = <codebook_s[c], a[8v .. 8v+8)>      (fp32, 3 stages x 256 x 32)
// so that a row's partial dot product over the slice is
//   sum_v  LUT[0][code0[v][r]][v] + LUT[1][code1[v][r]][v] + LUT[2][code2[v][r]][v].
// One table serves every matrix applied to the same vector: all of a token's
// experts' gate and up rows (the codebooks are per layer), or a pair's down rows.
//
// Codes are stored position-major (rows contiguous for one position and
// stage).  A producer warp stages the codes of one 512-row group into a
// double-buffered ring of shared memory, a group ahead of the lookups: four TMA
// boxes of [3 stages][32 positions][128 rows] (12 KB each, one instruction
// apiece) with the 128-byte swizzle, so that each (stage, position) run of
// 128 rows is one contiguous DRAM read and the lanes' 8-byte code reads
// (lane l reads line l of a stage) spread over the banks.  The boxes' tensor
// map is the matrix's; its address is patched on the device whenever the
// matrix changes.
//
// Tables are built on the tensor cores (build_table): per stage the product
// of the slice's 32 x 8 elements and the 256 x 8 codebook, one
// mma.sync.m16n8k8 per 16 positions x 8 codes, the elements split into f16
// hi + lo pairs after a power-of-two rescale.
//
// Lookups.  Lane l of a consumer warp owns position l of the slice: the 32
// lanes of a lookup read 32 different banks whatever the codes are.  The
// table sits at a 64 KB-aligned shared address L and keeps stages 0 and 1 in
// the two halves of 256-byte rows -- entry (s, c, l) at L + c * 256 + 128 s +
// 4 l, stage 2 at L + 65,536 + c * 256 + 4 l -- so one byte permute that puts
// code c into byte 1 of the lane's base address (L + 4 l, byte 1 zero) is
// already the entry's shared address.  The code ring's twelve-kilobyte boxes
// fill the space either side of the table.
// Each of the 16 consumer warps takes 32 rows of the staged group and
// reduces its 32 per-lane row values over the lanes with a reduce-scatter.
// Lane l accumulates in register j the row j XOR (a lane-dependent mask):
// the code word it loads, the half of the word and the byte it picks are
// chosen by its own lane bits, so four of the five halving steps swap no
// registers before their shuffle; lane l ends with one row's slice sum.
//
// Work: units are (vector, slice, matrix, 512-row group) in this order; each
// persistent CTA takes one contiguous range of units and rebuilds the table
// when the (vector, slice) changes (about once or twice per CTA at decode
// sizes) while the producer keeps staging codes; the gate/up kernel builds its
// first table before it waits for the routing kernels.  Slice sums go to
// pair-indexed partial buffers; the down kernel finishes h (the slice sums of
// gate and up, then the activation) while it loads its vector, and the
// combine adds the down kernel's slice sums, so no separate reduction pass
// runs.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <utility>

#include "moe_internal.cuh"
#include "tc_ops.cuh"

namespace moe {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kPos = 32;                              // vector positions per slice
constexpr int kGroupRows = 512;                       // rows per staged group
constexpr int kBoxRows = 128;                         // rows per TMA box (one 128-byte swizzle line)
constexpr int kBoxesPerGroup = kGroupRows / kBoxRows;  // 4
constexpr int kRowsPerWarp = kGroupRows / kConsumerWarps;  // 32
constexpr int kBoxBytes = 3 * kPos * kBoxRows;        // 12,288
constexpr int kBufs = 2;
constexpr int kMapSlots = 8;  // per-CTA global tensor maps: a slot is reused after 8 matrix changes
constexpr uint32_t kLutBytes = 131072;  // stages 0 and 1 interleaved (64 KB), stage 2 (64 KB, half used)
constexpr uint32_t kVecBytes = 8 * kPos * sizeof(float);  // 1,024: the vector's slice
constexpr uint32_t kUpOff = kVecBytes;                    // down: the up half's slice sums while h is formed
constexpr uint32_t kMapOff = kUpOff + kVecBytes;          // 128-byte tensor map being patched
constexpr uint32_t kBarOff = kMapOff + 128;
constexpr uint32_t kValidOff = kBarOff + 2 * kBufs * sizeof(uint64_t);  // [kBufs] the staged group has a record
constexpr uint32_t kMiscBytes = kValidOff + kBufs * sizeof(int);
constexpr int kMaxPartsInFlight = 8;  // down: gate/up slice sums loaded at once per element of h
constexpr int kBoxes = kBufs * kBoxesPerGroup;  // 8 boxes of 12 KB, 1024-byte aligned (128-byte swizzle atoms)
constexpr size_t kSmem = 232448;                // all of it: the table, the boxes and the rest are placed at run time
static_assert(kLutBytes + kBoxes * kBoxBytes + kMiscBytes <= kSmem, "shared memory per CTA");  // placement checked at run time
constexpr int kMaxSmsRvq = 160;

// Where the table, the boxes and the small items go in this CTA's shared
// window [s0, s0 + kSmem): the table at the first 64 KB boundary, boxes in
// 1024-byte aligned runs before and after it, the small items in what is left
// of either gap.  Offsets are from the start of the dynamic shared memory.
struct SmemPlan {
  uint32_t lut;
  uint32_t box1, n1, box2;  // boxes n < n1 at box1 + n * kBoxBytes, the rest from box2
  uint32_t misc;
  bool ok;
  __device__ uint32_t box(int n) const {
    return n < (int)n1 ? box1 + n * kBoxBytes : box2 + (n - n1) * kBoxBytes;
  }
};

__device__ SmemPlan plan_smem(uint32_t s0) {
  SmemPlan p;
  const uint32_t end = s0 + (uint32_t)kSmem;
  const uint32_t t = (s0 + 65535u) & ~65535u;
  p.lut = t - s0;
  const uint32_t a1 = (s0 + 1023u) & ~1023u;
  p.n1 = t >= a1 ? min((uint32_t)kBoxes, (t - a1) / kBoxBytes) : 0u;
  p.box1 = a1 - s0;
  p.box2 = t + kLutBytes - s0;
  const uint32_t after1 = a1 + p.n1 * kBoxBytes;          // first byte after the boxes before the table
  const uint32_t after2 = t + kLutBytes + (kBoxes - p.n1) * kBoxBytes;
  bool misc_ok = true;
  if (after1 + kMiscBytes <= t)
    p.misc = after1 - s0;
  else if (after2 + kMiscBytes <= end)
    p.misc = after2 - s0;
  else
    misc_ok = false;
  p.ok = misc_ok && after2 <= end;
  return p;
}

__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float lds_f32_128(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1+128];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds_u64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}

// The codebooks (one or two of 3 x 256 codewords, 16 bytes each) sit in the
// unused upper halves of the table's stage-2 rows: codeword i at table byte
// 65,536 + (i / 8) * 256 + 128 + (i % 8) * 16.
__device__ __forceinline__ uint32_t cb_offset(int i) {
  return 65536u + (uint32_t)(i >> 3) * 256u + 128u + (uint32_t)(i & 7) * 16u;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

struct RGeom {
  int K;         // contraction length of the matrices
  int rows;      // rows of one matrix
  int kv;        // K / 8 vector positions
  int ns;        // slices: ceil(kv / 32)
  int nvec;      // vectors: tokens (gate/up) or pairs (down)
  int kcombo;    // gate/up: 1 when gate and up share a codebook (one table serves both), else 2
  int nseg;      // matrices per (vector, table): gate/up ks * 2 / kcombo, down 1
  int gpm;       // 512-row groups per matrix
  int ks;        // pairs per token
  int ns_gu;     // down: the gate/up kernel's slice count (its partials per row)
  size_t mat_bytes;  // one matrix: 3 * rows * K / 8 (gate and up: ff x d; down: d x ff)
};

RGeom make_geom(int mode, const FfnArgs& a) {
  RGeom g;
  g.K = mode == 0 ? a.d : a.ff;
  g.rows = mode == 0 ? a.ff : a.d;
  g.kv = g.K / 8;
  g.ns = (g.kv + kPos - 1) / kPos;
  g.ks = a.k;
  g.nvec = mode == 0 ? a.T : a.T * a.k;
  g.kcombo = mode == 0 ? (a.cb[0] == a.cb[1] ? 1 : 2) : 1;
  g.nseg = mode == 0 ? a.k * (2 / g.kcombo) : 1;
  g.gpm = (g.rows + kGroupRows - 1) / kGroupRows;
  g.ns_gu = (a.d / 8 + kPos - 1) / kPos;
  g.mat_bytes = (size_t)3 * a.ff * a.d / 8;
  return g;
}

// One unit: its table (vector, kind-of-table, slice) and its rows.
struct Unit {
  long long combo;
  int vi, kc, slice;
  int p, kind;  // pair and matrix (0 gate, 1 up, 2 down)
  int r0, nrows;
};

// Walks the units of a CTA's range in order without divisions (one set of
// divisions at the start).
struct UnitIter {
  long long combo;
  int slice, kc, vi, seg, grp;
  __device__ void init(const RGeom& g, long long u) {
    const long long per_combo = (long long)g.nseg * g.gpm;
    combo = u / per_combo;
    const int rem = (int)(u - combo * per_combo);
    seg = rem / g.gpm;
    grp = rem % g.gpm;
    slice = (int)(combo % g.ns);
    kc = (int)((combo / g.ns) % g.kcombo);
    vi = (int)(combo / ((long long)g.ns * g.kcombo));
  }
  __device__ void next(const RGeom& g) {
    if (++grp < g.gpm) return;
    grp = 0;
    if (++seg < g.nseg) return;
    seg = 0;
    ++combo;
    if (++slice < g.ns) return;
    slice = 0;
    if (++kc < g.kcombo) return;
    kc = 0;
    ++vi;
  }
  template <int MODE>
  __device__ Unit unit(const RGeom& g) const {
    Unit t;
    t.combo = combo;
    t.slice = slice;
    t.kc = kc;
    t.vi = vi;
    if (MODE == 0) {  // one table serves both kinds (segments alternate gate, up) or one kind (kc)
      t.p = vi * g.ks + (g.kcombo == 1 ? seg >> 1 : seg);
      t.kind = g.kcombo == 1 ? seg & 1 : kc;
    } else {
      t.p = vi;
      t.kind = 2;
    }
    t.r0 = grp * kGroupRows;
    t.nrows = min(kGroupRows, g.rows - t.r0);
    return t;
  }
};

// The record of pair p, or null (reported) when it is unusable.
__device__ __forceinline__ const uint8_t* pair_record(const FfnArgs& a, const int32_t* pair_expert, int p,
                                                     bool report) {
  const int e = pair_expert[p];
  const uint8_t* rec = (e >= 0 && e < a.E) ? a.records[e] : nullptr;
  if (rec == nullptr || (reinterpret_cast<uintptr_t>(rec) & 15u)) {
    if (report)
      dev_error(a.err, (e < 0 || e >= a.E) ? MOE_ERR_BAD_EXPERT_INDEX
                                           : (rec == nullptr ? MOE_ERR_MISSING_EXPERT : MOE_ERR_INVALID_ARG), e);
    return nullptr;
  }
  return rec;
}

// Shared address of the entry for the code in byte (sel >> 4 & 3) of w: that
// byte replaces byte 1 of the lane's base address (L + 4 l, whose byte 1 is
// zero) -> L + c * 256 + 4 l.
__device__ __forceinline__ uint32_t lut_addr(uint32_t w, uint32_t base, uint32_t sel) {
  return __byte_perm(w, base, sel);
}

// Sum over the 32 lanes of 32 values whose registers are XOR-permuted by the
// lane bits 4..1 (register j of lane l holds row j ^ mask(l)): four halving
// steps add the partner's upper half straight into the lower half; the last
// (lane bit 0) swaps as usual.  Lane l ends with row mask(l)'s sum in v[0].
__device__ __forceinline__ void reduce_scatter32_xor(float (&v)[32], int lane) {
#pragma unroll
  for (int m = 16; m >= 2; m >>= 1) {
#pragma unroll
    for (int i = 0; i < m; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i + m], m);
  }
  const bool upper = (lane & 1) != 0;
  const float send = upper ? v[0] : v[1];
  const float keep = upper ? v[1] : v[0];
  v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
}

__device__ __forceinline__ void mma1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

// fp32 2^e for -126 <= e <= 127.
__device__ __forceinline__ float pow2_i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// Power-of-two shift s with mx * 2^-s in [2^14, 2^15) (0 for mx 0 or not finite).
__device__ __forceinline__ int f16_shift(float mx) {
  int sh = 0;
  if (mx > 0.f && mx < INFINITY) sh = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127 - 14;
  return max(-100, min(100, sh));
}

// The table of one (vector, slice) on the tensor cores: per stage, LUT = P C^T
// with P [32 positions][8 dims] the slice of the vector and C [256 codes][8]
// the codebook, as mma.sync.m16n8k8 (M = 16 positions, N = 8 codes, K = 8
// dims).  A position's 8 elements are rescaled by a power of two (its largest
// magnitude into [2^14, 2^15)) and split into an f16 pair hi + lo, so every
// product is exact and the two MMAs' fp32 sum carries about 22 significant
// bits of the elements; the codewords are exact f16.  Warp w takes the 8-code
// N tiles w, w + 16, ... (96 per table) for both position halves.  The lane
// holding an entry is not the lane that owns its position in the lookups, so
// the stores pair up lanes: store q writes position half q ^ (t >> 1), which
// puts 16 different positions (banks) into every store instruction.
//   cb_base: shared address of codeword 0 of the table's codebook, holes
//   addressed by cb_offset() relative to it.
__device__ __forceinline__ void build_table(uint8_t* lut, uint32_t cb_base, const float* vec, int warp, int lane) {
  const int g = lane >> 2, t = lane & 3;
  uint32_t ahi[2][2], alo[2][2];  // [position half][row g, row g + 8]
  float unscale[2][2];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int pos = 16 * mt + 8 * h + g;
      const float2 e = *reinterpret_cast<const float2*>(vec + 8 * pos + 2 * t);
      float mx = fmaxf(fabsf(e.x), fabsf(e.y));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));  // the 4 lanes holding the position
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const int sh = f16_shift(mx);
      const float inv = pow2_i(-sh);
      unscale[mt][h] = pow2_i(sh);
      const float x0 = e.x * inv, x1 = e.y * inv;
      const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
      ahi[mt][h] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
      const __half l0 = __float2half_rn(x0 - __half2float(h0)), l1 = __float2half_rn(x1 - __half2float(h1));
      alo[mt][h] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
    }
  const int up = t >> 1;
#pragma unroll 2
  for (int j = warp; j < 3 * 32; j += kConsumerWarps) {
    const int st = j >> 5, c0 = (j & 31) * 8;  // stage and first code of the N tile
    // B: codeword c0 + g, elements 2t, 2t + 1
    const uint32_t bf = lds_u32(cb_base + cb_offset(st * 256 + c0 + g) + 4u * (uint32_t)t);
    float d[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
      for (int i = 0; i < 4; ++i) d[mt][i] = 0.f;
      mma1688(d[mt], ahi[mt][0], ahi[mt][1], bf);
      mma1688(d[mt], alo[mt][0], alo[mt][1], bf);
      d[mt][0] *= unscale[mt][0];
      d[mt][1] *= unscale[mt][0];
      d[mt][2] *= unscale[mt][1];
      d[mt][3] *= unscale[mt][1];
    }
    // entry (stage st, code c, position p) at st < 2 ? c * 256 + 128 st + 4 p : 65536 + c * 256 + 4 p
    uint8_t* row = lut + (st < 2 ? 128 * st : 65536) + (size_t)(c0 + 2 * t) * 256;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int mt = q ^ up;
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const float v = mt ? d[1][2 * h + b] : d[0][2 * h + b];
          *reinterpret_cast<float*>(row + b * 256 + 4 * (16 * mt + 8 * h + g)) = v;
        }
    }
  }
}

// MODE 0: gate/up (vectors = tokens; a table of kind kc, or of both kinds when
// they share a codebook); MODE 1: down (vectors = pairs).
//   gpart[((p * 2 + kind) * ns_gu + slice) * ff + row]
//   dpart[(p * ns + slice) * d + row]
template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    rvq3_kernel(const FfnArgs a, const RGeom g, const int32_t* pair_expert, float* gpart, float* dpart,
                const __grid_constant__ CUtensorMap tmpl, CUtensorMap* gmaps) {
  extern __shared__ __align__(1024) uint8_t rsm[];
  const uint32_t s0 = tc::saddr(rsm);
  const SmemPlan plan = plan_smem(s0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (!plan.ok) {  // the shared window cannot hold the layout: nothing was touched
    if (tid == 0) dev_error(a.err, MOE_ERR_UNSUPPORTED, (int)s0);
    return;
  }
  uint8_t* lut = rsm + plan.lut;                                   // the table (layout above)
  float* vec = reinterpret_cast<float*>(rsm + plan.misc);          // [256] the vector's slice
  uint8_t* smap = rsm + plan.misc + kMapOff;                       // the tensor map being patched
  uint64_t* full = reinterpret_cast<uint64_t*>(rsm + plan.misc + kBarOff);  // [kBufs]
  uint64_t* empty = full + kBufs;                                           // [kBufs]
  volatile int* bvalid = reinterpret_cast<volatile int*>(rsm + plan.misc + kValidOff);  // [kBufs]
  // box i of buffer b: rsm + plan.box(b * kBoxesPerGroup + i), [3][32][128] bytes
  if (tid == 0) {
    for (int b = 0; b < kBufs; ++b) {
      mbar_init(&full[b], 1);
      mbar_init(&empty[b], kConsumerWarps);
    }
    fence_mbar_init();
  }
  if (warp == kConsumerWarps) reinterpret_cast<uint32_t*>(smap)[lane] = reinterpret_cast<const uint32_t*>(&tmpl)[lane];
  __syncthreads();
  // Work that depends on nothing the previous kernel writes runs before the
  // wait on it: the codebooks, the gate/up kernel's first table (the layer
  // input was complete before the routing kernels ran), and the down kernel's
  // whole producer, which stages codes for routing written before the gate/up
  // kernel passed its own wait (into tensor-map slots of its own).  Each role
  // waits where it first needs the previous kernel's output, and releases the
  // dependent launch only after that wait: the down kernel's producer relies
  // on the gate/up kernel's wait having returned before it starts.
  const long long total = (long long)g.nvec * g.kcombo * g.ns * g.nseg * g.gpm;
  const long long ub = total * blockIdx.x / gridDim.x, ue = total * (blockIdx.x + 1) / gridDim.x;
  const int nu = (int)(ue - ub);

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------------- producer
    for (int i = 16 * lane; i < a.E; i += 16 * 32)  // the record table into L2 while the routing is made
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a.records + i));
    if (MODE == 0) pdl_wait();
    pdl_launch_dependents();
    int cur_p = -1, cur_kind = -1, slot = -1;
    const uint8_t* rec = nullptr;
    CUtensorMap* my_maps = gmaps + ((size_t)MODE * kMaxSmsRvq + blockIdx.x) * kMapSlots;  // per kernel and CTA
    int issued = 0;
    UnitIter it;
    it.init(g, ub);
    for (int n = 0; n < nu; ++n, it.next(g)) {
      const Unit t = it.unit<MODE>(g);
      if (t.p != cur_p) {
        rec = pair_record(a, pair_expert, t.p, lane == 0);
        cur_p = t.p;
        cur_kind = -1;
      }
      const int b = n % kBufs;
      int ok = 1;
      if (lane == 0 && n >= kBufs && !mbar_wait(&empty[b], ((n / kBufs) - 1) & 1, a.err)) ok = 0;
      if (__shfl_sync(0xffffffffu, ok, 0) == 0) break;
      if (lane == 0) bvalid[b] = rec != nullptr;  // published by the arrival below
      if (rec == nullptr) {  // nothing to stage: complete the phase without bytes
        if (lane == 0) mbar_arrive(&full[b]);
      } else {
        if (t.kind != cur_kind) {  // the matrix's tensor map, in a slot no copy in flight still uses
          cur_kind = t.kind;
          slot = (slot + 1) % kMapSlots;
          if (lane == 0) tc::tensormap_set_address(smap, rec + (size_t)t.kind * g.mat_bytes);
          __syncwarp();
          tc::tensormap_publish(my_maps + slot, smap);
          if (lane == 0) tc::tensormap_acquire(my_maps + slot);
          __syncwarp();
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[b], (uint32_t)(kBoxesPerGroup * kBoxBytes));
          // boxes at (row r0 + 128 i, position v0, stage 0); rows past the matrix read zeros
#pragma unroll
          for (int i = 0; i < kBoxesPerGroup; ++i)
            tc::tma_load_3d(rsm + plan.box(b * kBoxesPerGroup + i), my_maps + slot, t.r0 + i * kBoxRows,
                            t.slice * kPos, 0, &full[b]);
        }
      }
      issued = n + 1;
    }
    // never leave with copies in flight
    if (lane == 0)
      for (int j = (issued > kBufs ? issued - kBufs : 0); j < issued; ++j)
        mbar_wait_drain(&full[j % kBufs], (j / kBufs) & 1, a.err);
    return;
  }

  // ------------------------------------------------------------------ consumers
  long long lut_combo = -1;
  bool alive = true;  // false after a wait ran out: the remaining units are skipped, barriers still met
  {  // the codebooks this kernel's tables use, into the table's spare bytes (read after the first build's barrier)
    const int ncb = MODE == 0 ? g.kcombo : 1;
    for (int i = tid; i < ncb * 3 * 256; i += kConsumerWarps * 32) {
      const int kc = i / (3 * 256);
      const uint4* src = reinterpret_cast<const uint4*>(MODE == 0 ? a.cb[kc] : a.cb[2]);
      *reinterpret_cast<uint4*>(lut + cb_offset(i)) = __ldg(src + (i - kc * 3 * 256));
    }
  }
  const uint32_t lut_s = s0 + plan.lut;
  const uint32_t base01 = s0 + plan.lut + 4u * (uint32_t)lane;  // stages 0 and 1 (+128)
  const uint32_t base2 = base01 + 65536u;                         // stage 2
  // the lane's register permutation: bit 4 of the row picks the 16-row chunk,
  // bit 3 the 8-byte half of it, bits 1-0 the byte (lane bits 4, 3, 2-1)
  const int l4 = (lane >> 4) & 1, l3 = (lane >> 3) & 1;
  const uint32_t jx = ((uint32_t)lane >> 1) & 3u;
  uint32_t sel[4];
#pragma unroll
  for (int J = 0; J < 4; ++J) sel[J] = 0x7604u | (((uint32_t)J ^ jx) << 4);
  const int r_local = warp * kRowsPerWarp;
  const int c0 = (r_local % kBoxRows) / 16;  // the warp's first 16-row chunk in its box
  static_assert(kBufs == 2, "two buffers");
  const uint32_t box_s0 = s0 + plan.box(r_local / kBoxRows), box_s1 = s0 + plan.box(kBoxesPerGroup + r_local / kBoxRows);
  const int row_of_lane = 16 * l4 + 8 * l3 + 4 * (lane & 1) + (int)jx;
  // byte offsets in a box of the lane's code words for stage 0: line lane (the
  // stage adds 32 lines, 4096 bytes, and leaves line & 7 unchanged), 16-byte
  // chunk (c0 + h ^ l4) swizzled by the line, half hf ^ l3 of it
  uint32_t qo[2][2];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
      qo[h][hf] = (uint32_t)(lane * kBoxRows + (((c0 + (h ^ l4)) ^ (lane & 7)) * 16) + 8 * (hf ^ l3));
  // a new (vector, slice): rebuild the table (uniform over the consumer warps)
  auto rebuild = [&](const Unit& t) {
    const int v0 = t.slice * kPos, nv = min(kPos, g.kv - v0);  // positions past kv: zero vector, zero entries
    named_bar_sync(1, kConsumerWarps * 32);  // the previous table's readers are done
    if (MODE == 0) {
      if (tid < 8 * kPos) vec[tid] = tid < 8 * nv ? load_act(a.x, a.x_dtype, (size_t)t.vi * a.d + 8 * v0 + tid) : 0.f;
    } else {  // h of pair vi: each thread sums one gate or up element's slice sums (ascending), then the activation
      float* up = reinterpret_cast<float*>(rsm + plan.misc + kUpOff);
      const int i = tid & (8 * kPos - 1), kind = tid >> 8;
      float sum = 0.f;
      if (i < 8 * nv) {
        const float* gp = gpart + ((size_t)t.vi * 2 + kind) * g.ns_gu * a.ff + 8 * v0 + i;
        for (int q0 = 0; q0 < g.ns_gu; q0 += kMaxPartsInFlight) {  // loads in flight together, added in order
          float pv[kMaxPartsInFlight];
#pragma unroll
          for (int q = 0; q < kMaxPartsInFlight; ++q)
            if (q0 + q < g.ns_gu) pv[q] = gp[(size_t)(q0 + q) * a.ff];
#pragma unroll
          for (int q = 0; q < kMaxPartsInFlight; ++q)
            if (q0 + q < g.ns_gu) sum += pv[q];
        }
      }
      (kind == 0 ? vec : up)[i] = sum;
      named_bar_sync(1, kConsumerWarps * 32);
      if (tid < 8 * kPos) vec[tid] = tid < 8 * nv ? act_fn(vec[tid], up[tid], a.act) : 0.f;
    }
    named_bar_sync(1, kConsumerWarps * 32);
    // the table's codebook: kind kc's codewords start kc * 768 / 8 holes further
    build_table(lut, lut_s + (uint32_t)(MODE == 0 ? t.kc * 3 * 256 / 8 * 256 : 0), vec, warp, lane);
    named_bar_sync(1, kConsumerWarps * 32);
  };
  UnitIter uit;
  uit.init(g, ub);
  if (MODE == 0 && nu > 0) {  // the first table needs only the layer input
    const Unit t0 = uit.unit<MODE>(g);
    rebuild(t0);
    lut_combo = t0.combo;
  }
  pdl_wait();
  pdl_launch_dependents();
  for (int n = 0; n < nu; ++n, uit.next(g)) {
    const Unit t = uit.unit<MODE>(g);
    if (t.combo != lut_combo) {
      rebuild(t);
      lut_combo = t.combo;
    }
    const int b = n % kBufs;
    if (alive && !mbar_wait(&full[b], (n / kBufs) & 1, a.err)) alive = false;
    const bool mine = alive && bvalid[b] != 0 && r_local < t.nrows;  // no record: the producer reported it
    uint2 q[3][2][2];  // stage s, chunk h, half hf (words 2 hf, 2 hf + 1) of the lane's permuted view
    if (mine) {
      const uint32_t box_s = b ? box_s1 : box_s0;
      // line (stage s, position lane) of the box; its 16-byte chunks are swizzled by the line index
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const uint32_t ad = box_s + qo[h][hf];
#pragma unroll
          for (int st = 0; st < 3; ++st) q[st][h][hf] = lds_u64(ad + (uint32_t)(st * kPos * kBoxRows));
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[b]);  // the codes are in registers: the buffer can be refilled
    if (!mine) continue;
    // register j = 16 h + 8 hf + 2 J + wd holds row 16 (h ^ l4) + 8 (hf ^ l3) + 4 wd + (J ^ jx);
    // positions past the matrix have all-zero table entries, so every lane adds
    float acc[32];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int wd = 0; wd < 2; ++wd) {
          const uint32_t w0 = wd ? q[0][h][hf].y : q[0][h][hf].x;
          const uint32_t w1 = wd ? q[1][h][hf].y : q[1][h][hf].x;
          const uint32_t w2 = wd ? q[2][h][hf].y : q[2][h][hf].x;
#pragma unroll
          for (int J = 0; J < 4; ++J)
            acc[16 * h + 8 * hf + 2 * J + wd] = lds_f32(lut_addr(w0, base01, sel[J])) +
                                                lds_f32_128(lut_addr(w1, base01, sel[J])) +
                                                lds_f32(lut_addr(w2, base2, sel[J]));
        }
    reduce_scatter32_xor(acc, lane);
    const int r = t.r0 + r_local + row_of_lane;
    if (MODE == 0)
      gpart[(((size_t)t.p * 2 + t.kind) * g.ns + t.slice) * a.ff + r] = acc[0];
    else
      dpart[((size_t)t.p * g.ns + t.slice) * a.d + r] = acc[0];
  }
}

// pair_expert[pair_ids[s]] = the expert whose bucket holds slot s (the
// standalone expert call, which gets buckets instead of the routing).
__global__ void pair_expert_kernel(const int32_t* offsets, const int32_t* pair_ids, int E, int32_t* pair_expert) {
  pdl_wait();
  pdl_launch_dependents();
  for (int e = blockIdx.x; e < E; e += gridDim.x)
    for (int s = offsets[e] + threadIdx.x; s < offsets[e + 1]; s += blockDim.x) pair_expert[pair_ids[s]] = e;
}

// y_pairs[p][i] = sum over slices of the down kernel's partial sums (ascending).
__global__ void sum_parts_kernel(const float* dpart, int ns, int d, long long n, float* y_pairs) {
  pdl_wait();
  pdl_launch_dependents();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long p = i / d, r = i % d;
    const float* src = dpart + (size_t)p * ns * d + r;
    float s = 0.f;
    for (int k = 0; k < ns; ++k) s += src[(size_t)k * d];
    y_pairs[i] = s;
  }
}

struct Parts {
  CUtensorMap* maps;
  float* gpart;
  float* dpart;
  int32_t* pair_expert;
};

// The partial area: per-CTA tensor-map slots (64-byte aligned), then the
// gate/up and down partial sums and the pair -> expert list.
constexpr size_t kMapFloats = (size_t)2 * kMaxSmsRvq * kMapSlots * sizeof(CUtensorMap) / sizeof(float);

Parts carve_parts(const FfnArgs& a) {
  const int P = a.T * a.k;
  const int ns_gu = (a.d / 8 + kPos - 1) / kPos, ns_dn = (a.ff / 8 + kPos - 1) / kPos;
  Parts pt;
  pt.maps = reinterpret_cast<CUtensorMap*>(a.partial);
  pt.gpart = a.partial + kMapFloats;
  pt.dpart = pt.gpart + (size_t)P * 2 * ns_gu * a.ff;
  pt.pair_expert = reinterpret_cast<int32_t*>(pt.dpart + (size_t)P * ns_dn * a.d);
  return pt;
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

// One matrix's codes as a 3-D byte tensor (row, position, stage): strides
// `rows` bytes (position) and kv * rows bytes (stage); one box = 128 rows x 32
// positions x 3 stages with the 128-byte swizzle.  The address is replaced
// per matrix on the device.
bool make_code_map(CUtensorMap* m, const void* any_base, const RGeom& g) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)g.rows, (cuuint64_t)g.kv, 3};
  cuuint64_t strides[2] = {(cuuint64_t)g.rows, (cuuint64_t)g.kv * g.rows};
  cuuint32_t box[3] = {kBoxRows, kPos, 3};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(any_base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t rvq3_partial_floats(int T, int k, int d, int ff) {
  const size_t P = (size_t)T * k;
  const size_t ns_gu = (d / 8 + kPos - 1) / kPos, ns_dn = (ff / 8 + kPos - 1) / kPos;
  return kMapFloats + P * (2 * ns_gu * ff + ns_dn * d + 1);  // tensor maps, partials, pair -> expert
}

int rvq3_down_parts(int d, int ff) {
  (void)d;
  return (ff / 8 + kPos - 1) / kPos;
}

float* rvq3_down_partials(const FfnArgs& a) { return carve_parts(a).dpart; }

cudaError_t launch_rvq3_ffn(const FfnArgs& a, const int32_t* pair_expert, bool y_out, int num_sms, bool pdl,
                            cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  const Parts pt = carve_parts(a);
  cudaError_t err;
  if (pair_expert == nullptr) {  // from the buckets
    err = launch("rvq3_pair_expert", pair_expert_kernel, dim3(num_sms), dim3(128), 0, s, pdl, a.offsets, a.pair_ids,
                 a.E, pt.pair_expert);
    if (err != cudaSuccess) return err;
    pair_expert = pt.pair_expert;
    pdl = true;
  }
  if (num_sms > kMaxSmsRvq) return cudaErrorInvalidValue;  // the map slots are sized for this many CTAs
  const RGeom g0 = make_geom(0, a), g1 = make_geom(1, a);
  CUtensorMap m0, m1;
  if (!make_code_map(&m0, pt.gpart, g0) || !make_code_map(&m1, pt.gpart, g1)) return cudaErrorInvalidValue;
  ensure_smem(rvq3_kernel<0>, kSmem);
  ensure_smem(rvq3_kernel<1>, kSmem);
  err = launch("rvq3_gate_up", rvq3_kernel<0>, dim3(num_sms), dim3(kThreads), kSmem, s, pdl, a, g0, pair_expert,
               pt.gpart, pt.dpart, m0, pt.maps);
  if (err != cudaSuccess) return err;
  err = launch("rvq3_down", rvq3_kernel<1>, dim3(num_sms), dim3(kThreads), kSmem, s, true, a, g1, pair_expert,
               pt.gpart, pt.dpart, m1, pt.maps);
  if (err != cudaSuccess || !y_out) return err;
  const long long n = (long long)a.T * a.k * a.d;
  return launch("rvq3_sum_parts", sum_parts_kernel, dim3(2 * num_sms), dim3(256), 0, s, true, pt.dpart, g1.ns, a.d, n,
                a.y_pairs);
}

}  // namespace moe

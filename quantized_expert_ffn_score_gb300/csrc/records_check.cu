// records_check.cu -- CRC-32 of expert records on the GPU, and the check of
// each record against an expected value (WASTE README, "How it works": every
// expert record carries a CRC32 of its payload, verified on request, so a
// truncated or spliced bank names the bad record instead of answering from
// wrong bytes).
//
// The checksum is the IEEE 802.3 / zlib CRC-32: reflected generator 0xEDB88320,
// register starting at all ones, result complemented.  It is linear over
// GF(2), which is what lets thousands of threads share one record:
//   * with the register starting at zero (the "raw" CRC R), leading zero bytes
//     change nothing, and R(A || B) = R(A) * x^(8|B|) xor R(B), the product
//     taken in GF(2)[x] modulo the generator;
//   * the standard value is CRC(M) = R(M) xor (0xFFFFFFFF * x^(8|M|)) xor 0xFFFFFFFF.
// A record of B bytes is read as if preceded by zeros up to a whole number of
// 4 KiB units.  Every warp takes one unit at a time, independently of the
// other warps: it reads the unit with coalesced 16-byte loads (each load
// instruction covers 512 contiguous bytes) into its own 4 KiB of shared
// memory, XOR-swizzled by 16-byte slot so that both the stores and the
// per-lane reads below are free of bank conflicts, while the loads of its next
// unit are in flight; each lane then folds its 128 contiguous bytes through byte tables
// (four bytes per step, the four tables giving a byte's effect after 4, 3, 2
// and 1 more bytes), multiplies the result by x to the number of bits that
// follow it in the unit, and the warp xors the lanes into the unit's raw CRC.
// A second kernel joins a record's units (one warp per record: each lane a
// contiguous run of units by Horner's rule, then shifted past the units after
// it) and completes the standard value.  The byte tables are stored once per
// lane (entry i of lane l at word 32 i + l), so every lane reads its own bank
// and the lookups never conflict; the products by the lane's fixed power of x
// are eight lookups of per-lane nibble tables.  In the reflected bit order
// used throughout, bit 31 - k of a 32-bit word is the coefficient of x^k.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr uint32_t kCrcPoly = 0xEDB88320u;
constexpr int kCrcWarps = 16;
constexpr int kCrcThreads = kCrcWarps * 32;
constexpr int kCrcLaneBytes = 128;             // contiguous bytes per lane and unit
constexpr int kCrcUnit = 32 * kCrcLaneBytes;   // 4 KiB per warp unit
// shared memory: byte tables [4][256][32] (128 KiB), the per-lane nibble
// tables of the lane's power of x [8][16][32] (16 KiB), then one unit per warp
// (64 KiB)
constexpr int kByteTabWords = 4 * 256 * 32;
constexpr int kNibTabWords = 8 * 16 * 32;
constexpr int kStageWords = kCrcWarps * kCrcUnit / 4;
constexpr size_t kCrcSmemBytes = (size_t)(kByteTabWords + kNibTabWords + kStageWords) * sizeof(uint32_t);

// Shared-memory slot of a unit's 16-byte piece k (0..255): the low three bits
// are xored with bits 3..5, so that 8 consecutive lanes touch 8 distinct
// 16-byte bank groups both when lane l stores pieces l + 32 j and when it
// reads pieces 8 l + i.
__device__ __forceinline__ int crc_slot(int k) { return k ^ ((k >> 3) & 7); }

// a * b modulo the generator: sum over the coefficients a_k of x^k * b.
__host__ __device__ inline uint32_t gf2_mulmod(uint32_t a, uint32_t b) {
  uint32_t p = 0;
  for (int k = 0; k < 32; ++k) {
    p ^= b & (0u - ((a >> (31 - k)) & 1u));
    b = (b >> 1) ^ (kCrcPoly & (0u - (b & 1u)));  // b * x
  }
  return p;
}

// x^(8 n) modulo the generator, by squaring.
__host__ __device__ inline uint32_t gf2_xpow8(unsigned long long n) {
  uint32_t r = 0x80000000u;     // x^0
  uint32_t base = 0x00800000u;  // x^8
  while (n) {
    if (n & 1ull) r = gf2_mulmod(r, base);
    base = gf2_mulmod(base, base);
    n >>= 1;
  }
  return r;
}

struct CrcArgs {
  const uint8_t* const* records;
  int n;
  long long bytes;  // B, a multiple of 16
  int units;        // ceil(B / kCrcUnit)
  long long pad;    // units * kCrcUnit - B virtual leading zero bytes
  uint32_t* unit_crc;        // [n][units] workspace
  const uint32_t* expected;  // [n] or null
  uint32_t* crc_out;         // [n] or null
  int* err;
  uint32_t lane_mul[32];     // x^(8 (bytes after lane l's piece in a unit))
  uint32_t unit_mul;         // x^(8 kCrcUnit)
  uint32_t init_term;        // 0xFFFFFFFF * x^(8 B): the all-ones start carried over B bytes
};

__device__ __forceinline__ bool record_usable(const uint8_t* p) {
  return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// Raw CRC of every (record, unit) work item; each warp strides over the items.
__global__ void __launch_bounds__(kCrcThreads, 1) crc_units_kernel(const CrcArgs a) {
  extern __shared__ uint32_t tab[];
  __shared__ uint32_t t[4][256];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // t[0][i]: byte i shifted through the register (one byte); t[j][i]: the same
  // followed by j zero bytes
  if (tid < 256) {
    uint32_t c = (uint32_t)tid;
    for (int b = 0; b < 8; ++b) c = (c >> 1) ^ (kCrcPoly & (0u - (c & 1u)));
    t[0][tid] = c;
  }
  __syncthreads();
  for (int j = 1; j < 4; ++j) {
    if (tid < 256) t[j][tid] = (t[j - 1][tid] >> 8) ^ t[0][t[j - 1][tid] & 0xFFu];
    __syncthreads();
  }
  for (int i = tid; i < kByteTabWords; i += kCrcThreads) tab[i] = t[i >> 13][(i >> 5) & 255];
  uint32_t* nib = tab + kByteTabWords;  // entry (j, v) of lane l: (v at nibble j) * lane_mul[l]
  for (int i = tid; i < kNibTabWords; i += kCrcThreads) {
    const int l = i & 31, v = (i >> 5) & 15, j = i >> 9;
    nib[i] = gf2_mulmod((uint32_t)v << (28 - 4 * j), a.lane_mul[l]);
  }
  __syncthreads();
  const uint32_t* T0 = tab + lane;              // one more byte
  const uint32_t* T1 = tab + 1 * 8192 + lane;   // two
  const uint32_t* T2 = tab + 2 * 8192 + lane;   // three
  const uint32_t* T3 = tab + 3 * 8192 + lane;   // four
  const uint32_t* N = nib + lane;
  // n * units < 2^31 (checked by the launcher): 32-bit work indices
  const unsigned total = (unsigned)a.n * (unsigned)a.units;
  const unsigned nwarps = gridDim.x * kCrcWarps;
  uint4* stage = reinterpret_cast<uint4*>(nib + kNibTabWords) + warp * (kCrcUnit / 16);
  // the coalesced loads of unit w: lane l's pieces l + 32 j (zeros where the
  // piece lies in the virtual leading zeros; nothing for an unusable record)
  auto fetch = [&](unsigned w, uint4 (&g)[8]) {
    const unsigned rec = w / (unsigned)a.units;
    const long long unit = (long long)(w - rec * (unsigned)a.units);
    const uint8_t* base = a.records[rec];
    const bool usable = record_usable(base);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const long long o = unit * kCrcUnit + 16 * (lane + 32 * j) - a.pad;  // pieces lie wholly in the padding or the record
      g[j] = usable && o >= 0 ? __ldg(reinterpret_cast<const uint4*>(base + o)) : make_uint4(0u, 0u, 0u, 0u);
    }
    return usable;
  };
  uint4 g[8];
  unsigned w = blockIdx.x * kCrcWarps + warp;
  bool usable = w < total && fetch(w, g);
  for (; w < total; w += nwarps) {
    __syncwarp();  // the previous unit's reads are done
#pragma unroll
    for (int j = 0; j < 8; ++j) stage[crc_slot(lane + 32 * j)] = g[j];
    __syncwarp();
    uint4 q[kCrcLaneBytes / 16];
#pragma unroll
    for (int i = 0; i < kCrcLaneBytes / 16; ++i) q[i] = stage[crc_slot(8 * lane + i)];
    const bool cur_usable = usable;
    if (w + nwarps < total) usable = fetch(w + nwarps, g);  // in flight during the folding below
    uint32_t part = 0;
    if (cur_usable) {
      uint32_t reg = 0;
#pragma unroll
      for (int j = 0; j < kCrcLaneBytes / 16; ++j) {
        const uint32_t wv[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          reg ^= wv[m];  // the word's first byte in memory is its low byte
          reg = T3[(reg & 0xFFu) << 5] ^ T2[((reg >> 8) & 0xFFu) << 5] ^ T1[((reg >> 16) & 0xFFu) << 5] ^
                T0[(reg >> 24) << 5];
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) part ^= N[((j << 4) | ((reg >> (28 - 4 * j)) & 15u)) << 5];
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) part ^= __shfl_xor_sync(0xffffffffu, part, s);
    }
    if (lane == 0) a.unit_crc[w] = part;
  }
}

// One warp per record: lane l joins units [l U / 32, (l + 1) U / 32) by
// Horner's rule and shifts the result past the units after them; the lanes'
// xor is the record's raw CRC, completed to the standard value.
__global__ void crc_finish_kernel(const CrcArgs a) {
  const int e = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (e >= a.n) return;
  const uint8_t* base = a.records[e];
  if (!record_usable(base)) {
    if (lane == 0) {
      dev_error(a.err, base == nullptr ? MOE_ERR_MISSING_EXPERT : MOE_ERR_BAD_RECORD, e);
      if (a.crc_out) a.crc_out[e] = 0u;
    }
    return;
  }
  const long long U = a.units;
  const long long u0 = U * lane / 32, u1 = U * (lane + 1) / 32;
  uint32_t r = 0;
  for (long long u = u0; u < u1; ++u) r = gf2_mulmod(r, a.unit_mul) ^ a.unit_crc[(size_t)e * U + u];
  r = gf2_mulmod(r, gf2_xpow8((unsigned long long)(U - u1) * kCrcUnit));
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) r ^= __shfl_xor_sync(0xffffffffu, r, s);
  r ^= a.init_term ^ 0xFFFFFFFFu;
  if (lane == 0) {
    if (a.crc_out) a.crc_out[e] = r;
    if (a.expected && a.expected[e] != r) dev_error(a.err, MOE_ERR_BAD_RECORD, e);
  }
}

}  // namespace

int records_crc_units(size_t record_bytes) { return (int)((record_bytes + kCrcUnit - 1) / kCrcUnit); }

cudaError_t launch_records_check(const uint8_t* const* records, int n, size_t record_bytes, const uint32_t* expected,
                                 uint32_t* crc_out, uint32_t* unit_ws, int* err, int num_sms, cudaStream_t s) {
  CrcArgs a;
  a.records = records;
  a.n = n;
  a.bytes = (long long)record_bytes;
  a.units = records_crc_units(record_bytes);
  a.pad = (long long)a.units * kCrcUnit - a.bytes;
  a.unit_crc = unit_ws;
  a.expected = expected;
  a.crc_out = crc_out;
  a.err = err;
  for (int l = 0; l < 32; ++l) a.lane_mul[l] = gf2_xpow8((unsigned long long)kCrcLaneBytes * (31 - l));
  a.unit_mul = gf2_xpow8(kCrcUnit);
  a.init_term = gf2_mulmod(0xFFFFFFFFu, gf2_xpow8((unsigned long long)record_bytes));
  if ((long long)n * a.units >= (1ll << 31)) return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem(crc_units_kernel, kCrcSmemBytes);
  if (e != cudaSuccess) return e;
  const long long warps = (long long)n * a.units;
  const long long ctas = (warps + kCrcWarps - 1) / kCrcWarps;
  const int grid = (int)(ctas < num_sms ? ctas : num_sms);
  e = launch("records_crc", crc_units_kernel, dim3(grid), dim3(kCrcThreads), kCrcSmemBytes, s, false, a);
  if (e != cudaSuccess) return e;
  return launch("records_crc_finish", crc_finish_kernel, dim3((n + 3) / 4), dim3(128), 0, s, false, a);
}

}  // namespace moe

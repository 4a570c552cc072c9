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
// 128 KiB segments.  One CTA takes one segment at a time: each lane folds its
// 128 contiguous bytes through byte tables (four bytes per step, the four
// tables giving a byte's effect after 4, 3, 2 and 1 more bytes), multiplies
// the result by x to the number of bits that follow it in the warp's 4 KiB
// step and the warp xors the lanes; steps, warps and finally segments are
// joined by the same product.  The tables are stored once per lane (entry i of
// lane l at word 32 i + l), so every lane reads its own bank and the lookups
// never conflict.  In the reflected bit order used throughout, bit 31 - k of a
// 32-bit word is the coefficient of x^k.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr uint32_t kCrcPoly = 0xEDB88320u;
constexpr int kCrcWarps = 16;
constexpr int kCrcThreads = kCrcWarps * 32;
constexpr int kCrcLaneBytes = 128;                          // contiguous bytes per lane and step
constexpr int kCrcStep = 32 * kCrcLaneBytes;                // 4 KiB per warp step
constexpr int kCrcStepsPerWarp = 2;
constexpr int kCrcSeg = kCrcWarps * kCrcStepsPerWarp * kCrcStep;  // 128 KiB per segment
constexpr size_t kCrcTableBytes = 4 * 256 * 32 * sizeof(uint32_t);  // 128 KiB: four tables per lane

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

struct CrcConsts {
  uint32_t lane_mul[32];         // x^(8 (bytes after lane l's piece in a step))
  uint32_t warp_mul[kCrcWarps];  // x^(8 (bytes after warp w's region in a segment))
  uint32_t step_mul;             // x^(8 kCrcStep)
  uint32_t seg_mul;              // x^(8 kCrcSeg)
  uint32_t init_term;            // 0xFFFFFFFF * x^(8 B): the all-ones start carried over B bytes
};

struct CrcArgs {
  const uint8_t* const* records;
  int n;
  long long bytes;  // B, a multiple of 16
  int segs;         // ceil(B / kCrcSeg)
  long long pad;    // segs * kCrcSeg - B virtual leading zero bytes
  uint32_t* seg_crc;  // [n][segs] workspace
  const uint32_t* expected;  // [n] or null
  uint32_t* crc_out;         // [n] or null
  int* err;
  CrcConsts c;
};

__device__ __forceinline__ bool record_usable(const uint8_t* p) {
  return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// Raw CRC of every (record, segment) work item; persistent CTAs.
__global__ void __launch_bounds__(kCrcThreads, 1) crc_segments_kernel(const CrcArgs a) {
  extern __shared__ uint32_t tab[];  // [4][256][32]
  __shared__ uint32_t t[4][256];
  __shared__ uint32_t wpart[kCrcWarps];
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
  for (int i = tid; i < 4 * 256 * 32; i += kCrcThreads) tab[i] = t[i >> 13][(i >> 5) & 255];
  __syncthreads();
  const uint32_t* T0 = tab + lane;              // one more byte
  const uint32_t* T1 = tab + 1 * 8192 + lane;   // two
  const uint32_t* T2 = tab + 2 * 8192 + lane;   // three
  const uint32_t* T3 = tab + 3 * 8192 + lane;   // four
  const uint32_t lane_mul = a.c.lane_mul[lane];
  const long long total = (long long)a.n * a.segs;
  for (long long w = blockIdx.x; w < total; w += gridDim.x) {
    const int rec = (int)(w / a.segs);
    const int seg = (int)(w - (long long)rec * a.segs);
    const uint8_t* base = a.records[rec];
    uint32_t run = 0;
    if (record_usable(base)) {
      const long long v0 = (long long)seg * kCrcSeg + (long long)warp * kCrcStepsPerWarp * kCrcStep;
      uint4 q[kCrcStepsPerWarp][kCrcLaneBytes / 16];
#pragma unroll
      for (int st = 0; st < kCrcStepsPerWarp; ++st) {
        const long long o = v0 + (long long)st * kCrcStep + lane * kCrcLaneBytes - a.pad;  // real offset
#pragma unroll
        for (int j = 0; j < kCrcLaneBytes / 16; ++j) {
          const long long oj = o + 16 * j;  // 16-byte chunks lie wholly in the padding or in the record
          q[st][j] = oj >= 0 ? __ldg(reinterpret_cast<const uint4*>(base + oj)) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int st = 0; st < kCrcStepsPerWarp; ++st) {
        uint32_t reg = 0;
#pragma unroll
        for (int j = 0; j < kCrcLaneBytes / 16; ++j) {
          const uint32_t wv[4] = {q[st][j].x, q[st][j].y, q[st][j].z, q[st][j].w};
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            reg ^= wv[m];  // the word's first byte in memory is its low byte
            reg = T3[(reg & 0xFFu) << 5] ^ T2[((reg >> 8) & 0xFFu) << 5] ^ T1[((reg >> 16) & 0xFFu) << 5] ^
                  T0[(reg >> 24) << 5];
          }
        }
        uint32_t part = gf2_mulmod(reg, lane_mul);
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) part ^= __shfl_xor_sync(0xffffffffu, part, s);
        run = gf2_mulmod(run, a.c.step_mul) ^ part;
      }
    }
    if (lane == 0) wpart[warp] = gf2_mulmod(run, a.c.warp_mul[warp]);
    __syncthreads();
    if (tid == 0) {
      uint32_t s = 0;
      for (int i = 0; i < kCrcWarps; ++i) s ^= wpart[i];
      a.seg_crc[w] = s;
    }
    __syncthreads();
  }
}

// One thread per record: join the segments, finish the standard CRC, compare.
__global__ void crc_finish_kernel(const CrcArgs a) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= a.n) return;
  const uint8_t* base = a.records[e];
  if (!record_usable(base)) {
    dev_error(a.err, base == nullptr ? MOE_ERR_MISSING_EXPERT : MOE_ERR_BAD_RECORD, e);
    if (a.crc_out) a.crc_out[e] = 0u;
    return;
  }
  uint32_t r = 0;
  for (int s = 0; s < a.segs; ++s) r = gf2_mulmod(r, a.c.seg_mul) ^ a.seg_crc[(size_t)e * a.segs + s];
  r ^= a.c.init_term ^ 0xFFFFFFFFu;
  if (a.crc_out) a.crc_out[e] = r;
  if (a.expected && a.expected[e] != r) dev_error(a.err, MOE_ERR_BAD_RECORD, e);
}

}  // namespace

int records_crc_segments(size_t record_bytes) { return (int)((record_bytes + kCrcSeg - 1) / kCrcSeg); }

cudaError_t launch_records_check(const uint8_t* const* records, int n, size_t record_bytes, const uint32_t* expected,
                                 uint32_t* crc_out, uint32_t* seg_ws, int* err, int num_sms, cudaStream_t s) {
  CrcArgs a;
  a.records = records;
  a.n = n;
  a.bytes = (long long)record_bytes;
  a.segs = records_crc_segments(record_bytes);
  a.pad = (long long)a.segs * kCrcSeg - a.bytes;
  a.seg_crc = seg_ws;
  a.expected = expected;
  a.crc_out = crc_out;
  a.err = err;
  for (int l = 0; l < 32; ++l) a.c.lane_mul[l] = gf2_xpow8((unsigned long long)kCrcLaneBytes * (31 - l));
  for (int w = 0; w < kCrcWarps; ++w)
    a.c.warp_mul[w] = gf2_xpow8((unsigned long long)kCrcStepsPerWarp * kCrcStep * (kCrcWarps - 1 - w));
  a.c.step_mul = gf2_xpow8(kCrcStep);
  a.c.seg_mul = gf2_xpow8(kCrcSeg);
  a.c.init_term = gf2_mulmod(0xFFFFFFFFu, gf2_xpow8((unsigned long long)record_bytes));
  cudaError_t e = ensure_smem(crc_segments_kernel, kCrcTableBytes);
  if (e != cudaSuccess) return e;
  const long long total = (long long)n * a.segs;
  const int grid = (int)(total < num_sms ? total : num_sms);
  e = launch("records_crc", crc_segments_kernel, dim3(grid), dim3(kCrcThreads), kCrcTableBytes, s, false, a);
  if (e != cudaSuccess) return e;
  return launch("records_crc_finish", crc_finish_kernel, dim3((n + 127) / 128), dim3(128), 0, s, false, a);
}

}  // namespace moe

/*
 * si_device.cu -- device-side fills of the seeded synthetic inputs (C ABI).
 *
 * Same arithmetic as si_host.c (both include si_rng.h), so a buffer filled here
 * is byte-identical to the host fill of the same (seed, stream, range).  Used to
 * materialise the expert banks (up to ~94 GB) directly in HBM.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "si_rng.h"

namespace {

__global__ void fill_normal_kernel(uint64_t key, double sigma, uint64_t offset, uint64_t n, int dtype,
                                   void* out) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
       i += (uint64_t)gridDim.x * blockDim.x) {
    float v = (float)(si_std_normal(key, offset + i) * sigma);
    if (dtype == 0)
      ((float*)out)[i] = v;
    else if (dtype == 1)
      ((uint16_t*)out)[i] = si_f32_to_bf16(v);
    else
      ((uint16_t*)out)[i] = si_f32_to_f16(v);
  }
}

__global__ void fill_bytes_kernel(uint64_t key, uint64_t offset, uint64_t n, uint8_t* out) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
       i += (uint64_t)gridDim.x * blockDim.x)
    out[i] = si_byte(key, offset + i);
}

/* One thread per 16-byte chunk of one record; a chunk never straddles a region
 * boundary because every region size is a multiple of 16 bytes. */
__global__ void fill_mxfp4_bank_kernel(uint64_t seed, uint64_t e0, uint64_t n_exp, uint64_t d, uint64_t ff,
                                       uint32_t lo, uint32_t hi, uint8_t* base, uint64_t stride) {
  const uint64_t rec = 3u * (ff * d / 2u + ff * d / 32u);
  const uint64_t chunks = rec / 16u;
  const uint64_t total = chunks * n_exp;
  for (uint64_t c = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; c < total;
       c += (uint64_t)gridDim.x * blockDim.x) {
    uint64_t e = c / chunks, off = (c % chunks) * 16u;
    uint64_t stream = SI_STREAM_RECORD + e0 + e;
    uint8_t b[16];
    if (si_mxfp4_is_scale(off, d, ff)) {
      uint64_t ks = si_key(seed, stream | SI_STREAM_SCALE_TAG);
      for (int j = 0; j < 16; ++j) b[j] = si_scale_byte(ks, off + j, lo, hi);
    } else {
      uint64_t kc = si_key(seed, stream);
      uint64_t w0 = si_u64(kc, off >> 3), w1 = si_u64(kc, (off >> 3) + 1u);
      for (int j = 0; j < 8; ++j) {
        b[j] = (uint8_t)(w0 >> (8 * j));
        b[8 + j] = (uint8_t)(w1 >> (8 * j));
      }
    }
    uint4 v;
    v.x = b[0] | (b[1] << 8) | (b[2] << 16) | ((uint32_t)b[3] << 24);
    v.y = b[4] | (b[5] << 8) | (b[6] << 16) | ((uint32_t)b[7] << 24);
    v.z = b[8] | (b[9] << 8) | (b[10] << 16) | ((uint32_t)b[11] << 24);
    v.w = b[12] | (b[13] << 8) | (b[14] << 16) | ((uint32_t)b[15] << 24);
    *reinterpret_cast<uint4*>(base + e * stride + off) = v;
  }
}

__global__ void fill_rvq3_bank_kernel(uint64_t seed, uint64_t e0, uint64_t n_exp, uint64_t rec,
                                      uint8_t* base, uint64_t stride) {
  const uint64_t chunks = rec / 16u;
  const uint64_t total = chunks * n_exp;
  for (uint64_t c = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; c < total;
       c += (uint64_t)gridDim.x * blockDim.x) {
    uint64_t e = c / chunks, off = (c % chunks) * 16u;
    uint64_t kc = si_key(seed, SI_STREAM_RECORD + e0 + e);
    uint4 v;
    uint64_t w0 = si_u64(kc, off >> 3), w1 = si_u64(kc, (off >> 3) + 1u);
    v.x = (uint32_t)w0;
    v.y = (uint32_t)(w0 >> 32);
    v.z = (uint32_t)w1;
    v.w = (uint32_t)(w1 >> 32);
    *reinterpret_cast<uint4*>(base + e * stride + off) = v;
  }
}

unsigned grid_for(uint64_t work) {
  uint64_t g = (work + 255u) / 256u;
  if (g > 152u * 64u) g = 152u * 64u;
  if (g == 0) g = 1;
  return (unsigned)g;
}

}  // namespace

extern "C" {

int si_dev_fill_normal(uint64_t seed, uint64_t stream, double sigma, uint64_t offset, uint64_t n, int dtype,
                       void* out, cudaStream_t s) {
  if (n == 0) return 0;
  fill_normal_kernel<<<grid_for(n), 256, 0, s>>>(si_key(seed, stream), sigma, offset, n, dtype, out);
  return (int)cudaGetLastError();
}

int si_dev_fill_bytes(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, uint8_t* out,
                      cudaStream_t s) {
  if (n == 0) return 0;
  fill_bytes_kernel<<<grid_for(n), 256, 0, s>>>(si_key(seed, stream), offset, n, out);
  return (int)cudaGetLastError();
}

/* Fills records of experts e0 .. e0+n_exp-1, record i at base + i*stride.
 * base and stride must be multiples of 16; d % 32 == 0 and ff % 32 == 0. */
int si_dev_fill_mxfp4_bank(uint64_t seed, uint64_t e0, uint64_t n_exp, uint64_t d, uint64_t ff, uint32_t lo,
                           uint32_t hi, uint8_t* base, uint64_t stride, cudaStream_t s) {
  if (((uintptr_t)base & 15u) || (stride & 15u) || (d & 31u) || (ff & 31u) || hi < lo) return -1;
  uint64_t rec = 3u * (ff * d / 2u + ff * d / 32u);
  fill_mxfp4_bank_kernel<<<grid_for(rec / 16u * n_exp), 256, 0, s>>>(seed, e0, n_exp, d, ff, lo, hi, base,
                                                                      stride);
  return (int)cudaGetLastError();
}

int si_dev_fill_rvq3_bank(uint64_t seed, uint64_t e0, uint64_t n_exp, uint64_t d, uint64_t ff, uint8_t* base,
                          uint64_t stride, cudaStream_t s) {
  if (((uintptr_t)base & 15u) || (stride & 15u) || (d & 31u) || (ff & 31u)) return -1;
  uint64_t rec = 9u * ff * d / 8u;
  fill_rvq3_bank_kernel<<<grid_for(rec / 16u * n_exp), 256, 0, s>>>(seed, e0, n_exp, rec, base, stride);
  return (int)cudaGetLastError();
}

}  // extern "C"

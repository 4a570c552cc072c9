/*
 * si_host.c -- host-side fills of the seeded synthetic inputs (C ABI).
 * The arithmetic lives in si_rng.h; this file only loops over indices.
 */
#include <stddef.h>
#include <stdint.h>

#include "si_rng.h"

/* dtype codes: 0 = float32, 1 = bfloat16, 2 = float16 */
void si_fill_normal(uint64_t seed, uint64_t stream, double sigma, uint64_t offset, uint64_t n,
                    int dtype, void* out) {
  uint64_t key = si_key(seed, stream);
  for (uint64_t i = 0; i < n; ++i) {
    float v = (float)(si_std_normal(key, offset + i) * sigma);
    if (dtype == 0)
      ((float*)out)[i] = v;
    else if (dtype == 1)
      ((uint16_t*)out)[i] = si_f32_to_bf16(v);
    else
      ((uint16_t*)out)[i] = si_f32_to_f16(v);
  }
}

void si_fill_bytes(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, uint8_t* out) {
  uint64_t key = si_key(seed, stream);
  for (uint64_t i = 0; i < n; ++i) out[i] = si_byte(key, offset + i);
}

uint64_t si_mxfp4_record_size(uint64_t d, uint64_t ff) { return 3u * (ff * d / 2u + ff * d / 32u); }

uint64_t si_rvq3_record_size(uint64_t d, uint64_t ff) { return 9u * ff * d / 8u; }

/* Fills bytes [offset, offset + n) of expert `expert`'s MXFP4 record. */
void si_fill_mxfp4_record(uint64_t seed, uint64_t expert, uint64_t d, uint64_t ff, uint32_t scale_lo,
                          uint32_t scale_hi, uint64_t offset, uint64_t n, uint8_t* out) {
  uint64_t stream = SI_STREAM_RECORD + expert;
  uint64_t kc = si_key(seed, stream);
  uint64_t ks = si_key(seed, stream | SI_STREAM_SCALE_TAG);
  for (uint64_t i = 0; i < n; ++i) {
    uint64_t off = offset + i;
    out[i] = si_mxfp4_is_scale(off, d, ff) ? si_scale_byte(ks, off, scale_lo, scale_hi) : si_byte(kc, off);
  }
}

/* Fills bytes [offset, offset + n) of expert `expert`'s RVQ3 record (uniform codes). */
void si_fill_rvq3_record(uint64_t seed, uint64_t expert, uint64_t offset, uint64_t n, uint8_t* out) {
  si_fill_bytes(seed, SI_STREAM_RECORD + expert, offset, n, out);
}

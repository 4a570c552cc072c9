/*
 * si_rng.h -- counter-based random source for the synthetic MoE-layer inputs.
 *
 * This header is the whole of the input generator's arithmetic.  It is compiled
 * twice: by the host C compiler into libseeded_inputs_host.so (used by the tests
 * and by the CPU oracle's drivers) and by nvcc into libseeded_inputs_cuda.so
 * (which fills device buffers directly, so that a 15.7 GB expert bank never has
 * to cross the PCIe/C2C link).  It holds none of the MoE layer's arithmetic: it
 * only turns (seed, stream, index) into bytes.
 *
 * Every step is integer arithmetic or a single correctly rounded IEEE operation
 * (double add/multiply of dyadic values, double->float conversion), so host and
 * device produce bit-identical values; a GPU test checks that.
 *
 * Generator: the SplitMix64 output function (Steele, Lea and Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014) applied to a counter,
 * i.e. value(key, i) = mix64(key + (i + 1) * golden_gamma).
 *
 * Normal variates use the Irwin-Hall construction: the sum of twelve uniform
 * 16-bit draws, centred, has mean 0 and variance 1 (to within 2^-32) and is an
 * exact dyadic rational, so it needs no transcendental function.
 */
#ifndef SEEDED_INPUTS_SI_RNG_H
#define SEEDED_INPUTS_SI_RNG_H

#include <stdint.h>

#ifdef __CUDACC__
#define SI_HD __host__ __device__ __forceinline__
#else
#define SI_HD static inline
#endif

#define SI_GOLDEN_GAMMA 0x9E3779B97F4A7C15ull

/* Stream identifiers (one independent sequence per synthetic tensor). */
#define SI_STREAM_X 1ull         /* activations x [T][d]                      */
#define SI_STREAM_ROUTER_W 2ull  /* router weight [E][d]                      */
#define SI_STREAM_CODEBOOK 16ull /* + stage: RVQ codebooks, fp16 [256][8]     */
#define SI_STREAM_RECORD 0x100000ull        /* + expert id: record code bytes */
#define SI_STREAM_SCALE_TAG 0x4000000000ull /* OR-ed in for E8M0 scale bytes  */

SI_HD uint64_t si_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

SI_HD uint64_t si_key(uint64_t seed, uint64_t stream) {
  return si_mix64(si_mix64(seed + SI_GOLDEN_GAMMA) ^ (stream * 0xD1B54A32D192ED03ull));
}

SI_HD uint64_t si_u64(uint64_t key, uint64_t i) {
  return si_mix64(key + (i + 1ull) * SI_GOLDEN_GAMMA);
}

/* Irwin-Hall(12) approximately standard normal variate number i of the stream. */
SI_HD double si_std_normal(uint64_t key, uint64_t i) {
  uint64_t a = si_u64(key, 3ull * i);
  uint64_t b = si_u64(key, 3ull * i + 1ull);
  uint64_t c = si_u64(key, 3ull * i + 2ull);
  uint64_t s = 0;
  for (int j = 0; j < 4; ++j) {
    s += (a >> (16 * j)) & 0xFFFFull;
    s += (b >> (16 * j)) & 0xFFFFull;
    s += (c >> (16 * j)) & 0xFFFFull;
  }
  /* sum of U_j = (v_j + 1/2) / 65536 over 12 draws, minus 6: exact in double */
  return ((double)s + 6.0) * (1.0 / 65536.0) - 6.0;
}

SI_HD uint32_t si_f32_bits(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  return v.u;
}

/* float -> bfloat16, round to nearest even (inputs here are finite). */
SI_HD uint16_t si_f32_to_bf16(float f) {
  uint32_t u = si_f32_bits(f);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* float -> IEEE binary16, round to nearest even, with subnormals and overflow. */
SI_HD uint16_t si_f32_to_f16(float f) {
  uint32_t u = si_f32_bits(f);
  uint32_t sign = (u >> 16) & 0x8000u;
  uint32_t a = u & 0x7FFFFFFFu;
  if (a >= 0x7F800000u) return (uint16_t)(sign | 0x7C00u | (a > 0x7F800000u ? 0x200u : 0u));
  if (a >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u); /* rounds to >= 65520: inf */
  if (a < 0x38800000u) {                                  /* below 2^-14: subnormal  */
    if (a < 0x33000000u) return (uint16_t)sign;           /* below 2^-25: zero       */
    uint32_t e = a >> 23;                                 /* 102..112                */
    uint32_t m = (a & 0x7FFFFFu) | 0x800000u;             /* 24-bit significand      */
    uint32_t shift = 126u - e;                            /* value = m * 2^(e-150)   */
    uint32_t q = m >> shift;                              /* units of 2^-24          */
    uint32_t rem = m & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1u);
    if (rem > half || (rem == half && (q & 1u))) q += 1u;
    return (uint16_t)(sign | q);
  }
  uint32_t r = a - 0x38000000u; /* rebias exponent 127 -> 15 */
  uint32_t q = r >> 13;
  uint32_t rem = r & 0x1FFFu;
  if (rem > 0x1000u || (rem == 0x1000u && (q & 1u))) q += 1u;
  return (uint16_t)(sign | q);
}

/* Byte j of a uniformly random byte stream. */
SI_HD uint8_t si_byte(uint64_t key, uint64_t j) {
  return (uint8_t)(si_u64(key, j >> 3) >> (8u * (uint32_t)(j & 7u)));
}

/* Scale byte j, uniform in [lo, hi] (hi >= lo). */
SI_HD uint8_t si_scale_byte(uint64_t key, uint64_t j, uint32_t lo, uint32_t hi) {
  return (uint8_t)(lo + (uint32_t)(si_u64(key, j) % (uint64_t)(hi - lo + 1u)));
}

/*
 * Expert record layouts the generator fills.  MXFP4 record (all sizes in bytes):
 *   gate.codes [ff][d/2] | gate.scales [ff][d/32] | up.codes [ff][d/2] |
 *   up.scales [ff][d/32] | down.codes [d][ff/2]   | down.scales [d][ff/32]
 * The generator only needs to know which byte ranges hold E8M0 scales.
 */
SI_HD int si_mxfp4_is_scale(uint64_t off, uint64_t d, uint64_t ff) {
  uint64_t mat = ff * d / 2u + ff * d / 32u; /* one matrix: codes + scales */
  uint64_t in_mat = off % mat;
  return in_mat >= ff * d / 2u;
}

SI_HD uint8_t si_mxfp4_record_byte(uint64_t seed, uint64_t expert, uint64_t d, uint64_t ff,
                                   uint32_t scale_lo, uint32_t scale_hi, uint64_t off) {
  uint64_t stream = SI_STREAM_RECORD + expert;
  if (si_mxfp4_is_scale(off, d, ff))
    return si_scale_byte(si_key(seed, stream | SI_STREAM_SCALE_TAG), off, scale_lo, scale_hi);
  return si_byte(si_key(seed, stream), off);
}

#endif /* SEEDED_INPUTS_SI_RNG_H */

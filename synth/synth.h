/*
 * synth.h -- seeded, counter-based synthetic input generator.
 *
 * This header is the single definition of every synthetic input used by the
 * tests, the oracle harness and the benchmark.  It is compiled twice: by gcc
 * for the host library (synth.c) and by nvcc for the device library
 * (synth_cuda.cu), so that a tensor of several GB can be generated directly
 * in device memory while the CPU oracle regenerates exactly the same bits for
 * the rows it needs.  It holds no arithmetic of the attention method itself:
 * only hashing, the mapping of a hash to a number, and the conversion of that
 * number to the storage format (bf16, e4m3).
 *
 * Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014; finaliser constants as in
 * S. Vigna's public-domain splitmix64.c).  Element i of a stream with state
 * `base` is mix64(base + (i + 1) * GAMMA), the i-th output of SplitMix64.
 *
 * Normal samples: the four 16-bit fields of one 64-bit output are summed
 * (Irwin-Hall with n = 4), centred and scaled by sqrt(3)/65536 in one IEEE
 * fp32 multiply of an exact integer, so the result is bit-identical on every
 * IEEE machine.  Mean 0, variance 1 (to 2^-32), support [-3.46, 3.46].
 */
#ifndef CSA2_SYNTH_H
#define CSA2_SYNTH_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYNTH_FN __host__ __device__ __forceinline__
#else
#define SYNTH_FN static inline
#endif

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ULL

SYNTH_FN uint64_t synth_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* State of the stream (seed, stream id). */
SYNTH_FN uint64_t synth_base(uint64_t seed, uint64_t stream) {
  uint64_t s = synth_mix64(seed + SYNTH_GAMMA);
  return synth_mix64(s ^ (stream * 0xD1B54A32D192ED03ULL + SYNTH_GAMMA));
}

SYNTH_FN uint64_t synth_u64(uint64_t base, uint64_t i) {
  return synth_mix64(base + (i + 1) * SYNTH_GAMMA);
}

/* Uniform fp32 in [0, 1) with 24 random bits. */
SYNTH_FN float synth_uniform(uint64_t base, uint64_t i) {
  return (float)(uint32_t)(synth_u64(base, i) >> 40) * 5.9604644775390625e-08f;
}

/* Approximately N(0,1): Irwin-Hall(4) of 16-bit fields, exact integer sum. */
SYNTH_FN float synth_normal(uint64_t base, uint64_t i) {
  uint64_t h = synth_u64(base, i);
  int32_t s = (int32_t)(h & 0xFFFFu) + (int32_t)((h >> 16) & 0xFFFFu) +
              (int32_t)((h >> 32) & 0xFFFFu) + (int32_t)((h >> 48) & 0xFFFFu) -
              131070;
  return (float)s * 2.642919309437275e-05f; /* sqrt(3) / 65536 */
}

SYNTH_FN uint32_t synth_f32_bits(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  return v.u;
}

/* fp32 -> bf16 bits, round to nearest even (inputs here are finite). */
SYNTH_FN uint16_t synth_bf16(float f) {
  uint32_t u = synth_f32_bits(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* fp32 -> OCP FP8 E4M3 code, round to nearest even, saturating at +-448.
 * E4M3: bias 7, 3 mantissa bits, subnormal quantum 2^-9, no infinities. */
SYNTH_FN uint8_t synth_e4m3(float x) {
  uint32_t u = synth_f32_bits(x);
  uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
  uint32_t au = u & 0x7FFFFFFFu;
  if (au == 0) return sign;
  int e = (int)(au >> 23) - 127;        /* floor(log2 |x|) for normal fp32 */
  if (e > 8) return sign | 0x7E;        /* |x| >= 512: saturate to 448 */
  int qexp = e < -6 ? -9 : e - 3;       /* quantum of the target binade */
  /* |x| / 2^qexp is exact; round it to an integer, ties to even. */
  uint32_t mant = (au & 0x7FFFFFu) | 0x800000u; /* |x| = mant * 2^(e-23) */
  int sh = (qexp - (e - 23));                    /* right shift, >= 20 */
  if (sh > 31) return sign;                      /* far below the quantum */
  uint32_t q = mant >> sh;
  uint32_t rem = mant & ((1u << sh) - 1u);
  uint32_t half = 1u << (sh - 1);
  if (rem > half || (rem == half && (q & 1u))) q += 1u;
  uint32_t code;
  if (qexp == -9) {
    code = q;                           /* q <= 8; q == 8 is 2^-6, code 0x08 */
  } else {
    int ee = e;
    if (q == 16u) { q = 8u; ee += 1; }
    if (ee + 7 > 15) return sign | 0x7E;
    code = ((uint32_t)(ee + 7) << 3) | (q - 8u);
    if (code > 0x7Eu) code = 0x7Eu;    /* 0x7F is NaN: saturate */
  }
  return (uint8_t)(sign | code);
}

/* Logical element id of row j, column d of sequence b in a [rows, D] tensor.
 * Independent of how the sequences are laid out in memory. */
SYNTH_FN uint64_t synth_row_elem(uint64_t b, uint64_t j, uint64_t D, uint64_t d) {
  return ((b << 32) | j) * D + d;
}

#endif /* CSA2_SYNTH_H */

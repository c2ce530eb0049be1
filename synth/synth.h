/*
 * synth.h — seeded, counter-based synthetic inputs for the routed MXFP4 MoE layer.
 *
 * This module makes INPUT BYTES only (activations, router weights, packed
 * expert weights).  It holds none of the layer's arithmetic: the CUDA library
 * and the fp64 oracle both consume the bytes it writes, and neither includes
 * this file.  Every function is a pure function of (seed, tag, index), written
 * with integer operations and exactly rounded IEEE operations only, so the host
 * build (gcc) and the device build (nvcc) produce identical bytes.
 *
 * Generator definitions (all public):
 *   - SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
 *     generators", OOPSLA 2014): output n of the stream with state S is
 *     mix64(S + (n + 1) * 0x9E3779B97F4A7C15).
 *   - Approximately standard-normal samples by the Irwin–Hall construction:
 *     the sum of twelve independent uniforms, centred.  Here the uniforms are
 *     16-bit integers, so z = (S - 393210) / 65536 with S the integer sum; z has
 *     mean 0, variance 1 - 2^-32, lies in [-6, 6] and is exact in binary64.
 *   - The block quantiser that turns a row of reals into MX blocks (32 values
 *     sharing one power-of-two scale, elements stored as 4-bit E2M1 codes) in
 *     the manner of the OCP Microscaling Formats (MX) v1.0 specification:
 *     shared exponent X = floor(log2(max|v|)) - 2 (the largest E2M1 magnitude is
 *     6 = 1.5 * 2^2), element code = v / 2^X rounded to the nearest E2M1 value,
 *     ties to the code with a zero mantissa bit, saturating at +-6.
 */
#ifndef MOE_SYNTH_H
#define MOE_SYNTH_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYN_FN static __host__ __device__ __forceinline__
#else
#define SYN_FN static inline
#endif

#define SYN_GAMMA 0x9E3779B97F4A7C15ULL

/* Stream tags: one independent stream per input tensor. */
#define SYN_TAG_X 1ULL
#define SYN_TAG_ROUTER 2ULL
#define SYN_TAG_PLANT 3ULL    /* directions for the planted wide-decode routing */
#define SYN_TAG_PERM 4ULL     /* expert permutations (Zipf ranks, planted sets) */
#define SYN_TAG_SHARED 0x100ULL /* + j, j = 0 gate, 1 up, 2 down */
#define SYN_TAG_EXPERT 0x10000ULL /* + 4*e + j, j = 0 gate, 1 up, 2 down */

SYN_FN uint64_t syn_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Key of the stream for (seed, tag). */
SYN_FN uint64_t syn_key(uint64_t seed, uint64_t tag) {
  return syn_mix64(syn_mix64(seed + SYN_GAMMA) ^ (tag * 0xD1B54A32D192ED03ULL));
}

/* Output i of the SplitMix64 stream whose state starts at key. */
SYN_FN uint64_t syn_u64(uint64_t key, uint64_t i) {
  return syn_mix64(key + (i + 1ULL) * SYN_GAMMA);
}

/* Sample i of the approximately-normal stream (Irwin–Hall of 12 uniform u16). */
SYN_FN double syn_normal(uint64_t key, uint64_t i) {
  int64_t sum = 0;
  for (int w = 0; w < 3; ++w) {
    uint64_t r = syn_u64(key, 3ULL * i + (uint64_t)w);
    sum += (int64_t)(r & 0xFFFFULL) + (int64_t)((r >> 16) & 0xFFFFULL) +
           (int64_t)((r >> 32) & 0xFFFFULL) + (int64_t)(r >> 48);
  }
  return (double)(2 * sum - 786420) / 131072.0;
}

/* Round a binary32 value to bfloat16, nearest-even (NaN kept quiet). */
SYN_FN uint16_t syn_bf16_rne(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  uint32_t u = v.u;
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
    return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* 2^n as binary64 for -1022 <= n <= 1023, built from its bits (exact). */
SYN_FN double syn_pow2(int n) {
  union { double d; uint64_t u; } v;
  v.u = (uint64_t)(n + 1023) << 52;
  return v.d;
}

/* floor(log2(a)) for a finite a > 0 in the normal binary64 range, from its bits. */
SYN_FN int syn_floor_log2(double a) {
  union { double d; uint64_t u; } v;
  v.d = a;
  return (int)((v.u >> 52) & 0x7FFu) - 1023;
}

/* Magnitude code of |r| on the E2M1 grid {0,.5,1,1.5,2,3,4,6}: nearest, ties to
 * the even code (zero mantissa bit), saturating at 6. */
SYN_FN uint32_t syn_e2m1_code(double a) {
  if (a <= 0.25) return 0u;
  if (a < 0.75) return 1u;
  if (a <= 1.25) return 2u;
  if (a < 1.75) return 3u;
  if (a <= 2.5) return 4u;
  if (a < 3.5) return 5u;
  if (a <= 5.0) return 6u;
  return 7u;
}

/* Quantise 32 reals into one MX block: 16 packed bytes (element 2i in the low
 * nibble of byte i, element 2i+1 in the high nibble) and one E8M0 scale byte. */
SYN_FN void syn_quant_block(const double* v, uint8_t* q, uint8_t* s) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) {
    double a = v[i] < 0.0 ? -v[i] : v[i];
    if (a > amax) amax = a;
  }
  if (amax == 0.0) {
    for (int i = 0; i < 16; ++i) q[i] = 0;
    *s = 0;
    return;
  }
  int X = syn_floor_log2(amax) - 2;
  int e = X + 127;
  if (e < 0) e = 0;
  if (e > 254) e = 254;
  double inv = syn_pow2(127 - e); /* 1 / 2^(e-127), exact */
  for (int i = 0; i < 16; ++i) {
    uint32_t byte = 0;
    for (int h = 0; h < 2; ++h) {
      double r = v[2 * i + h] * inv;
      double a = r < 0.0 ? -r : r;
      uint32_t c = syn_e2m1_code(a);
      if (r < 0.0 && c != 0u) c |= 8u;
      byte |= c << (4 * h);
    }
    q[i] = (uint8_t)byte;
  }
  *s = (uint8_t)e;
}

/* Expert weight value (before quantisation): 0.02 * z. */
SYN_FN double syn_weight(uint64_t key, uint64_t i) { return syn_normal(key, i) * 0.02; }

/* Quantise block b (32 consecutive columns) of row r of a rows x cols matrix
 * whose reals are syn_weight(key, r*cols + c). */
SYN_FN void syn_mx_block(uint64_t key, int64_t cols, int64_t r, int64_t b, uint8_t* q, uint8_t* s) {
  double v[32];
  for (int i = 0; i < 32; ++i) v[i] = syn_weight(key, (uint64_t)(r * cols + b * 32 + i));
  syn_quant_block(v, q, s);
}

#endif /* MOE_SYNTH_H */

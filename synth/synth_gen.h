/*
 * Seeded synthetic inputs for the routed MoE layer.
 *
 * This header is the single definition of the counter-based generator that
 * both the CPU oracle and the GPU-side input fill kernels use.  It holds no
 * step of the layer's arithmetic (no routing, no quantisation, no GEMM): it
 * only turns (seed, tensor id, element index) into numbers.
 *
 *  - mix64 is the SplitMix64 finaliser (Steele, Lea and Flood, "Fast
 *    splittable pseudorandom number generators", OOPSLA 2014), used as a
 *    stateless hash of a 64-bit counter.
 *  - A standard-normal stand-in is the Irwin-Hall sum of twelve 24-bit
 *    uniforms minus 6.  The sum is an exact integer; it is rounded to fp32
 *    once, so the value is bit-identical on every IEEE machine.  Its tails
 *    are bounded at +-6, which is the only way it differs from N(0,1) here.
 *
 * Compiles as C99 (host) and as CUDA (host + device).
 */
#ifndef SYNTH_GEN_H
#define SYNTH_GEN_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYNTH_FN static __host__ __device__ __forceinline__
#else
#define SYNTH_FN static inline
#endif

/* Tensor ids: each input tensor draws from its own stream. */
enum {
  SYNTH_T_X = 1,        /* token activations x [T,H]              */
  SYNTH_T_ROUTER = 2,   /* router weight W_r [E,H]                */
  SYNTH_T_BIAS = 3,     /* router bias b [E]                      */
  SYNTH_T_OUTLIER = 4,  /* choice of outlier token rows           */
  SYNTH_T_RANK = 5,     /* popularity rank of each expert (Zipf)  */
  SYNTH_T_GATE = 10,    /* W_gate [E,F,H] master values           */
  SYNTH_T_UP = 11,      /* W_up   [E,F,H] master values           */
  SYNTH_T_DOWN = 12     /* W_down [E,H,F] master values           */
};

SYNTH_FN uint64_t synth_mix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Base counter of one tensor's stream. */
SYNTH_FN uint64_t synth_key(uint64_t seed, uint32_t tensor) {
  return synth_mix64(synth_mix64(seed) ^ ((uint64_t)tensor * 0xD1B54A32D192ED03ULL));
}

/* One 24-bit uniform integer in [0, 2^24) for element i of a stream. */
SYNTH_FN uint32_t synth_u24(uint64_t key, uint64_t i) {
  return (uint32_t)(synth_mix64(key + i) >> 40);
}

/* Raw 64-bit hash of element i (used to rank rows / experts). */
SYNTH_FN uint64_t synth_h64(uint64_t key, uint64_t i) {
  return synth_mix64(key + i);
}

/*
 * Irwin-Hall(12) - 6 for element i: six hashes, two 24-bit fields each.
 * Returns the exact integer sum minus 6*2^24, so z = result * 2^-24.
 */
SYNTH_FN int32_t synth_normal_fixed(uint64_t key, uint64_t i) {
  uint64_t base = key + i * 6ULL;
  int32_t s = 0;
  for (int j = 0; j < 6; ++j) {
    uint64_t r = synth_mix64(base + (uint64_t)j);
    s += (int32_t)(r >> 40);
    s += (int32_t)((r >> 16) & 0xFFFFFFULL);
  }
  return s - 6 * (1 << 24);
}

/* The fp32 normal stand-in: one rounding of the exact integer, then an
 * exact power-of-two scale. */
SYNTH_FN float synth_normal(uint64_t key, uint64_t i) {
  return (float)synth_normal_fixed(key, i) * 5.9604644775390625e-08f; /* 2^-24 */
}

/* fp32 -> bf16 bits, round to nearest even (finite inputs). */
SYNTH_FN uint16_t synth_bf16_bits(float f) {
  union { float f; uint32_t u; } c;
  c.f = f;
  uint32_t lsb = (c.u >> 16) & 1u;
  return (uint16_t)((c.u + 0x7FFFu + lsb) >> 16);
}

#endif /* SYNTH_GEN_H */

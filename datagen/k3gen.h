/*
 * k3gen.h -- seeded, counter-based synthetic input generator.
 *
 * This module is the only code shared by the fp64 oracle and the GPU tests/bench.
 * It holds none of the LatentMoE arithmetic: it only turns (seed, stream, index)
 * into integers, uniform reals and normal reals, and rounds a drawn real to its
 * storage type.  Every tensor element can be regenerated on its own, so a caller
 * that needs one expert out of 896 regenerates just that expert.
 *
 * Definition (fixed; changing it changes every synthetic input):
 *   mix64(z)      = splitmix64 finaliser (Steele, Lea, Flood, "Fast splittable
 *                   pseudorandom number generators", OOPSLA 2014).
 *   key(seed,str) = mix64(seed * G + mix64(str + C0)),   G = 0x9E3779B97F4A7C15
 *   draw(key,i)   = mix64(key + (i + 1) * G)
 *   byte i of a uniform-u8 tensor      = byte (i & 7) of draw(key, i >> 3)
 *   element i of an integer [lo, hi]   = lo + draw(key, i) mod (hi - lo + 1)
 *   uniform real in [a, b)             = a + (b - a) * (draw >> 11) * 2^-53
 *   normal N(0, sigma^2), element i    = sigma * sqrt(-2 ln u1) * cos(2 pi u2),
 *        u1 = ((draw(key, 2i) >> 11) + 1) * 2^-53,  u2 = (draw(key, 2i+1) >> 11) * 2^-53
 *        (Box and Muller, 1958; computed in fp64 on the host only)
 *
 * The integer parts are usable from CUDA device code (K3GEN_HD); the real-valued
 * draws use libm and are host-only.
 */
#ifndef K3GEN_H
#define K3GEN_H

#include <stdint.h>

#if defined(__CUDACC__)
#define K3GEN_HD static __host__ __device__ __forceinline__
#else
#define K3GEN_HD static inline
#endif

#define K3GEN_GOLDEN 0x9E3779B97F4A7C15ULL
#define K3GEN_C0 0x632BE59BD9B4E019ULL

K3GEN_HD uint64_t k3gen_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

K3GEN_HD uint64_t k3gen_key(uint64_t seed, uint64_t stream) {
  return k3gen_mix64(seed * K3GEN_GOLDEN + k3gen_mix64(stream + K3GEN_C0));
}

K3GEN_HD uint64_t k3gen_draw(uint64_t key, uint64_t i) {
  return k3gen_mix64(key + (i + 1) * K3GEN_GOLDEN);
}

/* byte i of a uniform-u8 tensor */
K3GEN_HD uint8_t k3gen_u8(uint64_t key, uint64_t i) {
  return (uint8_t)(k3gen_draw(key, i >> 3) >> (8 * (i & 7)));
}

/* element i of a uniform integer tensor on [lo, hi] (stored as u8 by callers) */
K3GEN_HD uint32_t k3gen_int(uint64_t key, uint64_t i, uint32_t lo, uint32_t hi) {
  return lo + (uint32_t)(k3gen_draw(key, i) % (uint64_t)(hi - lo + 1));
}

/* Stream ids of the tensors of one LatentMoE layer.  Expert tensors get their own
 * stream per (expert, tensor), so any expert can be regenerated alone. */
enum {
  K3GEN_S_X = 1,      /* activations x [T, H] (or z [T, L] for the single-expert case) */
  K3GEN_S_WR = 2,     /* router weight [E, H] */
  K3GEN_S_BIAS = 3,   /* router score-correction bias [E] */
  K3GEN_S_WD = 4,     /* latent down [L, H] */
  K3GEN_S_WU = 5,     /* latent up [H, L] */
  K3GEN_S_XBASE = 6,  /* base vectors of the temporal-locality chunk */
  K3GEN_S_XNOISE = 7, /* per-token perturbations of the temporal-locality chunk */
  K3GEN_S_SGU = 8,    /* shared experts: fused gate and up rows [2 Is, H] */
  K3GEN_S_SDN = 9,    /* shared experts: fused down matrix [H, Is] */
  K3GEN_S_EXPERT0 = 0x1000
};
/* which: 0 gate packed, 1 gate scales, 2 up packed, 3 up scales, 4 down packed, 5 down scales */
K3GEN_HD uint64_t k3gen_expert_stream(uint32_t expert, uint32_t which) {
  return (uint64_t)K3GEN_S_EXPERT0 + (uint64_t)expert * 8u + which;
}

#endif /* K3GEN_H */

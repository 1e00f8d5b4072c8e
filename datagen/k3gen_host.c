/*
 * k3gen_host.c -- host-side fills for the seeded synthetic inputs (see k3gen.h).
 * Exported with C linkage for the Python wrapper in this directory.  OpenMP
 * threads only split the index range; every element depends on its index alone,
 * so the result does not depend on the thread count.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include "k3gen.h"

static const double K3GEN_TWO_PI = 6.283185307179586476925286766559;

void k3gen_fill_u8(uint64_t seed, uint64_t stream, uint64_t n, uint8_t* out) {
  const uint64_t key = k3gen_key(seed, stream);
  const int64_t words = (int64_t)(n >> 3);
#pragma omp parallel for schedule(static)
  for (int64_t w = 0; w < words; ++w) {
    uint64_t r = k3gen_draw(key, (uint64_t)w);
    memcpy(out + 8 * w, &r, 8); /* little-endian: byte j of r is element 8w+j */
  }
  for (uint64_t i = (uint64_t)words << 3; i < n; ++i) out[i] = k3gen_u8(key, i);
}

void k3gen_fill_int_u8(uint64_t seed, uint64_t stream, uint64_t n, uint32_t lo, uint32_t hi,
                       uint8_t* out) {
  const uint64_t key = k3gen_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = (uint8_t)k3gen_int(key, (uint64_t)i, lo, hi);
}

static double k3gen_unit(uint64_t r) { return (double)(r >> 11) * 0x1.0p-53; }

void k3gen_fill_uniform_f64(uint64_t seed, uint64_t stream, uint64_t n, double lo, double hi,
                            double* out) {
  const uint64_t key = k3gen_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i)
    out[i] = lo + (hi - lo) * k3gen_unit(k3gen_draw(key, (uint64_t)i));
}

void k3gen_fill_normal_f64(uint64_t seed, uint64_t stream, uint64_t n, double sigma, double* out) {
  const uint64_t key = k3gen_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) {
    double u1 = ((double)(k3gen_draw(key, 2 * (uint64_t)i) >> 11) + 1.0) * 0x1.0p-53;
    double u2 = k3gen_unit(k3gen_draw(key, 2 * (uint64_t)i + 1));
    out[i] = sigma * sqrt(-2.0 * log(u1)) * cos(K3GEN_TWO_PI * u2);
  }
}

/* Storage rounding of a drawn real to bf16, round-to-nearest-even.  The double is
 * first narrowed to float with round-to-odd (truncate toward zero, then set the
 * last bit if anything was discarded); float keeps 16 more bits than bf16, so the
 * second rounding (RNE on the float bits) gives the correctly rounded result
 * (Boldo and Melquiond, "Emulation of FMA and correctly rounded sums: proved
 * algorithms using rounding to odd", IEEE TC 2008). */
static uint16_t k3gen_bf16_bits(double d) {
  float f = (float)d;
  uint32_t b;
  memcpy(&b, &f, 4);
  if ((b & 0x7F800000u) == 0x7F800000u) return (uint16_t)((b >> 16) | ((b & 0xFFFFu) ? 0x40u : 0u));
  if ((double)f != d) {
    if ((b & 0x7FFFFFFFu) == 0u) return (uint16_t)(b >> 16); /* far below bf16's smallest subnormal */
    if (fabs((double)f) > fabs(d)) b -= 1; /* narrowing went away from zero: step back toward zero */
    b |= 1u;
  }
  uint32_t lsb = (b >> 16) & 1u;
  b += 0x7FFFu + lsb;
  return (uint16_t)(b >> 16);
}

void k3gen_round_bf16(uint64_t n, const double* in, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = k3gen_bf16_bits(in[i]);
}

void k3gen_round_f32(uint64_t n, const double* in, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = (float)in[i];
}

int k3gen_abi_version(void) { return 1; }

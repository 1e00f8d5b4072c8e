// k3_common.cuh -- device helpers shared by the k3moe kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/k3moe.h"

#define K3_DEVI __device__ __forceinline__

namespace k3 {

// ------------------------------------------------------------------ async global->shared copies
K3_DEVI uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// 16-byte copy, bypassing L1 (weights are streamed once)
K3_DEVI void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src));
}
// 8-byte copy
K3_DEVI void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(dst), "l"(src));
}
// 4-byte copy
K3_DEVI void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src));
}
K3_DEVI void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
K3_DEVI void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Shared-memory reads as plain C++ loads (the compiler may schedule them freely
// between the memory barriers that cp_async_wait / __syncwarp / __syncthreads are).
K3_DEVI uint32_t lds32(uint32_t a) {
  return *reinterpret_cast<const uint32_t*>(__cvta_shared_to_generic(a));
}
K3_DEVI uint2 lds64(uint32_t a) { return *reinterpret_cast<const uint2*>(__cvta_shared_to_generic(a)); }

// read-only 16-byte / 8-byte global loads for activations (small, reused: keep in L1)
K3_DEVI uint4 ldg128(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
K3_DEVI uint2 ldg64(const void* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }

// ------------------------------------------------------------------ tensor-core MMA (m16n8k16)
// D = A * B + C, A 16x16 row-major fragment (4 regs), B 16x8 col fragment (2 regs), fp32 accumulate.
// (pure register operations: not volatile, so the compiler can interleave them)
K3_DEVI void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1, const float (&c)[4]) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
        "f"(c[3]));
}
K3_DEVI void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1, const float (&c)[4]) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
        "f"(c[3]));
}

// d = a * b + c on two fp32 lanes at once (packed FMA)
K3_DEVI void ffma2(float& d0, float& d1, float a0, float a1, float b, float c0, float c1) {
  uint64_t rd;
  const uint64_t ra = ((uint64_t)__float_as_uint(a1) << 32) | __float_as_uint(a0);
  const uint64_t rb = ((uint64_t)__float_as_uint(b) << 32) | __float_as_uint(b);
  const uint64_t rc = ((uint64_t)__float_as_uint(c1) << 32) | __float_as_uint(c0);
  asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  d0 = __uint_as_float((uint32_t)rd);
  d1 = __uint_as_float((uint32_t)(rd >> 32));
}

// ------------------------------------------------------------------ MXFP4 decode
// Four packed bytes (8 E2M1 codes, low nibble first) -> four f16x2 words holding the
// exact E2M1 values; word i holds the codes of byte i (low nibble in the low half).
K3_DEVI void e2m1x8_to_f16x8(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n"
      ".reg .b8 b0, b1, b2, b3;\n"
      "mov.b32 {b0, b1, b2, b3}, %4;\n"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n"
      "}\n"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}

// E8M0 scale byte -> f32 value 2^(s-127): normal for 1..254, the subnormal 2^-127 for 0, NaN for 255.
K3_DEVI float ue8m0_to_f32(uint32_t s) {
  uint32_t bits = (s == 0u) ? 0x00400000u : ((s == 255u) ? 0x7FC00000u : (s << 23));
  return __uint_as_float(bits);
}
// Fast form used inside the GEMVs: byte k of a 4-byte word w placed in the f32
// exponent field (2 integer ops).  Equal to ue8m0_to_f32 for bytes 1..254; byte 0
// gives 0 instead of 2^-127 (a difference below 6*2^-127 per weight, far under fp32
// resolution of any sum it enters) and byte 255 gives +inf instead of NaN (the
// result is non-finite either way).
template <int K>
K3_DEVI float ue8m0_byte_to_f32(uint32_t w) {
  if constexpr (K == 3) {
    return __uint_as_float((w >> 1) & 0x7F800000u);
  } else {
    return __uint_as_float((w << (23 - 8 * K)) & 0x7F800000u);
  }
}

// ------------------------------------------------------------------ numerics
K3_DEVI float sigmoidf_(float a) { return 1.0f / (1.0f + expf(-a)); }
// SiTU-GLU, 4 tanh(g/4) sigmoid(g) * 25 tanh(u/25)
K3_DEVI float situf(float g, float u) { return 4.0f * tanhf(g * 0.25f) * sigmoidf_(g) * (25.0f * tanhf(u / 25.0f)); }

// e^x - 1 to a few ulp without cancellation near 0: the Taylor series through x^9 for
// |x| < 1/2 (truncation below 1e-9 relative), expf(x) - 1 elsewhere.
K3_DEVI float expm1_k3(float x) {
  float t = 1.0f / 362880.0f;
  t = fmaf(t, x, 1.0f / 40320.0f);
  t = fmaf(t, x, 1.0f / 5040.0f);
  t = fmaf(t, x, 1.0f / 720.0f);
  t = fmaf(t, x, 1.0f / 120.0f);
  t = fmaf(t, x, 1.0f / 24.0f);
  t = fmaf(t, x, 1.0f / 6.0f);
  t = fmaf(t, x, 0.5f);
  t = fmaf(t, x, 1.0f);
  const float small = t * x;
  return (fabsf(x) < 0.5f) ? small : expf(x) - 1.0f;
}
// SiTU-GLU from two exponentials per element pair:  with P = e^(g/2), A = P - 1 and
// B = e^(2u/25) - 1,
//   tanh(g/4) = A / (A + 2),  sigmoid(g) = P^2 / (P^2 + 1),  tanh(u/25) = B / (B + 2),
// so h = 100 * A/(A+2) * P^2/(P^2+1) * B/(B+2).  A comes from the series near g = 0 (no
// cancellation in e^(g/2) - 1) and P from expf elsewhere (no cancellation in A + 1 for
// negative g, where sigmoid(g) is tiny): a few f32 ulp everywhere until P^2 underflows
// (g < -87, |h| < 1e-36).  g is clamped to 80 and u/25 to [-40, 40], where every factor
// is already 1 (or -1) in f32; NaN passes through.
K3_DEVI float situ_fast(float g, float u) {
  g = (g > 80.0f) ? 80.0f : g;
  float v = u * 0.08f;  // 2u/25
  v = (v > 80.0f) ? 80.0f : ((v < -80.0f) ? -80.0f : v);
  const float x = 0.5f * g;
  const float A = expm1_k3(x), B = expm1_k3(v);
  const float P = (fabsf(x) < 0.5f) ? A + 1.0f : expf(x);
  const float P2 = P * P;
  return 100.0f * __fdividef(A, A + 2.0f) * __fdividef(P2, P2 + 1.0f) * __fdividef(B, B + 2.0f);
}

// 2^e as f32 for e in [-126, 127]
K3_DEVI float pow2f(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// Exponent p of a token's f16 activation row: max|z| * 2^p lies in [2^14, 2^15) (0 for an
// all-zero or non-finite row).  `maxbits` is the f32 bit pattern of max|z| over the row
// (z values are bf16, so its low 16 bits are zero).
K3_DEVI int act_exp_from_max(uint32_t maxbits) {
  const uint32_t mx = maxbits >> 16;
  int pw = 0;
  if (mx != 0u && mx < 0x7F80u) {
    const int ex = (int)(mx >> 7);               // biased exponent field of the largest |z|
    const int E2 = (ex == 0) ? -127 : ex - 127;  // floor(log2) (subnormal: below -126)
    pw = 14 - E2;
  }
  return pw;
}

K3_DEVI uint16_t f32_to_bf16_bits(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&b);
}
K3_DEVI float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// Eight bf16 values -> eight f16 values times 2^pw (two exact power-of-two factors, one
// rounding to f16): the activation operand of the f16 MMAs, from the bf16 row itself.
K3_DEVI uint4 bf16x8_to_f16x8(uint4 v, int pw) {
  const float f1 = pow2f(pw >> 1), f2 = pow2f(pw - (pw >> 1));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t r[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __half2 h = __floats2half2_rn(__uint_as_float(w[k] << 16) * f1 * f2,
                                        __uint_as_float(w[k] & 0xFFFF0000u) * f1 * f2);
    r[k] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

// ------------------------------------------------------------------ programmatic dependent launch
// Wait until the previous kernel in the stream has completed and its writes are
// visible (no-op when the kernel was launched without the programmatic attribute).
K3_DEVI void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
// Allow the next kernel in the stream to start launching.
K3_DEVI void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// ------------------------------------------------------------------ token batches
// One batch of up to MX_MAX_NB tokens routed to one expert (written by the
// permutation, read by the expert kernels): the expert's six vendor tensors, the
// batch's first sorted slot and size, and its tokens.  128 bytes.
constexpr int MX_MAX_NB = 16;
struct __align__(16) MxBatch {
  const uint8_t* w[6];  // gate_q, gate_s, up_q, up_s, down_q, down_s
  int32_t slot0, n;
  int32_t tok[MX_MAX_NB];
  int32_t pad[2];
};
static_assert(sizeof(MxBatch) == 128, "batch record is 128 bytes");

// ------------------------------------------------------------------ status word
K3_DEVI void flag_status(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

}  // namespace k3

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
K3_DEVI void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
K3_DEVI void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

K3_DEVI uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(a));
  return v;
}
K3_DEVI uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}

// read-only 16-byte / 8-byte global loads for activations (small, reused: keep in L1)
K3_DEVI uint4 ldg128(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
K3_DEVI uint2 ldg64(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.b32 {%0, %1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

// ------------------------------------------------------------------ tensor-core MMA (m16n8k16)
// D = A * B + C, A 16x16 row-major fragment (4 regs), B 16x8 col fragment (2 regs), fp32 accumulate.
K3_DEVI void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1, const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
        "f"(c[3]));
}
K3_DEVI void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1, const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
        "f"(c[3]));
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

// ------------------------------------------------------------------ numerics
K3_DEVI float sigmoidf_(float a) { return 1.0f / (1.0f + expf(-a)); }
// SiTU-GLU, 4 tanh(g/4) sigmoid(g) * 25 tanh(u/25)
K3_DEVI float situf(float g, float u) { return 4.0f * tanhf(g * 0.25f) * sigmoidf_(g) * (25.0f * tanhf(u / 25.0f)); }

K3_DEVI uint16_t f32_to_bf16_bits(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&b);
}
K3_DEVI float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// ------------------------------------------------------------------ status word
K3_DEVI void flag_status(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

}  // namespace k3

// k3_shared.cuh -- the shared experts beside the routed block (colibri PR #684, engine
// commit: "2 fused shared experts"; colibri PR #676, architecture bullets: SiTU-GLU).
//
// Two SiTU-GLU experts on the hidden width, their weights fused along the intermediate
// dimension (gate rows, then up rows of one [2 Is, H] matrix; one [H, Is] down matrix), so
// one fused expert computes the sum of both.  Three launches, on the same dense kernels as
// the latent projections (weight-streaming GEMVs below the tensor-core threshold, tcgen05
// GEMMs from it):
//   [g | u] = x . Wgu^T  (fp32, [T, 2 Is]);  h = bf16(SiTU(g, u))  ([T, Is], this file);
//   out += h . Wdn^T     (the accumulating epilogue adds to the routed block's output).
#pragma once

#include "k3_common.cuh"

namespace k3 {

// h[t][j] = bf16(SiTU(gu[t][j], gu[t][Is + j])); four elements per thread
__global__ void __launch_bounds__(256) k3_shared_glu_kernel(const float* __restrict__ gu, int T, int Is,
                                                            uint16_t* __restrict__ h) {
  grid_dep_wait();
  grid_dep_launch();
  const int q = Is / 4;
  const size_t n = (size_t)T * q;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / q), j = (int)(i % q) * 4;
    const float4 g = *reinterpret_cast<const float4*>(gu + (size_t)t * 2 * Is + j);
    const float4 u = *reinterpret_cast<const float4*>(gu + (size_t)t * 2 * Is + Is + j);
    const uint32_t lo = (uint32_t)f32_to_bf16_bits(situ_fast(g.x, u.x)) |
                        ((uint32_t)f32_to_bf16_bits(situ_fast(g.y, u.y)) << 16);
    const uint32_t hi = (uint32_t)f32_to_bf16_bits(situ_fast(g.z, u.z)) |
                        ((uint32_t)f32_to_bf16_bits(situ_fast(g.w, u.w)) << 16);
    *reinterpret_cast<uint2*>(h + (size_t)t * Is + j) = make_uint2(lo, hi);
  }
}

}  // namespace k3

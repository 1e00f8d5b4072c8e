/*
 * k3gen_cuda.cu -- device-side fill of the integer-valued synthetic tensors
 * (uniform u8 and uniform integer bytes), bit-identical to the host fill in
 * k3gen_host.c because both evaluate the same integer hash from k3gen.h.
 * Used to materialise the 896-expert MXFP4 pool (about 15.7 GB) directly in HBM.
 * Holds no LatentMoE arithmetic.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "k3gen.h"

/* One thread writes 8 consecutive bytes of one tensor of one expert.
 * Tensor `which` of expert e lives at base + e * expert_stride + offset, n bytes. */
__global__ void k3gen_pool_kernel(uint8_t* base, uint64_t expert_stride, uint64_t offset, uint64_t n,
                                  uint32_t n_experts, uint64_t seed, uint32_t which, int is_int,
                                  uint32_t lo, uint32_t hi) {
  const uint64_t words = (n + 7) / 8;
  const uint64_t total = words * n_experts;
  for (uint64_t idx = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t e = (uint32_t)(idx / words);
    const uint64_t w = idx - (uint64_t)e * words;
    const uint64_t key = k3gen_key(seed, k3gen_expert_stream(e, which));
    uint8_t* dst = base + e * expert_stride + offset + 8 * w;
    uint8_t v[8];
    if (is_int) {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = (uint8_t)k3gen_int(key, 8 * w + j, lo, hi);
    } else {
      uint64_t r = k3gen_draw(key, w);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = (uint8_t)(r >> (8 * j));
    }
    const uint64_t rem = n - 8 * w;
    if (rem >= 8 && ((uintptr_t)dst & 7) == 0) {
      uint64_t packed = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) packed |= (uint64_t)v[j] << (8 * j);
      *(uint64_t*)dst = packed;
    } else {
      for (uint64_t j = 0; j < rem && j < 8; ++j) dst[j] = v[j];
    }
  }
}

extern "C" int k3gen_cuda_fill_pool(void* base, uint64_t expert_stride, uint64_t offset, uint64_t n,
                                    uint32_t n_experts, uint64_t seed, uint32_t which, int is_int,
                                    uint32_t lo, uint32_t hi, void* stream) {
  if (!base || n == 0 || n_experts == 0) return 1;
  if (is_int && hi < lo) return 1;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int threads = 256;
  const int blocks = (sms > 0 ? sms : 132) * 8;
  k3gen_pool_kernel<<<blocks, threads, 0, (cudaStream_t)stream>>>((uint8_t*)base, expert_stride, offset, n,
                                                                   n_experts, seed, which, is_int, lo, hi);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

// k3_front.cuh -- the decode step's routing and latent down projection in one launch (one
// token): the router logits come from the kernel before it (a one-token GEMV); here one
// CTA routes the token as soon as they are complete while all the other CTAs stream the
// latent down projection, which does not depend on them.
#pragma once

#include "k3_common.cuh"
#include "k3_gemv.cuh"
#include "k3_gemv_bulk.cuh"
#include "k3_route.cuh"
#include "k3_tc.cuh"

namespace k3 {

constexpr int FR_THREADS = PERM_WARPS * 32;  // 512: the routing CTA's size, shared by all CTAs
constexpr int FR_UNR = 4;                    // 16-byte loads in flight per lane (two CTAs per SM)

struct FrontParams {
  DenseParams d;   // W0 = latent down [L, H] (z), R0 = L, act = x [1, H]; R1 = 0
  TopkParams tp;   // T = 1, logits written by the previous kernel
  PermParams pp;   // T = 1
};

__host__ __device__ constexpr int front_smem_bytes(int H, int E) {
  return (H * 4 > RouteSmem::bytes(E)) ? H * 4 : RouteSmem::bytes(E);
}

// CTA 0 routes: it waits for the previous kernel (the router logits; programmatic
// dependent launch), then runs the one-token routing with all its threads (top-k,
// permutation, expert batch records).  CTAs 1.. stream the latent rows without waiting for
// it (x and the weights are inputs of the layer): each owns a slice of the rows, which its
// warps take from a shared-memory counter; a row is read with 16-byte non-caching loads
// into registers (the next row's first loads issued before the current one is reduced) and
// multiplied with x held as f32 in shared memory.  The kernel ends after the routing CTA,
// so it also ends after the router kernel.
__global__ void __launch_bounds__(FR_THREADS, 2) k3_front_kernel(FrontParams f) {
  extern __shared__ __align__(16) uint8_t fsm[];
  __shared__ int next_row;
  const DenseParams& p = f.d;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = p.K, KV = K / 8;
  const int L = p.R0;
  if (blockIdx.x == 0) {
    // ------------------------------------------------------------ routing CTA
    grid_dep_wait();
    grid_dep_launch();
    route_one_token_block(f.tp, f.pp, fsm, lane, warp);
    return;
  }
  // -------------------------------------------------------------- streaming CTAs
  float* xs = reinterpret_cast<float*>(fsm);  // x as f32, H values
  const int G = gridDim.x - 1, b = blockIdx.x - 1;
  const int r0 = (int)(((long long)L * b) / G), n = (int)(((long long)L * (b + 1)) / G) - r0;
  auto row_of = [&](int i) { return r0 + i; };
  auto row_ptr = [&](int r) -> const uint4* { return reinterpret_cast<const uint4*>(p.W0 + (size_t)r * K); };
  if (threadIdx.x == 0) next_row = 0;
  for (int v = threadIdx.x; v < K / 2; v += blockDim.x) {
    const uint32_t xx = __ldg(reinterpret_cast<const uint32_t*>(p.act) + v);
    reinterpret_cast<float2*>(xs)[v] = make_float2(__uint_as_float(xx << 16), __uint_as_float(xx & 0xFFFF0000u));
  }
  __syncthreads();
  grid_dep_launch();
  auto grab = [&]() {
    int i = 0;
    if (lane == 0) i = atomicAdd(&next_row, 1);
    return __shfl_sync(0xffffffffu, i, 0);
  };
  uint4 w[FR_UNR];
  auto load_chunk = [&](const uint4* wv, int vb) {
#pragma unroll
    for (int u = 0; u < FR_UNR; ++u) {
      const int v = vb + lane + 32 * u;
      w[u] = (v < KV) ? ldg_stream(wv + v) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  int i = grab();
  if (i < n) load_chunk(row_ptr(row_of(i)), 0);
  while (i < n) {
    const int r = row_of(i);
    const int inext = grab();
    const uint4* wv = row_ptr(r);
    const uint4* wnext = (inext < n) ? row_ptr(row_of(inext)) : nullptr;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    for (int v0 = 0; v0 < KV; v0 += 32 * FR_UNR) {
      uint4 cur[FR_UNR];
#pragma unroll
      for (int u = 0; u < FR_UNR; ++u) cur[u] = w[u];
      const int vn = v0 + 32 * FR_UNR;
      if (vn < KV) load_chunk(wv, vn);
      else if (wnext) load_chunk(wnext, 0);
#pragma unroll
      for (int u = 0; u < FR_UNR; ++u) {
        const int v = v0 + lane + 32 * u;
        if (v < KV) {
          const float4 xa = reinterpret_cast<const float4*>(xs)[2 * v];
          const float4 xb = reinterpret_cast<const float4*>(xs)[2 * v + 1];
          a0 = fmaf(__uint_as_float(cur[u].x << 16), xa.x, a0);
          a1 = fmaf(__uint_as_float(cur[u].x & 0xFFFF0000u), xa.y, a1);
          a2 = fmaf(__uint_as_float(cur[u].y << 16), xa.z, a2);
          a3 = fmaf(__uint_as_float(cur[u].y & 0xFFFF0000u), xa.w, a3);
          a0 = fmaf(__uint_as_float(cur[u].z << 16), xb.x, a0);
          a1 = fmaf(__uint_as_float(cur[u].z & 0xFFFF0000u), xb.y, a1);
          a2 = fmaf(__uint_as_float(cur[u].w << 16), xb.z, a2);
          a3 = fmaf(__uint_as_float(cur[u].w & 0xFFFF0000u), xb.w, a3);
        }
      }
    }
    float sum = (a0 + a1) + (a2 + a3);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0) {
      const uint16_t zb = f32_to_bf16_bits(sum);
      p.out1[r] = zb;
      atomicMax(p.zmax, __float_as_uint(fabsf(bf16_bits_to_f32(zb))));
    }
    i = inext;
  }
}

}  // namespace k3

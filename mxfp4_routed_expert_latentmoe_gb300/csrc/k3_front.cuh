// k3_front.cuh -- the decode step's front in one launch (one token): router logits and
// the latent down projection streamed together, with the routing run as soon as the
// logits are complete, while the latent rows are still streaming.
#pragma once

#include "k3_common.cuh"
#include "k3_gemv.cuh"
#include "k3_gemv_bulk.cuh"
#include "k3_route.cuh"

namespace k3 {

// cnt[0]: router rows done, cnt[1]: latent rows done (zero on entry: they live in the
// status region that every forward clears)
struct FrontParams {
  DenseParams d;   // W0 = router weight [E, H] (logits), W1 = latent down [L, H] (z), act = x [1, H]
  TopkParams tp;   // T = 1
  PermParams pp;   // T = 1
  Z16Params zp;    // T = 1
  uint32_t* cnt;
};

// Every CTA owns a slice of the router rows and a slice of the latent rows; its warps take
// the slice's rows in that order from a shared-memory counter (the router rows of all CTAs
// are therefore done early).  A row is read with 16-byte non-caching loads into registers
// (the next row's first loads issued before the current one is reduced) and multiplied
// with x held as f32 in shared memory.  After storing a row's result, lane 0 publishes it
// (fence, then a count in global memory); the warp that completes the last router row
// runs top-k, the permutation and the expert batch records for the token, and the warp
// that completes the last latent row converts z to the f16 operand of the expert GEMVs.
// A warp busy routing leaves its CTA's remaining rows to the other warps.  No thread waits
// on another: the last-arriving warp of each phase does the dependent work.
__global__ void __launch_bounds__(D1_WARPS * 32, 2) k3_front1_kernel(FrontParams f) {
  extern __shared__ __align__(16) float xs[];  // x as f32, H values
  __shared__ TopkScratch S;
  __shared__ int next_row;
  const DenseParams& p = f.d;
  const int lane = threadIdx.x & 31;
  const int K = p.K, KV = K / 8;
  const int E = p.R0, L = p.R1, G = gridDim.x, b = blockIdx.x;
  const int e0 = (int)(((long long)E * b) / G), e1 = (int)(((long long)E * (b + 1)) / G);
  const int z0 = (int)(((long long)L * b) / G), z1 = (int)(((long long)L * (b + 1)) / G);
  const int ne = e1 - e0, n = ne + (z1 - z0);
  // i-th row of this CTA: router rows first (global row index, router rows before latent rows)
  auto row_of = [&](int i) { return (i < ne) ? e0 + i : E + z0 + (i - ne); };
  auto row_ptr = [&](int r) -> const uint4* {
    return reinterpret_cast<const uint4*>((r < E) ? p.W0 + (size_t)r * K : p.W1 + (size_t)(r - E) * K);
  };
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
  uint4 w[D1_UNR];
  auto load_chunk = [&](const uint4* wv, int vb) {
#pragma unroll
    for (int u = 0; u < D1_UNR; ++u) {
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
    for (int v0 = 0; v0 < KV; v0 += 32 * D1_UNR) {
      uint4 cur[D1_UNR];
#pragma unroll
      for (int u = 0; u < D1_UNR; ++u) cur[u] = w[u];
      const int vn = v0 + 32 * D1_UNR;
      if (vn < KV) load_chunk(wv, vn);
      else if (wnext) load_chunk(wnext, 0);
#pragma unroll
      for (int u = 0; u < D1_UNR; ++u) {
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
    int last = 0;  // 1: this warp finished the last router row, 2: the last latent row
    if (lane == 0) {
      if (r < E) {
        p.out0[r] = sum;
        __threadfence();
        last = (atomicAdd(f.cnt, 1u) == (uint32_t)E - 1u) ? 1 : 0;
      } else {
        const uint16_t zb = f32_to_bf16_bits(sum);
        p.out1[r - E] = zb;
        atomicMax(p.zmax, __float_as_uint(fabsf(bf16_bits_to_f32(zb))));
        __threadfence();
        last = (atomicAdd(f.cnt + 1, 1u) == (uint32_t)L - 1u) ? 2 : 0;
      }
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last == 1) {  // every router logit is written and visible: route the token
      __threadfence();
      topk_token(f.tp, 0, nullptr, nullptr, S, lane);
      permute_warp(f.pp, lane);
    } else if (last == 2) {  // z and its max are complete: the f16 operand of the expert GEMVs
      __threadfence();
      z16_token(f.zp, 0, lane);
    }
    i = inext;
  }
}

}  // namespace k3

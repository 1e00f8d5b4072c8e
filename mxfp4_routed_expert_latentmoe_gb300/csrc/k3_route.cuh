// k3_route.cuh -- router top-k, chunk expert-union permutation, activation prep,
// combine + RMSNorm, and the MXFP4 dequant check kernel.
#pragma once

#include "k3_common.cuh"

namespace k3 {

// ============================================================================ top-k
// One warp per token.  Sigmoid scores and biased scores in fp32 from fp32 logits;
// the K + REFINE_EXTRA best candidates by biased score are picked (ties to the lower
// id); every candidate whose biased score lies within `tau` of a neighbour, in a
// near-tie cluster that reaches the top K + 1, gets its logit recomputed exactly in
// fp64 from the bf16 inputs; candidates are then ranked on the refined values.
constexpr int TOPK_WARPS = 4;
constexpr int REFINE_EXTRA = 8;
constexpr int TOPK_MAX_P = 64 + REFINE_EXTRA;
constexpr int TOPK_MAX_E = 2048;

struct TopkParams {
  const float* logits;  // [T, E]
  const float* bias;    // [E]
  const uint16_t* x;    // [T, H]
  const uint16_t* wr;   // [E, H]
  int T, E, K, H;
  float tau;
  int32_t* ids;  // [T, K]
  float* w;      // [T, K]
  int32_t* ids_out;
  float* w_out;
  uint32_t* status;
};

__global__ void __launch_bounds__(TOPK_WARPS * 32) k3_topk_kernel(TopkParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = blockIdx.x * TOPK_WARPS + warp;
  if (t >= p.T) return;
  float* sb = reinterpret_cast<float*>(smem) + warp * (2 * p.E);  // biased scores (consumed)
  float* sr = sb + p.E;                                            // raw scores
  __shared__ float cv[TOPK_WARPS][TOPK_MAX_P];
  __shared__ float cs[TOPK_WARPS][TOPK_MAX_P];
  __shared__ int ci[TOPK_WARPS][TOPK_MAX_P];
  __shared__ double rv[TOPK_WARPS][TOPK_MAX_P];
  __shared__ double rs[TOPK_WARPS][TOPK_MAX_P];
  __shared__ int rf[TOPK_WARPS][TOPK_MAX_P];

  // sb: NaN marks an expert already taken; a NaN score ranks last (-inf)
  for (int e = lane; e < p.E; e += 32) {
    const float s = sigmoidf_(p.logits[(size_t)t * p.E + e]);
    const float v = s + p.bias[e];
    sr[e] = s;
    sb[e] = (v == v) ? v : -INFINITY;
  }
  __syncwarp();
  const int P = min(p.E, p.K + REFINE_EXTRA);
  for (int k = 0; k < P; ++k) {
    float best = -INFINITY;
    int bid = 0x7fffffff;
    for (int e = lane; e < p.E; e += 32) {
      const float v = sb[e];
      if (v != v) continue;
      if (v > best || (v == best && e < bid)) {
        best = v;
        bid = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bid, off);
      if (ov > best || (ov == best && oi < bid)) {
        best = ov;
        bid = oi;
      }
    }
    if (lane == 0) {
      cv[warp][k] = best;
      ci[warp][k] = bid;
      cs[warp][k] = sr[bid];
      sb[bid] = __int_as_float(0x7fc00000);
    }
    __syncwarp();
  }
  // near-tie clusters: consecutive candidates closer than tau are linked; a cluster
  // is refined when it starts at or before position K (it can change the top K or
  // their order)
  if (lane == 0) {
    int start = 0;
    for (int k = 0; k < P; ++k) {
      const bool linked_prev = k > 0 && (cv[warp][k - 1] - cv[warp][k]) < p.tau;
      const bool linked_next = k + 1 < P && (cv[warp][k] - cv[warp][k + 1]) < p.tau;
      if (!linked_prev) start = k;
      rf[warp][k] = (linked_prev || linked_next) && start <= p.K;
    }
    if (P < p.E && rf[warp][P - 1]) flag_status(p.status, K3MOE_DEV_TIE_WINDOW);
  }
  __syncwarp();
  for (int k = 0; k < P; ++k) {
    if (!rf[warp][k]) continue;  // warp-uniform
    const int e = ci[warp][k];
    double acc = 0.0;
    const uint16_t* xr = p.x + (size_t)t * p.H;
    const uint16_t* wrr = p.wr + (size_t)e * p.H;
    for (int h = lane; h < p.H; h += 32)
      acc = fma((double)bf16_bits_to_f32(xr[h]), (double)bf16_bits_to_f32(wrr[h]), acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      const double s = 1.0 / (1.0 + exp(-acc));
      rs[warp][k] = s;
      rv[warp][k] = s + (double)p.bias[e];
    }
    __syncwarp();
  }
  if (lane == 0) {
    // rank the P candidates on (refined value when refined, else the fp32 value) desc, id asc
    for (int k = 0; k < P; ++k) {
      if (!rf[warp][k]) {
        rv[warp][k] = (double)cv[warp][k];
        rs[warp][k] = (double)cs[warp][k];
      }
    }
    for (int a = 0; a < p.K; ++a) {
      int b = a;
      for (int c = a + 1; c < P; ++c) {
        const double vc = rv[warp][c], vb = rv[warp][b];
        if (vc > vb || (vc == vb && ci[warp][c] < ci[warp][b])) b = c;
      }
      if (b != a) {
        double tv = rv[warp][a]; rv[warp][a] = rv[warp][b]; rv[warp][b] = tv;
        double ts = rs[warp][a]; rs[warp][a] = rs[warp][b]; rs[warp][b] = ts;
        int ti = ci[warp][a]; ci[warp][a] = ci[warp][b]; ci[warp][b] = ti;
      }
    }
    float sum = 0.f;
    for (int k = 0; k < p.K; ++k) sum += (float)rs[warp][k];
    for (int k = 0; k < p.K; ++k) {
      const int id = ci[warp][k];
      const float wk = (float)rs[warp][k] / sum;
      p.ids[(size_t)t * p.K + k] = id;
      p.w[(size_t)t * p.K + k] = wk;
      if (p.ids_out) p.ids_out[(size_t)t * p.K + k] = id;
      if (p.w_out) p.w_out[(size_t)t * p.K + k] = wk;
    }
  }
}

// ============================================================================ permutation
// Single CTA stable counting sort of the T*K routed slots by expert (the chunk's
// expert union with per-expert position lists).  Each warp owns a contiguous range
// of slots and a private histogram; positions are handed out in slot order inside
// a warp (warp-synchronous ranking with __match_any_sync) and in warp order across
// warps, so the result is the stable sort by (expert, t*K + k).
constexpr int PERM_WARPS = 16;

struct PermParams {
  const int32_t* ids;  // [T*K], or null: every slot routes to fixed_expert
  int fixed_expert;
  int T, K, E, NB;
  int32_t* counts;     // [E]
  int32_t* offsets;    // [E+1]
  int32_t* slot_of;    // [T*K] sorted slot -> flat index t*K+k
  int32_t* slot_tok;   // [T*K] sorted slot -> token
  int32_t* inv;        // [T*K] flat index -> sorted slot
  int32_t* uniq;       // [E]
  int32_t* n_uniq;     // [1]
  int32_t* nb_prefix;  // [E+1] over unique experts: prefix of ceil(count/NB)
  uint32_t* status;
};

// exclusive scan of 4 values per thread over a 512-thread block (values in order
// thread 0 v0..v3, thread 1 v0..v3, ...); returns the block total
K3_DEVI int block_scan4(int (&v)[4], int* wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int loc = v[0] + v[1] + v[2] + v[3];
  int inc = loc;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int x = (lane < PERM_WARPS) ? wsum[lane] : 0;
    int xi = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, xi, off);
      if (lane >= off) xi += o;
    }
    if (lane < PERM_WARPS) wsum[lane] = xi - x;  // exclusive warp offsets
    if (lane == PERM_WARPS - 1) wsum[PERM_WARPS] = xi;
  }
  __syncthreads();
  int run = wsum[warp] + inc - loc;
  const int total = wsum[PERM_WARPS];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int x = v[q];
    v[q] = run;
    run += x;
  }
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(PERM_WARPS * 32) k3_permute_kernel(PermParams p) {
  extern __shared__ __align__(16) int32_t hist[];  // [PERM_WARPS][E]
  __shared__ int wsum[PERM_WARPS + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = p.T * p.K;
  const int chunk = (n + PERM_WARPS - 1) / PERM_WARPS;
  const int b0 = min(n, warp * chunk), b1 = min(n, b0 + chunk);

  for (int i = threadIdx.x; i < PERM_WARPS * p.E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (int i = b0 + lane; i < b1; i += 32) {
    int e = p.ids ? p.ids[i] : p.fixed_expert;
    if (e < 0 || e >= p.E) {
      flag_status(p.status, K3MOE_DEV_BAD_ID);
      e = min(max(e, 0), p.E - 1);
    }
    atomicAdd(&hist[warp * p.E + e], 1);
  }
  __syncthreads();
  // per expert: warp-major running offsets, and the expert's count
  int cnt[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e = threadIdx.x * 4 + q;
    int run = 0;
    if (e < p.E) {
      for (int w = 0; w < PERM_WARPS; ++w) {
        const int c = hist[w * p.E + e];
        hist[w * p.E + e] = run;
        run += c;
      }
      p.counts[e] = run;
    }
    cnt[q] = run;
  }
  int off[4] = {cnt[0], cnt[1], cnt[2], cnt[3]};
  const int tot = block_scan4(off, wsum);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e = threadIdx.x * 4 + q;
    if (e < p.E) {
      p.offsets[e] = off[q];
      for (int w = 0; w < PERM_WARPS; ++w) hist[w * p.E + e] += off[q];
    }
  }
  if (threadIdx.x == 0) p.offsets[p.E] = tot;
  __syncthreads();
  // stable placement
  for (int base = b0; base < b1; base += 32) {
    const int i = base + lane;
    const bool valid = i < b1;
    int e = -1;
    if (valid) {
      e = p.ids ? p.ids[i] : p.fixed_expert;
      e = min(max(e, 0), p.E - 1);
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int leader = __ffs(peers) - 1;
    int pos = 0;
    if (valid) {
      pos = hist[warp * p.E + e] + rank;
      p.slot_of[pos] = i;
      p.slot_tok[pos] = i / p.K;
      p.inv[i] = pos;
    }
    __syncwarp();
    if (valid && lane == leader) hist[warp * p.E + e] += __popc(peers);
    __syncwarp();
  }
  // unique experts (ascending) and their token-batch prefix
  int flag[4], nbv[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) flag[q] = cnt[q] > 0 ? 1 : 0;
  const int nu = block_scan4(flag, wsum);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e = threadIdx.x * 4 + q;
    nbv[q] = 0;
    if (e < p.E && cnt[q] > 0) p.uniq[flag[q]] = e;
  }
  if (threadIdx.x == 0) *p.n_uniq = nu;
  __syncthreads();
  // nb over unique experts in order: thread handles unique indices 4*tid .. 4*tid+3
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int u = threadIdx.x * 4 + q;
    nbv[q] = (u < nu) ? (p.counts[p.uniq[u]] + p.NB - 1) / p.NB : 0;
  }
  const int nbt = block_scan4(nbv, wsum);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int u = threadIdx.x * 4 + q;
    if (u < nu) p.nb_prefix[u] = nbv[q];
  }
  if (threadIdx.x == 0) p.nb_prefix[nu] = nbt;
}

// ============================================================================ activation prep
// z [T, L] bf16 -> z16 [T, L] f16 = z * 2^p with p chosen so max|z_t| * 2^p lies in
// [2^14, 2^15) (exact power-of-two scaling; keeps bf16 values exact in f16).
struct Z16Params {
  const uint16_t* z;
  int T, L;
  __half* z16;
  int32_t* pow2;
};

__global__ void k3_z16_kernel(Z16Params p) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= p.T) return;
  const uint16_t* zr = p.z + (size_t)t * p.L;
  uint32_t mx = 0;
  for (int c = lane; c < p.L; c += 32) mx = max(mx, (uint32_t)(zr[c] & 0x7FFFu));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  int pw = 0;
  if (mx != 0u && mx < 0x7F80u) {
    const int ex = (int)(mx >> 7);  // biased exponent field of the largest |z|
    const int E2 = (ex == 0) ? -127 : ex - 127;  // floor(log2) (subnormal: below -126)
    pw = 14 - E2;
  }
  if (lane == 0) p.pow2[t] = pw;
  __half* o = p.z16 + (size_t)t * p.L;
  for (int c = lane; c < p.L; c += 32) o[c] = __float2half_rn(scalbnf(bf16_bits_to_f32(zr[c]), pw));
}

// ============================================================================ combine + RMSNorm
struct CombineParams {
  const float* o;      // [T*K slots, L] expert outputs in sorted-slot order
  const int32_t* inv;  // [T*K] flat (t, k) -> sorted slot
  const float* w;      // [T, K]
  const float* gamma;  // [L]
  int T, K, L;
  float eps;
  float* y;            // [T, L] f32 combined
  uint16_t* yhat;      // [T, L] bf16
};

constexpr int COMB_THREADS = 256;

__global__ void __launch_bounds__(COMB_THREADS) k3_combine_norm_kernel(CombineParams p) {
  extern __shared__ __align__(16) float ybuf[];  // [L]
  __shared__ float part[COMB_THREADS / 32];
  const int t = blockIdx.x;
  float ss = 0.f;
  for (int c = threadIdx.x; c < p.L; c += blockDim.x) {
    float y = 0.f;
    for (int k = 0; k < p.K; ++k) {
      const int slot = p.inv[(size_t)t * p.K + k];
      y = fmaf(p.w[(size_t)t * p.K + k], p.o[(size_t)slot * p.L + c], y);
    }
    ybuf[c] = y;
    ss = fmaf(y, y, ss);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += part[w];
  const float r = 1.0f / sqrtf(tot / (float)p.L + p.eps);
  for (int c = threadIdx.x; c < p.L; c += blockDim.x) {
    const float y = ybuf[c];
    p.y[(size_t)t * p.L + c] = y;
    p.yhat[(size_t)t * p.L + c] = f32_to_bf16_bits(p.gamma[c] * (y * r));
  }
}

// ============================================================================ dequant check
__global__ void k3_dequant_kernel(const uint8_t* q, const uint8_t* s, int O, int I, float* out) {
  const size_t words = (size_t)O * (I / 8);  // 4 packed bytes = 8 values per thread
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < words; i += (size_t)gridDim.x * blockDim.x) {
    const size_t o = i / (I / 8), c8 = i - o * (I / 8);
    const uint32_t w = *reinterpret_cast<const uint32_t*>(q + o * (I / 2) + c8 * 4);
    const float sc = ue8m0_to_f32(s[o * (I / 32) + (c8 * 8) / 32]);
    uint32_t h[4];
    e2m1x8_to_f16x8(w, h);
    float v[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[k]));
      v[2 * k] = f.x * sc;
      v[2 * k + 1] = f.y * sc;
    }
    float4* dst = reinterpret_cast<float4*>(out + o * I + c8 * 8);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

}  // namespace k3

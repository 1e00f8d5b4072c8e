// k3_gemv.cuh -- weight-streaming "skinny" kernels for small token counts per weight
// matrix (decode, chunked prefill).  Every weight byte of a selected matrix is read
// from HBM once per call (per n-batch of tokens); tokens ride along as the N
// dimension of m16n8k16 tensor-core MMAs.
//
// Work decomposition (both kernels):
//   * item  = 16 consecutive output rows of one matrix x one batch of up to NB tokens;
//   * the reduction dimension K is split across the warps of a CTA (a fixed slice
//     per warp); every warp streams its slice of the item's rows into its own
//     shared-memory ring with cp.async (16-byte copies, STAGES deep), so the copies
//     of later items are in flight while earlier ones are reduced;
//   * per-warp partial sums meet in shared memory and are added in warp order
//     (deterministic), then the epilogue applies the output transform.
//
// MXFP4 kernel (k3_mx_gemv): each 32-element scale group is decoded in registers
// with cvt.rn.f16x2.e2m1x2 (exact E2M1 values), multiplied on the tensor core with
// f16 activations into a fresh fp32 fragment, and folded into the fp32 accumulator
// with the group's power-of-two scale (exact), so any scale byte is supported.
// Activations enter as f16 pre-scaled by a power of two (exact for bf16 inputs in
// range): z by a per-token 2^p that puts max|z| in [2^14, 2^15), h by 2^8.
#pragma once

#include "k3_common.cuh"

namespace k3 {

// ============================================================================ MXFP4 GEMV
constexpr int MX_GPW = 8;                      // 32-element groups per warp slice (256 elements)
constexpr int MX_ROWS = 16;                    // rows per item
constexpr int MX_Q_BYTES = MX_ROWS * MX_GPW * 16;  // packed bytes per matrix per stage (2048)
constexpr int MX_S_BYTES = MX_ROWS * MX_GPW;       // scale bytes per matrix per stage (128)
constexpr int MX_MAX_THREADS = 512;

enum { MX_GATEUP = 0, MX_DOWN = 1 };

struct MxGemvParams {
  const uint8_t* const* q0;  // gate (GATEUP) / down (DOWN) packed tables
  const uint8_t* const* s0;
  const uint8_t* const* q1;  // up (GATEUP)
  const uint8_t* const* s1;
  int R;  // rows per matrix
  int K;  // reduction length
  const int32_t* uniq;
  const int32_t* n_uniq;
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* nb_prefix;  // [n_uniq + 1] prefix of per-expert token batches
  const int32_t* slot_tok;   // sorted slot -> token
  const __half* act;         // GATEUP: z16 [T, K]; DOWN: h16 [slots, K]
  const int32_t* act_pow;    // GATEUP: per-token exponent p (z16 = z * 2^p)
  void* out;                 // GATEUP: h16 [slots, R] (h * 2^8); DOWN: o f32 [slots, R]
};

template <int M, int STAGES>
struct MxLayout {
  static constexpr int STAGE_BYTES = M * (MX_Q_BYTES + MX_S_BYTES);
  static constexpr int WARP_BYTES = STAGES * STAGE_BYTES;
};

struct MxItem {
  int e, row0, slot0, n;
};

K3_DEVI void mx_item(const MxGemvParams& p, int tiles, int NB, int i, MxItem& it) {
  const int gb = i / tiles;
  const int tile = i - gb * tiles;
  int lo = 0, hi = *p.n_uniq;  // nb_prefix[lo] <= gb < nb_prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.nb_prefix[mid] <= gb) lo = mid;
    else hi = mid;
  }
  const int e = p.uniq[lo];
  const int b = gb - p.nb_prefix[lo];
  it.e = e;
  it.row0 = tile * MX_ROWS;
  it.slot0 = p.offsets[e] + b * NB;
  it.n = min(NB, p.counts[e] - b * NB);
}

template <int M, int STAGES>
K3_DEVI void mx_issue(const MxGemvParams& p, const MxItem& it, int warp, int lane, int ngroups, uint32_t stage) {
  const size_t qrow = (size_t)p.K / 2, srow = (size_t)p.K / 32;
  const bool sc_async = (p.K % 256) == 0;
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const uint8_t* q = (m == 0 ? p.q0 : p.q1)[it.e];
    const uint8_t* s = (m == 0 ? p.s0 : p.s1)[it.e];
    const uint32_t sq = stage + m * (MX_Q_BYTES + MX_S_BYTES);
    const uint32_t ss = sq + MX_Q_BYTES;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = lane + 32 * i;
      const int r = c >> 3, j = c & 7;
      if (j < ngroups) {
        const int row = min(it.row0 + r, p.R - 1);
        cp_async16(sq + r * 128 + ((j ^ (r & 7)) << 4), q + (size_t)row * qrow + (size_t)warp * 128 + j * 16);
      }
    }
    if (lane < MX_ROWS) {
      const int row = min(it.row0 + lane, p.R - 1);
      const uint8_t* src = s + (size_t)row * srow + (size_t)warp * MX_GPW;
      if (sc_async) {
        cp_async8(ss + lane * 8, src);
      } else {  // partial slice or unaligned scale rows: plain byte copies (small shapes only)
        uint8_t* dst = (uint8_t*)__cvta_shared_to_generic(ss + lane * 8);
        for (int j = 0; j < MX_GPW; ++j) dst[j] = (j < ngroups) ? src[j] : (uint8_t)127;
      }
    }
  }
}

template <int MODE, int NBLK, int STAGES>
__global__ void __launch_bounds__(MX_MAX_THREADS) k3_mx_gemv_kernel(MxGemvParams p) {
  constexpr int M = (MODE == MX_GATEUP) ? 2 : 1;
  constexpr int NB = 8 * NBLK;
  using Lay = MxLayout<M, STAGES>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int ngroups = min(MX_GPW, p.K / 32 - warp * MX_GPW);
  const uint32_t wbase = smem_u32(smem) + warp * Lay::WARP_BYTES;
  float* red = reinterpret_cast<float*>(smem + nwarps * Lay::WARP_BYTES);

  const int tiles = p.R / MX_ROWS;
  const int total = tiles * p.nb_prefix[*p.n_uniq];
  const int n_mine = (total > (int)blockIdx.x) ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  // prologue
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < n_mine) {
      MxItem it;
      mx_item(p, tiles, NB, blockIdx.x + s * gridDim.x, it);
      mx_issue<M, STAGES>(p, it, warp, lane, ngroups, wbase + s * Lay::STAGE_BYTES);
    }
    cp_async_commit();
  }

  for (int s = 0; s < n_mine; ++s) {
    {
      const int sn = s + STAGES - 1;
      if (sn < n_mine) {
        MxItem itn;
        mx_item(p, tiles, NB, blockIdx.x + sn * gridDim.x, itn);
        mx_issue<M, STAGES>(p, itn, warp, lane, ngroups, wbase + (sn % STAGES) * Lay::STAGE_BYTES);
      }
      cp_async_commit();
    }
    MxItem it;
    mx_item(p, tiles, NB, blockIdx.x + s * gridDim.x, it);
    cp_async_wait<STAGES - 1>();
    __syncwarp();

    const uint32_t stage = wbase + (s % STAGES) * Lay::STAGE_BYTES;
    float acc[M][NBLK][4];
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
      for (int nb = 0; nb < NBLK; ++nb)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[m][nb][q] = 0.f;

    if (ngroups > 0) {
      // activation pointers of this lane's token column in every 8-token block
      const __half* bptr[NBLK];
      bool bval[NBLK];
#pragma unroll
      for (int nb = 0; nb < NBLK; ++nb) {
        const int col = nb * 8 + g;
        bval[nb] = col < it.n;
        const int slot = it.slot0 + (bval[nb] ? col : 0);
        const int row = (MODE == MX_GATEUP) ? p.slot_tok[slot] : slot;
        bptr[nb] = p.act + (size_t)row * p.K + warp * 256 + 8 * t;
      }
      uint2 sc_lo[M], sc_hi[M];
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const uint32_t ss = stage + m * (MX_Q_BYTES + MX_S_BYTES) + MX_Q_BYTES;
        sc_lo[m] = lds64(ss + g * 8);
        sc_hi[m] = lds64(ss + (g + 8) * 8);
      }
#pragma unroll
      for (int j = 0; j < MX_GPW; ++j) {
        if (j < ngroups) {
          uint32_t a0[M][4], a1[M][4];
          float slo[M], shi[M];
#pragma unroll
          for (int m = 0; m < M; ++m) {
            const uint32_t sq = stage + m * (MX_Q_BYTES + MX_S_BYTES);
            const uint32_t off = ((j ^ g) << 4) + 4 * t;
            const uint32_t wlo = lds32(sq + g * 128 + off);
            const uint32_t whi = lds32(sq + (g + 8) * 128 + off);
            uint32_t plo[4], phi[4];
            e2m1x8_to_f16x8(wlo, plo);
            e2m1x8_to_f16x8(whi, phi);
            // K order inside the group: this thread's 8 elements 8t..8t+7 feed
            // MMA 0 slots {2t,2t+1 | 2t+8,2t+9} = elements {8t,8t+1 | 8t+2,8t+3} and
            // MMA 1 the same slots with elements {8t+4,8t+5 | 8t+6,8t+7}
            a0[m][0] = plo[0]; a0[m][1] = phi[0]; a0[m][2] = plo[1]; a0[m][3] = phi[1];
            a1[m][0] = plo[2]; a1[m][1] = phi[2]; a1[m][2] = plo[3]; a1[m][3] = phi[3];
            const uint32_t blo = (j < 4) ? sc_lo[m].x : sc_lo[m].y;
            const uint32_t bhi = (j < 4) ? sc_hi[m].x : sc_hi[m].y;
            slo[m] = ue8m0_to_f32((blo >> (8 * (j & 3))) & 0xFFu);
            shi[m] = ue8m0_to_f32((bhi >> (8 * (j & 3))) & 0xFFu);
          }
#pragma unroll
          for (int nb = 0; nb < NBLK; ++nb) {
            if (nb * 8 < it.n) {
              uint4 b = make_uint4(0u, 0u, 0u, 0u);
              if (bval[nb]) b = ldg128(bptr[nb] + 32 * j);
#pragma unroll
              for (int m = 0; m < M; ++m) {
                const float z4[4] = {0.f, 0.f, 0.f, 0.f};
                float d[4];
                mma_f16(d, a0[m], b.x, b.y, z4);
                mma_f16(d, a1[m], b.z, b.w, d);
                acc[m][nb][0] = fmaf(d[0], slo[m], acc[m][nb][0]);
                acc[m][nb][1] = fmaf(d[1], slo[m], acc[m][nb][1]);
                acc[m][nb][2] = fmaf(d[2], shi[m], acc[m][nb][2]);
                acc[m][nb][3] = fmaf(d[3], shi[m], acc[m][nb][3]);
              }
            }
          }
        }
      }
    }
    __syncwarp();
    // per-warp partials -> shared memory: red[warp][m][nb][row 16][col 8]
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
      for (int nb = 0; nb < NBLK; ++nb) {
        float* r = red + ((warp * M + m) * NBLK + nb) * 128;
        *reinterpret_cast<float2*>(r + g * 8 + 2 * t) = make_float2(acc[m][nb][0], acc[m][nb][1]);
        *reinterpret_cast<float2*>(r + (g + 8) * 8 + 2 * t) = make_float2(acc[m][nb][2], acc[m][nb][3]);
      }
    __syncthreads();
    for (int idx = threadIdx.x; idx < MX_ROWS * it.n; idx += blockDim.x) {
      const int row = idx & 15, col = idx >> 4, nb = col >> 3, cc = col & 7;
      float v[M];
#pragma unroll
      for (int m = 0; m < M; ++m) {
        float sum = 0.f;
        for (int w = 0; w < nwarps; ++w) sum += red[((w * M + m) * NBLK + nb) * 128 + row * 8 + cc];
        v[m] = sum;
      }
      const int slot = it.slot0 + col;
      if (MODE == MX_GATEUP) {
        const int pw = p.act_pow[p.slot_tok[slot]];
        const float gg = scalbnf(v[0], -pw), uu = scalbnf(v[M - 1], -pw);
        const float h = __uint_as_float((uint32_t)f32_to_bf16_bits(situf(gg, uu)) << 16);  // bf16 rounding
        reinterpret_cast<__half*>(p.out)[(size_t)slot * p.R + it.row0 + row] = __float2half_rn(h * 256.0f);
      } else {
        reinterpret_cast<float*>(p.out)[(size_t)slot * p.R + it.row0 + row] = v[0] * (1.0f / 256.0f);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
}

// ============================================================================ bf16 GEMV
constexpr int DN_CHUNK = 64;  // elements per row per stage
constexpr int DN_WARPS = 8;
constexpr int DN_STAGE_BYTES = 16 * DN_CHUNK * 2;  // 2048

enum { DN_PROJ = 0, DN_PLAIN = 1 };

struct DenseParams {
  const uint16_t* W0;
  int R0;
  const uint16_t* W1;
  int R1;
  int K;
  const uint16_t* act;  // [T, K] bf16
  int T;
  float* out0;      // PROJ: logits [T, R0]; PLAIN: out [T, R0]
  uint16_t* out1;   // PROJ: z [T, R1] bf16
  uint32_t* zmax;   // PROJ: per-token max |z| (f32 bits)
};

// smem row layout: 16-byte chunk j of row r sits at position j ^ (2 * (r & 3)); with the
// per-thread 8-byte reads of an m16n8k16 fragment this keeps both half-warps conflict-free
K3_DEVI uint32_t dn_pos(int r, int j) { return r * 128 + ((j ^ (2 * (r & 3))) << 4); }

template <int STAGES>
K3_DEVI void dn_issue(const DenseParams& p, const uint16_t* W, int R, int row0, int chunk, int lane, uint32_t stage) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = lane + 32 * i;
    const int r = c >> 3, j = c & 7;
    const int row = min(row0 + r, R - 1);
    cp_async16(stage + dn_pos(r, j), W + (size_t)row * p.K + (size_t)chunk * DN_CHUNK + j * 8);
  }
}

template <int EPI, int NBLK, int STAGES>
__global__ void __launch_bounds__(DN_WARPS * 32) k3_dense_gemv_kernel(DenseParams p) {
  constexpr int NB = 8 * NBLK;
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t wbase = smem_u32(smem) + warp * STAGES * DN_STAGE_BYTES;
  float* red = reinterpret_cast<float*>(smem + DN_WARPS * STAGES * DN_STAGE_BYTES);

  const int tiles0 = (p.R0 + 15) / 16, tiles1 = (p.R1 + 15) / 16, tiles = tiles0 + tiles1;
  const int nbatch = (p.T + NB - 1) / NB;
  const int total = tiles * nbatch;
  const int n_mine = (total > (int)blockIdx.x) ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int nchunks = p.K / DN_CHUNK;
  const int cpw = (nchunks + DN_WARPS - 1) / DN_WARPS;
  const int c0 = warp * cpw;
  const int units = n_mine * cpw;

  auto unit_issue = [&](int u) {
    const int k = u / cpw, c = u - k * cpw;
    const int chunk = c0 + c;
    if (chunk < nchunks) {
      const int i = blockIdx.x + k * gridDim.x;
      const int tile = i % tiles;
      const bool m1 = tile >= tiles0;
      dn_issue<STAGES>(p, m1 ? p.W1 : p.W0, m1 ? p.R1 : p.R0, (m1 ? tile - tiles0 : tile) * 16, chunk, lane,
                       wbase + (u % STAGES) * DN_STAGE_BYTES);
    }
  };

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < units) unit_issue(s);
    cp_async_commit();
  }

  float acc[NBLK][4];
  for (int u = 0; u < units; ++u) {
    if (u + STAGES - 1 < units) unit_issue(u + STAGES - 1);
    cp_async_commit();
    const int k = u / cpw, c = u - k * cpw;
    const int i = blockIdx.x + k * gridDim.x;
    const int tile = i % tiles, bt = i / tiles;
    const int t0 = bt * NB;
    const int n = min(NB, p.T - t0);
    if (c == 0) {
#pragma unroll
      for (int nb = 0; nb < NBLK; ++nb)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[nb][q] = 0.f;
    }
    cp_async_wait<STAGES - 1>();
    __syncwarp();
    const int chunk = c0 + c;
    if (chunk < nchunks) {
      const uint32_t stage = wbase + (u % STAGES) * DN_STAGE_BYTES;
#pragma unroll
      for (int s = 0; s < DN_CHUNK / 16; ++s) {
        const int j = 2 * s + (t >> 1);
        const uint2 alo = lds64(stage + dn_pos(g, j) + (t & 1) * 8);
        const uint2 ahi = lds64(stage + dn_pos(g + 8, j) + (t & 1) * 8);
        const uint32_t a[4] = {alo.x, ahi.x, alo.y, ahi.y};
#pragma unroll
        for (int nb = 0; nb < NBLK; ++nb) {
          if (nb * 8 < n) {
            const int col = nb * 8 + g;
            uint2 b = make_uint2(0u, 0u);
            if (col < n) b = ldg64(p.act + (size_t)(t0 + col) * p.K + (size_t)chunk * DN_CHUNK + 16 * s + 4 * t);
            mma_bf16(acc[nb], a, b.x, b.y, acc[nb]);
          }
        }
      }
    }
    __syncwarp();
    if (c == cpw - 1) {  // item complete: reduce across warps, epilogue
#pragma unroll
      for (int nb = 0; nb < NBLK; ++nb) {
        float* r = red + (warp * NBLK + nb) * 128;
        *reinterpret_cast<float2*>(r + g * 8 + 2 * t) = make_float2(acc[nb][0], acc[nb][1]);
        *reinterpret_cast<float2*>(r + (g + 8) * 8 + 2 * t) = make_float2(acc[nb][2], acc[nb][3]);
      }
      __syncthreads();
      const bool m1 = tile >= tiles0;
      const int R = m1 ? p.R1 : p.R0;
      const int row0 = (m1 ? tile - tiles0 : tile) * 16;
      for (int idx = threadIdx.x; idx < 16 * n; idx += blockDim.x) {
        const int row = idx & 15, col = idx >> 4, nb = col >> 3, cc = col & 7;
        if (row0 + row >= R) continue;
        float sum = 0.f;
        for (int w = 0; w < DN_WARPS; ++w) sum += red[(w * NBLK + nb) * 128 + row * 8 + cc];
        const int tok = t0 + col;
        if (EPI == DN_PROJ && m1) {
          const uint16_t zb = f32_to_bf16_bits(sum);
          p.out1[(size_t)tok * p.R1 + row0 + row] = zb;
          atomicMax(p.zmax + tok, __float_as_uint(fabsf(bf16_bits_to_f32(zb))));
        } else {
          p.out0[(size_t)tok * p.R0 + row0 + row] = sum;
        }
      }
      __syncthreads();
    }
  }
  cp_async_wait<0>();
}

}  // namespace k3

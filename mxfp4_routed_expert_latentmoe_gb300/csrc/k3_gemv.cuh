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
constexpr int MX_REC_BYTES = 128;                  // batch record copy per stage
constexpr int MX_MAX_THREADS = 512;

enum { MX_GATEUP = 0, MX_DOWN = 1 };

struct MxGemvParams {
  const MxBatch* batches;    // token batches (one expert each), written by the permutation
  const int32_t* n_batches;  // number of batches
  int R;                     // rows per matrix
  int K;                     // reduction length
  const __half* act;         // GATEUP: z16 [T, K]; DOWN: h16 [slots, K]
  const int32_t* act_pow;    // GATEUP: per-token exponent p (z16 = z * 2^p)
  const uint16_t* act_bf16;  // GATEUP, bulk kernel: z [T, K] bf16 read directly (act unused), or NULL
  const uint32_t* act_max;   // with act_bf16: per-token max|z| (f32 bits), which fixes p
  void* out;                 // GATEUP: h16 [slots, R] (h * 2^8); DOWN: o f32 [slots, R]
  uint32_t* status;          // device status word (bounded waits of the bulk-copy kernel)
};

template <int M, int STAGES>
struct MxLayout {
  static constexpr int STAGE_BYTES = M * (MX_Q_BYTES + MX_S_BYTES) + MX_REC_BYTES;
  static constexpr int WARP_BYTES = STAGES * STAGE_BYTES;
};

// lanes 0..15 each hold one 8-byte word of a batch record
K3_DEVI uint64_t mx_load_record(const MxGemvParams& p, int tiles, int i, int lane) {
  const int gb = i / tiles;
  return lane < 16 ? reinterpret_cast<const uint64_t*>(p.batches + gb)[lane] : 0ull;
}

// issue the cp.async copies of item i (record `rec`, lane-distributed) into `stage`
template <int MODE, int M>
K3_DEVI void mx_issue(const MxGemvParams& p, int tiles, int i, uint64_t rec, int warp, int lane, int ngroups,
                      uint32_t stage) {
  const size_t qrow = (size_t)p.K / 2, srow = (size_t)p.K / 32;
  const bool sc_async = (p.K % 256) == 0;
  const int row0 = (i % tiles) * MX_ROWS;
  constexpr int WOFF = (MODE == MX_GATEUP) ? 0 : 4;
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const uint8_t* q = reinterpret_cast<const uint8_t*>(__shfl_sync(0xffffffffu, rec, WOFF + 2 * m));
    const uint8_t* s = reinterpret_cast<const uint8_t*>(__shfl_sync(0xffffffffu, rec, WOFF + 2 * m + 1));
    const uint32_t sq = stage + m * (MX_Q_BYTES + MX_S_BYTES);
    const uint32_t ss = sq + MX_Q_BYTES;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int c = lane + 32 * k;
      const int r = c >> 3, j = c & 7;
      if (j < ngroups)
        cp_async16(sq + r * 128 + ((j ^ (r & 7)) << 4), q + (size_t)(row0 + r) * qrow + (size_t)warp * 128 + j * 16);
    }
    if (lane < MX_ROWS) {
      const uint8_t* src = s + (size_t)(row0 + lane) * srow + (size_t)warp * MX_GPW;
      if (sc_async) {
        cp_async8(ss + lane * 8, src);
      } else {  // partial slice or unaligned scale rows: plain byte copies (small shapes only)
        uint8_t* dst = (uint8_t*)__cvta_shared_to_generic(ss + lane * 8);
        for (int j = 0; j < MX_GPW; ++j) dst[j] = (j < ngroups) ? src[j] : (uint8_t)127;
      }
    }
  }
  // the record rides with the stage (word 15, padding in memory, carries the row tile)
  if (lane < 16) {
    const uint64_t v = (lane == 15) ? (uint64_t)(uint32_t)row0 : rec;
    *reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(stage + M * (MX_Q_BYTES + MX_S_BYTES) + 8 * lane)) = v;
  }
}

// PRE: the expert weights of the first items are requested before waiting for the
// previous kernel (programmatic dependent launch); only the activations wait.
// FULL: every warp's K slice is a whole 8 groups (K a multiple of 256).
template <int MODE, int NBLK, int STAGES, bool PRE, bool FULL>
__global__ void __launch_bounds__(MX_MAX_THREADS) k3_mx_gemv_kernel(MxGemvParams p) {
  constexpr int M = (MODE == MX_GATEUP) ? 2 : 1;
  using Lay = MxLayout<M, STAGES>;
  constexpr int RED = M * NBLK * 128;  // floats of one warp's partial sums
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int col_pw[2][MX_MAX_NB];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int ngroups = FULL ? MX_GPW : min(MX_GPW, p.K / 32 - warp * MX_GPW);
  const uint32_t wbase = smem_u32(smem) + warp * Lay::WARP_BYTES;
  float* red = reinterpret_cast<float*>(smem + nwarps * Lay::WARP_BYTES);  // [2][nwarps][RED]
  const int tiles = p.R / MX_ROWS;

  if (!PRE) grid_dep_wait();
  const int total = tiles * (*p.n_batches);
  const int n_mine = (total > (int)blockIdx.x) ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  // prologue: the first STAGES-1 items
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < n_mine) {
      const int i = blockIdx.x + s * gridDim.x;
      mx_issue<MODE, M>(p, tiles, i, mx_load_record(p, tiles, i, lane), warp, lane, ngroups,
                        wbase + s * Lay::STAGE_BYTES);
    }
    cp_async_commit();
  }
  uint64_t rec_next = (STAGES - 1 < n_mine) ? mx_load_record(p, tiles, blockIdx.x + (STAGES - 1) * gridDim.x, lane)
                                            : 0ull;
  if (PRE) grid_dep_wait();
  grid_dep_launch();

  // single-token batches of the same token (decode) share their activation fragments:
  // this warp's 8 groups stay in registers across items
  constexpr bool CACHE_B = (MODE == MX_GATEUP) && (NBLK == 1);
  uint4 bcache[CACHE_B ? MX_GPW : 1];
  int bkey = -1;

  for (int s = 0; s < n_mine; ++s) {
    {
      const int sn = s + STAGES - 1;
      if (sn < n_mine)
        mx_issue<MODE, M>(p, tiles, blockIdx.x + sn * gridDim.x, rec_next, warp, lane, ngroups,
                          wbase + (sn % STAGES) * Lay::STAGE_BYTES);
      cp_async_commit();
      if (sn + 1 < n_mine) rec_next = mx_load_record(p, tiles, blockIdx.x + (sn + 1) * gridDim.x, lane);
    }
    cp_async_wait<STAGES - 1>();
    __syncwarp();

    const uint8_t* stp = smem + warp * Lay::WARP_BYTES + (s % STAGES) * Lay::STAGE_BYTES;
    const int32_t* rec = reinterpret_cast<const int32_t*>(stp + M * (MX_Q_BYTES + MX_S_BYTES));
    const int slot0 = rec[12], n = rec[13], row0 = rec[30];
    if (MODE == MX_GATEUP && warp == 0 && lane < n) col_pw[s & 1][lane] = p.act_pow[rec[14 + lane]];

    float acc[M][NBLK][4];
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
      for (int nb = 0; nb < NBLK; ++nb)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[m][nb][q] = 0.f;

    if (FULL || ngroups > 0) {
      // activation row of this lane's token column in every 8-token block (columns
      // past the batch repeat its last token: their results are never stored)
      const __half* bptr[NBLK];
#pragma unroll
      for (int nb = 0; nb < NBLK; ++nb) {
        const int col = min(nb * 8 + g, n - 1);
        const int row = (MODE == MX_GATEUP) ? rec[14 + col] : slot0 + col;
        bptr[nb] = p.act + (size_t)row * p.K + warp * 256 + 8 * t;
      }
      if (CACHE_B) {
        const int key = (n == 1) ? rec[14] : -1;
        if (key < 0 || key != bkey) {
#pragma unroll
          for (int j = 0; j < MX_GPW; ++j)
            if (FULL || j < ngroups) bcache[CACHE_B ? j : 0] = ldg128(bptr[0] + 32 * j);
          bkey = key;
        }
      }
      uint2 sc_lo[M], sc_hi[M];
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const uint8_t* ss = stp + m * (MX_Q_BYTES + MX_S_BYTES) + MX_Q_BYTES;
        sc_lo[m] = *reinterpret_cast<const uint2*>(ss + g * 8);
        sc_hi[m] = *reinterpret_cast<const uint2*>(ss + (g + 8) * 8);
      }
#pragma unroll
      for (int j = 0; j < MX_GPW; ++j) {
        if (FULL || j < ngroups) {
          uint32_t a0[M][4], a1[M][4];
          float slo[M], shi[M];
#pragma unroll
          for (int m = 0; m < M; ++m) {
            const uint8_t* sq = stp + m * (MX_Q_BYTES + MX_S_BYTES);
            const int off = ((j ^ g) << 4) + 4 * t;
            const uint32_t wlo = *reinterpret_cast<const uint32_t*>(sq + g * 128 + off);
            const uint32_t whi = *reinterpret_cast<const uint32_t*>(sq + (g + 8) * 128 + off);
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
            if ((j & 3) == 0) { slo[m] = ue8m0_byte_to_f32<0>(blo); shi[m] = ue8m0_byte_to_f32<0>(bhi); }
            if ((j & 3) == 1) { slo[m] = ue8m0_byte_to_f32<1>(blo); shi[m] = ue8m0_byte_to_f32<1>(bhi); }
            if ((j & 3) == 2) { slo[m] = ue8m0_byte_to_f32<2>(blo); shi[m] = ue8m0_byte_to_f32<2>(bhi); }
            if ((j & 3) == 3) { slo[m] = ue8m0_byte_to_f32<3>(blo); shi[m] = ue8m0_byte_to_f32<3>(bhi); }
          }
#pragma unroll
          for (int nb = 0; nb < NBLK; ++nb) {
            if (NBLK == 1 || nb * 8 < n) {
              const uint4 b = CACHE_B ? bcache[CACHE_B ? j : 0] : ldg128(bptr[nb] + 32 * j);
#pragma unroll
              for (int m = 0; m < M; ++m) {
                const float z4[4] = {0.f, 0.f, 0.f, 0.f};
                float d[4];
                mma_f16(d, a0[m], b.x, b.y, z4);
                mma_f16(d, a1[m], b.z, b.w, d);
                ffma2(acc[m][nb][0], acc[m][nb][1], d[0], d[1], slo[m], acc[m][nb][0], acc[m][nb][1]);
                ffma2(acc[m][nb][2], acc[m][nb][3], d[2], d[3], shi[m], acc[m][nb][2], acc[m][nb][3]);
              }
            }
          }
        }
      }
    }
    // per-warp partials -> shared memory: red[s & 1][warp][m][nb][row 16][col 8]; the
    // buffer alternates between items, so one barrier per item suffices
    float* rb = red + ((s & 1) * nwarps + warp) * RED;
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
      for (int nb = 0; nb < NBLK; ++nb) {
        float* r = rb + (m * NBLK + nb) * 128;
        *reinterpret_cast<float2*>(r + g * 8 + 2 * t) = make_float2(acc[m][nb][0], acc[m][nb][1]);
        *reinterpret_cast<float2*>(r + (g + 8) * 8 + 2 * t) = make_float2(acc[m][nb][2], acc[m][nb][3]);
      }
    __syncthreads();
    const float* rs = red + (s & 1) * nwarps * RED;
    for (int idx = threadIdx.x; idx < MX_ROWS * n; idx += blockDim.x) {
      const int row = idx & 15, col = idx >> 4, nb = col >> 3, cc = col & 7;
      float v[M];
#pragma unroll
      for (int m = 0; m < M; ++m) {
        float sum = 0.f;
        for (int w = 0; w < nwarps; ++w) sum += rs[w * RED + (m * NBLK + nb) * 128 + row * 8 + cc];
        v[m] = sum;
      }
      const int slot = slot0 + col;
      if (MODE == MX_GATEUP) {
        const int pw = col_pw[s & 1][col];
        const float gg = scalbnf(v[0], -pw), uu = scalbnf(v[M - 1], -pw);
        const float h = __uint_as_float((uint32_t)f32_to_bf16_bits(situf(gg, uu)) << 16);  // bf16 rounding
        reinterpret_cast<__half*>(p.out)[(size_t)slot * p.R + row0 + row] = __float2half_rn(h * 256.0f);
      } else {
        reinterpret_cast<float*>(p.out)[(size_t)slot * p.R + row0 + row] = v[0] * (1.0f / 256.0f);
      }
    }
  }
  cp_async_wait<0>();
}

// ============================================================================ bf16 GEMV
constexpr int DN_CHUNK = 64;  // elements per row per stage
constexpr int DN_WARPS = 8;
constexpr int DN_A_BYTES = 16 * DN_CHUNK * 2;  // 2048: 16 weight rows

enum { DN_PROJ = 0, DN_PLAIN = 1, DN_ACC = 2 };  // ACC: out0 += the product

struct DenseParams {
  const uint16_t* W0;
  int R0;
  const uint16_t* W1;
  int R1;
  int K;
  const uint16_t* act;  // [T, K] bf16
  int T;
  float* out0;      // PROJ: logits [T, R0]; PLAIN: out [T, R0]; ACC: out [T, R0], added to
  uint16_t* out1;   // PROJ: z [T, R1] bf16
  uint32_t* zmax;   // PROJ: per-token max |z| (f32 bits)
  uint32_t* status; // device status word (bounded waits that run out)
};

// bytes of one stage: 16 weight rows and NB activation rows of one 64-element chunk
__host__ __device__ constexpr int dn_stage_bytes(int nblk) { return DN_A_BYTES + 8 * nblk * DN_CHUNK * 2; }

// smem row layout: 16-byte chunk j of row r sits at position j ^ (2 * (r & 3)); with the
// per-thread 8-byte reads of an m16n8k16 fragment this keeps both half-warps conflict-free
K3_DEVI uint32_t dn_pos(int r, int j) { return r * 128 + ((j ^ (2 * (r & 3))) << 4); }

template <int NBLK>
K3_DEVI void dn_issue(const DenseParams& p, const uint16_t* W, int R, int row0, int t0, int n, int chunk, int lane,
                      uint32_t stage) {
  const size_t k0 = (size_t)chunk * DN_CHUNK;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = lane + 32 * i;
    const int r = c >> 3, j = c & 7;
    const int row = min(row0 + r, R - 1);
    cp_async16(stage + dn_pos(r, j), W + (size_t)row * p.K + k0 + j * 8);
  }
  // activation rows of the batch (rows past n keep stale data: their columns are never stored)
#pragma unroll
  for (int i = 0; i < NBLK * 2; ++i) {
    const int c = lane + 32 * i;
    const int r = c >> 3, j = c & 7;
    if (r < n) cp_async16(stage + DN_A_BYTES + dn_pos(r, j), p.act + (size_t)(t0 + r) * p.K + k0 + j * 8);
  }
}

template <int EPI, int NBLK, int STAGES>
__global__ void __launch_bounds__(DN_WARPS * 32) k3_dense_gemv_kernel(DenseParams p) {
  constexpr int NB = 8 * NBLK;
  constexpr int SB = dn_stage_bytes(NBLK);
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t wbase = smem_u32(smem) + warp * STAGES * SB;
  float* red = reinterpret_cast<float*>(smem + DN_WARPS * STAGES * SB);

  const int tiles0 = (p.R0 + 15) / 16, tiles1 = (p.R1 + 15) / 16, tiles = tiles0 + tiles1;
  const int nbatch = (p.T + NB - 1) / NB;
  const int total = tiles * nbatch;
  const int n_mine = (total > (int)blockIdx.x) ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int nchunks = p.K / DN_CHUNK;
  const int cpw = (nchunks + DN_WARPS - 1) / DN_WARPS;
  const int c0 = warp * cpw;
  const int units = n_mine * cpw;

  auto unit_rows = [&](int u, const uint16_t*& W, int& R, int& row0, int& t0, int& n) {
    const int i = blockIdx.x + (u / cpw) * gridDim.x;
    const int tile = i % tiles, bt = i / tiles;
    const bool m1 = tile >= tiles0;
    W = m1 ? p.W1 : p.W0;
    R = m1 ? p.R1 : p.R0;
    row0 = (m1 ? tile - tiles0 : tile) * 16;
    t0 = bt * NB;
    n = min(NB, p.T - t0);
  };
  auto unit_issue = [&](int u) {
    const int chunk = c0 + u % cpw;
    if (chunk < nchunks) {
      const uint16_t* W;
      int R, row0, t0, n;
      unit_rows(u, W, R, row0, t0, n);
      dn_issue<NBLK>(p, W, R, row0, t0, n, chunk, lane, wbase + (u % STAGES) * SB);
    }
  };

  // the weights of the first stages do not depend on the previous kernel: pull them
  // into L2 before waiting for it
  for (int u = 0; u < STAGES - 1 && u < units; ++u) {
    const int chunk = c0 + u % cpw;
    if (chunk < nchunks && lane < 16) {
      const uint16_t* W;
      int R, row0, t0, n;
      unit_rows(u, W, R, row0, t0, n);
      const uint16_t* a = W + (size_t)min(row0 + lane, R - 1) * p.K + (size_t)chunk * DN_CHUNK;
      asm volatile("prefetch.global.L2 [%0];\n" ::"l"(a));
    }
  }
  grid_dep_wait();
  grid_dep_launch();
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < units) unit_issue(s);
    cp_async_commit();
  }

  float acc[NBLK][4];
  for (int u = 0; u < units; ++u) {
    if (u + STAGES - 1 < units) unit_issue(u + STAGES - 1);
    cp_async_commit();
    const int c = u % cpw;
    const int i = blockIdx.x + (u / cpw) * gridDim.x;
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
      const uint8_t* stp = smem + warp * STAGES * SB + (u % STAGES) * SB;
#pragma unroll
      for (int s = 0; s < DN_CHUNK / 16; ++s) {
        const int j = 2 * s + (t >> 1);
        const uint2 alo = *reinterpret_cast<const uint2*>(stp + dn_pos(g, j) + (t & 1) * 8);
        const uint2 ahi = *reinterpret_cast<const uint2*>(stp + dn_pos(g + 8, j) + (t & 1) * 8);
        const uint32_t a[4] = {alo.x, ahi.x, alo.y, ahi.y};
#pragma unroll
        for (int nb = 0; nb < NBLK; ++nb) {
          if (NBLK == 1 || nb * 8 < n) {
            const uint2 b = *reinterpret_cast<const uint2*>(stp + DN_A_BYTES + dn_pos(nb * 8 + g, j) + (t & 1) * 8);
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
        } else if (EPI == DN_ACC) {
          p.out0[(size_t)tok * p.R0 + row0 + row] += sum;
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

// k3_gemv_bulk.cuh -- MXFP4 weight-streaming GEMV with bulk (TMA engine) copies, for
// small token counts per expert (decode, chunked prefill) when K is a multiple of 256.
//
// Same arithmetic as k3_mx_gemv_kernel (k3_gemv.cuh): item = 16 rows of one matrix
// (gate and up together for GATEUP) x one batch of up to 8 * NBLK tokens; K split into
// 256-element slices, one per compute warp; each 32-element scale group is decoded with
// cvt.rn.f16x2.e2m1x2, multiplied on the tensor core (m16n8k16, f16 in, fp32 out) and
// folded into the fp32 accumulator with the group's power-of-two scale.
//
// What differs is how bytes move and how partial sums meet:
//   warp 0       producer: the item's 16 rows are contiguous in each matrix; lanes
//                0..7 (and 8..15 for the up matrix) each issue one cp.async.bulk of a
//                pair of rows into shared memory, pairs padded by 16 bytes (the fragment
//                reads of 8 rows then meet at most 2-way bank conflicts), plus one bulk
//                copy of the 16 rows' scale bytes per matrix; completion is counted in
//                bytes on the stage's mbarrier.  The copies run on the TMA engine, so the
//                bytes in flight are not limited by per-warp load queues; the engine takes
//                about one copy instruction per ~100 cycles, hence pairs of rows (measured
//                per item: 34 single-row copies took ~3300 cycles);
//   warp 1       reducer: adds the compute warps' partial sums in warp order
//                (deterministic), applies the epilogue (SiTU-GLU for GATEUP) and stores;
//   warps 2..    compute: one 256-element K slice each.
// Stages (STAGES deep), partial-sum buffers (2) and their hand-offs are mbarriers; no
// block-wide barrier is taken per item.  Every wait is bounded (about 2^32 cycles, with a
// per-CTA abort flag): a wait that runs out sets K3MOE_DEV_TIMEOUT and all roles drain
// their issued copies and return.
#pragma once

#include "k3_common.cuh"
#include "k3_gemv.cuh"
#include "k3_tc.cuh"

namespace k3 {

constexpr int MXB_MAX_WARPS = 14;  // compute warps: K <= 3584 (larger K uses k3_mx_gemv_kernel)

K3_DEVI void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// 0, through an instruction the compiler cannot see through: a value computed from x that
// the hardware can produce only once x is available
K3_DEVI uint32_t opaque_zero(uint32_t x) {
  uint32_t z;
  asm volatile("and.b32 %0, %1, 0;\n" : "=r"(z) : "r"(x));
  return z;
}
// the same with an L2 eviction-priority policy (createpolicy)
K3_DEVI void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}


template <int MODE>
struct MxbLayout {
  static constexpr int M = (MODE == MX_GATEUP) ? 2 : 1;
  // per stage: M x (8 padded row pairs + 16 rows of scale bytes), then the 128-byte batch record
  __host__ __device__ static constexpr int pair_stride(int K) { return K + 16; }
  __host__ __device__ static constexpr int mat_bytes(int K) { return (MX_ROWS / 2) * pair_stride(K) + MX_ROWS * (K / 32); }
  __host__ __device__ static constexpr int stage_bytes(int K) { return M * mat_bytes(K) + 128; }
  __host__ __device__ static constexpr int red_floats(int W, int nblk) { return W * M * nblk * 128; }
  static constexpr int META = 48;  // ints per partial-sum buffer: slot0, n, row0, tok[16], pow[16]
  __host__ __device__ static constexpr int smem_bytes(int K, int stages, int nblk) {
    return 128 + stages * stage_bytes(K) + 2 * red_floats(K / 256, nblk) * 4 + 2 * META * 4 + 256;
  }
};

// PRE: the first stages' weight copies are issued before waiting for the previous kernel
// (programmatic dependent launch); valid when the batch records were written at least
// two kernels earlier.
template <int MODE, int NBLK, int STAGES, bool PRE>
__global__ void __launch_bounds__((2 + MXB_MAX_WARPS) * 32) k3_mxb_gemv_kernel(MxGemvParams p) {
  using Lay = MxbLayout<MODE>;
  constexpr int M = Lay::M;
  constexpr int RED = M * NBLK * 128;  // floats of one warp's partial sums
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ int abort_sh;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int W = (int)(blockDim.x >> 5) - 2;  // compute warps (K / 256)
  const int K = p.K, PS = Lay::pair_stride(K), MB = Lay::mat_bytes(K), SB = Lay::stage_bytes(K);
  const uint32_t base = (smem_u32(smem_raw) + 127u) & ~127u;
  uint8_t* base_ptr = smem_raw + (base - smem_u32(smem_raw));
  const uint32_t red_s = base + STAGES * SB;  // [2][W][RED] f32
  float* red = reinterpret_cast<float*>(base_ptr + STAGES * SB);
  int* meta = reinterpret_cast<int*>(base_ptr + STAGES * SB + 2 * W * RED * 4);  // [2][META]
  const uint32_t bars = red_s + 2 * W * RED * 4 + 2 * Lay::META * 4;
  auto full = [&](int s) { return bars + 8 * s; };
  auto empty = [&](int s) { return bars + 8 * (STAGES + s); };
  auto rfull = [&](int b) { return bars + 8 * (2 * STAGES + b); };
  auto rempty = [&](int b) { return bars + 8 * (2 * STAGES + 2 + b); };
  volatile int* abort_flag = &abort_sh;
  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), W);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(rfull(b), W);
      mbar_init(rempty(b), 1);
    }
    fence_barrier_init();
  }
  __syncthreads();

  const int tiles = p.R / MX_ROWS;
  const size_t qrow = (size_t)K / 2, srow = (size_t)K / 32;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = l2_policy_evict_first();  // expert weights are read once per call
    if (!PRE) grid_dep_wait();
    const int total = tiles * (*p.n_batches);
    const int n_mine = (total > (int)blockIdx.x) ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    constexpr int WOFF = (MODE == MX_GATEUP) ? 0 : 4;
    // lanes 0..5 hold the six tensor pointers of the item's batch record, loaded one
    // item ahead so the copies are not held up by the record's latency
    auto rec_word = [&](int s2) -> uint64_t {
      if (s2 >= n_mine || lane >= 6) return 0ull;
      return reinterpret_cast<const uint64_t*>(p.batches + (blockIdx.x + s2 * gridDim.x) / tiles)[lane];
    };
    uint64_t wnext = rec_word(0);
    int s = 0;
    for (; s < n_mine; ++s) {
      if (PRE && s == STAGES) grid_dep_wait();
      const int st = s % STAGES;
      const uint64_t wcur = wnext;
      wnext = rec_word(s + 1);
      if (!__all_sync(0xffffffffu, mbar_wait(empty(st), ((s / STAGES) & 1) ^ 1, abort_flag))) break;
      const int i = blockIdx.x + s * gridDim.x;
      const MxBatch* rec = p.batches + i / tiles;
      const size_t row0 = (size_t)(i % tiles) * MX_ROWS;
      const uint32_t sbase = base + st * SB;
      if (lane == 0) mbar_expect_tx(full(st), (uint32_t)(M * MX_ROWS * (qrow + srow) + 128));
      __syncwarp();
      const int mq = (lane < 8 * M) ? (lane >> 3) : ((lane >= 16 && lane < 16 + M) ? lane - 16 : 0);
      const uint8_t* qptr = reinterpret_cast<const uint8_t*>(__shfl_sync(0xffffffffu, wcur, WOFF + 2 * mq));
      const uint8_t* sptr = reinterpret_cast<const uint8_t*>(__shfl_sync(0xffffffffu, wcur, WOFF + 2 * mq + 1));
      if (lane < 8 * M) {  // row pair lane & 7 of matrix lane >> 3
        const int pr = lane & 7;
        bulk_g2s_hint(sbase + mq * MB + pr * PS, qptr + (row0 + 2 * pr) * qrow, (uint32_t)(2 * qrow), full(st), pol);
      } else if (lane >= 16 && lane < 16 + M) {  // scale bytes of matrix lane - 16
        bulk_g2s_hint(sbase + mq * MB + (MX_ROWS / 2) * PS, sptr + row0 * srow, (uint32_t)(MX_ROWS * srow), full(st),
                      pol);
      }
      if (lane == 31) bulk_g2s(sbase + M * MB, rec, 128, full(st));
    }
    if (PRE && s < STAGES) grid_dep_wait();
    grid_dep_launch();
    // drain: every issued stage must land before the CTA exits
    for (int t = (s > STAGES ? s - STAGES : 0); t < s; ++t) {
      volatile int never = 0;
      mbar_wait(full(t % STAGES), (t / STAGES) & 1, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ reducer + epilogue
    grid_dep_wait();
    grid_dep_launch();
    const int total = tiles * (*p.n_batches);
    const int n_mine = (total > (int)blockIdx.x) ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    for (int s = 0; s < n_mine; ++s) {
      const int b = s & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(rfull(b), (s >> 1) & 1, abort_flag))) break;
      const int* mt = meta + b * Lay::META;
      const int slot0 = mt[0], n = mt[1], row0 = mt[2];
      const float* rs = red + b * W * RED;
      // one token: the 16 rows' sums on all 32 lanes, each half of the warp over half of the
      // compute warps' partials (lane and lane + 16 hold the same row), then added
      const bool halves = (n == 1);
      for (int idx = halves ? (lane & 15) : lane; idx < MX_ROWS * n; idx += 32) {
        const int row = idx & 15, col = idx >> 4, nb = col >> 3, cc = col & 7;
        float v[M];
#pragma unroll
        for (int mm = 0; mm < M; ++mm) {
          float sum = 0.f;
          if (halves) {
#pragma unroll 4
            for (int w = lane >> 4; w < W; w += 2) sum += rs[w * RED + (mm * NBLK + nb) * 128 + row * 8 + cc];
            sum += __shfl_xor_sync(0xffffffffu, sum, 16);
          } else {
#pragma unroll 6
            for (int w = 0; w < W; ++w) sum += rs[w * RED + (mm * NBLK + nb) * 128 + row * 8 + cc];
          }
          v[mm] = sum;
        }
        if (halves && lane >= 16) continue;
        const int slot = slot0 + col;
        if (MODE == MX_GATEUP) {
          const int pw = mt[19 + col];
          const float f1 = pow2f(-(pw >> 1)), f2 = pow2f((pw >> 1) - pw);  // exact 2^-p
          const float gg = v[0] * f1 * f2, uu = v[M - 1] * f1 * f2;
          const float h = __uint_as_float((uint32_t)f32_to_bf16_bits(situ_fast(gg, uu)) << 16);  // bf16 rounding
          reinterpret_cast<__half*>(p.out)[(size_t)slot * p.R + row0 + row] = __float2half_rn(h * 256.0f);
        } else {
          reinterpret_cast<float*>(p.out)[(size_t)slot * p.R + row0 + row] = v[0] * (1.0f / 256.0f);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(rempty(b));
    }
  } else {
    // ------------------------------------------------------------ compute warps
    const int c = warp - 2;  // K slice
    const int g = lane >> 2, t = lane & 3;
    const bool bf_in = (MODE == MX_GATEUP) && p.act_bf16 != nullptr;  // activations read as bf16 z
    grid_dep_wait();
    grid_dep_launch();
    const int total = tiles * (*p.n_batches);
    const int n_mine = (total > (int)blockIdx.x) ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    // single-token batches keep this warp's activation fragments in registers while
    // consecutive items use the same activation row (GATEUP: the same token, every item of
    // a one-token call; DOWN would need the same slot, i.e. the same expert, which a CTA's
    // consecutive items almost never share: it keeps the registers for the early release)
    constexpr bool CACHE_B = (NBLK == 1) && MODE == MX_GATEUP;
    uint4 bcache[CACHE_B ? MX_GPW : 1];
    int bkey = -1;
    for (int s = 0; s < n_mine; ++s) {
      const int st = s % STAGES;
      if (!__all_sync(0xffffffffu, mbar_wait(full(st), (s / STAGES) & 1, abort_flag))) break;
      const uint8_t* stp = base_ptr + st * SB;
      const MxBatch* rec = reinterpret_cast<const MxBatch*>(stp + M * MB);
      const int slot0 = rec->slot0, n = rec->n;
      // warp 0 passes the item's bookkeeping to the reducer (fetched now, stored with the
      // partial sums): token ids and, for GATEUP, their activation exponents
      int my_tok = 0, my_pow = 0;
      if (c == 0 && lane < n) {
        my_tok = rec->tok[lane];
        if (MODE == MX_GATEUP) my_pow = bf_in ? act_exp_from_max(p.act_max[my_tok]) : p.act_pow[my_tok];
      }

      float acc[M][NBLK][4];
#pragma unroll
      for (int m = 0; m < M; ++m)
#pragma unroll
        for (int nb = 0; nb < NBLK; ++nb)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[m][nb][q] = 0.f;
      // activation row of this lane's token column in every 8-token block (columns past
      // the batch repeat its last token: their results are never stored)
      // (GATEUP from bf16 z: 8 bf16 values become the f16 operand, scaled by the token's 2^p)
      const __half* bptr[NBLK];
      const uint16_t* bptr16[NBLK];
      int brow[NBLK];
#pragma unroll
      for (int nb = 0; nb < NBLK; ++nb) {
        const int col = min(nb * 8 + g, n - 1);
        const int row = (MODE == MX_GATEUP) ? rec->tok[col] : slot0 + col;
        brow[nb] = row;
        bptr[nb] = p.act + (size_t)row * K + c * 256 + 8 * t;
        bptr16[nb] = (MODE == MX_GATEUP && bf_in) ? p.act_bf16 + (size_t)row * K + c * 256 + 8 * t : nullptr;
      }
      // the token's 2^p is read when its row is read (the max comes from the previous kernel)
      auto load_b = [&](int nb, int j, int pw) -> uint4 {
        if (MODE == MX_GATEUP && bf_in) return bf16x8_to_f16x8(ldg128(bptr16[nb] + 32 * j), pw);
        return ldg128(bptr[nb] + 32 * j);
      };
      auto row_pow = [&](int nb) { return (MODE == MX_GATEUP && bf_in) ? act_exp_from_max(__ldg(p.act_max + brow[nb])) : 0; };
      if (CACHE_B) {
        const int key = (n == 1) ? ((MODE == MX_GATEUP) ? rec->tok[0] : slot0) : -1;
        if (key < 0 || key != bkey) {
          const int pw = row_pow(0);
#pragma unroll
          for (int j = 0; j < MX_GPW; ++j) bcache[CACHE_B ? j : 0] = load_b(0, j, pw);
          bkey = key;
        }
      }
      int bpw[NBLK];
#pragma unroll
      for (int nb = 0; nb < NBLK; ++nb) bpw[nb] = (CACHE_B || !(MODE == MX_GATEUP && bf_in)) ? 0 : row_pow(nb);
      uint2 sc_lo[M], sc_hi[M];
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const uint8_t* ss = stp + m * MB + (MX_ROWS / 2) * PS + c * MX_GPW;
        sc_lo[m] = *reinterpret_cast<const uint2*>(ss + g * srow);
        sc_hi[m] = *reinterpret_cast<const uint2*>(ss + (g + 8) * srow);
      }
      // this warp's packed words of the item (row r sits at pair r / 2, half r % 2), all
      // loaded into registers first: the stage goes back to the producer before the decode
      // and the MMAs, so the copies in flight do not wait for the compute
      constexpr bool EARLY = true;
      uint32_t wlo_[MX_GPW][M], whi_[MX_GPW][M];
      if (EARLY) {
#pragma unroll
        for (int j = 0; j < MX_GPW; ++j)
#pragma unroll
          for (int m = 0; m < M; ++m) {
            const uint8_t* sq = stp + m * MB + c * 128 + j * 16 + 4 * t + (g >> 1) * PS + (g & 1) * (K / 2);
            wlo_[j][m] = *reinterpret_cast<const uint32_t*>(sq);
            whi_[j][m] = *reinterpret_cast<const uint32_t*>(sq + 4 * PS);
          }
      }
      if (EARLY) {
        // every lane's loads have landed (the fold reads each loaded register, and the warp
        // reduction reads each lane's fold) before lane 0 releases the stage
        uint32_t chk = 0u;
#pragma unroll
        for (int m = 0; m < M; ++m) chk ^= sc_lo[m].x ^ sc_lo[m].y ^ sc_hi[m].x ^ sc_hi[m].y;
#pragma unroll
        for (int j = 0; j < MX_GPW; ++j)
#pragma unroll
          for (int m = 0; m < M; ++m) chk ^= wlo_[j][m] ^ whi_[j][m];
        const uint32_t zero = __reduce_or_sync(0xffffffffu, opaque_zero(chk));
        if (lane == 0) mbar_arrive(empty(st) + zero);
      }
#pragma unroll
      for (int j = 0; j < MX_GPW; ++j) {
        uint32_t a0[M][4], a1[M][4];
        float slo[M], shi[M];
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const uint8_t* sq = stp + m * MB + c * 128 + j * 16 + 4 * t + (g >> 1) * PS + (g & 1) * (K / 2);
          const uint32_t wlo = EARLY ? wlo_[j][m] : *reinterpret_cast<const uint32_t*>(sq);
          const uint32_t whi = EARLY ? whi_[j][m] : *reinterpret_cast<const uint32_t*>(sq + 4 * PS);
          uint32_t plo[4], phi[4];
          e2m1x8_to_f16x8(wlo, plo);
          e2m1x8_to_f16x8(whi, phi);
          // K order inside the group: this thread's 8 elements 8t..8t+7 feed MMA 0 slots
          // {2t,2t+1 | 2t+8,2t+9} = elements {8t,8t+1 | 8t+2,8t+3} and MMA 1 the same
          // slots with elements {8t+4,8t+5 | 8t+6,8t+7}
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
            const uint4 bv = CACHE_B ? bcache[CACHE_B ? j : 0] : load_b(nb, j, bpw[nb]);
#pragma unroll
            for (int m = 0; m < M; ++m) {
              const float z4[4] = {0.f, 0.f, 0.f, 0.f};
              float d[4];
              mma_f16(d, a0[m], bv.x, bv.y, z4);
              mma_f16(d, a1[m], bv.z, bv.w, d);
              ffma2(acc[m][nb][0], acc[m][nb][1], d[0], d[1], slo[m], acc[m][nb][0], acc[m][nb][1]);
              ffma2(acc[m][nb][2], acc[m][nb][3], d[2], d[3], shi[m], acc[m][nb][2], acc[m][nb][3]);
            }
          }
        }
      }
      if (!EARLY) {
        // the stage's bytes are consumed: hand it back to the producer
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(st));
      }
      // partial sums -> red[s & 1][c][m][nb][row 16][col 8] once the reducer released it
      const int b = s & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(rempty(b), ((s >> 1) & 1) ^ 1, abort_flag))) break;
      float* rb = red + (b * W + c) * RED;
      if (c == 0) {
        int* mt = meta + b * Lay::META;
        if (lane == 0) {
          mt[0] = slot0;
          mt[1] = n;
          mt[2] = ((blockIdx.x + s * gridDim.x) % tiles) * MX_ROWS;
        }
        if (lane < n) {
          mt[3 + lane] = my_tok;
          mt[19 + lane] = my_pow;
        }
      }
#pragma unroll
      for (int m = 0; m < M; ++m)
#pragma unroll
        for (int nb = 0; nb < NBLK; ++nb) {
          float* r = rb + (m * NBLK + nb) * 128;
          *reinterpret_cast<float2*>(r + g * 8 + 2 * t) = make_float2(acc[m][nb][0], acc[m][nb][1]);
          *reinterpret_cast<float2*>(r + (g + 8) * 8 + 2 * t) = make_float2(acc[m][nb][2], acc[m][nb][3]);
        }
      __syncwarp();
      if (lane == 0) mbar_arrive(rfull(b));
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) flag_status(p.status, K3MOE_DEV_TIMEOUT);
}

}  // namespace k3

namespace k3 {

// ============================================================================ bf16 GEMV, one token
// out[r] = W[r, :] . x for the rows of W0 (then W1) with a single activation row x (the
// decode step's latent projections).  Each CTA owns a contiguous range of rows and its
// warps take them in turn; a warp reads a whole row with 16-byte non-caching loads, eight
// per lane in flight (4 KB per warp, the next chunk issued before the current one is
// used), straight into registers, multiplies with x held in
// shared memory as f32 and sums in fp32, lanes combined by a fixed butterfly.  Plain
// vector loads from many warps keep enough bytes in flight per SM to stream at the HBM
// copy rate (bulk copies of a few KB issued by one thread reach barely half of it).
constexpr int D1_WARPS = 8;   // warps per CTA
constexpr int D1_UNR = 8;     // 16-byte loads in flight per lane

K3_DEVI uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <int EPI>
__global__ void __launch_bounds__(D1_WARPS * 32, 2) k3_dense_gemv1_kernel(DenseParams p) {
  extern __shared__ __align__(16) float xs[];  // x as f32, K values
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = p.K, KV = K / 8;  // 16-byte vectors per row
  const int R = p.R0 + p.R1;
  const int r0 = (int)(((long long)R * blockIdx.x) / gridDim.x);
  const int r1 = (int)(((long long)R * (blockIdx.x + 1)) / gridDim.x);
  auto row_ptr = [&](int r) -> const uint4* {
    return reinterpret_cast<const uint4*>((r < p.R0) ? p.W0 + (size_t)r * K : p.W1 + (size_t)(r - p.R0) * K);
  };
  // the first row's first loads do not depend on the previous kernel: issue them before
  // waiting for it
  uint4 w[D1_UNR];
  int r = r0 + warp;
  if (r < r1) {
    const uint4* wv = row_ptr(r);
#pragma unroll
    for (int u = 0; u < D1_UNR; ++u) {
      const int v = lane + 32 * u;
      w[u] = (v < KV) ? ldg_stream(wv + v) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  grid_dep_wait();
  grid_dep_launch();
  for (int v = threadIdx.x; v < K / 2; v += blockDim.x) {
    const uint32_t xx = __ldg(reinterpret_cast<const uint32_t*>(p.act) + v);
    reinterpret_cast<float2*>(xs)[v] = make_float2(__uint_as_float(xx << 16), __uint_as_float(xx & 0xFFFF0000u));
  }
  __syncthreads();
  for (; r < r1; r += D1_WARPS) {
    const uint4* wv = row_ptr(r);
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    for (int v0 = 0; v0 < KV; v0 += 32 * D1_UNR) {
      uint4 cur[D1_UNR];
#pragma unroll
      for (int u = 0; u < D1_UNR; ++u) cur[u] = w[u];
      // next chunk (of this row, else of the warp's next row) in flight while this one is used
      const int vn = v0 + 32 * D1_UNR;
      const bool more = vn < KV;
      const uint4* wn = more ? wv : ((r + D1_WARPS < r1) ? row_ptr(r + D1_WARPS) : nullptr);
      const int vb = more ? vn : 0;
      if (wn) {
#pragma unroll
        for (int u = 0; u < D1_UNR; ++u) {
          const int v = vb + lane + 32 * u;
          w[u] = (v < KV) ? ldg_stream(wn + v) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
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
    if (lane == 0) {
      if (EPI == DN_PROJ && r >= p.R0) {
        const uint16_t zb = f32_to_bf16_bits(sum);
        p.out1[r - p.R0] = zb;
        atomicMax(p.zmax, __float_as_uint(fabsf(bf16_bits_to_f32(zb))));
      } else if (EPI == DN_ACC) {
        p.out0[r] += sum;
      } else {
        p.out0[r] = sum;
      }
    }
  }
}

}  // namespace k3

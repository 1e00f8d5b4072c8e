// k3_tc.cuh -- tensor-core (tcgen05 / TMEM / TMA) GEMMs for large token counts.
//
// D[M, N] = A[M, K] . B[N, K]^T, both operands K-major bf16, fp32 accumulation in
// tensor memory.  One CTA per SM, persistent over output tiles of 128 x 256:
//   warp 0      TMA producer: A and B k-blocks (64 wide, 128-byte swizzle) into a
//               STAGES-deep shared-memory ring (mbarrier full/empty pairs);
//   warp 1      allocates 512 TMEM columns (two 256-column accumulators) and issues
//               tcgen05.mma (M 128, N 256, K 16) from one elected lane; completion
//               of each k-block frees its stage (tcgen05.commit -> empty), completion
//               of a tile hands its accumulator to the epilogue;
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quarter, conversion, stores;
//               the accumulator is released for the tile after next.
// Every mbarrier wait is bounded (about 2 s of clock); a wait that runs out sets
// K3MOE_DEV_TIMEOUT in the status word and all roles drain and exit (TMEM is freed).
#pragma once

#include <cuda.h>

#include "k3_common.cuh"

namespace k3 {

// ---------------------------------------------------------------------------- PTX wrappers
K3_DEVI void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
K3_DEVI void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
K3_DEVI void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
K3_DEVI bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// As mbar_try_wait, but a thread whose phase is still open is suspended until the
// phase completes or about `ns` nanoseconds pass (so waiting warps leave the issue
// slots to the warps doing work).
K3_DEVI bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity.  Returns false when the CTA's
// abort flag is set (by this or another thread) or the wait exceeds `limit` cycles
// (~2^32 in the kernels; the self-test uses a short one).
K3_DEVI bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, long long limit = (1ll << 32)) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait_sleep(bar, parity, 10000u)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      *abort_flag = 1;
      return false;
    }
  }
}

// Non-suspending test of the phase with the given parity.
K3_DEVI bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// As mbar_wait, for the single thread that issues MMAs: hardware-suspending try_wait
// without a time hint (the thread resumes when the phase completes), so that a waiting
// issuer takes no issue slots from the warps that decode the next stage on its
// sub-partition (a test_wait spin loop had cost them a large share of the integer pipe).
K3_DEVI bool mbar_wait_issue(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_test(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > (1ll << 32)) {
      *abort_flag = 1;
      return false;
    }
  }
}

K3_DEVI void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          dst),
      "l"(map), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
// an L2 policy that makes the lines a copy brings in the first to be evicted (the weight
// streams of the decode GEMVs: read once per call)
K3_DEVI uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}
K3_DEVI void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(map) : "memory");
}
// Tensor maps rewritten on the device: the global address of a map held in shared memory,
// the warp-wide copy of that map to global memory with a release fence for the tensor-map
// proxy, and the acquire fence before a copy uses the global map.
K3_DEVI void tmap_replace_addr(uint32_t smem_map, const void* gaddr) {
  asm volatile("tensormap.replace.tile.global_address.shared::cta.b1024.b64 [%0], %1;\n" ::"r"(smem_map), "l"(gaddr)
               : "memory");
}
K3_DEVI void tmap_store_release(void* gmem_map, uint32_t smem_map) {
  asm volatile(
      "tensormap.cp_fenceproxy.global.shared::cta.tensormap::generic.release.gpu.sync.aligned [%0], [%1], 128;\n" ::"l"(
          gmem_map),
      "r"(smem_map)
      : "memory");
}
K3_DEVI void tmap_acquire(const void* gmem_map) {
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;\n" ::"l"(gmem_map) : "memory");
}
K3_DEVI void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
// arrival on the barrier once all of this thread's earlier cp.async copies have landed (the
// barrier's expected count includes it)
K3_DEVI void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}

K3_DEVI void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
K3_DEVI void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory"); }
K3_DEVI void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}
K3_DEVI void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
K3_DEVI void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
// make generic-proxy shared-memory writes visible to the async proxy (tensor core reads)
K3_DEVI void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
K3_DEVI void fence_barrier_init() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 in, fp32 accumulate)
K3_DEVI void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.u32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive on `bar` once all previously issued tcgen05.mma of this thread have completed
K3_DEVI void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar) : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns (this warp's lane quarter)
K3_DEVI void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns
K3_DEVI void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
K3_DEVI void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, rows of 128 bytes with the 128-byte
// swizzle, 8-row groups 1024 bytes apart (the layout TMA writes with SWIZZLE_128B and a
// 64 x bf16 inner box).  Advancing along K inside the 128-byte row adds to the address.
K3_DEVI uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                            // leading-dimension byte offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;                  // stride-dimension byte offset
  d |= (uint64_t)1 << 46;                            // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;                            // 128-byte swizzle
  return d;
}
// Instruction descriptor, kind::f16: bf16 A and B (K-major), fp32 D, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------------------- dense GEMM
constexpr int TC_BM = 128, TC_BN = 256, TC_BK = 64, TC_STAGES = 4;
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;  // 16 KB
constexpr int TC_B_BYTES = TC_BN * TC_BK * 2;  // 32 KB
constexpr int TC_STAGE_BYTES = TC_A_BYTES + TC_B_BYTES;
constexpr int TC_THREADS = 192;
constexpr int TC_SMEM = 1024 + TC_STAGES * TC_STAGE_BYTES + 256;  // alignment slack, ring, barriers

enum { TC_PROJ = 0, TC_PLAIN = 1, TC_ACC = 2 };  // ACC: out0 += the product

struct TcDenseParams {
  int M;       // rows of A (tokens)
  int N0, N1;  // output features from B map 0 and from B map 1 (0: none)
  int K;       // reduction length (multiple of 64)
  float* out0;     // PROJ: logits [M, N0]; PLAIN: out [M, N0]; ACC: out [M, N0], added to
  uint16_t* out1;  // PROJ: z [M, N1] bf16
  uint32_t* zmax;  // PROJ: per-row max |z| (f32 bits)
  uint32_t* status;
  // split-K (few rows: too few output tiles to fill the GPU): ksplit > 1 CTAs share each
  // tile, each over kblocks / ksplit of the k-blocks, and write raw fp32 partial sums to
  // part [ksplit][M][N0 + N1]; k3_tc_splitk_reduce_kernel adds them in order and applies
  // the epilogue
  int ksplit;
  float* part;
};

template <int EPI>
__global__ void __launch_bounds__(TC_THREADS, 1)
    k3_tc_dense_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB0,
                       const __grid_constant__ CUtensorMap mapB1, TcDenseParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1024-byte alignment
  const uint32_t bars = base + TC_STAGES * TC_STAGE_BYTES;
  auto full_bar = [&](int s) { return bars + 8 * s; };
  auto empty_bar = [&](int s) { return bars + 8 * (TC_STAGES + s); };
  auto tfull_bar = [&](int b) { return bars + 8 * (2 * TC_STAGES + b); };
  auto tempty_bar = [&](int b) { return bars + 8 * (2 * TC_STAGES + 2 + b); };
  const uint32_t done_bar = bars + 8 * (2 * TC_STAGES + 4);
  volatile int* abort_flag = &abort_sh;

  const int m_tiles = (p.M + TC_BM - 1) / TC_BM;
  const int n_t0 = (p.N0 + TC_BN - 1) / TC_BN, n_t1 = (p.N1 + TC_BN - 1) / TC_BN;
  const int otiles = m_tiles * (n_t0 + n_t1);  // output tiles
  const int ks = p.ksplit > 1 ? p.ksplit : 1;
  const int tiles = otiles * ks;               // work units: output tile x k-range
  const int kblocks = p.K / TC_BK / ks;        // k-blocks per work unit

  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int s = 0; s < TC_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 128);
    }
    mbar_init(done_bar, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB0);
    if (p.N1 > 0) tma_prefetch_desc(&mapB1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  grid_dep_wait();
  grid_dep_launch();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int it = 0;
      for (int tile = blockIdx.x; tile < tiles && !*abort_flag; tile += gridDim.x) {
        const int ot = tile % otiles, kb0 = (tile / otiles) * kblocks;
        const int tm = ot % m_tiles, tn = ot / m_tiles;
        const bool b1 = tn >= n_t0;
        const CUtensorMap* mb = b1 ? &mapB1 : &mapB0;
        const int n0 = (b1 ? tn - n_t0 : tn) * TC_BN;
        for (int kb = kb0; kb < kb0 + kblocks; ++kb, ++it) {
          const int s = it % TC_STAGES;
          if (!mbar_wait(empty_bar(s), ((it / TC_STAGES) & 1) ^ 1, abort_flag)) break;
          const uint32_t st = base + s * TC_STAGE_BYTES;
          mbar_expect_tx(full_bar(s), TC_STAGE_BYTES);
          tma_load_2d(st, &mapA, kb * TC_BK, tm * TC_BM, full_bar(s));
          tma_load_2d(st + TC_A_BYTES, mb, kb * TC_BK, n0, full_bar(s));
        }
      }
      // drain: every issued stage must have landed before the CTA exits
      for (int s = 0; s < TC_STAGES; ++s) {
        const int last = it - 1 - ((it - 1 - s) % TC_STAGES + TC_STAGES) % TC_STAGES;  // last issue into stage s
        if (last >= 0 && last < it) {
          volatile int never = 0;
          mbar_wait(full_bar(s), (last / TC_STAGES) & 1, &never);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(TC_BM, TC_BN);
      int it = 0, lt = 0;
      for (int tile = blockIdx.x; tile < tiles && !*abort_flag; tile += gridDim.x, ++lt) {
        const int b = lt & 1;
        if (!mbar_wait(tempty_bar(b), ((lt >> 1) & 1) ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + b * TC_BN;
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {  // k-blocks of the work unit, counted from 0
          const int s = it % TC_STAGES;
          if (!mbar_wait(full_bar(s), (it / TC_STAGES) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = base + s * TC_STAGE_BYTES;
#pragma unroll
          for (int k = 0; k < TC_BK / 16; ++k)
            tc_mma(d, sdesc_sw128(st + k * 32), sdesc_sw128(st + TC_A_BYTES + k * 32), idesc, (kb | k) != 0);
          tc_commit(empty_bar(s));
        }
        if (!ok) break;
        tc_commit(tfull_bar(b));
      }
      // all MMAs issued by this thread have completed once done_bar flips
      tc_commit(done_bar);
      volatile int never = 0;
      mbar_wait(done_bar, 0, &never);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int lt = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++lt) {
      const int b = lt & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(tfull_bar(b), (lt >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      const int ot = tile % otiles, kq = tile / otiles;
      const int tm = ot % m_tiles, tn = ot / m_tiles;
      const bool b1 = tn >= n_t0;
      const int n0 = (b1 ? tn - n_t0 : tn) * TC_BN;
      const int row = tm * TC_BM + q * 32 + lane;
      const int N = b1 ? p.N1 : p.N0;
      float zm = 0.f;
#pragma unroll 1
      for (int c = 0; c < TC_BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + b * TC_BN + c * 32, r);
        tmem_ld_wait();
        const int col0 = n0 + c * 32;
        if (row < p.M && col0 < N) {
          if (ks > 1) {
            // raw partial sums of this k-range: part[kq][row][(N0 if b1) + col]
            const int NT = p.N0 + p.N1;
            float* dst = p.part + ((size_t)kq * p.M + row) * NT + (b1 ? p.N0 : 0) + col0;
            if (col0 + 32 <= N && (NT % 4) == 0 && (p.N0 % 4) == 0) {
#pragma unroll
              for (int v = 0; v < 8; ++v)
                reinterpret_cast<float4*>(dst)[v] =
                    make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
            } else {
              for (int e = 0; e < 32 && col0 + e < N; ++e) dst[e] = __uint_as_float(r[e]);
            }
          } else if (EPI == TC_PROJ && b1) {
            uint16_t* dst = p.out1 + (size_t)row * p.N1 + col0;
            if (col0 + 32 <= N) {
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const uint16_t lo = f32_to_bf16_bits(__uint_as_float(r[8 * v + 2 * e]));
                  const uint16_t hi = f32_to_bf16_bits(__uint_as_float(r[8 * v + 2 * e + 1]));
                  zm = fmaxf(zm, fmaxf(fabsf(bf16_bits_to_f32(lo)), fabsf(bf16_bits_to_f32(hi))));
                  w[e] = (uint32_t)lo | ((uint32_t)hi << 16);
                }
                reinterpret_cast<uint4*>(dst)[v] = make_uint4(w[0], w[1], w[2], w[3]);
              }
            } else {
              for (int e = 0; e < 32 && col0 + e < N; ++e) {
                const uint16_t h = f32_to_bf16_bits(__uint_as_float(r[e]));
                zm = fmaxf(zm, fabsf(bf16_bits_to_f32(h)));
                dst[e] = h;
              }
            }
          } else {
            float* dst = p.out0 + (size_t)row * p.N0 + col0;
            if (col0 + 32 <= N && (p.N0 % 4) == 0) {
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                float4 o = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                       __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                if (EPI == TC_ACC) {
                  const float4 prev = reinterpret_cast<const float4*>(dst)[v];
                  o = make_float4(prev.x + o.x, prev.y + o.y, prev.z + o.z, prev.w + o.w);
                }
                reinterpret_cast<float4*>(dst)[v] = o;
              }
            } else {
              for (int e = 0; e < 32 && col0 + e < N; ++e)
                dst[e] = (EPI == TC_ACC) ? dst[e] + __uint_as_float(r[e]) : __uint_as_float(r[e]);
            }
          }
        }
      }
      if (EPI == TC_PROJ && b1 && ks == 1 && row < p.M) atomicMax(p.zmax + row, __float_as_uint(zm));
      tc_fence_before();
      mbar_arrive(tempty_bar(b));
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) flag_status(p.status, K3MOE_DEV_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Split-K epilogue: CTA (row, column chunk of TC_RED_COLS); out = sum of the ksplit
// partials in order, then the dense epilogue (PLAIN: out0; ACC: out0 +=; PROJ: logits for
// the first N0 columns, z (bf16) and the row's max |z| for the next N1)
constexpr int TC_RED_COLS = 1024;
template <int EPI>
__global__ void __launch_bounds__(256) k3_tc_splitk_reduce_kernel(TcDenseParams p) {
  grid_dep_wait();
  grid_dep_launch();
  const int row = blockIdx.x, NT = p.N0 + p.N1;
  const int c_end = min(NT, (int)(blockIdx.y + 1) * TC_RED_COLS);
  __shared__ float wmax[8];
  float zm = 0.f;
  for (int c = blockIdx.y * TC_RED_COLS + threadIdx.x; c < c_end; c += blockDim.x) {
    float sum = 0.f;
    for (int kq = 0; kq < p.ksplit; ++kq) sum += p.part[((size_t)kq * p.M + row) * NT + c];
    if (c < p.N0) {
      float* o = p.out0 + (size_t)row * p.N0 + c;
      *o = (EPI == TC_ACC) ? *o + sum : sum;
    } else {
      const uint16_t zb = f32_to_bf16_bits(sum);
      p.out1[(size_t)row * p.N1 + (c - p.N0)] = zb;
      zm = fmaxf(zm, fabsf(bf16_bits_to_f32(zb)));
    }
  }
  if (EPI == TC_PROJ && p.N1 > 0) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) zm = fmaxf(zm, __shfl_xor_sync(0xffffffffu, zm, off));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = zm;
    __syncthreads();
    if (threadIdx.x == 0) {
      float m = 0.f;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, wmax[w]);
      atomicMax(p.zmax + row, __float_as_uint(m));
    }
  }
}

}  // namespace k3

namespace k3 {

// ---------------------------------------------------------------------------- grouped MXFP4 GEMM
// Per token batch (up to TM_NB tokens of one expert) and 128-row tile of the expert's
// weight matrix:  D[rows, tokens] = W[rows, K] . Act[tokens, K]^T  with
//   A = W decoded by producer warps from the vendor MXFP4 bytes into TENSOR MEMORY
//       (tcgen05.st; row i in lane i, two bf16 per 32-bit column, K along columns):
//       integer operations place each E2M1 code's sign, exponent and mantissa bits in
//       a bf16 word (the value v * 2^-126, exact, subnormal for the code 0.5), and one
//       bf16x2 multiply by a power of two (two when the scale byte exceeds 128) gives
//       v * 2^(s-127), exact in bf16 for every scale byte 0..252 (every e2m1 value
//       times 2^k with k in [-127, 125] is a bf16 number);
//       the vendor bytes reach shared memory through a chunk ring filled by a copy warp
//       (TMA for the packed bytes, through tensor maps whose global address is set to
//       the tile's expert tensor on the device; cp.async for the scale bytes);
//   B = the batch's activation rows in slot order (the bf16 values themselves) loaded
//       by TMA into shared memory (128-byte swizzle);
//   fp32 accumulation in TMEM (kind::f16 with bf16 A and B, M 128, N = tokens rounded
//   up to 16).
// Both operands hold the K dimension in the same interleaved order: within every group
// of 8 consecutive elements, positions 0..7 hold elements 0, 4, 1, 5, 2, 6, 3, 7 (the
// order in which one 32-bit word of packed codes decodes into four bf16 pairs with
// the same shifts in both halves).  A dot product does not depend on the order of its
// terms' positions, so the products are those of the natural order; the activation
// rows are written in this order by the gather (z) and by the gate/up epilogue (h).
// Keeping A out of shared memory leaves shared-memory bandwidth to B and the raw bytes
// (with A in shared memory the decoded tile is written and then read again by the
// tensor core, which made the kernel shared-memory bound at these small N).
// GATEUP: two matrices (gate rows, up rows) share B; the epilogue applies SiTU-GLU,
// rounds h to bf16 and stores it in slot order (interleaved K order, for the down
// GEMM).  DOWN: one matrix; the epilogue stores o (fp32) in slot order.
constexpr int TM_ROWS = 128;       // weight rows per MMA (M)
constexpr int TM_BLOCKS = 2;       // row blocks per tile, each with its own accumulator and MMA issuer
constexpr int TM_NB = 96;          // tokens per batch (MMA N <= 96): bounded by TMEM columns
constexpr int TM_BK = 64;          // k-block
constexpr int TM_PRODUCERS = 16;   // decode warps
constexpr int TM_EPI = 8;         // epilogue warps: two per TMEM lane quarter, alternate 16-column chunks
constexpr int TM_COPY_WARP = 3 + TM_EPI + TM_PRODUCERS;  // packed-weight TMA copies
constexpr int TM_THREADS = (TM_COPY_WARP + 1) * 32;
constexpr int TM_B_BYTES = TM_NB * TM_BK * 2;  // 12 KB
constexpr int TM_AKB = 2;          // k-blocks per A stage (one barrier round trip per stage)

// Tile = 2 row blocks of 128 weight rows x one token batch.  GATEUP: block 0 = gate rows
// 128 t .. 128 t + 127, block 1 = the same rows of the up matrix; DOWN: blocks 0 and 1 =
// rows 256 t .. 256 t + 255 of the down matrix.  Two blocks, two accumulators and two
// issuing threads: one thread issues a kind::f16 MMA no faster than about every 100
// cycles at these N, two in parallel double the tensor-core rate.
template <int MODE>
struct TmLayout {
  static constexpr int MROWS = TM_BLOCKS * TM_ROWS;   // 256 weight rows per tile
  static constexpr int TILE_ROWS = (MODE == 0) ? TM_ROWS : MROWS;  // output rows per tile
  // TMEM columns: one accumulator buffer (2 blocks x TM_NB), then SA A stages of
  // TM_AKB k-blocks (64 columns = 128 f16 per block per stage).  The epilogue empties the
  // accumulators into shared memory (GATEUP) or global memory (DOWN) at once, so one
  // buffer suffices and the columns go to A stages, which the MMA-completion -> decode ->
  // MMA chain needs.
  static constexpr int ACC = TM_BLOCKS * TM_NB;
  static constexpr int SA = 2;
  static constexpr int A_COLS = TM_AKB * 32;          // per block per stage
  static constexpr int A_COL0 = ACC;
  static_assert(A_COL0 + SA * TM_BLOCKS * A_COLS <= 512, "TMEM columns");
  // B slots (one k-block each, shared memory) in NBS groups of TM_AKB: group st % NBS
  // holds stage st's token tiles, so TMA runs up to NBS stages ahead (NBS >= SA)
  static constexpr int SB = (MODE == 0) ? 4 : 8;
  static constexpr int NBS = SB / TM_AKB;
  static_assert(SB % TM_AKB == 0 && NBS >= SA, "B slot groups");
  // raw chunks: CKB k-blocks = CKB * 32 bytes of every row
  static constexpr int CKB = 4;
  static constexpr int ROWB = CKB * 32;                // raw bytes per row per chunk
  static constexpr int GPR = ROWB / 16;                // 16-byte granules per row per chunk
  static_assert(CKB % TM_AKB == 0, "chunks hold whole A stages");
  static constexpr int RC = (MODE == 0) ? 2 : 3;      // raw chunks in flight
  static constexpr int RAW_SLOT = MROWS * ROWB;
  static constexpr int SC_SLOT = MROWS * CKB * 2;     // two scale bytes per row per k-block
  // GATEUP staging of the accumulators: per epilogue thread up to 3 chunks x (16 g + 16 u)
  static constexpr int STG_WORDS = (MODE == 0) ? (TM_NB / 16 / 2) * 32 : 0;
  static constexpr int STG = STG_WORDS * TM_EPI * 32 * 4;
  // barriers (512 bytes), then a shared-memory copy of each block's packed-weight tensor map
  static constexpr int SMEM = 1024 + SB * TM_B_BYTES + RC * (RAW_SLOT + SC_SLOT) + STG + 512 + TM_BLOCKS * 128;
};

// CTAs of one grouped-GEMM launch at most (sizes the per-warp tensor-map workspace)
constexpr int TM_MAX_CTAS = 256;

struct TcMoeParams {
  const MxBatch* batches;    // token batches of up to TM_NB tokens (one expert each)
  const int32_t* n_batches;
  int R;                     // rows per matrix (I for gate/up, L for down)
  int K;                     // reduction length (L or I)
  void* out;                 // GATEUP: h [slots, R] bf16 (interleaved K order); DOWN: o f32 [slots, R]
  uint32_t* status;
  void* tmaps;               // packed-weight tensor maps, [TM_MAX_CTAS][TM_BLOCKS][2] x 128 bytes
};

// Eight E2M1 codes (one 32-bit word of packed bytes, low nibble first: codes c0..c7 of
// eight consecutive elements) -> four bf16x2 words holding v * 2^-126 for the code
// pairs [c0 c4] [c1 c5] [c2 c6] [c3 c7] (low half first).  A code s e1 e0 m shifted
// into bits 15 (sign) and 8..6 (exponent bits 1..0, mantissa bit 6) is the bf16 number
// v * 2^-126: for e > 0 the exponent field e gives 2^(e-127) (1 + m/2) = 2^(e-1) (1 + m/2)
// * 2^-126, and for e = 0 the subnormal m * 2^-127 = (m/2) * 2^-126.  The multiply by
// 0x1040 (or 0x104 for a high nibble) copies the masked nibble of both halves to bit
// offsets +6 and +12 at once (no carries between the copies); the mask keeps the sign
// from the second copy and the magnitude from the first.
K3_DEVI void e2m1x8_to_bf16x8_il(uint32_t w, uint32_t (&o)[4]) {
  const uint32_t w8 = w >> 8;
  o[0] = ((w & 0x000F000Fu) * 0x1040u) & 0x81C081C0u;
  o[1] = ((w & 0x00F000F0u) * 0x104u) & 0x81C081C0u;
  o[2] = ((w8 & 0x000F000Fu) * 0x1040u) & 0x81C081C0u;
  o[3] = ((w8 & 0x00F000F0u) * 0x104u) & 0x81C081C0u;
}

// d = a * b on two bf16 lanes, round to nearest (exact for power-of-two b unless the
// product leaves the bf16 range)
K3_DEVI uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// position of element j (0..7) of an 8-element group in the interleaved K order
K3_DEVI int il_pos(int j) { return (j < 4) ? 2 * j : 2 * (j - 4) + 1; }

// An empty statement reading 16 registers: keeps the source of an in-flight tcgen05.st
// allocated (the compiler does not know the store reads them until tcgen05.wait::st)
K3_DEVI void keep_regs16(const uint32_t (&r)[16]) {
  asm volatile("" ::"r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
               "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]));
}
// TMEM store: each lane of the warp writes 16 consecutive 32-bit columns of its own lane
// of the warp's lane quarter
K3_DEVI void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
K3_DEVI void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16
K3_DEVI void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.u32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}


template <int MODE>
__global__ void __launch_bounds__(TM_THREADS, 1) k3_tc_moe_kernel(const __grid_constant__ CUtensorMap mapB,
                                                                  const __grid_constant__ CUtensorMap mapA,
                                                                  TcMoeParams p) {
  using Lay = TmLayout<MODE>;
  constexpr int SA = Lay::SA, SB = Lay::SB, RC = Lay::RC, MROWS = Lay::MROWS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // B stages [SB][TM_NB rows][128 bytes]
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t raw_base = base + SB * TM_B_BYTES;         // [RC][MROWS rows][ROWB bytes]
  const uint32_t sraw_base = raw_base + RC * Lay::RAW_SLOT;  // [RC][MROWS rows][2 CKB bytes]
  const uint32_t stg_base = sraw_base + RC * Lay::SC_SLOT;  // [STG_WORDS][epilogue thread] f32
  const uint32_t bars = stg_base + Lay::STG;
  const uint32_t smaps = bars + 512;  // [TM_BLOCKS][128 bytes] tensor maps
  // Stage st = TM_AKB k-blocks: A in TMEM slot st % SA, B in shared-memory group st % NBS.
  // full(g): the stage in group g is ready -- all producer warps stored their A rows
  // (one arrival each) and the TMA landed its B tiles (the TMA thread's arrival with the
  // byte count) -- so an issuer tests one barrier per stage; kdone(g): both issuers' MMAs
  // of the stage in group g completed, which frees its B group and (NBS >= SA) its A slot:
  // one commit per stage serves both rings.
  constexpr int NBS = Lay::NBS;
  auto full = [&](int g) { return bars + 8 * g; };
  auto kdone = [&](int g) { return bars + 8 * (NBS + g); };
  constexpr int NB0 = 2 * NBS;
  auto tfull = [&](int b) { return bars + 8 * (NB0 + b); };
  auto tempty = [&](int b) { return bars + 8 * (NB0 + 2 + b); };
  const uint32_t done_bar = bars + 8 * (NB0 + 4);
  // raw_full(s): the packed and scale bytes of the chunk in slot s landed (the copy warp's
  // lane 0 arrives with the TMA byte count, each of its lanes once its scale copies land);
  // raw_empty(s): every producer warp is done with the slot's chunk
  auto raw_full = [&](int s) { return bars + 8 * (NB0 + 5 + s); };
  auto raw_empty = [&](int s) { return bars + 8 * (NB0 + 5 + RC + s); };
  static_assert(8 * (NB0 + 5 + 2 * RC) <= 512, "barrier space");
  volatile int* abort_flag = &abort_sh;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int g = 0; g < NBS; ++g) {
      mbar_init(full(g), TM_PRODUCERS + 1);  // producer warps + the TMA thread
      mbar_init(kdone(g), TM_BLOCKS);        // one commit per issuer
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull(b), TM_BLOCKS);
      mbar_init(tempty(b), TM_EPI * 32);
    }
    mbar_init(done_bar, TM_BLOCKS);
    for (int r = 0; r < RC; ++r) {
      mbar_init(raw_full(r), 1 + 32);
      mbar_init(raw_empty(r), TM_PRODUCERS);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&mapB);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  grid_dep_wait();
  grid_dep_launch();

  const int mtiles = p.R / Lay::TILE_ROWS;
  const int tiles = mtiles * (*p.n_batches);
  const int kblocks = p.K / TM_BK;
  // weight tensor (index into MxBatch::w) and first row of block mm of row tile tm
  auto blk_tensor = [](int mm) { return (MODE == 0) ? 2 * mm : 4; };
  auto blk_row0 = [](int tm, int mm) { return (MODE == 0) ? (size_t)tm * TM_ROWS : (size_t)tm * MROWS + mm * TM_ROWS; };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (B)
    if (lane == 0) {
      int bs = 0;  // stages loaded
      for (int tile = blockIdx.x; tile < tiles && !*abort_flag; tile += gridDim.x) {
        const int slot0 = p.batches[tile / mtiles].slot0;
        for (int kb = 0; kb < kblocks; kb += TM_AKB, ++bs) {
          // group bs % NBS last held stage bs - NBS
          const int g = bs % NBS;
          if (!mbar_wait(kdone(g), ((bs / NBS) & 1) ^ 1, abort_flag)) break;
          mbar_expect_tx(full(g), TM_AKB * TM_B_BYTES);
#pragma unroll
          for (int kk = 0; kk < TM_AKB; ++kk)
            tma_load_2d(base + (g * TM_AKB + kk) * TM_B_BYTES, &mapB, (kb + kk) * TM_BK, slot0, full(g));
        }
      }
      // drain issued loads: the stage's phase completes once its bytes landed (and the
      // producers arrived).  After an abort the producers may never arrive: wait a bounded
      // time, far beyond a copy's latency, instead.
      const bool aborted = *abort_flag != 0;
      for (int g = 0; g < NBS; ++g) {
        const int last = bs - 1 - ((bs - 1 - g) % NBS + NBS) % NBS;
        if (last >= 0 && last < bs) {
          if (!aborted) {
            volatile int never = 0;
            mbar_wait(full(g), (last / NBS) & 1, &never);
          } else {
            const long long t0 = clock64();
            while (!mbar_test(full(g), (last / NBS) & 1) && clock64() - t0 < (1ll << 21)) {
            }
          }
        }
      }
    }
  } else if (warp <= TM_BLOCKS) {
    // ------------------------------------------------------------ MMA issuers (warp 1: block 0, warp 2: block 1)
    if (lane == 0) {
      const int mm = warp - 1;
      // B descriptors differ only in their start-address field: add (offset >> 4) to the
      // stage-0 descriptor (addresses stay below 2^18, so the 14-bit field never carries)
      const uint64_t dB = sdesc_sw128(base);
      int it = 0, lt = 0;
      for (int tile = blockIdx.x; tile < tiles && !*abort_flag; tile += gridDim.x, ++lt) {
        const int n = p.batches[tile / mtiles].n;
        const int N = (n + 15) & ~15;
        const uint32_t idesc = idesc_bf16(TM_ROWS, N);  // bf16 x bf16 -> f32
        if (!mbar_wait_issue(tempty(0), (lt & 1) ^ 1, abort_flag)) break;  // accumulators emptied
        tc_fence_after();
        const uint32_t d = tmem + mm * TM_NB;
        bool ok = true;
        for (int kb = 0; kb < kblocks; kb += TM_AKB, it += TM_AKB) {
          const int st = it / TM_AKB, sa = st % SA, g = st % NBS;
          if (!mbar_wait_issue(full(g), (st / NBS) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ta = tmem + Lay::A_COL0 + (sa * TM_BLOCKS + mm) * Lay::A_COLS;
#pragma unroll
          for (int kk = 0; kk < TM_AKB; ++kk) {
            const uint64_t db = dB + ((uint32_t)((g * TM_AKB + kk) * TM_B_BYTES) >> 4);
#pragma unroll
            for (int k = 0; k < TM_BK / 16; ++k)
              tc_mma_ts(d, ta + kk * 32 + 8 * k, db + 2 * k, idesc, (kb | kk | k) != 0);
          }
          tc_commit(kdone(g));
        }
        if (!ok) break;
        tc_commit(tfull(0));
      }
      tc_commit(done_bar);
      volatile int never = 0;
      mbar_wait(done_bar, 0, &never);
    }
  } else if (warp < 3 + TM_EPI) {
    // ------------------------------------------------------------ epilogue (warps 3..10)
    // warp w reads TMEM lane quarter w % 4 (32 weight rows) and the 16-column chunks
    // e, e + 2, e + 4 of the batch's tokens (e = 0 for warps 3..6, 1 for 7..10).  It first
    // empties its accumulator chunks (GATEUP: into its own shared-memory words; DOWN:
    // straight to the output) and releases TMEM, then (GATEUP) applies SiTU-GLU while the
    // next tile's MMAs run.
    const int q = warp & 3;
    const int e0 = (warp - 3) >> 2;
    const int et = threadIdx.x - 3 * 32;  // epilogue thread 0..255
    float* stg = reinterpret_cast<float*>(base_ptr + (stg_base - base)) + et;  // word k at stg[k * 256]
    int lt = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++lt) {
      // warp-uniform outcome: the tcgen05.ld below must be executed by all 32 lanes
      if (!__all_sync(0xffffffffu, mbar_wait(tfull(0), lt & 1, abort_flag))) break;
      tc_fence_after();
      const MxBatch* rec = p.batches + tile / mtiles;
      const int slot0 = rec->slot0, n = rec->n;
      const int tm = tile % mtiles;
      const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int c = e0, k = 0; c * 16 < n; c += 2, ++k) {
        uint32_t r0[16], r1[16];
        tmem_ld16(tq + c * 16, r0);
        tmem_ld16(tq + TM_NB + c * 16, r1);
        tmem_ld_wait();
        if (MODE == 0) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            stg[(k * 32 + j) * (TM_EPI * 32)] = __uint_as_float(r0[j]);
            stg[(k * 32 + 16 + j) * (TM_EPI * 32)] = __uint_as_float(r1[j]);
          }
        } else {
          const int row0 = tm * MROWS + q * 32 + lane;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = c * 16 + j;
            if (col < n) {
              float* o = reinterpret_cast<float*>(p.out) + (size_t)(slot0 + col) * p.R + row0;
              o[0] = __uint_as_float(r0[j]);
              o[TM_ROWS] = __uint_as_float(r1[j]);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty(0));
      if (MODE == 0) {
        // h element `row` of each token, stored at its place in the interleaved K order
        const int row = tm * TM_ROWS + q * 32 + lane;
        const int hcol = (row & ~7) + il_pos(row & 7);
#pragma unroll 1
        for (int c = e0, k = 0; c * 16 < n; c += 2, ++k) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = c * 16 + j;
            if (col < n) {
              const float gg = stg[(k * 32 + j) * (TM_EPI * 32)];
              const float uu = stg[(k * 32 + 16 + j) * (TM_EPI * 32)];
              reinterpret_cast<uint16_t*>(p.out)[(size_t)(slot0 + col) * p.R + hcol] =
                  f32_to_bf16_bits(situ_fast(gg, uu));  // bf16 rounding of h
            }
          }
        }
      }
    }
  } else if (warp == TM_COPY_WARP) {
    // ------------------------------------------------------------ packed-weight copies (warp 27)
    // The packed bytes of a tile travel in chunks of CKB k-blocks (ROWB bytes of each of its
    // 256 rows) through a ring of RC slots: per chunk one TMA copy per block (128 rows x
    // ROWB bytes; the 128-byte swizzle puts 16-byte granule c of row r at c ^ (r & 7), the
    // layout the decode reads), issued once all producer warps are done with the slot.
    // The tensor maps take the tile's expert tensors as global addresses, rewritten on the
    // device when the tile changes; two per block in global memory, used by alternate tiles,
    // so a map is rewritten only after every copy of the tile before last has landed.
    constexpr int CKB = Lay::CKB, ROWB = Lay::ROWB;
    static_assert(ROWB == 128, "the TMA 128-byte swizzle matches the granule layout for 128-byte rows");
    const int kchunks = kblocks / CKB;
    const int my_tiles = (tiles > (int)blockIdx.x) ? (tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int nchunks = my_tiles * kchunks;
    uint8_t* gmaps = reinterpret_cast<uint8_t*>(p.tmaps) + (size_t)blockIdx.x * (TM_BLOCKS * 2 * 128);
    auto gmap = [&](int b, int par) { return gmaps + (b * 2 + par) * 128; };
#pragma unroll
    for (int b = 0; b < TM_BLOCKS; ++b)
      reinterpret_cast<uint32_t*>(base_ptr + (smaps + b * 128 - base))[lane] = reinterpret_cast<const uint32_t*>(&mapA)[lane];
    __syncwarp();
    const size_t srow = (size_t)p.K / 32;
    const uint8_t* sc_t[TM_BLOCKS] = {nullptr, nullptr};  // the tile's scale tensors, at its first row
    int cur_tile = -1, par = 1, tm = 0, n_issued = 0;
#pragma unroll 1
    for (int jc = 0; jc < nchunks && !*abort_flag; ++jc) {
      const int slot = jc % RC;
      // the slot's previous chunk (jc - RC) has been decoded by every producer warp
      if (jc >= RC && !__all_sync(0xffffffffu, mbar_wait(raw_empty(slot), ((jc / RC) - 1) & 1, abort_flag))) break;
      const int tile = blockIdx.x + (jc / kchunks) * gridDim.x, kc = jc % kchunks;
      if (tile != cur_tile) {  // warp-uniform
        const MxBatch* rec = p.batches + tile / mtiles;
        const uint8_t* q0 = rec->w[blk_tensor(0)];
        const uint8_t* q1 = rec->w[blk_tensor(1)];
        if (((reinterpret_cast<uintptr_t>(q0) | reinterpret_cast<uintptr_t>(q1)) & 15u) != 0) {
          // a TMA source must be 16-byte aligned: abandon the call
          if (lane == 0) flag_status(p.status, K3MOE_DEV_ALIGN);
          *abort_flag = 1;
          break;
        }
        par ^= 1;
        if (lane == 0) {
          tmap_replace_addr(smaps, q0);
          tmap_replace_addr(smaps + 128, q1);
        }
        __syncwarp();
        tmap_store_release(gmap(0, par), smaps);
        tmap_store_release(gmap(1, par), smaps + 128);
        if (lane == 0) {
          tmap_acquire(gmap(0, par));
          tmap_acquire(gmap(1, par));
        }
        cur_tile = tile;
        tm = tile % mtiles;
#pragma unroll
        for (int b = 0; b < TM_BLOCKS; ++b) sc_t[b] = rec->w[blk_tensor(b) + 1] + blk_row0(tm, b) * srow;
      }
      // scale bytes: 2 CKB per row, rows lane + 32 i of the slot's 256, by cp.async; each
      // lane's arrival on raw_full fires once they land
#pragma unroll
      for (int i = 0; i < MROWS / 32; ++i) {
        const int r = lane + 32 * i, b = r / TM_ROWS;
        const uint8_t* ssrc = sc_t[b] + (size_t)(r % TM_ROWS) * srow + kc * (2 * CKB);
        const uint32_t sdst = sraw_base + slot * Lay::SC_SLOT + r * (2 * CKB);
        if constexpr (CKB == 4) cp_async8(sdst, ssrc);
        else cp_async4(sdst, ssrc);
      }
      cp_async_mbar_arrive(raw_full(slot));
      if (lane == 0) {
        mbar_expect_tx(raw_full(slot), TM_BLOCKS * TM_ROWS * ROWB);
#pragma unroll
        for (int b = 0; b < TM_BLOCKS; ++b)
          tma_load_2d(raw_base + slot * Lay::RAW_SLOT + b * TM_ROWS * ROWB, reinterpret_cast<const CUtensorMap*>(gmap(b, par)),
                      kc * ROWB, (int)blk_row0(tm, b), raw_full(slot));
      }
      n_issued = jc + 1;
    }
    // let every issued copy land before the CTA exits (after an abort some are never
    // consumed): the lanes' cp.async, then bounded waits on the last RC chunks
    cp_async_wait<0>();
    if (lane == 0) {
      for (int j = (n_issued > RC ? n_issued - RC : 0); j < n_issued; ++j) {
        const long long t0 = clock64();
        while (!mbar_test(raw_full(j % RC), (j / RC) & 1) && clock64() - t0 < (1ll << 21)) {
        }
      }
    }
  } else {
    // ------------------------------------------------------------ decode producers (warps 11..26)
    // A chunk's packed and scale bytes come from the copy warp (raw_full / raw_empty);
    // 16-byte granules are XOR-swizzled by row so the decode reads are free of bank
    // conflicts.
    // Decode: a warp owns the TMEM lane quarter warp % 4 (32 rows) of one block and one of
    // the two 32-element scale groups of every k-block (16 TMEM columns): warps 11..14
    // block 0 group 0, 15..18 block 1 group 0, 19..22 block 0 group 1, 23..26 block 1
    // group 1; each thread decodes its row's group.
    static_assert(TM_PRODUCERS == 4 * TM_BLOCKS * 2, "four lane quarters x two blocks x two groups");
    const int pw = warp - (3 + TM_EPI);
    const int qd = warp & 3;
    const int mb = (pw >> 2) % TM_BLOCKS;
    const int kg = pw / (4 * TM_BLOCKS);           // scale group within a k-block
    const int ri = mb * TM_ROWS + qd * 32 + lane;  // row of the tile (over both blocks)
    constexpr int CKB = Lay::CKB, ROWB = Lay::ROWB, GPR = Lay::GPR;
    // granule c of row r sits at position c ^ swz(r): conflict-free reads of 8 consecutive rows
    auto swz = [](int r) { return (GPR == 8) ? (r & 7) : ((r >> 1) & 3); };
    const int kchunks = kblocks / CKB;
    const int my_tiles = (tiles > (int)blockIdx.x) ? (tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int nchunks = my_tiles * kchunks;
    static_assert(CKB == 4 && TM_AKB == 2, "a chunk is two A stages of two k-blocks");
    // byte offsets of this thread's granule (its group of k-block kq) inside its row's
    // ROWB raw bytes, and the byte selector that gathers its four scale bytes (bytes
    // 2 kq + kg of the row's 8 per chunk)
    int goff[CKB];
#pragma unroll
    for (int kq = 0; kq < CKB; ++kq) goff[kq] = ((2 * kq + kg) ^ swz(ri)) << 4;
    const uint32_t ssel = kg ? 0x7531u : 0x6420u;
    bool stop = false;
#pragma unroll 1
    for (int jc = 0; jc < nchunks && !stop; ++jc) {
      // chunk jc's packed and scale bytes (the copy warp's) have landed
      if (!__all_sync(0xffffffffu, mbar_wait(raw_full(jc % RC), (jc / RC) & 1, abort_flag))) {
        stop = true;
        break;
      }
      const uint8_t* src = base_ptr + (raw_base - base) + (jc % RC) * Lay::RAW_SLOT + ri * ROWB;
      const uint2 sc8 = *reinterpret_cast<const uint2*>(base_ptr + (sraw_base - base) + (jc % RC) * Lay::SC_SLOT +
                                                        ri * (2 * CKB));
      // the decoded words are v * 2^-126, so a group's factor is 2^(s-1): a bf16 power of
      // two with exponent field s + 126 when s <= 128.  A chunk in which any thread of the
      // warp has a larger byte takes 2^127 first and then 2^(s-128) (exponent field s - 1)
      // for its bytes above 128 (1 for the others); each product is exact.
      const uint32_t s4 = __byte_perm(sc8.x, sc8.y, ssel);  // byte kq: scale byte of k-block kq
      bool bg = false;
#pragma unroll
      for (int kq = 0; kq < CKB; ++kq) bg |= ((s4 >> (8 * kq)) & 0xFFu) > 128u;
      const bool big = __any_sync(0xffffffffu, bg);  // warp-uniform
      uint32_t f1[CKB], f2[CKB];
      if (!big) {
        const uint32_t e4 = s4 + 0x7E7E7E7Eu;  // bytes s + 126 <= 254: no carries
#pragma unroll
        for (int kq = 0; kq < CKB; ++kq) {
          f1[kq] = __byte_perm(e4, 0u, 0x4040u | (kq << 8) | kq) << 7;  // [e, e] in both exponent fields
          f2[kq] = 0x3F803F80u;                                          // 1.0
        }
      } else {
#pragma unroll
        for (int kq = 0; kq < CKB; ++kq) {
          const uint32_t sb = (s4 >> (8 * kq)) & 0xFFu;
          f1[kq] = (((sb > 128u) ? 254u : sb + 126u) << 7) * 0x10001u;
          f2[kq] = (((sb > 128u) ? sb - 1u : 127u) << 7) * 0x10001u;
        }
      }
      // decode this thread's group of k-block kq (32 elements of row ri) into out[]: 16
      // bf16x2 columns in the interleaved K order
      auto decode = [&](int kq, uint32_t (&out)[16]) {
        const uint4 cq = *reinterpret_cast<const uint4*>(src + goff[kq]);
        const uint32_t w4[4] = {cq.x, cq.y, cq.z, cq.w};
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {  // 8 elements = 4 packed bytes -> 4 bf16x2 columns
          uint32_t h[4];
          e2m1x8_to_bf16x8_il(w4[cc], h);
#pragma unroll
          for (int e = 0; e < 4; ++e) out[cc * 4 + e] = bf16x2_mul(h[e], f1[kq]);
        }
        if (big) {
#pragma unroll
          for (int i = 0; i < 16; ++i) out[i] = bf16x2_mul(out[i], f2[kq]);
        }
      };
      // a tcgen05.st keeps its source registers until tcgen05.wait::st: the stage's second
      // k-block is decoded into other registers while the first one's store is in flight
      uint32_t a[16], a2[16];
#pragma unroll
      for (int h = 0; h < CKB / TM_AKB; ++h) {
        const int st = jc * (CKB / TM_AKB) + h, sa = st % SA;  // A stage and its slot
        const uint32_t ta =
            tmem + ((uint32_t)(qd * 32) << 16) + Lay::A_COL0 + (sa * TM_BLOCKS + mb) * Lay::A_COLS + kg * 16;
        decode(h * TM_AKB, a);
        // the slot's previous stage (st - SA) must have been consumed by the MMAs
        const int j = st - SA;
        if (j >= 0 && !__all_sync(0xffffffffu, mbar_wait(kdone(j % NBS), (j / NBS) & 1, abort_flag))) {
          stop = true;
          break;
        }
        tc_fence_after();
        tmem_st16(ta, a);
        decode(h * TM_AKB + 1, a2);
        tmem_st16(ta + 32, a2);
        tmem_st_wait();
        keep_regs16(a);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(full(st % NBS));
      }
      // the warp's reads of this chunk's packed bytes are done (its last decode came before
      // the TMEM store and the arrival above): the slot may be refilled
      if (!stop && lane == 0) mbar_arrive(raw_empty(jc % RC));
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) flag_status(p.status, K3MOE_DEV_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace k3

namespace k3 {

// Self-test of the bounded waits: an mbarrier that nothing arrives on.  Warp 0 waits with
// a short limit, runs out, sets the CTA's abort flag; warp 1 waits on the same barrier
// with the kernels' long limit and leaves through the abort flag.  The kernel then reports
// K3MOE_DEV_TIMEOUT as every kernel with a bounded wait does, and returns normally.
__global__ void k3_selftest_timeout_kernel(uint32_t* status, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_sh;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    abort_sh = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort_flag = &abort_sh;
  bool ok = true;
  if (warp == 0) ok = mbar_wait(smem_u32(&bar), 0, abort_flag, limit);
  else if (warp == 1) ok = mbar_wait(smem_u32(&bar), 0, abort_flag);
  (void)ok;
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) flag_status(status, K3MOE_DEV_TIMEOUT);
}

}  // namespace k3

// k3_mx8.cuh -- the grouped expert GEMM on block-scaled tcgen05.mma (kind::mxf8f6f4):
// the MXFP4 weights as stored against MXFP8 activation rows, no weight decode on the SMs.
// Two uses: the exact path's split form (SPLIT = 1: each bf16 activation as two MXFP8 terms
// hi + lo that hold it exactly, two MMAs per k-block into one accumulator; see the split
// helpers below), and the low-precision-activation variant (SPLIT = 0: one MXFP8 term).
//
// The variant follows the per-32-group quantized-activation kernel of colibri PR #676
// ("What's in the commits" item 7) and colibri PR #684 (quant.h commit: matmul_mxfp4_i8),
// in the tensor core's own microscaling form: activations become OCP MX MXFP8 (E4M3
// elements, one E8M0 scale byte per 32 consecutive elements along the contraction), the
// weights stay E2M1 with their E8M0 scale bytes, and one MMA instruction applies both
// scales per 32-element k-block:
//   D[m, n] += sum_k  w[m, k] 2^(sw[m, k/32] - 127) * a[n, k] 2^(sa[n, k/32] - 127).
// Every product of an E2M1 and an E4M3 value is exact; fp32 accumulation.
//
// Operand layouts (measured on sm_103a with a layout probe, one MMA at a time):
//   A (weights, M = 128 rows): shared memory, K-major, 128-byte swizzle; a 16-byte
//     granule holds 16 E2M1 codes in its first 8 bytes (low nibble first) and 8 bytes
//     of padding -- the layout a TMA copy of type 16U4_ALIGN16B writes from the packed
//     vendor rows (it counts the 64 packed bytes of a 128-element row, not the 128 it
//     writes).  A 128-byte smem row is 128 elements = 4 MMAs of K 32 (32 bytes each).
//   B (activations, N tokens): shared memory, K-major, 128-byte swizzle, one E4M3 byte
//     per element.
//   scale of A row m for the k-block selected by the instruction's A scale id (0..3):
//     TMEM lane m, column sfa + m / 32, byte `id` of the 32-bit word.
//   scale of B column n for the k-block of the B scale id: TMEM lane 32 q + n % 32 of
//     EVERY lane quarter q (each quarter of the datapath reads its own copy), column
//     sfb + n / 32, byte `id`.
// So four consecutive k-blocks share one word per row (or token), and a stage of 128
// elements takes one column per 32 rows of A and one per 32 tokens of B.
//
// Roles (one CTA per SM, persistent over tiles; a tile = two 128-row blocks of one
// expert's weight rows x one token batch of up to TM_NB tokens, the batches of the
// exact path's permutation):
//   warp 0      loads: per stage one 16U4 TMA copy per block (tensor maps whose global
//               address is rewritten on the device to the tile's expert tensors) and one
//               TMA copy of the batch's activation rows per term, into a STAGES-deep ring;
//   warps 1, 2  MMA issuers, block 0 and block 1 (4 MMAs of K 32 per stage and term);
//   warps 3..6  scale writers: each holds one TMEM lane quarter; per stage it loads the
//               weight scale words of its 32 rows (both blocks) and the activation scale
//               words of the batch's tokens (k-block-major, coalesced), several stages
//               ahead, and stores them into the stage's scale columns (tcgen05.st);
//   warps 7..22 epilogue, double-buffered accumulators, four warps per TMEM lane quarter
//               on alternate 8-token chunks: GATEUP applies SiTU-GLU and rounds h to bf16,
//               then (variant) quantizes it to MXFP8 (one scale per 32 features of a token
//               = the 32 lanes of a warp) and stores codes and scales, or (split form)
//               stores the bf16 h, in slot order for the down GEMM; DOWN stores o (fp32)
//               in slot order.
// Every mbarrier wait is bounded; on expiry K3MOE_DEV_TIMEOUT is set and all roles drain.
#pragma once

#include <cuda_fp8.h>

#include "k3_tc.cuh"

namespace k3 {

constexpr int X8_ROWS = TM_ROWS;       // weight rows per MMA block (M)
constexpr int X8_BLOCKS = 2;           // row blocks per tile (two issuers, two accumulators)
constexpr int X8_NB = TM_NB;           // tokens per batch (the large-batch layout)
constexpr int X8_BK = 128;             // contraction elements per stage
constexpr int X8_STAGES = 4;           // stages of the large-batch layout
// small batches (at most 32, or 16, tokens): smaller B tiles leave room for a fifth (sixth)
// stage of weight bytes in flight (needs contraction lengths of at least that many stages)
constexpr int X8_NB_SMALL = 32, X8_STAGES_SMALL = 5;
constexpr int X8_NB_TINY = 16, X8_STAGES_TINY = 6;
constexpr int X8_A_BYTES = X8_ROWS * 128;  // shared-memory bytes of one block's stage
constexpr int X8_A_TX = X8_ROWS * 64;      // bytes the copy reads (packed E2M1)
constexpr int X8_EPI = 16;
constexpr int X8_SCALE_W0 = 3;
constexpr int X8_EPI_W0 = X8_SCALE_W0 + 4;
constexpr int X8_THREADS = (X8_EPI_W0 + X8_EPI) * 32;
constexpr int X8_PREF = 4;  // stages of scale words in flight per scale writer
// SPLIT = 0: one MXFP8 activation term (the lossy variant); SPLIT = 1: two terms hi + lo
// that hold the bf16 activations exactly (see k3_split_rows_kernel).  NB: tokens per batch
// (MMA N at most), STAGES: the ring's depth.
// TMEM columns: accumulators [buffer][block][NB], then per stage SFA block 0 (4), SFA
// block 1 (4), SFB of each activation term (4 each: up to 128 tokens)
template <int SPLIT, int NB, int STAGES>
struct X8Lay {
  static constexpr int TERMS = 1 + SPLIT;
  static constexpr int B_BYTES = NB * 128;  // one activation term's stage (NB rows x 128 bytes)
  static constexpr int STAGE_BYTES = X8_BLOCKS * X8_A_BYTES + TERMS * B_BYTES;
  static constexpr int ACC_COLS = X8_BLOCKS * NB;
  static constexpr int SF0 = 2 * ACC_COLS;
  static constexpr int SF_COLS = 4 * (X8_BLOCKS + TERMS);
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + 512 + X8_BLOCKS * 2 * 128;
  static_assert(NB % 16 == 0 && NB <= 128, "the B scale columns hold 128 tokens");
  static_assert(SF0 + STAGES * SF_COLS <= 512, "TMEM columns");
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
  static_assert(8 * (2 * STAGES + 5) <= 512, "barrier space");
  static_assert(STAGE_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "128-byte swizzle atoms stay 1024-byte aligned");
};

struct Mx8Params {
  const MxBatch* batches;   // token batches of up to NB tokens (one expert each)
  const int32_t* n_batches;
  int R;                    // rows per weight matrix (I for gate/up, L for down)
  int K;                    // contraction length (L or I), a multiple of 128, >= 128 * STAGES
  // activation terms (one, or hi then lo when split): codes [terms][slots][K] E4M3 (the
  // operand's tensor map), rows in slot order; scale bytes k-block-major (act_scale_idx)
  const uint8_t* act_s;
  int slots;                // slots (rows of one activation term)
  void* out;                // GATEUP: h codes [slots, R] E4M3 (one term) or h [slots, R] bf16
                            // (split: k3_split_rows_kernel makes its terms); DOWN: o [slots, R] f32
  uint8_t* out_s;           // GATEUP, one term: h scale bytes, k-block-major (act_scale_idx)
  uint32_t* status;
  void* tmaps;              // packed-weight tensor maps, [TM_MAX_CTAS][X8_BLOCKS][2] x 128 bytes
};

// instruction descriptor, kind::mxf8f6f4 with block scaling: A E2M1, B E4M3, E8M0 scales,
// fp32 D, M 128, N; the scale ids select the k-block's byte of the scale words
__host__ __device__ constexpr uint32_t idesc_mx8(int N, int sf_id) {
  return ((uint32_t)sf_id << 4) | (5u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
         ((uint32_t)(X8_ROWS >> 4) << 24) | ((uint32_t)sf_id << 29);
}

K3_DEVI void tc_mma_mx8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                        uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.u32 p, %6, 0;\n"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
K3_DEVI void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
K3_DEVI void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};\n" ::"r"(taddr), "r"(v) : "memory");
}
K3_DEVI void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(taddr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// ---------------------------------------------------------------------------- MXFP8 quantization
// E8M0 scale byte of a 32-element group from its largest magnitude: 127 + floor(log2 amax)
// - 8 (8: the largest E4M3 exponent), clamped to [0, 254]; 0 for an all-zero group
K3_DEVI uint32_t mx8_scale_byte(float amax) {
  if (!(amax > 0.f)) return 0u;
  const uint32_t b = __float_as_uint(amax);
  const int e = (int)(b >> 23);  // amax > 0: sign bit clear
  const int fl = e ? e - 127 : (31 - __clz((int)(b & 0x7FFFFFu))) - 149;  // floor(log2 amax)
  const int s = fl - 8 + 127;
  return (uint32_t)(s < 0 ? 0 : (s > 254 ? 254 : s));
}
// 2^(127 - s) for a scale byte s <= 254 (2^-127 is an fp32 subnormal)
K3_DEVI float mx8_inv_scale(uint32_t s) {
  return s < 254u ? __uint_as_float((254u - s) << 23) : __uint_as_float(0x00400000u);
}
// v -> nearest E4M3 code (ties to even), saturating at +-448
K3_DEVI uint32_t e4m3_code(float v) { return (uint32_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3); }
K3_DEVI uint32_t e4m3x4_codes(float a, float b, float c, float d) {
  const uint32_t lo = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

// Activation scale bytes are stored k-block-major: the four bytes of row r for the
// 32-element groups 4w .. 4w + 3 form 32-bit word w of the rows (word index w * rows + r),
// so that a stage's scale words for a batch's consecutive rows are consecutive in memory
// (one coalesced load per 32 tokens).  rows = terms x slots (term t's row s is t x slots + s).
K3_DEVI size_t act_scale_idx(size_t row, int g, size_t rows) { return ((size_t)(g >> 2) * rows + row) * 4 + (g & 3); }

// ---------------------------------------------------------------------------- exact two-term split
// A bf16 value x of a 32-element group is written as x = hi + lo with two MXFP8 terms:
//   hi: E4M3 codes at the scale 2^(s_hi - 127), the smallest power of two that keeps the
//       group's largest magnitude within 448 (the OCP shared exponent, raised by one where
//       that element would saturate), nearest even;
//   lo: the residual x - hi (exact in fp32) as E4M3 codes at the fixed scale s_lo = s_hi - 4.
// In units of the hi scale an element of binade 2^k (k >= -6, the normal E4M3 range) has
// 8 significant bits, hi keeps the top 4 and the residual is a multiple of 2^(k-7) of
// magnitude at most 2^(k-4) <= 16: 16 times that (its lo value) is at most 256 <= 448 with at
// most 4 significant bits and a step of at least 2^-9, the finest E4M3 step, so lo holds
// it exactly and hi + lo == x for every element within 2^14 of the group's largest.  A
// smaller element is held to within 2^-14 of the hi scale (under 2^-21 of the group's
// largest), below the fp32 accumulation error of the contraction.  E2M1 x E4M3 products
// are exact on the tensor core, so the two block-scaled MMAs of a k-block reproduce the
// bf16 operand's products.
K3_DEVI uint32_t split_hi_scale(float amax) {
  uint32_t s = mx8_scale_byte(amax);
  if (s < 254u && amax * mx8_inv_scale(s) > 448.0f) ++s;
  return s;
}
K3_DEVI uint32_t split_lo_scale(uint32_t s_hi) { return s_hi >= 4u ? s_hi - 4u : 0u; }
// 2^(s - 127) for a scale byte s (2^-127 is an f32 subnormal)
K3_DEVI float e8m0_value(uint32_t s) { return s ? __uint_as_float(s << 23) : __uint_as_float(0x00400000u); }
// two elements: the codes of hi and lo at the group's scales (inv_hi = 2^(127 - s_hi),
// sc_hi = 2^(s_hi - 127), inv_lo = 2^(127 - s_lo)), two codes per 16 bits (x0 low)
K3_DEVI void split_pair(float x0, float x1, float inv_hi, float sc_hi, float inv_lo, uint32_t& c_hi,
                        uint32_t& c_lo) {
  c_hi = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(x0 * inv_hi, x1 * inv_hi), __NV_SATFINITE, __NV_E4M3);
  const __half2_raw hv = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)c_hi, __NV_E4M3);
  const float2 v = __half22float2(__half2(hv));  // exact: every E4M3 value is an f16 value
  const float r0 = x0 - v.x * sc_hi, r1 = x1 - v.y * sc_hi;  // exact
  c_lo = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(r0 * inv_lo, r1 * inv_lo), __NV_SATFINITE, __NV_E4M3);
}

// A 32-element group (bf16 pairs in w[16], low element first) -> its two terms' codes (8
// words each, byte j of word i = element 4 i + j) and scale bytes
K3_DEVI void split_group(const uint32_t (&w)[16], uint32_t (&ch)[8], uint32_t (&cl)[8], uint32_t& s_hi,
                         uint32_t& s_lo) {
  uint32_t mx = 0u;  // largest |x| as bf16 magnitude bits (they order as integers)
#pragma unroll
  for (int j = 0; j < 16; ++j) mx = max(mx, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
  s_hi = split_hi_scale(__uint_as_float(mx << 16));
  s_lo = split_lo_scale(s_hi);
  const float inv_hi = mx8_inv_scale(s_hi), sc_hi = e8m0_value(s_hi), inv_lo = mx8_inv_scale(s_lo);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t h0, l0, h1, l1;
    split_pair(__uint_as_float(w[2 * j] << 16), __uint_as_float(w[2 * j] & 0xFFFF0000u), inv_hi, sc_hi, inv_lo, h0,
               l0);
    split_pair(__uint_as_float(w[2 * j + 1] << 16), __uint_as_float(w[2 * j + 1] & 0xFFFF0000u), inv_hi, sc_hi,
               inv_lo, h1, l1);
    ch[j] = (h0 & 0xFFFFu) | (h1 << 16);
    cl[j] = (l0 & 0xFFFFu) | (l1 << 16);
  }
}

// bf16 rows -> the two split terms of every routed slot: codes [2][slots][L] (hi rows,
// then lo rows), scale bytes of the 2 slots rows k-block-major (act_scale_idx).  The row of
// slot s is row slot_tok[s] of x (z: the gather into slot order), or row s itself when
// slot_tok is null (h, already in slot order).  One thread per 32-element group (L / 32 a
// multiple of 4, so the four groups of one scale word sit on four consecutive lanes of a
// warp, and the first of them stores the word); the first n_placed slots are the routed
// ones.
__global__ void __launch_bounds__(256) k3_split_rows_kernel(const uint16_t* __restrict__ x,
                                                            const int32_t* __restrict__ slot_tok,
                                                            const int32_t* __restrict__ n_placed, int slots, int L,
                                                            uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  grid_dep_wait();
  grid_dep_launch();
  const int G = L / 32;
  const int np = min(*n_placed, slots);
  const size_t total = (size_t)np * G;  // a multiple of 4
  const int lane = threadIdx.x & 31;
  uint32_t* sw = reinterpret_cast<uint32_t*>(scales);
  // whole warps run every iteration (the word's bytes are gathered by shuffles); a quad of
  // lanes is entirely inside or entirely past the end
  for (size_t i0 = (size_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31u); i0 < total;
       i0 += (size_t)gridDim.x * blockDim.x) {
    const size_t i = i0 + lane;
    const bool in = i < total;
    const int slot = in ? (int)(i / G) : 0, g = in ? (int)(i % G) : 0;
    uint32_t s_hi = 0u, s_lo = 0u;
    if (in) {
      const int row = slot_tok ? __ldg(slot_tok + slot) : slot;
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)row * L + g * 32);
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 v = __ldg(src + j);
        w[4 * j] = v.x; w[4 * j + 1] = v.y; w[4 * j + 2] = v.z; w[4 * j + 3] = v.w;
      }
      uint32_t ch[8], cl[8];
      split_group(w, ch, cl, s_hi, s_lo);
      uint4* dh = reinterpret_cast<uint4*>(codes + (size_t)slot * L + g * 32);
      uint4* dl = reinterpret_cast<uint4*>(codes + ((size_t)slots + slot) * L + g * 32);
      dh[0] = make_uint4(ch[0], ch[1], ch[2], ch[3]);
      dh[1] = make_uint4(ch[4], ch[5], ch[6], ch[7]);
      dl[0] = make_uint4(cl[0], cl[1], cl[2], cl[3]);
      dl[1] = make_uint4(cl[4], cl[5], cl[6], cl[7]);
    }
    // the quad's four scale bytes (groups 4w .. 4w + 3 of one slot) into one word per term
    const int q0 = lane & ~3;
    uint32_t wh = 0u, wl = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      wh |= __shfl_sync(0xffffffffu, s_hi, q0 + j) << (8 * j);
      wl |= __shfl_sync(0xffffffffu, s_lo, q0 + j) << (8 * j);
    }
    if (in && (lane & 3) == 0) {
      const size_t rows = 2 * (size_t)slots, wq = (size_t)(g >> 2);
      sw[wq * rows + slot] = wh;
      sw[wq * rows + slots + slot] = wl;
    }
  }
}

// z rows (bf16, token order) -> MXFP8 rows in slot order: codes [slots, L], scale bytes
// k-block-major (act_scale_idx).  One thread per 32-element group; the four groups of a
// scale word sit on four consecutive lanes (L / 32 a multiple of 4) and the first of them
// stores the word.
__global__ void __launch_bounds__(256) k3_gather_mx8_kernel(const uint16_t* __restrict__ z,
                                                            const int32_t* __restrict__ slot_tok,
                                                            const int32_t* __restrict__ n_placed, int slots, int L,
                                                            uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  grid_dep_wait();
  grid_dep_launch();
  const int G = L / 32;
  const int np = min(*n_placed, slots);
  const size_t total = (size_t)np * G;  // a multiple of 4
  const int lane = threadIdx.x & 31;
  uint32_t* sw = reinterpret_cast<uint32_t*>(scales);
  // whole warps run every iteration (the word's bytes are gathered by shuffles); a quad of
  // lanes is entirely inside or entirely past the end
  for (size_t i0 = (size_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31u); i0 < total;
       i0 += (size_t)gridDim.x * blockDim.x) {
    const size_t i = i0 + lane;
    const bool in = i < total;
    const int slot = in ? (int)(i / G) : 0, g = in ? (int)(i % G) : 0;
    uint32_t s = 0u;
    if (in) {
      const int t = __ldg(slot_tok + slot);
      const uint4* src = reinterpret_cast<const uint4*>(z + (size_t)t * L + g * 32);
      uint4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = __ldg(src + j);
      const uint32_t* w = reinterpret_cast<const uint32_t*>(v);
      float x[32];
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        x[2 * j] = __uint_as_float(w[j] << 16);
        x[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        amax = fmaxf(amax, fmaxf(fabsf(x[2 * j]), fabsf(x[2 * j + 1])));
      }
      s = mx8_scale_byte(amax);
      const float inv = mx8_inv_scale(s);
      uint32_t c[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        c[j] = e4m3x4_codes(x[4 * j] * inv, x[4 * j + 1] * inv, x[4 * j + 2] * inv, x[4 * j + 3] * inv);
      uint4* dst = reinterpret_cast<uint4*>(codes + (size_t)slot * L + g * 32);
      dst[0] = make_uint4(c[0], c[1], c[2], c[3]);
      dst[1] = make_uint4(c[4], c[5], c[6], c[7]);
    }
    const int q0 = lane & ~3;
    uint32_t word = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) word |= __shfl_sync(0xffffffffu, s, q0 + j) << (8 * j);
    if (in && (lane & 3) == 0) sw[(size_t)(g >> 2) * slots + slot] = word;
  }
}

// ---------------------------------------------------------------------------- grouped GEMM
template <int MODE, int SPLIT, int NB, int STAGES>
__global__ void __launch_bounds__(X8_THREADS, 1) k3_mx8_moe_kernel(const __grid_constant__ CUtensorMap mapB,
                                                                   const __grid_constant__ CUtensorMap mapA,
                                                                   Mx8Params p) {
  using Lay = X8Lay<SPLIT, NB, STAGES>;
  constexpr int TERMS = Lay::TERMS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // stage s: A block 0, A block 1, B term(s)
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bars = base + STAGES * Lay::STAGE_BYTES;
  const uint32_t smaps = bars + 512;  // [X8_BLOCKS][128 bytes] tensor-map images
  auto stage_a = [&](int s, int b) { return base + s * Lay::STAGE_BYTES + b * X8_A_BYTES; };
  auto stage_b = [&](int s, int t) { return base + s * Lay::STAGE_BYTES + X8_BLOCKS * X8_A_BYTES + t * Lay::B_BYTES; };
  // full(s): the stage's copies landed (the load thread's arrival with the byte count) and
  // the four scale writers stored its scale words; kdone(s): both issuers' MMAs of the
  // stage completed (frees its shared memory and scale columns); tfull / tempty: the
  // accumulator buffer holds a finished tile / was read by all epilogue threads
  auto full = [&](int s) { return bars + 8 * s; };
  auto kdone = [&](int s) { return bars + 8 * (STAGES + s); };
  auto tfull = [&](int b) { return bars + 8 * (2 * STAGES + b); };
  auto tempty = [&](int b) { return bars + 8 * (2 * STAGES + 2 + b); };
  const uint32_t done_bar = bars + 8 * (2 * STAGES + 4);
  volatile int* abort_flag = &abort_sh;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1 + 4);
      mbar_init(kdone(s), X8_BLOCKS);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull(b), X8_BLOCKS);
      mbar_init(tempty(b), X8_EPI * 32);
    }
    mbar_init(done_bar, X8_BLOCKS);
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

  const int mtiles = p.R / (MODE == 0 ? X8_ROWS : X8_BLOCKS * X8_ROWS);
  const int tiles = mtiles * (*p.n_batches);
  const int kst = p.K / X8_BK;  // stages per tile (>= STAGES)
  const int my_tiles = (tiles > (int)blockIdx.x) ? (tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int nst = my_tiles * kst;
  // weight tensors of block b (index into MxBatch::w: packed, then scales) and the first row
  // of block b of row tile tm
  auto blk_tensor = [](int b) { return (MODE == 0) ? 2 * b : 4; };
  auto blk_row0 = [](int tm, int b) {
    return (MODE == 0) ? tm * X8_ROWS : tm * (X8_BLOCKS * X8_ROWS) + b * X8_ROWS;
  };
  auto sf_col = [&](int s) { return tmem + Lay::SF0 + s * Lay::SF_COLS; };

  if (warp == 0) {
    // ------------------------------------------------------------ loads
    uint8_t* gmaps = reinterpret_cast<uint8_t*>(p.tmaps) + (size_t)blockIdx.x * (X8_BLOCKS * 2 * 128);
    auto gmap = [&](int b, int par) { return gmaps + (b * 2 + par) * 128; };
#pragma unroll
    for (int b = 0; b < X8_BLOCKS; ++b)
      reinterpret_cast<uint32_t*>(base_ptr + (smaps + b * 128 - base))[lane] =
          reinterpret_cast<const uint32_t*>(&mapA)[lane];
    __syncwarp();
    int par = 1, slot0 = 0, tm = 0, issued = 0;
#pragma unroll 1
    for (int j = 0; j < nst; ++j) {
      const int s = j % STAGES, ks = j % kst;
      // the stage's previous contents (j - STAGES) have been consumed by the MMAs
      if (j >= STAGES &&
          !__all_sync(0xffffffffu, mbar_wait(kdone(s), ((j / STAGES) - 1) & 1, abort_flag)))
        break;
      if (ks == 0) {
        // a new tile: point the block maps of this tile's parity at its expert tensors.  The
        // copies of the tile before last (same parity) have all landed: the wait above was
        // for a stage of the previous tile or later (a tile has >= STAGES stages).
        const int tile = blockIdx.x + (j / kst) * gridDim.x;
        const MxBatch* rec = p.batches + tile / mtiles;
        const uint8_t* q0 = rec->w[blk_tensor(0)];
        const uint8_t* q1 = rec->w[blk_tensor(1)];
        const uint8_t* s0 = rec->w[blk_tensor(0) + 1];
        const uint8_t* s1 = rec->w[blk_tensor(1) + 1];
        if ((((reinterpret_cast<uintptr_t>(q0) | reinterpret_cast<uintptr_t>(q1)) & 31u) |
             ((reinterpret_cast<uintptr_t>(s0) | reinterpret_cast<uintptr_t>(s1)) & 3u)) != 0) {
          // the 4-bit copies need 32-byte aligned rows, the scale words 4-byte aligned ones
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
        slot0 = rec->slot0;
        tm = tile % mtiles;
      }
      if (lane == 0) {
        mbar_expect_tx(full(s), X8_BLOCKS * X8_A_TX + TERMS * Lay::B_BYTES);
#pragma unroll
        for (int b = 0; b < X8_BLOCKS; ++b)
          tma_load_2d(stage_a(s, b), reinterpret_cast<const CUtensorMap*>(gmap(b, par)), ks * X8_BK, blk_row0(tm, b),
                      full(s));
        // term t's rows start at row t * slots of the operand
#pragma unroll
        for (int t = 0; t < TERMS; ++t) tma_load_2d(stage_b(s, t), &mapB, ks * X8_BK, t * p.slots + slot0, full(s));
      }
      issued = j + 1;
    }
    // let every issued copy land before the CTA exits: bounded waits on the last stages'
    // byte counts (their phases complete once the copies and the scale writers are done;
    // after an abort the writers may never arrive, so only a bounded time is spent)
    if (lane == 0) {
      for (int j = (issued > STAGES ? issued - STAGES : 0); j < issued; ++j) {
        const long long t0 = clock64();
        while (!mbar_test(full(j % STAGES), (j / STAGES) & 1) && clock64() - t0 < (1ll << 22)) {
        }
      }
    }
  } else if (warp <= X8_BLOCKS) {
    // ------------------------------------------------------------ MMA issuers
    if (lane == 0) {
      const int mm = warp - 1;
      const uint64_t dA0 = sdesc_sw128(stage_a(0, mm)), dB0 = sdesc_sw128(stage_b(0, 0));
      int j = 0, lt = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x, ++lt) {
        const int n = p.batches[tile / mtiles].n;
        const int N = (n + 15) & ~15;
        const int buf = lt & 1;
        if (!mbar_wait_issue(tempty(buf), ((lt >> 1) & 1) ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * Lay::ACC_COLS + mm * NB;
        for (int ks = 0; ks < kst; ++ks, ++j) {
          const int s = j % STAGES;
          if (!mbar_wait_issue(full(s), (j / STAGES) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t da = dA0 + ((uint32_t)(s * Lay::STAGE_BYTES) >> 4);
          const uint64_t db = dB0 + ((uint32_t)(s * Lay::STAGE_BYTES) >> 4);
          const uint32_t sfa = sf_col(s) + 4 * mm, sfb = sf_col(s) + 4 * X8_BLOCKS;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            tc_mma_mx8(d, da + 2 * kk, db + 2 * kk, idesc_mx8(N, kk), sfa, sfb, (ks | kk) != 0);
            // the lo term: same weights, its own rows and scale columns, same accumulator
            if (SPLIT)
              tc_mma_mx8(d, da + 2 * kk, db + (Lay::B_BYTES >> 4) + 2 * kk, idesc_mx8(N, kk), sfa, sfb + 4, 1u);
          }
          tc_commit(kdone(s));
        }
        if (!ok) break;
        tc_commit(tfull(buf));
      }
      tc_commit(done_bar);
      volatile int never = 0;
      mbar_wait(done_bar, 0, &never);
    }
  } else if (warp < X8_EPI_W0) {
    // ------------------------------------------------------------ scale writers
    // Lane quarter q: weight rows 32 q + lane of both blocks, and the lanes 32 q + lane
    // of the activation scale columns (token 32 c + lane in column c).  The scale words of
    // stage j + X8_PREF - 1 are loaded while stage j's are stored.
    const int q = warp & 3;
    const int KB = p.K / 32;  // scale bytes per row
    const uint32_t tq = (uint32_t)(q * 32) << 16;
    constexpr int W = 2 + 3 * TERMS;  // SFA of both blocks, then 3 words of SFB per term
    auto load = [&](int j, uint32_t (&w)[W]) {
      if (j >= nst) return;
      const int tile = blockIdx.x + (j / kst) * gridDim.x, ks = j % kst;
      const MxBatch* rec = p.batches + tile / mtiles;
      const int tm = tile % mtiles;
#pragma unroll
      for (int b = 0; b < X8_BLOCKS; ++b) {
        const uint8_t* sp = rec->w[blk_tensor(b) + 1] + (size_t)(blk_row0(tm, b) + q * 32 + lane) * KB + 4 * ks;
        w[b] = __ldg(reinterpret_cast<const uint32_t*>(sp));
      }
      const int n = rec->n, slot0 = rec->slot0;
#pragma unroll
      for (int t = 0; t < TERMS; ++t)
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          const int col = c * 32 + lane;
          w[2 + 3 * t + c] =
              (col < n && slot0 + col < p.slots)
                  ? __ldg(reinterpret_cast<const uint32_t*>(p.act_s) + (size_t)ks * TERMS * p.slots +
                          (size_t)t * p.slots + slot0 + col)
                  : 0x7F7F7F7Fu;  // columns past the batch: scale 1, outputs unused
        }
    };
    uint32_t ring[X8_PREF][W];
#pragma unroll
    for (int u = 0; u < X8_PREF - 1; ++u) load(u, ring[u]);
    bool ok = true;
#pragma unroll 1
    for (int j0 = 0; j0 < nst && ok; j0 += X8_PREF) {
#pragma unroll
      for (int u = 0; u < X8_PREF; ++u) {
        const int j = j0 + u;
        if (j >= nst) break;
        load(j + X8_PREF - 1, ring[(u + X8_PREF - 1) % X8_PREF]);
        const int s = j % STAGES;
        if (j >= STAGES &&
            !__all_sync(0xffffffffu, mbar_wait(kdone(s), ((j / STAGES) - 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t c0 = sf_col(s) + tq;
        tmem_st1(c0 + q, ring[u][0]);
        tmem_st1(c0 + 4 + q, ring[u][1]);
        tmem_st4(c0 + 8, ring[u][2], ring[u][3], ring[u][4], 0x7F7F7F7Fu);
        if constexpr (SPLIT) tmem_st4(c0 + 12, ring[u][5], ring[u][6], ring[u][7], 0x7F7F7F7Fu);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(full(s));
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 7..22)
    // warp w reads TMEM lane quarter w % 4 (32 weight rows of each block) and the 8-token
    // chunks e, e + 4, ... of the batch (e = (w - 7) / 4): four warps per lane quarter share
    // a tile's tokens within one chunk of each other (gate/up: SiTU-GLU and the MXFP8
    // encoding are most of the epilogue's work)
    const int q = warp & 3;
    const int e0 = (warp - X8_EPI_W0) >> 2;
    int lt = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++lt) {
      const int buf = lt & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(tfull(buf), (lt >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      const MxBatch* rec = p.batches + tile / mtiles;
      const int slot0 = rec->slot0, n = rec->n;
      const int tm = tile % mtiles;
      const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16) + buf * Lay::ACC_COLS;
#pragma unroll 1
      for (int c = e0; c * 8 < n; c += X8_EPI / 4) {
        uint32_t r0[8], r1[8];
        tmem_ld8(tq + c * 8, r0);
        tmem_ld8(tq + NB + c * 8, r1);
        tmem_ld_wait();
        if (MODE == 0) {
          // h of feature `feat` for 8 tokens; the 32 features of the warp are one MXFP8 group
          const int feat = tm * X8_ROWS + q * 32 + lane;
          uint8_t* hq = reinterpret_cast<uint8_t*>(p.out);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int col = c * 8 + jj;  // warp-uniform
            if (col >= n) break;
            const uint16_t hb = f32_to_bf16_bits(situ_fast(__uint_as_float(r0[jj]), __uint_as_float(r1[jj])));
            const size_t slot = (size_t)(slot0 + col);
            if constexpr (SPLIT) {
              // bf16 h in slot order; its two terms are made by a separate pass (the split
              // here would double the epilogue's work, which bounds this kernel)
              reinterpret_cast<uint16_t*>(p.out)[slot * p.R + feat] = hb;
            } else {
              const float h = bf16_bits_to_f32(hb);
              // largest |h| of the group: the bit patterns of non-negative floats order as integers
              const float m = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(h))));
              const uint32_t sb = mx8_scale_byte(m);
              const uint32_t code = e4m3_code(h * mx8_inv_scale(sb));
              hq[slot * p.R + feat] = (uint8_t)code;
              if (lane == 0) p.out_s[act_scale_idx(slot, feat >> 5, p.slots)] = (uint8_t)sb;
            }
          }
        } else {
          const int row0 = tm * (X8_BLOCKS * X8_ROWS) + q * 32 + lane;
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int col = c * 8 + jj;
            if (col < n) {
              float* o = reinterpret_cast<float*>(p.out) + (size_t)(slot0 + col) * p.R + row0;
              o[0] = __uint_as_float(r0[jj]);
              o[X8_ROWS] = __uint_as_float(r1[jj]);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty(buf));
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

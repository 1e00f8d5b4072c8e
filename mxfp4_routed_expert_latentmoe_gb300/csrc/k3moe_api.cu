// k3moe_api.cu -- C ABI of the LatentMoE routed-expert block (see include/k3moe.h):
// host-side validation, workspace carving and the launch sequence.  No allocation,
// no synchronisation (except k3moe_device_status, which is documented to sync).
#include <atomic>
#include <cstring>
#include <mutex>
#include <utility>

#include "k3_common.cuh"
#include "k3_gemv.cuh"
#include "k3_gemv_bulk.cuh"
#include "k3_route.cuh"
#include "k3_tc.cuh"
#include "k3_front.cuh"
#include "k3_mx8.cuh"
#include "k3_shared.cuh"

namespace {

using namespace k3;

constexpr float kTieTau = 3e-5f;
constexpr int kMaxDevices = 64;
constexpr int kTcMinTokensDefault = 9;  // measured crossover on GB300 at K3 shapes (bench.py --sweep)
constexpr int kSplitKMaxT = 512;        // the projections split K only when they have few output tiles
// exact tensor-core experts: two-term MXFP8 split below this many tokens, bf16 weight decode
// from it on.  Default: the split at every token count (measured on GB300 at K3 shapes, the
// whole forward: 9 tokens 586 us split against 766 us decode, 1024 tokens 3633 against
// 4716, 4096 tokens 4854 against 5780, 8192 tokens 9284 against 10833; bench.py --sweep)
constexpr int kSplitMaxTokensDefault = 1 << 30;

size_t align256(size_t b) { return (b + 255) / 256 * 256; }
int tc_min_t();
bool split_experts(const k3moe_dims& d, int T);

struct WsLayout {
  size_t status, logits, ids, w, zmax, zpow, counts, offsets, slot_of, slot_tok, inv, uniq, n_uniq, nb_prefix,
      n_batches, cta_cnt, cta_base, batches, z, z16, h16, o, y, yhat, cpart, ccount, act, tmaps, zero_end, total;
  size_t part = 0, part_bytes = 0;
  size_t hterm = 0;  // the split form's two terms of h
};

WsLayout ws_layout(const k3moe_dims& d, int T) {
  WsLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  };
  const size_t Tz = (size_t)T, E = (size_t)d.n_experts, K = (size_t)d.top_k, Lt = (size_t)d.latent,
               I = (size_t)d.inter;
  const size_t slots = Tz * K;
  // the words every forward clears come first (one memset): status word and kernel
  // counters, per-token max |z|, combine arrival counters
  L.status = take(256);
  L.zmax = take(Tz * 4);
  L.ccount = take(Tz * 4);
  L.zero_end = off;
  L.logits = take(Tz * E * 4);
  L.ids = take(slots * 4);
  L.w = take(slots * 4);
  L.zpow = take(Tz * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.slot_of = take(slots * 4);
  L.slot_tok = take(slots * 4);
  L.inv = take(slots * 4);
  L.uniq = take(E * 4);
  L.n_uniq = take(4);
  L.nb_prefix = take((E + 1) * 4);
  L.n_batches = take(4);
  // multi-CTA permutation: per-CTA expert counts and first positions
  const size_t nct = (slots + PERM_SPAN - 1) / PERM_SPAN;
  L.cta_cnt = take(nct * E * 4);
  L.cta_base = take(nct * E * 4);
  // token batches of at least 8 tokens: at most ceil(slots / 8) + min(E, slots) of them
  L.batches = take((slots / 8 + 1 + (E < slots ? E : slots)) * sizeof(MxBatch));
  L.z = take(Tz * Lt * 2);
  L.z16 = take(Tz * Lt * 2);
  // bf16 h (weight-decode and split forms), or the h codes and scale bytes of the MXFP8
  // variant (one term); the split form's two terms of h follow in their own region (2 slots I
  // codes + 2 slots I / 32 scale bytes)
  const bool split = split_experts(d, T);
  L.h16 = take(slots * I * 2);
  L.hterm = take(split ? slots * I * 2 + slots * I / 16 : 0);
  L.o = take(slots * Lt * 4);
  L.y = take(Tz * Lt * 4);
  L.yhat = take(Tz * Lt * 2);
  L.cpart = take(Tz * COMB_MAX_SPLIT * 4);
  // slot-order bf16 activation rows for the tensor-core expert path (large T only)
  const bool tc = T >= tc_min_t();
  // (bf16 rows; or the variant's codes and scale bytes; or the split's two terms of each)
  L.act = take(tc ? slots * Lt * 2 + (split ? slots * Lt / 16 : 0) : 0);
  L.tmaps = take(tc ? (size_t)TM_MAX_CTAS * TM_BLOCKS * 2 * 128 : 0);  // packed-weight tensor maps
  // split-K partial sums of the projections (few tokens on the tensor-core path)
  L.part_bytes = (tc && T <= kSplitKMaxT) ? (size_t)8 * T * std::max<size_t>((size_t)E + Lt, d.hidden) * 4 : 0;
  L.part = take(L.part_bytes);
  L.total = off;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool top_p_on(const k3moe_dims& d) { return d.top_p > 0.0f && d.top_p < 1.0f; }

k3moe_status check_dims(const k3moe_dims* d) {
  if (!d) return K3MOE_ERR_ARG;
  if (d->hidden <= 0 || d->latent <= 0 || d->inter <= 0 || d->n_experts <= 0 || d->top_k <= 0)
    return K3MOE_ERR_SHAPE;
  if (d->hidden % 64 || d->latent % 64 || d->inter % 64) return K3MOE_ERR_SHAPE;
  if (d->n_experts > TOPK_MAX_E || d->top_k > 64 || d->top_k > d->n_experts) return K3MOE_ERR_SHAPE;
  if (d->latent > 32768 || d->inter > 32768 || d->hidden > 65536) return K3MOE_ERR_SHAPE;
  if (!(d->rms_eps >= 0.0f) || d->rms_eps > 1.0f) return K3MOE_ERR_ARG;
  if (!(d->top_p >= 0.0f)) return K3MOE_ERR_ARG;
  if (top_p_on(*d) && d->top_k + REFINE_EXTRA > 32) return K3MOE_ERR_SHAPE;
  if (d->act_mxfp8 != 0 && d->act_mxfp8 != 1) return K3MOE_ERR_ARG;
  // the variant's grouped GEMM: 256-row tiles and at least X8_STAGES stages of 128 elements
  if (d->act_mxfp8 && (d->latent % 256 || d->inter % 256 || d->latent < X8_BK * X8_STAGES ||
                       d->inter < X8_BK * X8_STAGES))
    return K3MOE_ERR_SHAPE;
  return K3MOE_OK;
}

struct DevInfo {
  int sms = 0;
  bool ok = false;
};
DevInfo g_dev[kMaxDevices];
std::atomic<bool> g_dev_init[kMaxDevices];

k3moe_status check_device(int* dev_out, int* sms_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return K3MOE_ERR_DEVICE;
  if (!g_dev_init[dev].load(std::memory_order_acquire)) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    g_dev[dev].sms = sms;
    g_dev[dev].ok = (major == 10 && minor == 3);
    g_dev_init[dev].store(true, std::memory_order_release);
  }
  if (!g_dev[dev].ok) return K3MOE_ERR_DEVICE;
  *dev_out = dev;
  *sms_out = g_dev[dev].sms;
  return K3MOE_OK;
}

// per (kernel, device): raise the kernel's dynamic shared memory limit whenever a
// launch needs more than any earlier one did
template <auto Kern>
bool set_smem(int dev, int bytes) {
  static std::atomic<int> granted[kMaxDevices];
  if (bytes <= 48 * 1024 || granted[dev].load(std::memory_order_acquire) >= bytes) return true;
  if (cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  int cur = granted[dev].load(std::memory_order_acquire);
  while (cur < bytes && !granted[dev].compare_exchange_weak(cur, bytes, std::memory_order_acq_rel)) {
  }
  return true;
}

// ---------------------------------------------------------------------------- TMA descriptors
// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load(std::memory_order_acquire);
  if (!f) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    f = reinterpret_cast<EncodeTiledFn>(p);
    fn.store(f, std::memory_order_release);
  }
  return f;
}

// row-major [rows, cols] bf16 matrix, boxes of box_rows x 64 with the 128-byte swizzle
bool map_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// row-major [rows, cols] byte matrix, boxes of box_rows x 128 bytes with the 128-byte swizzle
bool map_u8(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// row-major [rows, cols] E2M1 matrix (cols 4-bit elements, packed two per byte, rows
// cols / 2 bytes apart), boxes of 128 rows x 128 elements; in shared memory each 16
// elements take a 16-byte granule (8 bytes of codes, 8 of padding), 128-byte swizzle
bool map_e2m1(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols / 2};
  const cuuint32_t box[2] = {128, 128};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------- launch helpers
// Launch with programmatic stream serialization: the kernel may start while its
// predecessor finishes; it waits (griddepcontrol.wait) before reading its inputs.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kern)(KArgs...), dim3 grid, dim3 block, int smem, cudaStream_t st, bool pdl,
                   Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ring depth per activation batch width: two CTAs per SM for NBLK 1 and 2
constexpr int dn_stages(int nblk) { return nblk == 1 ? 4 : 3; }
constexpr int dn_smem(int nblk) {
  return DN_WARPS * dn_stages(nblk) * dn_stage_bytes(nblk) + DN_WARPS * nblk * 128 * 4;
}

template <int EPI, int NBLK>
cudaError_t launch_dense_t(const DenseParams& p, int dev, int sms, cudaStream_t st, bool pdl) {
  constexpr int STAGES = dn_stages(NBLK);
  constexpr int smem = dn_smem(NBLK);
  if (!set_smem<k3_dense_gemv_kernel<EPI, NBLK, STAGES>>(dev, smem)) return cudaErrorInvalidValue;
  const int per_sm = (2 * smem + 2048 <= 228 * 1024) ? 2 : 1;
  const int tiles = (p.R0 + 15) / 16 + (p.R1 + 15) / 16;
  const int total = tiles * ((p.T + 8 * NBLK - 1) / (8 * NBLK));
  const int grid = total < per_sm * sms ? total : per_sm * sms;
  if (grid <= 0) return cudaSuccess;
  return launch(k3_dense_gemv_kernel<EPI, NBLK, STAGES>, dim3(grid), dim3(DN_WARPS * 32), smem, st, pdl, p);
}

// one token: rows streamed by plain vector loads (k3_dense_gemv1_kernel), x as f32 in
// shared memory
template <int EPI>
cudaError_t launch_dense1(const DenseParams& p, int dev, int sms, cudaStream_t st, bool pdl,
                          int rows_per_cta = 2 * D1_WARPS) {
  const int smem = p.K * 4;
  if (!set_smem<k3_dense_gemv1_kernel<EPI>>(dev, smem)) return cudaErrorInvalidValue;
  const int per_sm = (2 * (smem + 1024) <= 228 * 1024) ? 2 : 1;  // registers allow two CTAs per SM
  const int R = p.R0 + p.R1;
  int grid = per_sm * sms;
  if (R < grid * rows_per_cta) grid = (R + rows_per_cta - 1) / rows_per_cta;
  return launch(k3_dense_gemv1_kernel<EPI>, dim3(grid), dim3(D1_WARPS * 32), smem, st, pdl, p);
}

bool dense1_ok(const DenseParams& p) {
  return p.T == 1 && p.K % 8 == 0 && p.K * 4 <= 227 * 1024 && a16(p.act) && a16(p.W0) && (p.R1 == 0 || a16(p.W1));
}

template <int EPI>
cudaError_t launch_dense(const DenseParams& p, int dev, int sms, cudaStream_t st, bool pdl) {
  if (dense1_ok(p)) return launch_dense1<EPI>(p, dev, sms, st, pdl);
  if (p.T <= 8) return launch_dense_t<EPI, 1>(p, dev, sms, st, pdl);
  if (p.T <= 16) return launch_dense_t<EPI, 2>(p, dev, sms, st, pdl);
  return launch_dense_t<EPI, 4>(p, dev, sms, st, pdl);
}

int mx_nblk(int T) { return T <= 8 ? 1 : 2; }

// the bulk-copy GEMV takes K multiples of 256 up to 256 * MXB_MAX_WARPS
bool mxb_ok(int K) { return K % 256 == 0 && K / 256 <= MXB_MAX_WARPS; }

// token count from which the projections and experts run on the tcgen05 GEMMs (the
// workspace layout follows it); process-wide, set by k3moe_set_tc_min_tokens
std::atomic<int> g_tc_min_t{kTcMinTokensDefault};
int tc_min_t() { return g_tc_min_t.load(std::memory_order_relaxed); }
// token count from which the combine runs one CTA per token with several columns a thread
constexpr int kCombRowMinT = 256;
// the grouped expert GEMM moves scale bytes four k-blocks (8 bytes) at a time, so it
// needs both expert contraction lengths to be multiples of 256; other shapes keep the
// weight-streaming kernels at every T
bool tc_experts(const k3moe_dims& d, int T) { return T >= tc_min_t() && d.latent % 256 == 0 && d.inter % 256 == 0; }
// operand form of the exact grouped GEMM: below g_split_max_t tokens (process-wide,
// k3moe_set_tc_split_max_tokens; by default at every count) the bf16 activations are split
// exactly into two MXFP8 terms for block-scaled MMAs over the stored weights
// (k3_mx8_moe_kernel<.., 1>); from it on the SMs decode the weights to bf16
// (k3_tc_moe_kernel).  The split needs both contraction lengths >= 512.
std::atomic<int> g_split_max_t{kSplitMaxTokensDefault};
bool split_experts(const k3moe_dims& d, int T) {
  return T < g_split_max_t.load(std::memory_order_relaxed) && !d.act_mxfp8 && tc_experts(d, T) &&
         d.latent >= X8_BK * X8_STAGES && d.inter >= X8_BK * X8_STAGES;
}

// grouped MXFP4 expert GEMM on tcgen05; act [slots, K] f16 in slot order
template <int MODE>
cudaError_t launch_tc_moe(const uint16_t* act, int slots, TcMoeParams p, int dev, int sms, cudaStream_t st, bool pdl) {
  CUtensorMap mb, ma;
  if (!map_bf16(&mb, act, slots, p.K, TM_NB)) return cudaErrorInvalidValue;
  // template of the packed-weight maps ([R, K/2] bytes, 128-row boxes): the kernel writes
  // each expert tensor's address into its copies; the workspace stands in until then
  if (!map_u8(&ma, p.tmaps, (uint64_t)p.R, (uint64_t)p.K / 2, TM_ROWS)) return cudaErrorInvalidValue;
  constexpr int smem = TmLayout<MODE>::SMEM;
  if (!set_smem<k3_tc_moe_kernel<MODE>>(dev, smem)) return cudaErrorInvalidValue;
  const int grid = sms < TM_MAX_CTAS ? sms : TM_MAX_CTAS;
  return launch(k3_tc_moe_kernel<MODE>, dim3(grid), dim3(TM_THREADS), smem, st, pdl, mb, ma, p);
}

// grouped expert GEMM of the MXFP8-activation variant; act [slots, K] E4M3 codes in slot order
template <int MODE, int SPLIT, int NB, int STAGES>
cudaError_t launch_mx8_t(const uint8_t* act, Mx8Params p, int dev, int sms, cudaStream_t st, bool pdl) {
  if (p.K < X8_BK * STAGES) return cudaErrorInvalidValue;  // a tile has at least STAGES stages
  CUtensorMap mb, ma;
  // the activation terms' rows, one after the other
  if (!map_u8(&mb, act, (uint64_t)(1 + SPLIT) * p.slots, (uint64_t)p.K, NB)) return cudaErrorInvalidValue;
  // template of the weight maps ([R, K] E2M1): the kernel writes each expert tensor's address
  // into its copies; the (256-byte aligned) workspace stands in until then
  if (!map_e2m1(&ma, p.tmaps, (uint64_t)p.R, (uint64_t)p.K)) return cudaErrorInvalidValue;
  constexpr int smem = X8Lay<SPLIT, NB, STAGES>::SMEM;
  if (!set_smem<k3_mx8_moe_kernel<MODE, SPLIT, NB, STAGES>>(dev, smem)) return cudaErrorInvalidValue;
  const int grid = sms < TM_MAX_CTAS ? sms : TM_MAX_CTAS;
  return launch(k3_mx8_moe_kernel<MODE, SPLIT, NB, STAGES>, dim3(grid), dim3(X8_THREADS), smem, st, pdl, mb, ma, p);
}

// the batches' token count (the permutation's NB) picks the layout: up to X8_NB_SMALL
// tokens the small-batch layout with its deeper ring
template <int MODE, int SPLIT>
cudaError_t launch_mx8_moe(const uint8_t* act, Mx8Params p, int nb, int dev, int sms, cudaStream_t st, bool pdl) {
  if (nb == X8_NB_TINY) return launch_mx8_t<MODE, SPLIT, X8_NB_TINY, X8_STAGES_TINY>(act, p, dev, sms, st, pdl);
  if (nb == X8_NB_SMALL)
    return launch_mx8_t<MODE, SPLIT, X8_NB_SMALL, X8_STAGES_SMALL>(act, p, dev, sms, st, pdl);
  if (nb == X8_NB) return launch_mx8_t<MODE, SPLIT, X8_NB, X8_STAGES>(act, p, dev, sms, st, pdl);
  return cudaErrorInvalidValue;
}

// tokens per batch of the block-scaled expert GEMMs: small batches (deeper ring) when few
// tokens reach each expert -- at K3 shapes, up to kTinyBatchT tokens an expert rarely gets
// more than 16 of them and up to kSmallBatchT more than 32 (one that does takes several
// batches) -- and both contractions are long enough for the deeper ring (measured: 9 to
// 512 tokens 4-8% faster than the 96-token layout)
constexpr int kSmallBatchT = 512, kTinyBatchT = 256;
int mx8_batch(const k3moe_dims& d, int T) {
  const int kmin = d.latent < d.inter ? d.latent : d.inter;
  if (T <= kTinyBatchT && kmin >= X8_BK * X8_STAGES_TINY) return X8_NB_TINY;
  if (T <= kSmallBatchT && kmin >= X8_BK * X8_STAGES_SMALL) return X8_NB_SMALL;
  return X8_NB;
}

// D[M, N0 (+N1)] = A[M, K] . [B0; B1]^T on tcgen05 (A, B bf16 row-major)
template <int EPI>
cudaError_t launch_tc_dense(const uint16_t* A, int M, int K, const uint16_t* B0, int N0, const uint16_t* B1, int N1,
                            TcDenseParams p, int dev, int sms, cudaStream_t st, bool pdl, float* part = nullptr,
                            size_t part_bytes = 0) {
  CUtensorMap ma, mb0, mb1;
  if (!map_bf16(&ma, A, M, K, TC_BM) || !map_bf16(&mb0, B0, N0, K, TC_BN)) return cudaErrorInvalidValue;
  if (N1 > 0) {
    if (!map_bf16(&mb1, B1, N1, K, TC_BN)) return cudaErrorInvalidValue;
  } else {
    mb1 = mb0;
  }
  p.M = M;
  p.N0 = N0;
  p.N1 = N1;
  p.K = K;
  if (!set_smem<k3_tc_dense_kernel<EPI>>(dev, TC_SMEM)) return cudaErrorInvalidValue;
  const int tiles = ((M + TC_BM - 1) / TC_BM) * ((N0 + TC_BN - 1) / TC_BN + (N1 + TC_BN - 1) / TC_BN);
  // few output tiles (few tokens): split K over up to 8 CTAs per tile, partial sums in
  // `part`, so that the weight stream is spread over the SMs
  p.ksplit = 1;
  p.part = part;
  const int kb = K / TC_BK;
  for (int ks = 8; ks >= 2 && part; ks >>= 1)
    if (2 * tiles <= sms && kb % ks == 0 && kb / ks >= TC_STAGES && (size_t)ks * M * (N0 + N1) * 4 <= part_bytes) {
      p.ksplit = ks;
      break;
    }
  const int units = tiles * p.ksplit;
  const int grid = units < sms ? units : sms;
  cudaError_t e = launch(k3_tc_dense_kernel<EPI>, dim3(grid), dim3(TC_THREADS), TC_SMEM, st, pdl, ma, mb0, mb1, p);
  if (e == cudaSuccess && p.ksplit > 1)
    e = launch(k3_tc_splitk_reduce_kernel<EPI>, dim3(M, (N0 + N1 + TC_RED_COLS - 1) / TC_RED_COLS), dim3(256), 0,
               st, true, p);
  return e;
}

template <int MODE, int NBLK, int STAGES, bool FULL>
cudaError_t launch_mx_s(const MxGemvParams& p, int dev, int sms, cudaStream_t st, bool pdl, int smem, int warps) {
  constexpr bool PRE = MODE == MX_DOWN;  // its batches were written two kernels earlier
  if (!set_smem<k3_mx_gemv_kernel<MODE, NBLK, STAGES, PRE, FULL>>(dev, smem)) return cudaErrorInvalidValue;
  const int per_sm = (2 * smem + 2048 <= 228 * 1024) ? 2 : 1;
  return launch(k3_mx_gemv_kernel<MODE, NBLK, STAGES, PRE, FULL>, dim3(sms * per_sm), dim3(warps * 32), smem, st, pdl,
                p);
}

template <int MODE, int NBLK>
cudaError_t launch_mx_t(const MxGemvParams& p, int dev, int sms, cudaStream_t st, bool pdl) {
  constexpr int M = MODE == MX_GATEUP ? 2 : 1;
  const int warps = (p.K / 32 + MX_GPW - 1) / MX_GPW;
  if (warps * 32 > MX_MAX_THREADS) return cudaErrorInvalidValue;
  const int red = 2 * warps * M * NBLK * 128 * 4;  // double-buffered partial sums
  const bool full = p.K % 256 == 0;
  const int smem3 = warps * MxLayout<M, 3>::WARP_BYTES + red;
  const int smem2 = warps * MxLayout<M, 2>::WARP_BYTES + red;
  if (smem3 <= 227 * 1024)
    return full ? launch_mx_s<MODE, NBLK, 3, true>(p, dev, sms, st, pdl, smem3, warps)
                : launch_mx_s<MODE, NBLK, 3, false>(p, dev, sms, st, pdl, smem3, warps);
  if (smem2 <= 227 * 1024)
    return full ? launch_mx_s<MODE, NBLK, 2, true>(p, dev, sms, st, pdl, smem2, warps)
                : launch_mx_s<MODE, NBLK, 2, false>(p, dev, sms, st, pdl, smem2, warps);
  return cudaErrorInvalidValue;
}

// bulk-copy GEMV: one CTA per SM, K / 256 compute warps + producer + reducer
template <int MODE, int NBLK, int STAGES>
cudaError_t launch_mxb(const MxGemvParams& p, int dev, int sms, cudaStream_t st, bool pdl) {
  constexpr bool PRE = MODE == MX_DOWN;  // its batches were written two kernels earlier
  const int smem = MxbLayout<MODE>::smem_bytes(p.K, STAGES, NBLK);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  if (!set_smem<k3_mxb_gemv_kernel<MODE, NBLK, STAGES, PRE>>(dev, smem)) return cudaErrorInvalidValue;
  // two CTAs per SM where shared memory and registers allow (more warps to hide the
  // per-item latency of the compute warps)
  cudaFuncAttributes fa{};
  if (cudaFuncGetAttributes(&fa, k3_mxb_gemv_kernel<MODE, NBLK, STAGES, PRE>) != cudaSuccess) return cudaErrorInvalidValue;
  const int threads = (2 + p.K / 256) * 32;
  const bool two = 2 * (smem + 2048) <= 228 * 1024 && 2 * threads * fa.numRegs <= 65536;
  return launch(k3_mxb_gemv_kernel<MODE, NBLK, STAGES, PRE>, dim3(two ? 2 * sms : sms), dim3(threads), smem, st, pdl,
                p);
}

template <int MODE>
cudaError_t launch_mx(const MxGemvParams& p, int nblk, int dev, int sms, cudaStream_t st, bool pdl) {
  if (mxb_ok(p.K)) {
    if constexpr (MODE == MX_GATEUP)
      return nblk == 1 ? launch_mxb<MODE, 1, 3>(p, dev, sms, st, pdl) : launch_mxb<MODE, 2, 2>(p, dev, sms, st, pdl);
    else
      return nblk == 1 ? launch_mxb<MODE, 1, 3>(p, dev, sms, st, pdl) : launch_mxb<MODE, 2, 6>(p, dev, sms, st, pdl);
  }
  return nblk == 1 ? launch_mx_t<MODE, 1>(p, dev, sms, st, pdl) : launch_mx_t<MODE, 2>(p, dev, sms, st, pdl);
}

cudaError_t launch_topk(const TopkParams& p, int dev, cudaStream_t st, bool pdl) {
  const int smem = TOPK_WARPS * 2 * p.E * 4;
  if (!set_smem<k3_topk_kernel>(dev, smem)) return cudaErrorInvalidValue;
  return launch(k3_topk_kernel, dim3((p.T + TOPK_WARPS - 1) / TOPK_WARPS), dim3(TOPK_WARPS * 32), smem, st, pdl, p);
}

cudaError_t launch_permute(const PermParams& p, int dev, cudaStream_t st, bool pdl) {
  const int smem = PERM_WARPS * p.E * 4;
  const int n = p.T * p.K;
  if (n <= 2 * PERM_SPAN) {  // one CTA
    if (!set_smem<k3_permute_kernel>(dev, smem)) return cudaErrorInvalidValue;
    return launch(k3_permute_kernel, dim3(1), dim3(PERM_WARPS * 32), smem, st, pdl, p);
  }
  const int nct = (n + PERM_SPAN - 1) / PERM_SPAN;
  if (!set_smem<k3_perm_hist_kernel>(dev, smem) || !set_smem<k3_perm_scatter_kernel>(dev, smem))
    return cudaErrorInvalidValue;
  cudaError_t e = launch(k3_perm_hist_kernel, dim3(nct), dim3(PERM_WARPS * 32), smem, st, pdl, p);
  if (e == cudaSuccess) e = launch(k3_perm_scan_kernel, dim3(1), dim3(PERM_WARPS * 32), 0, st, pdl, p, nct);
  if (e == cudaSuccess) e = launch(k3_perm_scatter_kernel, dim3(nct), dim3(PERM_WARPS * 32), smem, st, pdl, p);
  if (e == cudaSuccess && p.ex.gate_q) {
    const int bound = n / 8 + 1 + (p.E < n ? p.E : n);  // records capacity of the workspace
    const int blocks = (bound + 255) / 256;
    e = launch(k3_perm_records_kernel, dim3(blocks < 1024 ? blocks : 1024), dim3(256), 0, st, pdl, p);
  }
  return e;
}

cudaError_t launch_z16(const Z16Params& p, cudaStream_t st, bool pdl) {
  return launch(k3_z16_kernel, dim3((p.T + 7) / 8), dim3(256), 0, st, pdl, p);
}

int tail_smem(int E) {
  const int a = PERM_WARPS * 2 * E * 4;  // per-warp top-k buffers; permutation histograms
  const int b = (E <= TOPK_BLOCK_N) ? RouteSmem::bytes(E) : 0;  // one-token routing
  return a > b ? a : b;
}
bool tail_fits(int T, int E) {
  return T <= TAIL_MAX_T && tail_smem(E) + (int)(PERM_WARPS * sizeof(TopkScratch)) + 1024 <= 227 * 1024;
}

// top-k, permutation and activation prep: one fused launch for small T, else three
cudaError_t launch_route_tail(const TopkParams& tp, const PermParams& pp, const Z16Params& zp, int dev, cudaStream_t st,
                              bool pdl) {
  if (tail_fits(tp.T, tp.E)) {
    const int smem = tail_smem(tp.E);
    if (!set_smem<k3_route_tail_kernel>(dev, smem)) return cudaErrorInvalidValue;
    return launch(k3_route_tail_kernel, dim3(1), dim3(PERM_WARPS * 32), smem, st, pdl, tp, pp, zp);
  }
  cudaError_t e = launch_topk(tp, dev, st, pdl);
  if (e == cudaSuccess) e = launch_permute(pp, dev, st, pdl);
  if (e == cudaSuccess) e = launch_z16(zp, st, pdl);
  return e;
}

// one token: router logits, latent down and routing in one launch (k3_front_kernel); the
// bulk gate/up GEMV then reads z itself
bool front_ok(const DenseParams& dp, const TopkParams& tp, bool z_direct) {
  return z_direct && dense1_ok(dp) && tp.T == 1 && tp.E <= TOPK_BLOCK_N && tp.K + REFINE_EXTRA <= 32;
}
cudaError_t launch_front(const FrontParams& f, int dev, int sms, cudaStream_t st, bool pdl) {
  const int smem = front_smem_bytes(f.d.K, f.tp.E);
  if (!set_smem<k3_front_kernel>(dev, smem)) return cudaErrorInvalidValue;
  return launch(k3_front_kernel, dim3(2 * sms), dim3(FR_THREADS), smem, st, pdl, f);
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t st, bool pdl) {
  // one CTA per token while a thread holds at most 8 float4 columns and there are enough
  // tokens to fill the GPU (few tokens: a row is split over several CTAs for more loads
  // in flight)
  const int L4 = p.L / 4;
  const bool g16 = (reinterpret_cast<uintptr_t>(p.gamma) & 15u) == 0;
  if (p.T < kCombRowMinT && L4 <= COMB_ROW_MAX_THREADS && g16) {
    // few tokens: one CTA per token, one float4 column per thread (all K rows' loads of a
    // column in flight at once), the norm reduced inside the CTA
    const int threads = (L4 + 31) / 32 * 32;
    return launch(k3_combine_row_kernel<1, COMB_ROW_MAX_THREADS, 8>, dim3(p.T), dim3(threads), 0, st, pdl, p);
  }
  if (p.T >= kCombRowMinT && L4 <= 8 * COMB_THREADS && g16) {
    const int cpt = L4 <= COMB_THREADS ? 1 : L4 <= 2 * COMB_THREADS ? 2 : L4 <= 4 * COMB_THREADS ? 4 : 8;
    const int threads = ((L4 + cpt - 1) / cpt + 31) / 32 * 32;
    switch (cpt) {
      case 1: return launch(k3_combine_row_kernel<1>, dim3(p.T), dim3(threads), 0, st, pdl, p);
      case 2: return launch(k3_combine_row_kernel<2>, dim3(p.T), dim3(threads), 0, st, pdl, p);
      case 4: return launch(k3_combine_row_kernel<4>, dim3(p.T), dim3(threads), 0, st, pdl, p);
      default: return launch(k3_combine_row_kernel<8>, dim3(p.T), dim3(threads), 0, st, pdl, p);
    }
  }
  const int split = (p.L / 4 + COMB_THREADS - 1) / COMB_THREADS;  // one float4 column per thread
  if (split > COMB_MAX_SPLIT) return cudaErrorInvalidValue;
  return launch(k3_combine_norm_kernel, dim3(p.T, split), dim3(COMB_THREADS), 0, st, pdl, p);
}

// records event i of a caller-supplied list (no-op when absent)
cudaError_t mark(void* const* events, int n_events, int i, cudaStream_t s) {
  if (!events || i >= n_events || !events[i]) return cudaSuccess;
  return cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s);
}

#define K3_TRY(expr)                                   \
  do {                                                 \
    if ((expr) != cudaSuccess) return K3MOE_ERR_CUDA;  \
  } while (0)

PermParams perm_params(const k3moe_dims& d, int T, int K, const int32_t* ids, int fixed, int NB, void* ws,
                       const WsLayout& L, const k3moe_experts* ex) {
  PermParams pp{};
  if (ex) pp.ex = *ex;
  pp.batches = at<MxBatch>(ws, L.batches);
  pp.n_batches = at<int32_t>(ws, L.n_batches);
  pp.ids = ids;
  pp.fixed_expert = fixed;
  pp.T = T;
  pp.K = K;
  pp.E = d.n_experts;
  pp.NB = NB;
  pp.counts = at<int32_t>(ws, L.counts);
  pp.offsets = at<int32_t>(ws, L.offsets);
  pp.slot_of = at<int32_t>(ws, L.slot_of);
  pp.slot_tok = at<int32_t>(ws, L.slot_tok);
  pp.inv = at<int32_t>(ws, L.inv);
  pp.uniq = at<int32_t>(ws, L.uniq);
  pp.n_uniq = at<int32_t>(ws, L.n_uniq);
  pp.nb_prefix = at<int32_t>(ws, L.nb_prefix);
  pp.status = at<uint32_t>(ws, L.status);
  pp.cta_cnt = at<int32_t>(ws, L.cta_cnt);
  pp.cta_base = at<int32_t>(ws, L.cta_base);
  return pp;
}

MxGemvParams mx_params(const k3moe_dims& d, const WsLayout& L, void* ws, int mode, const __half* act, void* out) {
  MxGemvParams p{};
  p.status = at<uint32_t>(ws, L.status);
  if (mode == MX_GATEUP) {
    p.R = d.inter;
    p.K = d.latent;
    p.act_pow = at<int32_t>(ws, L.zpow);
  } else {
    p.R = d.latent;
    p.K = d.inter;
  }
  p.batches = at<MxBatch>(ws, L.batches);
  p.n_batches = at<int32_t>(ws, L.n_batches);
  p.act = act;
  p.out = out;
  return p;
}

bool experts_ok(const k3moe_experts* ex) {
  return ex && ex->gate_q && ex->gate_s && ex->up_q && ex->up_s && ex->down_q && ex->down_s;
}

}  // namespace

extern "C" {

size_t k3moe_workspace_bytes(const k3moe_dims* dims, int32_t T) {
  if (check_dims(dims) != K3MOE_OK || T < 0) return 0;
  return ws_layout(*dims, T).total;
}

k3moe_status k3moe_route(const k3moe_dims* dims, int32_t T, const uint16_t* x, const uint16_t* wr, const float* bias,
                         int32_t* ids, float* w, void* ws, size_t ws_bytes, void* stream) {
  k3moe_status st = check_dims(dims);
  if (st != K3MOE_OK) return st;
  if (T < 0) return K3MOE_ERR_ARG;
  if (T == 0) return K3MOE_OK;
  if (!x || !wr || !bias || !ids || !w || !ws) return K3MOE_ERR_ARG;
  if (!a16(x) || !a16(wr) || !a16(bias) || !a16(ids) || !a16(w) || !a16(ws)) return K3MOE_ERR_ALIGN;
  const k3moe_dims d = *dims;
  const WsLayout L = ws_layout(d, T);
  if (ws_bytes < L.total) return K3MOE_ERR_WORKSPACE;
  int dev, sms;
  if ((st = check_device(&dev, &sms)) != K3MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  K3_TRY(cudaMemsetAsync(at<void>(ws, L.status), 0, 256, s));
  if (T >= tc_min_t()) {
    TcDenseParams tcp{};
    tcp.out0 = at<float>(ws, L.logits);
    tcp.status = at<uint32_t>(ws, L.status);
    K3_TRY(launch_tc_dense<TC_PLAIN>(x, T, d.hidden, wr, d.n_experts, nullptr, 0, tcp, dev, sms, s, false,
                                     at<float>(ws, L.part), L.part_bytes));
  } else {
    DenseParams dp{};
    dp.W0 = wr; dp.R0 = d.n_experts; dp.W1 = nullptr; dp.R1 = 0; dp.K = d.hidden; dp.act = x; dp.T = T;
    dp.out0 = at<float>(ws, L.logits);
    dp.status = at<uint32_t>(ws, L.status);
    K3_TRY(launch_dense<DN_PROJ>(dp, dev, sms, s, false));
  }
  TopkParams tp{};
  tp.logits = at<float>(ws, L.logits); tp.bias = bias; tp.x = x; tp.wr = wr;
  tp.T = T; tp.E = d.n_experts; tp.K = d.top_k; tp.H = d.hidden; tp.tau = kTieTau;
  tp.top_p = top_p_on(d) ? d.top_p : 0.f;
  tp.ids = ids; tp.w = w; tp.status = at<uint32_t>(ws, L.status);
  K3_TRY(launch_topk(tp, dev, s, true));
  return K3MOE_OK;
}

k3moe_status k3moe_forward_profiled(const k3moe_dims* dims, int32_t T, const uint16_t* x, const uint16_t* wr,
                                    const float* bias, const uint16_t* w_down, const uint16_t* w_up,
                                    const float* norm_w, const k3moe_experts* experts, float* out, int32_t* ids_out,
                                    float* w_out, void* ws, size_t ws_bytes, void* stream, void* const* events,
                                    int32_t n_events) {
  k3moe_status st = check_dims(dims);
  if (st != K3MOE_OK) return st;
  if (T < 0) return K3MOE_ERR_ARG;
  if (T == 0) return K3MOE_OK;
  if (!x || !wr || !bias || !w_down || !w_up || !norm_w || !experts_ok(experts) || !out || !ws) return K3MOE_ERR_ARG;
  if (!a16(x) || !a16(wr) || !a16(bias) || !a16(w_down) || !a16(w_up) || !a16(norm_w) || !a16(out) || !a16(ws) ||
      (ids_out && !a16(ids_out)) || (w_out && !a16(w_out)))
    return K3MOE_ERR_ALIGN;
  const k3moe_dims d = *dims;
  const WsLayout L = ws_layout(d, T);
  if (ws_bytes < L.total) return K3MOE_ERR_WORKSPACE;
  int dev, sms;
  if ((st = check_device(&dev, &sms)) != K3MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* status = at<uint32_t>(ws, L.status);

  if (n_events < 0 || (n_events > 0 && !events)) return K3MOE_ERR_ARG;
  const bool pdl = n_events == 0;  // phase events between kernels would serialise them anyway
  K3_TRY(mark(events, n_events, 0, s));
  K3_TRY(cudaMemsetAsync(status, 0, L.zero_end - L.status, s));  // status, counters, z max, combine counts
  // routing parameters (top-k with double-f32 near-tie refinement, chunk expert union,
  // activation operand prep)
  TopkParams tp{};
  tp.logits = at<float>(ws, L.logits); tp.bias = bias; tp.x = x; tp.wr = wr;
  tp.T = T; tp.E = d.n_experts; tp.K = d.top_k; tp.H = d.hidden; tp.tau = kTieTau;
  tp.top_p = top_p_on(d) ? d.top_p : 0.f;
  tp.ids = at<int32_t>(ws, L.ids); tp.w = at<float>(ws, L.w); tp.ids_out = ids_out; tp.w_out = w_out;
  tp.status = status;
  const bool tc = tc_experts(d, T);
  const bool split = split_experts(d, T);
  const int nblk = mx_nblk(T);
  // tokens per expert batch: the block-scaled GEMMs' (split form, variant), the
  // weight-decode GEMM's, or the weight-streaming kernels'
  const int NB = (split || (tc && d.act_mxfp8)) ? mx8_batch(d, T) : (tc ? TM_NB : 8 * nblk);
  const PermParams pp = perm_params(d, T, d.top_k, at<int32_t>(ws, L.ids), 0, NB, ws, L, experts);
  // one token: the bulk gate/up GEMV reads z (bf16) and its max itself (converting it once
  // per warp), so no f16 copy of z is made; batches of several tokens convert per item and
  // keep the copy made in the routing kernel
  const bool z_direct = T == 1 && mxb_ok(d.latent);
  const Z16Params zp{at<uint16_t>(ws, L.z), z_direct ? 0 : T, d.latent, at<__half>(ws, L.z16), at<int32_t>(ws, L.zpow)};
  const int slots = T * d.top_k;
  DenseParams dp{};
  dp.W0 = wr; dp.R0 = d.n_experts; dp.W1 = w_down; dp.R1 = d.latent; dp.K = d.hidden; dp.act = x; dp.T = T;
  dp.out0 = at<float>(ws, L.logits); dp.out1 = at<uint16_t>(ws, L.z); dp.zmax = at<uint32_t>(ws, L.zmax);
  dp.status = status;
  if (!tc && front_ok(dp, tp, z_direct) && 2 * (front_smem_bytes(dp.K, d.n_experts) + 1024) <= 228 * 1024) {
    // one token: the router logits (one warp per row), then routing and latent down in one
    // launch that starts while the router kernel runs (the latent rows do not depend on it;
    // the routing waits for it); the route phase has no launch of its own
    DenseParams rp = dp;
    rp.W1 = nullptr;
    rp.R1 = 0;
    K3_TRY(launch_dense1<DN_PLAIN>(rp, dev, sms, s, false, D1_WARPS));
    DenseParams zd = dp;
    zd.W0 = w_down;
    zd.R0 = d.latent;
    zd.W1 = nullptr;
    zd.R1 = 0;
    FrontParams fp{zd, tp, pp};
    K3_TRY(launch_front(fp, dev, sms, s, pdl));
    K3_TRY(mark(events, n_events, 1, s));
  } else {
    // router logits and latent down in one weight-streaming pass over x
    if (T >= tc_min_t()) {
      TcDenseParams tcp{};
      tcp.out0 = at<float>(ws, L.logits); tcp.out1 = at<uint16_t>(ws, L.z); tcp.zmax = at<uint32_t>(ws, L.zmax);
      tcp.status = status;
      K3_TRY(launch_tc_dense<TC_PROJ>(x, T, d.hidden, wr, d.n_experts, w_down, d.latent, tcp, dev, sms, s, false,
                                      at<float>(ws, L.part), L.part_bytes));
    } else {
      K3_TRY(launch_dense<DN_PROJ>(dp, dev, sms, s, false));
    }
    K3_TRY(mark(events, n_events, 1, s));
    if (tc) {
      // top-k, permutation, then the activation rows in expert-sorted slot order for the
      // grouped GEMM (the f16 copy of z that the weight-streaming kernels read is not needed)
      K3_TRY(launch_topk(tp, dev, s, pdl));
      K3_TRY(launch_permute(pp, dev, s, pdl));
      if (split) {
        // z's two exact MXFP8 terms in slot order (codes, then the scale bytes)
        uint8_t* a8 = at<uint8_t>(ws, L.act);
        const size_t groups = (size_t)slots * (d.latent / 32);
        const int gblocks = (int)((groups + 255) / 256 < (size_t)sms * 8 ? (groups + 255) / 256 : (size_t)sms * 8);
        K3_TRY(launch(k3_split_rows_kernel, dim3(gblocks), dim3(256), 0, s, pdl,
                      (const uint16_t*)at<uint16_t>(ws, L.z), (const int32_t*)at<int32_t>(ws, L.slot_tok),
                      (const int32_t*)(at<int32_t>(ws, L.offsets) + d.n_experts), slots, (int)d.latent, a8,
                      a8 + (size_t)2 * slots * d.latent));
      } else if (d.act_mxfp8) {
        // z quantized to MXFP8 rows in slot order (codes, then the scale bytes)
        uint8_t* a8 = at<uint8_t>(ws, L.act);
        const size_t groups = (size_t)slots * (d.latent / 32);
        const int gblocks = (int)((groups + 255) / 256 < (size_t)sms * 8 ? (groups + 255) / 256 : (size_t)sms * 8);
        K3_TRY(launch(k3_gather_mx8_kernel, dim3(gblocks), dim3(256), 0, s, pdl, (const uint16_t*)at<uint16_t>(ws, L.z),
                      (const int32_t*)at<int32_t>(ws, L.slot_tok),
                      (const int32_t*)(at<int32_t>(ws, L.offsets) + d.n_experts), slots, (int)d.latent, a8,
                      a8 + (size_t)slots * d.latent));
      } else {
        // bf16 rows in slot order (interleaved K order)
        const int per = d.latent / 8;
        const size_t items = (size_t)slots * per;
        const int gblocks = (int)((items + 255) / 256 < (size_t)sms * 8 ? (items + 255) / 256 : (size_t)sms * 8);
        K3_TRY(launch(k3_gather_rows_kernel, dim3(gblocks), dim3(256), 0, s, pdl,
                      (const uint16_t*)at<uint16_t>(ws, L.z), (const int32_t*)at<int32_t>(ws, L.slot_tok),
                      (const int32_t*)(at<int32_t>(ws, L.offsets) + d.n_experts), slots, (int)d.latent,
                      at<uint16_t>(ws, L.act)));
      }
    } else {
      K3_TRY(launch_route_tail(tp, pp, zp, dev, s, pdl));
    }
  }
  K3_TRY(mark(events, n_events, 2, s));
  // experts
  if (split) {
    // exact: the bf16 z and h as two MXFP8 terms each, block-scaled MMAs on the stored
    // MXFP4 weights (terms' codes [2][slots][K], then their scale bytes [2][slots][K / 32])
    const uint8_t* a8 = at<uint8_t>(ws, L.act);
    uint16_t* hb = at<uint16_t>(ws, L.h16);
    uint8_t* h8 = at<uint8_t>(ws, L.hterm);
    Mx8Params gp{at<MxBatch>(ws, L.batches), at<int32_t>(ws, L.n_batches), d.inter, d.latent,
                 a8 + (size_t)2 * slots * d.latent, slots, hb, nullptr, status, at<void>(ws, L.tmaps)};
    K3_TRY((launch_mx8_moe<0, 1>(a8, gp, NB, dev, sms, s, pdl)));
    // h (bf16, slot order) -> its two terms for the down GEMM
    const size_t hgroups = (size_t)slots * (d.inter / 32);
    const int hblocks = (int)((hgroups + 255) / 256 < (size_t)sms * 8 ? (hgroups + 255) / 256 : (size_t)sms * 8);
    K3_TRY(launch(k3_split_rows_kernel, dim3(hblocks), dim3(256), 0, s, pdl, (const uint16_t*)hb,
                  (const int32_t*)nullptr, (const int32_t*)(at<int32_t>(ws, L.offsets) + d.n_experts), slots,
                  (int)d.inter, h8, h8 + (size_t)2 * slots * d.inter));
    K3_TRY(mark(events, n_events, 3, s));
    Mx8Params dp2{at<MxBatch>(ws, L.batches), at<int32_t>(ws, L.n_batches), d.latent, d.inter,
                  h8 + (size_t)2 * slots * d.inter, slots, at<void>(ws, L.o), nullptr, status, at<void>(ws, L.tmaps)};
    K3_TRY((launch_mx8_moe<1, 1>(h8, dp2, NB, dev, sms, s, pdl)));
  } else if (tc && d.act_mxfp8) {
    // MXFP8 activations, block-scaled MMAs on the stored MXFP4 weights; h leaves the gate/up
    // epilogue as MXFP8 rows in slot order (codes, then the scale bytes)
    const uint8_t* a8 = at<uint8_t>(ws, L.act);
    uint8_t* h8 = at<uint8_t>(ws, L.h16);
    Mx8Params gp{at<MxBatch>(ws, L.batches), at<int32_t>(ws, L.n_batches), d.inter, d.latent,
                 a8 + (size_t)slots * d.latent, slots, h8, h8 + (size_t)slots * d.inter, status, at<void>(ws, L.tmaps)};
    K3_TRY((launch_mx8_moe<0, 0>(a8, gp, NB, dev, sms, s, pdl)));
    K3_TRY(mark(events, n_events, 3, s));
    Mx8Params dp2{at<MxBatch>(ws, L.batches), at<int32_t>(ws, L.n_batches), d.latent, d.inter,
                  h8 + (size_t)slots * d.inter, slots, at<void>(ws, L.o), nullptr, status, at<void>(ws, L.tmaps)};
    K3_TRY((launch_mx8_moe<1, 0>(h8, dp2, NB, dev, sms, s, pdl)));
  } else if (tc) {
    TcMoeParams gp{at<MxBatch>(ws, L.batches), at<int32_t>(ws, L.n_batches), d.inter, d.latent,
                   at<void>(ws, L.h16), status, at<void>(ws, L.tmaps)};
    K3_TRY(launch_tc_moe<0>(at<uint16_t>(ws, L.act), slots, gp, dev, sms, s, pdl));
    K3_TRY(mark(events, n_events, 3, s));
    TcMoeParams dp2{at<MxBatch>(ws, L.batches), at<int32_t>(ws, L.n_batches), d.latent, d.inter,
                    at<void>(ws, L.o), status, at<void>(ws, L.tmaps)};
    K3_TRY(launch_tc_moe<1>(at<uint16_t>(ws, L.h16), slots, dp2, dev, sms, s, pdl));
  } else {
    MxGemvParams gu = mx_params(d, L, ws, MX_GATEUP, at<__half>(ws, L.z16), at<void>(ws, L.h16));
    if (z_direct) {
      gu.act_bf16 = at<uint16_t>(ws, L.z);
      gu.act_max = at<uint32_t>(ws, L.zmax);
    }
    K3_TRY(launch_mx<MX_GATEUP>(gu, nblk, dev, sms, s, pdl));
    K3_TRY(mark(events, n_events, 3, s));
    K3_TRY(launch_mx<MX_DOWN>(mx_params(d, L, ws, MX_DOWN, at<__half>(ws, L.h16), at<void>(ws, L.o)), nblk, dev,
                              sms, s, pdl));
  }
  K3_TRY(mark(events, n_events, 4, s));
  // combine + RMSNorm
  CombineParams cp{at<float>(ws, L.o),     at<int32_t>(ws, L.inv),  at<float>(ws, L.w),
                   norm_w,                 T,                       d.top_k,
                   d.latent,               d.rms_eps,               at<float>(ws, L.y),
                   at<uint16_t>(ws, L.yhat), at<float>(ws, L.cpart), at<uint32_t>(ws, L.ccount)};
  K3_TRY(launch_combine(cp, s, pdl));
  K3_TRY(mark(events, n_events, 5, s));
  // latent up
  if (T >= tc_min_t()) {
    TcDenseParams tcp{};
    tcp.out0 = out;
    tcp.status = status;
    K3_TRY(launch_tc_dense<TC_PLAIN>(at<uint16_t>(ws, L.yhat), T, d.latent, w_up, d.hidden, nullptr, 0, tcp, dev, sms,
                                     s, pdl, at<float>(ws, L.part), L.part_bytes));
  } else {
    DenseParams up{};
    up.W0 = w_up; up.R0 = d.hidden; up.K = d.latent; up.act = at<uint16_t>(ws, L.yhat); up.T = T; up.out0 = out;
    up.status = status;
    K3_TRY(launch_dense<DN_PLAIN>(up, dev, sms, s, pdl));
  }
  K3_TRY(mark(events, n_events, 6, s));
  return K3MOE_OK;
}

k3moe_status k3moe_forward(const k3moe_dims* dims, int32_t T, const uint16_t* x, const uint16_t* wr,
                           const float* bias, const uint16_t* w_down, const uint16_t* w_up, const float* norm_w,
                           const k3moe_experts* experts, float* out, int32_t* ids_out, float* w_out, void* ws,
                           size_t ws_bytes, void* stream) {
  return k3moe_forward_profiled(dims, T, x, wr, bias, w_down, w_up, norm_w, experts, out, ids_out, w_out, ws,
                                ws_bytes, stream, nullptr, 0);
}

// ---------------------------------------------------------------------------- shared experts
namespace {
struct SharedLayout {
  size_t status, gu, h, total;
};
SharedLayout shared_layout(const k3moe_dims& d, int T, int Is) {
  SharedLayout L{};
  size_t off = 0;
  auto take = [&](size_t b) {
    const size_t o = off;
    off += align256(b);
    return o;
  };
  L.status = take(256);
  L.gu = take((size_t)T * 2 * Is * 4);
  L.h = take((size_t)T * Is * 2);
  L.total = off;
  return L;
}
bool shared_ok(const k3moe_dims* d, int Is) {
  return check_dims(d) == K3MOE_OK && Is > 0 && Is % 64 == 0 && Is <= 65536;
}
}  // namespace

k3moe_status k3moe_expert_forward(const k3moe_dims* dims, int32_t T, const uint16_t* z, int32_t expert,
                                  const k3moe_experts* experts, float* out, void* ws, size_t ws_bytes, void* stream) {
  k3moe_status st = check_dims(dims);
  if (st != K3MOE_OK) return st;
  if (T < 0 || expert < 0 || expert >= dims->n_experts) return K3MOE_ERR_ARG;
  if (T == 0) return K3MOE_OK;
  if (!z || !experts_ok(experts) || !out || !ws) return K3MOE_ERR_ARG;
  if (!a16(z) || !a16(out) || !a16(ws)) return K3MOE_ERR_ALIGN;
  const k3moe_dims d = *dims;
  const WsLayout L = ws_layout(d, T);
  if (ws_bytes < L.total) return K3MOE_ERR_WORKSPACE;
  int dev, sms;
  if ((st = check_device(&dev, &sms)) != K3MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  K3_TRY(cudaMemsetAsync(at<void>(ws, L.status), 0, 256, s));
  const int nblk = mx_nblk(T);
  K3_TRY(launch_permute(perm_params(d, T, 1, nullptr, expert, 8 * nblk, ws, L, experts), dev, s, false));
  Z16Params zp{z, T, d.latent, at<__half>(ws, L.z16), at<int32_t>(ws, L.zpow)};
  K3_TRY(launch_z16(zp, s, true));
  K3_TRY(launch_mx<MX_GATEUP>(mx_params(d, L, ws, MX_GATEUP, at<__half>(ws, L.z16), at<void>(ws, L.h16)), nblk, dev,
                              sms, s, true));
  // one expert: sorted slots are the tokens in order, so the down output lands in `out` directly
  K3_TRY(launch_mx<MX_DOWN>(mx_params(d, L, ws, MX_DOWN, at<__half>(ws, L.h16), out), nblk, dev, sms, s, true));
  return K3MOE_OK;
}

size_t k3moe_shared_workspace_bytes(const k3moe_dims* dims, int32_t T, int32_t inter_s) {
  if (!shared_ok(dims, inter_s) || T < 0) return 0;
  return shared_layout(*dims, T, inter_s).total;
}

k3moe_status k3moe_shared_forward(const k3moe_dims* dims, int32_t T, int32_t inter_s, const uint16_t* x,
                                  const uint16_t* w_gate_up, const uint16_t* w_down, float* out, void* ws,
                                  size_t ws_bytes, void* stream) {
  k3moe_status st = check_dims(dims);
  if (st != K3MOE_OK) return st;
  if (!shared_ok(dims, inter_s)) return K3MOE_ERR_SHAPE;
  if (T < 0) return K3MOE_ERR_ARG;
  if (T == 0) return K3MOE_OK;
  if (!x || !w_gate_up || !w_down || !out || !ws) return K3MOE_ERR_ARG;
  if (!a16(x) || !a16(w_gate_up) || !a16(w_down) || !a16(out) || !a16(ws)) return K3MOE_ERR_ALIGN;
  const k3moe_dims d = *dims;
  const int Is = inter_s, H = d.hidden;
  const SharedLayout L = shared_layout(d, T, Is);
  if (ws_bytes < L.total) return K3MOE_ERR_WORKSPACE;
  int dev, sms;
  if ((st = check_device(&dev, &sms)) != K3MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* status = at<uint32_t>(ws, L.status);
  float* gu = at<float>(ws, L.gu);
  uint16_t* h = at<uint16_t>(ws, L.h);
  K3_TRY(cudaMemsetAsync(status, 0, 256, s));
  const bool tc = T >= tc_min_t();
  // [g | u] = x . Wgu^T
  if (tc) {
    TcDenseParams tcp{};
    tcp.out0 = gu;
    tcp.status = status;
    K3_TRY(launch_tc_dense<TC_PLAIN>(x, T, H, w_gate_up, 2 * Is, nullptr, 0, tcp, dev, sms, s, false));
  } else {
    DenseParams dp{};
    dp.W0 = w_gate_up; dp.R0 = 2 * Is; dp.K = H; dp.act = x; dp.T = T; dp.out0 = gu; dp.status = status;
    K3_TRY(launch_dense<DN_PLAIN>(dp, dev, sms, s, false));
  }
  // h = bf16(SiTU(g, u))
  const size_t items = (size_t)T * (Is / 4);
  const int gblocks = (int)((items + 255) / 256 < (size_t)sms * 8 ? (items + 255) / 256 : (size_t)sms * 8);
  K3_TRY(launch(k3_shared_glu_kernel, dim3(gblocks), dim3(256), 0, s, true, (const float*)gu, (int)T, Is, h));
  // out += h . Wdn^T
  if (tc) {
    TcDenseParams tcp{};
    tcp.out0 = out;
    tcp.status = status;
    K3_TRY(launch_tc_dense<TC_ACC>(h, T, Is, w_down, H, nullptr, 0, tcp, dev, sms, s, true));
  } else {
    DenseParams dp{};
    dp.W0 = w_down; dp.R0 = H; dp.K = Is; dp.act = h; dp.T = T; dp.out0 = out; dp.status = status;
    K3_TRY(launch_dense<DN_ACC>(dp, dev, sms, s, true));
  }
  return K3MOE_OK;
}

k3moe_status k3moe_dequant_mxfp4(const uint8_t* q, const uint8_t* sc, int32_t O, int32_t I, float* out, void* stream) {
  if (O < 0 || I < 0) return K3MOE_ERR_ARG;
  if (I % 32) return K3MOE_ERR_SHAPE;
  if ((size_t)O * (size_t)I == 0) return K3MOE_OK;
  if (!q || !sc || !out) return K3MOE_ERR_ARG;
  if (!a16(q) || !a16(out)) return K3MOE_ERR_ALIGN;
  int dev, sms;
  k3moe_status st = check_device(&dev, &sms);
  if (st != K3MOE_OK) return st;
  const size_t words = (size_t)O * (I / 8);
  size_t grid = (words + 255) / 256;
  if (grid > (size_t)sms * 16) grid = (size_t)sms * 16;
  k3_dequant_kernel<<<(unsigned)grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(q, sc, O, I, out);
  return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}

k3moe_status k3moe_permute(const k3moe_dims* dims, int32_t T, const int32_t* ids, int32_t* counts, int32_t* offsets,
                           int32_t* slot_of, int32_t* uniq, int32_t* n_uniq, void* ws, size_t ws_bytes,
                           void* stream) {
  k3moe_status st = check_dims(dims);
  if (st != K3MOE_OK) return st;
  if (T < 0) return K3MOE_ERR_ARG;
  if (!ids || !counts || !offsets || !slot_of || !uniq || !n_uniq || !ws) return K3MOE_ERR_ARG;
  if (!a16(ids) || !a16(counts) || !a16(offsets) || !a16(slot_of) || !a16(uniq) || !a16(n_uniq) || !a16(ws))
    return K3MOE_ERR_ALIGN;
  const k3moe_dims d = *dims;
  const WsLayout L = ws_layout(d, T);
  if (ws_bytes < L.total) return K3MOE_ERR_WORKSPACE;
  int dev, sms;
  if ((st = check_device(&dev, &sms)) != K3MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  K3_TRY(cudaMemsetAsync(at<void>(ws, L.status), 0, 256, s));
  PermParams pp = perm_params(d, T, d.top_k, ids, 0, 8, ws, L, nullptr);
  pp.counts = counts;
  pp.offsets = offsets;
  pp.slot_of = slot_of;
  pp.uniq = uniq;
  pp.n_uniq = n_uniq;
  K3_TRY(launch_permute(pp, dev, s, false));
  return K3MOE_OK;
}

int32_t k3moe_set_tc_min_tokens(int32_t t) {
  if (t < 1) return -1;
  return g_tc_min_t.exchange(t);
}

int32_t k3moe_tc_min_tokens(void) { return tc_min_t(); }

int32_t k3moe_set_tc_split_max_tokens(int32_t t) {
  if (t < 0) return -1;
  return g_split_max_t.exchange(t);
}

int32_t k3moe_tc_split_max_tokens(void) { return g_split_max_t.load(std::memory_order_relaxed); }

k3moe_status k3moe_selftest_wait_timeout(void* ws, size_t ws_bytes, int64_t limit_cycles, void* stream) {
  if (!ws || ws_bytes < 256 || limit_cycles <= 0 || limit_cycles > (1ll << 32)) return K3MOE_ERR_ARG;
  if (!a16(ws)) return K3MOE_ERR_ALIGN;
  int dev, sms;
  const k3moe_status st = check_device(&dev, &sms);
  if (st != K3MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  K3_TRY(cudaMemsetAsync(ws, 0, 256, s));
  k3_selftest_timeout_kernel<<<1, 64, 0, s>>>(static_cast<uint32_t*>(ws), (long long)limit_cycles);
  K3_TRY(cudaGetLastError());
  return K3MOE_OK;
}

void* k3moe_workspace_view(const k3moe_dims* dims, int32_t T, void* ws, int32_t which) {
  if (check_dims(dims) != K3MOE_OK || T < 0 || !ws) return nullptr;
  const WsLayout L = ws_layout(*dims, T);
  switch (which) {
    case 0: return at<void>(ws, L.z);
    case 1: return at<void>(ws, L.yhat);
    case 2: return at<void>(ws, L.y);
    case 3: return at<void>(ws, L.logits);
    case 4: return at<void>(ws, L.h16);
    case 5: return at<void>(ws, L.o);
    default: break;
  }
  // MXFP8 rows: the variant's one term, or the exact split's two (hi rows, then lo rows)
  const size_t terms = dims->act_mxfp8 ? 1 : (split_experts(*dims, T) ? 2 : 0);
  if (!terms) return nullptr;
  const size_t slots = (size_t)T * dims->top_k;
  switch (which) {
    case 6: return at<void>(ws, L.act);
    case 7: return at<uint8_t>(ws, L.act) + terms * slots * dims->latent;
    case 8: return at<void>(ws, terms == 2 ? L.hterm : L.h16);
    case 9: return at<uint8_t>(ws, terms == 2 ? L.hterm : L.h16) + terms * slots * dims->inter;
    default: return nullptr;
  }
}

}  // extern "C"

// ---------------------------------------------------------------------------- allocation-free entry
// Scratch for k3moe_forward_noalloc: a fixed array in device memory that every GPU
// loading this library holds until the process exits.
static __device__ __align__(256) uint8_t g_k3_noalloc_scratch[K3MOE_NOALLOC_SCRATCH_BYTES];

namespace {
// Device address of the scratch array per device, with the id of the context it was
// looked up in (host code cannot use the array's name as a device pointer, and a reset
// device gets a new context whose copy of the array may live elsewhere).
struct NoallocSlot {
  void* ptr = nullptr;
  unsigned long long ctx_id = 0;
};
NoallocSlot g_noalloc[kMaxDevices];
std::atomic<bool> g_noalloc_ready[kMaxDevices];
std::mutex g_noalloc_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// id of the calling thread's current context (0 when none is current or the driver
// entry points are unavailable)
unsigned long long current_ctx_id() {
  static std::atomic<CtxGetCurrentFn> get_cur{nullptr};
  static std::atomic<CtxGetIdFn> get_id{nullptr};
  CtxGetCurrentFn fc = get_cur.load(std::memory_order_acquire);
  CtxGetIdFn fi = get_id.load(std::memory_order_acquire);
  if (!fc || !fi) {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult q1{}, q2{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess)
      return 0;
    fc = reinterpret_cast<CtxGetCurrentFn>(a);
    fi = reinterpret_cast<CtxGetIdFn>(b);
    get_cur.store(fc, std::memory_order_release);
    get_id.store(fi, std::memory_order_release);
  }
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (fc(&c) != CUDA_SUCCESS || !c || fi(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// The scratch array's device address on the current device.  Looked up with
// cudaGetSymbolAddress on the first call per device, and again only if the current
// context is no longer the one of that lookup (a device reset in between).
k3moe_status noalloc_scratch(void** out) {
  int dev = 0, sms = 0;
  k3moe_status st = check_device(&dev, &sms);
  if (st != K3MOE_OK) return st;
  const unsigned long long cur = current_ctx_id();
  if (g_noalloc_ready[dev].load(std::memory_order_acquire) && (cur == 0 || cur == g_noalloc[dev].ctx_id)) {
    *out = g_noalloc[dev].ptr;
    return K3MOE_OK;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_k3_noalloc_scratch) != cudaSuccess || !p) {
    (void)cudaGetLastError();  // leave no pending error behind for the caller's next check
    return K3MOE_ERR_CUDA;
  }
  g_noalloc[dev].ptr = p;
  g_noalloc[dev].ctx_id = current_ctx_id();  // the lookup made the device's context current
  g_noalloc_ready[dev].store(true, std::memory_order_release);
  *out = p;
  return K3MOE_OK;
}
}  // namespace

extern "C" {

k3moe_status k3moe_forward_noalloc(const k3moe_dims* dims, int32_t T, const uint16_t* x, const uint16_t* wr,
                                   const float* bias, const uint16_t* w_down, const uint16_t* w_up,
                                   const float* norm_w, const k3moe_experts* experts, float* out, int32_t* ids_out,
                                   float* w_out, void* stream) {
  k3moe_status st = check_dims(dims);
  if (st != K3MOE_OK) return st;
  if (T < 0) return K3MOE_ERR_ARG;
  if (T == 0) return K3MOE_OK;
  if (ws_layout(*dims, T).total > K3MOE_NOALLOC_SCRATCH_BYTES) return K3MOE_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != K3MOE_OK) return st;
  return k3moe_forward(dims, T, x, wr, bias, w_down, w_up, norm_w, experts, out, ids_out, w_out, scratch,
                       K3MOE_NOALLOC_SCRATCH_BYTES, stream);
}

k3moe_status k3moe_device_status(const void* ws, uint32_t* host_out, void* stream) {
  if (!host_out) return K3MOE_ERR_ARG;
  if (!ws) {  // the allocation-free entry point's scratch on the current device
    void* scratch = nullptr;
    const k3moe_status st = noalloc_scratch(&scratch);
    if (st != K3MOE_OK) return st;
    ws = scratch;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  K3_TRY(cudaMemcpyAsync(host_out, ws, 4, cudaMemcpyDeviceToHost, s));
  K3_TRY(cudaStreamSynchronize(s));
  return K3MOE_OK;
}

const char* k3moe_status_str(k3moe_status st) {
  switch (st) {
    case K3MOE_OK: return "ok";
    case K3MOE_ERR_ARG: return "invalid argument";
    case K3MOE_ERR_SHAPE: return "unsupported shape";
    case K3MOE_ERR_ALIGN: return "pointer not 16-byte aligned";
    case K3MOE_ERR_WORKSPACE: return "workspace too small";
    case K3MOE_ERR_DEVICE: return "current device is not compute capability 10.3";
    case K3MOE_ERR_CUDA: return "CUDA launch or copy failed";
  }
  return "unknown status";
}

int32_t k3moe_abi_version(void) { return 3; }

}  // extern "C"

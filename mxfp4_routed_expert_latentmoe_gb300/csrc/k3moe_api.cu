// k3moe_api.cu -- C ABI of the LatentMoE routed-expert block (see include/k3moe.h):
// host-side validation, workspace carving and the launch sequence.  No allocation,
// no synchronisation (except k3moe_device_status, which is documented to sync).
#include <atomic>
#include <cstring>

#include "k3_common.cuh"
#include "k3_gemv.cuh"
#include "k3_route.cuh"

namespace {

using namespace k3;

constexpr float kTieTau = 3e-5f;
constexpr int kMaxDevices = 64;

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

struct WsLayout {
  size_t status, logits, ids, w, zmax, zpow, counts, offsets, slot_of, slot_tok, inv, uniq, n_uniq, nb_prefix, z,
      z16, h16, o, y, yhat, total;
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
  L.status = take(256);
  L.logits = take(Tz * E * 4);
  L.ids = take(slots * 4);
  L.w = take(slots * 4);
  L.zmax = take(Tz * 4);
  L.zpow = take(Tz * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.slot_of = take(slots * 4);
  L.slot_tok = take(slots * 4);
  L.inv = take(slots * 4);
  L.uniq = take(E * 4);
  L.n_uniq = take(4);
  L.nb_prefix = take((E + 1) * 4);
  L.z = take(Tz * Lt * 2);
  L.z16 = take(Tz * Lt * 2);
  L.h16 = take(slots * I * 2);
  L.o = take(slots * Lt * 4);
  L.y = take(Tz * Lt * 4);
  L.yhat = take(Tz * Lt * 2);
  L.total = off;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

k3moe_status check_dims(const k3moe_dims* d) {
  if (!d) return K3MOE_ERR_ARG;
  if (d->hidden <= 0 || d->latent <= 0 || d->inter <= 0 || d->n_experts <= 0 || d->top_k <= 0)
    return K3MOE_ERR_SHAPE;
  if (d->hidden % 64 || d->latent % 64 || d->inter % 64) return K3MOE_ERR_SHAPE;
  if (d->n_experts > TOPK_MAX_E || d->top_k > 64 || d->top_k > d->n_experts) return K3MOE_ERR_SHAPE;
  if (d->latent > 32768 || d->inter > 32768 || d->hidden > 65536) return K3MOE_ERR_SHAPE;
  if (!(d->rms_eps >= 0.0f) || d->rms_eps > 1.0f) return K3MOE_ERR_ARG;
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

// ---------------------------------------------------------------------------- launch helpers
constexpr int kDnStages = 5;
constexpr int kMxStages = 3;

int dn_smem(int nblk) { return DN_WARPS * kDnStages * DN_STAGE_BYTES + DN_WARPS * nblk * 128 * 4; }

template <int EPI, int NBLK>
cudaError_t launch_dense_t(const DenseParams& p, int dev, int sms, cudaStream_t st) {
  auto kern = k3_dense_gemv_kernel<EPI, NBLK, kDnStages>;
  const int smem = dn_smem(NBLK);
  if (!set_smem<k3_dense_gemv_kernel<EPI, NBLK, kDnStages>>(dev, smem)) return cudaErrorInvalidValue;
  const int tiles = (p.R0 + 15) / 16 + (p.R1 + 15) / 16;
  const int total = tiles * ((p.T + 8 * NBLK - 1) / (8 * NBLK));
  const int grid = total < 2 * sms ? total : 2 * sms;
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, DN_WARPS * 32, smem, st>>>(p);
  return cudaGetLastError();
}

template <int EPI>
cudaError_t launch_dense(const DenseParams& p, int dev, int sms, cudaStream_t st) {
  if (p.T <= 8) return launch_dense_t<EPI, 1>(p, dev, sms, st);
  if (p.T <= 16) return launch_dense_t<EPI, 2>(p, dev, sms, st);
  return launch_dense_t<EPI, 4>(p, dev, sms, st);
}

int mx_nblk(int T) { return T <= 8 ? 1 : 2; }

template <int MODE, int NBLK>
cudaError_t launch_mx_t(const MxGemvParams& p, int dev, int sms, cudaStream_t st) {
  constexpr int M = MODE == MX_GATEUP ? 2 : 1;
  auto kern = k3_mx_gemv_kernel<MODE, NBLK, kMxStages>;
  const int warps = (p.K / 32 + MX_GPW - 1) / MX_GPW;
  const int smem = warps * MxLayout<M, kMxStages>::WARP_BYTES + warps * M * NBLK * 128 * 4;
  if (warps * 32 > MX_MAX_THREADS || smem > 227 * 1024) return cudaErrorInvalidValue;
  if (!set_smem<k3_mx_gemv_kernel<MODE, NBLK, kMxStages>>(dev, smem)) return cudaErrorInvalidValue;
  const int per_sm = (2 * smem + 2048 <= 228 * 1024) ? 2 : 1;
  kern<<<sms * per_sm, warps * 32, smem, st>>>(p);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_mx(const MxGemvParams& p, int nblk, int dev, int sms, cudaStream_t st) {
  return nblk == 1 ? launch_mx_t<MODE, 1>(p, dev, sms, st) : launch_mx_t<MODE, 2>(p, dev, sms, st);
}

cudaError_t launch_topk(const TopkParams& p, int dev, cudaStream_t st) {
  const int smem = TOPK_WARPS * 2 * p.E * 4;
  if (!set_smem<k3_topk_kernel>(dev, smem)) return cudaErrorInvalidValue;
  k3_topk_kernel<<<(p.T + TOPK_WARPS - 1) / TOPK_WARPS, TOPK_WARPS * 32, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_permute(const PermParams& p, int dev, cudaStream_t st) {
  const int smem = PERM_WARPS * p.E * 4;
  if (!set_smem<k3_permute_kernel>(dev, smem)) return cudaErrorInvalidValue;
  k3_permute_kernel<<<1, PERM_WARPS * 32, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_z16(const Z16Params& p, cudaStream_t st) {
  k3_z16_kernel<<<(p.T + 7) / 8, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_combine(const CombineParams& p, int dev, cudaStream_t st) {
  const int smem = p.L * 4;
  if (!set_smem<k3_combine_norm_kernel>(dev, smem)) return cudaErrorInvalidValue;
  k3_combine_norm_kernel<<<p.T, COMB_THREADS, smem, st>>>(p);
  return cudaGetLastError();
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
                       const WsLayout& L) {
  PermParams pp{};
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
  return pp;
}

MxGemvParams mx_params(const k3moe_dims& d, const WsLayout& L, void* ws, const k3moe_experts& ex, int mode,
                       const __half* act, void* out) {
  MxGemvParams p{};
  if (mode == MX_GATEUP) {
    p.q0 = ex.gate_q; p.s0 = ex.gate_s; p.q1 = ex.up_q; p.s1 = ex.up_s;
    p.R = d.inter; p.K = d.latent;
    p.act_pow = at<int32_t>(ws, L.zpow);
  } else {
    p.q0 = ex.down_q; p.s0 = ex.down_s; p.q1 = ex.down_q; p.s1 = ex.down_s;
    p.R = d.latent; p.K = d.inter;
  }
  p.uniq = at<int32_t>(ws, L.uniq);
  p.n_uniq = at<int32_t>(ws, L.n_uniq);
  p.counts = at<int32_t>(ws, L.counts);
  p.offsets = at<int32_t>(ws, L.offsets);
  p.nb_prefix = at<int32_t>(ws, L.nb_prefix);
  p.slot_tok = at<int32_t>(ws, L.slot_tok);
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
  DenseParams dp{};
  dp.W0 = wr; dp.R0 = d.n_experts; dp.W1 = nullptr; dp.R1 = 0; dp.K = d.hidden; dp.act = x; dp.T = T;
  dp.out0 = at<float>(ws, L.logits);
  K3_TRY(launch_dense<DN_PROJ>(dp, dev, sms, s));
  TopkParams tp{};
  tp.logits = at<float>(ws, L.logits); tp.bias = bias; tp.x = x; tp.wr = wr;
  tp.T = T; tp.E = d.n_experts; tp.K = d.top_k; tp.H = d.hidden; tp.tau = kTieTau;
  tp.ids = ids; tp.w = w; tp.status = at<uint32_t>(ws, L.status);
  K3_TRY(launch_topk(tp, dev, s));
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
  K3_TRY(mark(events, n_events, 0, s));
  K3_TRY(cudaMemsetAsync(status, 0, 256, s));
  K3_TRY(cudaMemsetAsync(at<void>(ws, L.zmax), 0, (size_t)T * 4, s));
  // router logits and latent down in one weight-streaming pass over x
  DenseParams dp{};
  dp.W0 = wr; dp.R0 = d.n_experts; dp.W1 = w_down; dp.R1 = d.latent; dp.K = d.hidden; dp.act = x; dp.T = T;
  dp.out0 = at<float>(ws, L.logits); dp.out1 = at<uint16_t>(ws, L.z); dp.zmax = at<uint32_t>(ws, L.zmax);
  K3_TRY(launch_dense<DN_PROJ>(dp, dev, sms, s));
  K3_TRY(mark(events, n_events, 1, s));
  // top-k with fp64 near-tie refinement
  TopkParams tp{};
  tp.logits = at<float>(ws, L.logits); tp.bias = bias; tp.x = x; tp.wr = wr;
  tp.T = T; tp.E = d.n_experts; tp.K = d.top_k; tp.H = d.hidden; tp.tau = kTieTau;
  tp.ids = at<int32_t>(ws, L.ids); tp.w = at<float>(ws, L.w); tp.ids_out = ids_out; tp.w_out = w_out;
  tp.status = status;
  K3_TRY(launch_topk(tp, dev, s));
  K3_TRY(mark(events, n_events, 2, s));
  // chunk expert union
  const int nblk = mx_nblk(T);
  K3_TRY(launch_permute(perm_params(d, T, d.top_k, at<int32_t>(ws, L.ids), 0, 8 * nblk, ws, L), dev, s));
  K3_TRY(mark(events, n_events, 3, s));
  // z -> f16 operand
  Z16Params zp{at<uint16_t>(ws, L.z), T, d.latent, at<__half>(ws, L.z16), at<int32_t>(ws, L.zpow)};
  K3_TRY(launch_z16(zp, s));
  K3_TRY(mark(events, n_events, 4, s));
  // experts
  const k3moe_experts ex = *experts;
  K3_TRY(launch_mx<MX_GATEUP>(mx_params(d, L, ws, ex, MX_GATEUP, at<__half>(ws, L.z16), at<void>(ws, L.h16)), nblk,
                              dev, sms, s));
  K3_TRY(mark(events, n_events, 5, s));
  K3_TRY(launch_mx<MX_DOWN>(mx_params(d, L, ws, ex, MX_DOWN, at<__half>(ws, L.h16), at<void>(ws, L.o)), nblk, dev,
                            sms, s));
  K3_TRY(mark(events, n_events, 6, s));
  // combine + RMSNorm
  CombineParams cp{at<float>(ws, L.o), at<int32_t>(ws, L.inv), at<float>(ws, L.w), norm_w, T, d.top_k, d.latent,
                   d.rms_eps, at<float>(ws, L.y), at<uint16_t>(ws, L.yhat)};
  K3_TRY(launch_combine(cp, dev, s));
  K3_TRY(mark(events, n_events, 7, s));
  // latent up
  DenseParams up{};
  up.W0 = w_up; up.R0 = d.hidden; up.K = d.latent; up.act = at<uint16_t>(ws, L.yhat); up.T = T; up.out0 = out;
  K3_TRY(launch_dense<DN_PLAIN>(up, dev, sms, s));
  K3_TRY(mark(events, n_events, 8, s));
  return K3MOE_OK;
}

k3moe_status k3moe_forward(const k3moe_dims* dims, int32_t T, const uint16_t* x, const uint16_t* wr,
                           const float* bias, const uint16_t* w_down, const uint16_t* w_up, const float* norm_w,
                           const k3moe_experts* experts, float* out, int32_t* ids_out, float* w_out, void* ws,
                           size_t ws_bytes, void* stream) {
  return k3moe_forward_profiled(dims, T, x, wr, bias, w_down, w_up, norm_w, experts, out, ids_out, w_out, ws,
                                ws_bytes, stream, nullptr, 0);
}

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
  K3_TRY(launch_permute(perm_params(d, T, 1, nullptr, expert, 8 * nblk, ws, L), dev, s));
  Z16Params zp{z, T, d.latent, at<__half>(ws, L.z16), at<int32_t>(ws, L.zpow)};
  K3_TRY(launch_z16(zp, s));
  const k3moe_experts ex = *experts;
  K3_TRY(launch_mx<MX_GATEUP>(mx_params(d, L, ws, ex, MX_GATEUP, at<__half>(ws, L.z16), at<void>(ws, L.h16)), nblk,
                              dev, sms, s));
  // one expert: sorted slots are the tokens in order, so the down output lands in `out` directly
  K3_TRY(launch_mx<MX_DOWN>(mx_params(d, L, ws, ex, MX_DOWN, at<__half>(ws, L.h16), out), nblk, dev, sms, s));
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
  PermParams pp = perm_params(d, T, d.top_k, ids, 0, 8, ws, L);
  pp.counts = counts;
  pp.offsets = offsets;
  pp.slot_of = slot_of;
  pp.uniq = uniq;
  pp.n_uniq = n_uniq;
  K3_TRY(launch_permute(pp, dev, s));
  return K3MOE_OK;
}

k3moe_status k3moe_device_status(const void* ws, uint32_t* host_out, void* stream) {
  if (!ws || !host_out) return K3MOE_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  K3_TRY(cudaMemcpyAsync(host_out, ws, 4, cudaMemcpyDeviceToHost, s));
  K3_TRY(cudaStreamSynchronize(s));
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
    default: return nullptr;
  }
}

}  // extern "C"

// ---------------------------------------------------------------------------- allocation-free entry
// Scratch for k3moe_forward_noalloc: a fixed array in device memory that every GPU
// loading this library holds until the process exits.
#define K3MOE_NOALLOC_SCRATCH_BYTES (4u << 20)
static __device__ __align__(256) uint8_t g_k3_noalloc_scratch[K3MOE_NOALLOC_SCRATCH_BYTES];

namespace {
// device address of the scratch array, looked up once per device (host code cannot
// use the array's name as a device pointer)
void* g_noalloc_ptr[kMaxDevices];
std::atomic<bool> g_noalloc_ready[kMaxDevices];
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
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return K3MOE_ERR_DEVICE;
  if (!g_noalloc_ready[dev].load(std::memory_order_acquire)) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_k3_noalloc_scratch) != cudaSuccess || !p) return K3MOE_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
    g_noalloc_ready[dev].store(true, std::memory_order_release);
  }
  return k3moe_forward(dims, T, x, wr, bias, w_down, w_up, norm_w, experts, out, ids_out, w_out, g_noalloc_ptr[dev],
                       K3MOE_NOALLOC_SCRATCH_BYTES, stream);
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

int32_t k3moe_abi_version(void) { return 1; }

}  // extern "C"

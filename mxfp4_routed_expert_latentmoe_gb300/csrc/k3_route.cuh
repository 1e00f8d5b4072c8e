// k3_route.cuh -- router top-k, chunk expert-union permutation, activation prep,
// combine + RMSNorm, and the MXFP4 dequant check kernel.
#pragma once

#include "k3_common.cuh"

namespace k3 {

// ============================================================================ top-k
// One warp per token.  Sigmoid scores and biased scores in fp32 from fp32 logits;
// the K + REFINE_EXTRA best candidates by biased score are picked (ties to the lower
// id) by a bitwise search for the threshold key (one warp-wide count per bit), ballot
// compaction and a warp sort; every candidate whose biased score lies within `tau` of a neighbour, in a
// near-tie cluster that reaches the top K + 1, gets its logit recomputed from the bf16
// inputs in double-f32 (about 48 significant bits); candidates are then ranked on the refined values.
// The ranking compares 64-bit integer images of the (exact) double values: the fp64
// unit is used only for the rare refinements.
// Logits are read through L2 (ld.global.cg): the fused one-token front kernel writes them
// in the same launch that routes, so the read-only path must not be used for them.
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
  float top_p;   // cumulative-weight pruning (K3_TOPP): 0 < top_p < 1, else 0 (off)
  int32_t* ids;  // [T, K]
  float* w;      // [T, K]
  int32_t* ids_out;
  float* w_out;
  uint32_t* status;
};

struct TopkScratch {         // per warp
  float cv[TOPK_MAX_P];      // fp32 biased score of candidate
  float cs[TOPK_MAX_P];      // raw score used for the weight
  int ci[TOPK_MAX_P];        // expert id
  int rf[TOPK_MAX_P];        // refine flag
  long long key[TOPK_MAX_P]; // ranking key
};

// exact double bit pattern of a float, by integer operations
K3_DEVI uint64_t f32_as_f64_bits(float f) {
  const uint32_t b = __float_as_uint(f);
  const uint64_t sign = (uint64_t)(b >> 31) << 63;
  uint32_t e = (b >> 23) & 0xFFu, m = b & 0x7FFFFFu;
  if (e == 0 && m == 0) return sign;
  if (e == 0xFFu) return sign | 0x7FF0000000000000ull | ((uint64_t)m << 29);
  int ee = (int)e;
  if (e == 0) {  // subnormal float: normalise
    const int sh = __clz(m) - 8;
    m = (m << sh) & 0x7FFFFFu;
    ee = 1 - sh;
  }
  return sign | ((uint64_t)(ee + 1023 - 127) << 52) | ((uint64_t)m << 29);
}
// order-preserving signed integer image of a (non-NaN) double bit pattern
K3_DEVI long long order_key(uint64_t bits) { return (long long)(bits ^ ((uint64_t)((long long)bits >> 63) >> 1)); }

// sb, sr: per-warp [E] buffers in shared memory
// Selection: every lane keeps the three best (value desc, id asc) of its experts
// e = lane + 32 i in registers; a tournament over the lanes' heads (warp argmax by
// shuffles) picks the next candidate, the winning lane pops its head, and rescans
// its experts only when its three are used up.
// monotone map of a float onto uint32 (larger float -> larger key), and back
K3_DEVI uint32_t f32_order(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
K3_DEVI float f32_from_order(uint32_t k) { return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k); }

// candidate selection with each lane's keys in registers (E <= 32 KPL): every load is
// issued before any arithmetic, and the per-bit counts run on registers
template <int KPL>
K3_DEVI void topk_select(const TopkParams& p, int t, TopkScratch& S, int lane, int P) {
  // keys of the biased scores (NaN ranks last, as -inf; -0 counts as +0); all loads first
  float lg[KPL], bs[KPL];
#pragma unroll
  for (int j = 0; j < KPL; ++j) {
    const int e = lane + 32 * j;
    lg[j] = (e < p.E) ? __ldcg(p.logits + (size_t)t * p.E + e) : 0.f;
    bs[j] = (e < p.E) ? __ldg(p.bias + e) : 0.f;
  }
  uint32_t kr[KPL];
  uint32_t kmax = 0u, kmin = 0xFFFFFFFFu;
#pragma unroll
  for (int j = 0; j < KPL; ++j) {
    // ranking keys only: a few-ulp sigmoid (near ties below tau are re-ranked in fp64)
    const float v = __fdividef(1.0f, 1.0f + __expf(-lg[j])) + bs[j];
    kr[j] = (lane + 32 * j < p.E) ? f32_order((v == v) ? v + 0.0f : -INFINITY) : 0u;  // 0: below every key
    if (lane + 32 * j < p.E) {
      kmax = max(kmax, kr[j]);
      kmin = min(kmin, kr[j]);
    }
  }
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  // the P-th largest key, bit by bit from the most significant bit in which keys differ
  // (one warp-wide count per bit)
  const uint32_t diff = kmax ^ kmin;
  uint32_t thr = diff ? (kmax & ~((2u << (31 - __clz(diff))) - 1u)) : kmax;
  for (int bit = diff ? 31 - __clz(diff) : -1; bit >= 0; --bit) {
    const uint32_t cand = thr | (1u << bit);
    int c[4] = {0, 0, 0, 0};  // independent partial counts (short dependency chains)
#pragma unroll
    for (int j = 0; j < KPL; ++j) c[j & 3] += (kr[j] >= cand) ? 1 : 0;
    if ((int)__reduce_add_sync(0xffffffffu, (uint32_t)(c[0] + c[1] + c[2] + c[3])) >= P) thr = cand;
  }
  // candidates: every key above the threshold, then keys equal to it in id order until P
  // (equal keys rank by lower id), compacted with ballots in id order
  int nsel = 0;
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
    for (int j = 0; j < KPL; ++j) {
      const int e = lane + 32 * j;
      const bool q = (e < p.E) && (pass == 0 ? (kr[j] > thr) : (kr[j] == thr));
      const unsigned m = __ballot_sync(0xffffffffu, q);
      const int pos = nsel + __popc(m & ((1u << lane) - 1u));
      if (q && pos < P) S.key[pos] = (long long)(((uint64_t)kr[j] << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)e));
      nsel = min(P, nsel + __popc(m));
    }
  }
}

// the same selection for E > 1024, keys kept in shared memory (kh: E words)
K3_DEVI void topk_select_smem(const TopkParams& p, int t, uint32_t* kh, TopkScratch& S, int lane, int P) {
  uint32_t kmax = 0u, kmin = 0xFFFFFFFFu;
  for (int e = lane; e < p.E; e += 32) {
    const float v = sigmoidf_(__ldcg(p.logits + (size_t)t * p.E + e)) + __ldg(p.bias + e);
    const uint32_t k = f32_order((v == v) ? v + 0.0f : -INFINITY);
    kh[e] = k;
    kmax = max(kmax, k);
    kmin = min(kmin, k);
  }
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  __syncwarp();
  const uint32_t diff = kmax ^ kmin;
  uint32_t thr = diff ? (kmax & ~((2u << (31 - __clz(diff))) - 1u)) : kmax;
  for (int bit = diff ? 31 - __clz(diff) : -1; bit >= 0; --bit) {
    const uint32_t cand = thr | (1u << bit);
    int c = 0;
    for (int e = lane; e < p.E; e += 32) c += (kh[e] >= cand) ? 1 : 0;
    if ((int)__reduce_add_sync(0xffffffffu, (uint32_t)c) >= P) thr = cand;
  }
  int nsel = 0;
  for (int pass = 0; pass < 2; ++pass) {
    for (int e0 = 0; e0 < p.E && nsel < P; e0 += 32) {
      const int e = e0 + lane;
      const uint32_t k = (e < p.E) ? kh[e] : 0u;
      const bool q = (e < p.E) && (pass == 0 ? (k > thr) : (k == thr));
      const unsigned m = __ballot_sync(0xffffffffu, q);
      const int pos = nsel + __popc(m & ((1u << lane) - 1u));
      if (q && pos < P) S.key[pos] = (long long)(((uint64_t)k << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)e));
      nsel = min(P, nsel + __popc(m));
    }
  }
}

// Logit of token t for expert e, refined: every bf16 x bf16 product is exact in f32; the
// products are summed in double-f32 (error-free two-sum per lane, then a two-sum
// butterfly), about 48 significant bits -- far below the tie window, on the f32 pipes
// (this GPU's fp64 rate is a small fraction of its f32 rate).  Same value on every lane.
K3_DEVI void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bp = s - a;
  e = (a - (s - bp)) + (b - bp);
}
K3_DEVI double refine_logit(const TopkParams& p, int t, int e, int lane) {
  const uint16_t* xr = p.x + (size_t)t * p.H;
  const uint16_t* wrr = p.wr + (size_t)e * p.H;
  float hi = 0.f, lo = 0.f;
  auto acc = [&](float pr) {
    float s, er;
    two_sum(hi, pr, s, er);
    hi = s;
    lo += er;
  };
  if ((p.H & 7) == 0 && ((reinterpret_cast<uintptr_t>(p.x) | reinterpret_cast<uintptr_t>(p.wr)) & 15u) == 0) {
    // 16-byte loads, eight per operand in flight per lane; four independent double-f32
    // accumulators (word j of each load feeds accumulator j), so the two-sum chains run
    // four at a time instead of one long dependent chain
    const uint4* xv = reinterpret_cast<const uint4*>(xr);
    const uint4* wv = reinterpret_cast<const uint4*>(wrr);
    const int nv = p.H >> 3;
    float h4[4] = {0.f, 0.f, 0.f, 0.f}, l4[4] = {0.f, 0.f, 0.f, 0.f};
    auto acc4 = [&](int j, float pr) {
      float s, er;
      two_sum(h4[j], pr, s, er);
      h4[j] = s;
      l4[j] += er;
    };
    for (int v0 = lane; v0 < nv; v0 += 32 * 8) {
      uint4 a[8], b[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int v = v0 + 32 * u;
        a[u] = (v < nv) ? __ldg(xv + v) : make_uint4(0u, 0u, 0u, 0u);
        b[u] = (v < nv) ? __ldg(wv + v) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t aw[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
        const uint32_t bw[4] = {b[u].x, b[u].y, b[u].z, b[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc4(j, __uint_as_float(aw[j] << 16) * __uint_as_float(bw[j] << 16));
          acc4(j, __uint_as_float(aw[j] & 0xFFFF0000u) * __uint_as_float(bw[j] & 0xFFFF0000u));
        }
      }
    }
    // the four accumulators into one (error-free sums of the leading parts)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float s, er;
      two_sum(hi, h4[j], s, er);
      hi = s;
      lo += l4[j] + er;
    }
  } else {
    for (int h = lane; h < p.H; h += 32) acc(bf16_bits_to_f32(__ldg(xr + h)) * bf16_bits_to_f32(__ldg(wrr + h)));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ohi = __shfl_xor_sync(0xffffffffu, hi, off), olo = __shfl_xor_sync(0xffffffffu, lo, off);
    float s, er;
    two_sum(hi, ohi, s, er);
    hi = s;
    lo = lo + olo + er;
  }
  return (double)hi + (double)lo;
}

// Everything after the candidate sort, for P <= 32, with candidate k in lane k's
// registers: near-tie clusters (neighbours by shuffles), fp64 refinement of the flagged
// candidates, re-ranking when any was refined, weights, stores.
// Returns the id of rank `lane` (lanes below K).
K3_DEVI int topk_finish_warp(const TopkParams& p, int t, uint64_t key, int lane, int P, const float* lg_smem = nullptr) {
  const bool in = lane < P;
  int id = in ? (int)(0xFFFFFFFFu - (uint32_t)key) : 0x7fffffff;
  const float cv = f32_from_order((uint32_t)(key >> 32));
  // the weight's score, from the logits copied to shared memory when the caller has them
  float cs = in ? sigmoidf_(lg_smem ? lg_smem[id] : __ldcg(p.logits + (size_t)t * p.E + id)) : 0.f;
  const float cv_prev = __shfl_up_sync(0xffffffffu, cv, 1);
  const float cv_next = __shfl_down_sync(0xffffffffu, cv, 1);
  const bool linked_prev = in && lane > 0 && (cv_prev - cv) < p.tau;
  const bool linked_next = in && lane + 1 < P && (cv - cv_next) < p.tau;
  // a cluster starts at an unlinked position; it is refined when it starts at or before K
  const unsigned unl = __ballot_sync(0xffffffffu, in && !linked_prev);
  const unsigned le = unl & ((2u << lane) - 1u);
  const int start = le ? 31 - __clz(le) : 0;
  const unsigned rmask = __ballot_sync(0xffffffffu, in && (linked_prev || linked_next) && start <= p.K);
  if (lane == 0 && P < p.E && ((rmask >> (P - 1)) & 1u)) flag_status(p.status, K3MOE_DEV_TIE_WINDOW);
  if (rmask) {
    long long rkey = in ? order_key(f32_as_f64_bits(cv)) : LLONG_MIN;
    for (unsigned m = rmask; m; m &= m - 1u) {
      const int k = __ffs(m) - 1;
      const int e = __shfl_sync(0xffffffffu, id, k);
      const double acc = refine_logit(p, t, e, lane);
      if (lane == k) {
        const double s = 1.0 / (1.0 + exp(-acc));
        cs = (float)s;
        rkey = order_key((uint64_t)__double_as_longlong(s + (double)p.bias[e]));
      }
    }
    // re-rank by (refined key desc, id asc): bitonic network carrying the score
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const long long ok = __shfl_xor_sync(0xffffffffu, rkey, stride);
        const int oi = __shfl_xor_sync(0xffffffffu, id, stride);
        const float os = __shfl_xor_sync(0xffffffffu, cs, stride);
        const bool o_better = ok > rkey || (ok == rkey && oi < id);
        const bool desc = ((lane & size) == 0);
        const bool lower = ((lane & stride) == 0);
        if ((lower == desc) ? o_better : !o_better) {
          rkey = ok;
          id = oi;
          cs = os;
        }
      }
    }
  }
  // weights of the first K: a fixed butterfly sum (the same on every lane), then w = s / sum
  float sum = (lane < p.K) ? cs : 0.f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  float wk = (lane < p.K) ? cs / sum : 0.f;
  if (p.top_p > 0.f) {
    // K3_TOPP: the K ordered by weight (equal weights keep their rank order), kept while the
    // weight before them is below top_p, renormalised over the kept raw scores; the others
    // become id -1, weight 0.  Lane j ends with the j-th largest weight.
    uint64_t key = (lane < p.K) ? (((uint64_t)f32_order(wk) << 32) | (uint64_t)(31 - lane)) : 0ull;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const uint64_t ok = __shfl_xor_sync(0xffffffffu, key, stride);
        const int oi = __shfl_xor_sync(0xffffffffu, id, stride);
        const float os = __shfl_xor_sync(0xffffffffu, cs, stride);
        const float ow = __shfl_xor_sync(0xffffffffu, wk, stride);
        const bool desc = ((lane & size) == 0), lower = ((lane & stride) == 0);
        if ((lower == desc) ? (ok > key) : (ok < key)) {
          key = ok;
          id = oi;
          cs = os;
          wk = ow;
        }
      }
    float incl = (lane < p.K) ? wk : 0.f;  // inclusive prefix of the ordered weights
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    const bool keep = lane < p.K && (lane == 0 || (incl - wk) < p.top_p);
    float ks = keep ? cs : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ks += __shfl_xor_sync(0xffffffffu, ks, off);
    wk = keep ? cs / ks : 0.f;
    if (!keep) id = -1;
  }
  if (lane < p.K) {
    p.ids[(size_t)t * p.K + lane] = id;
    p.w[(size_t)t * p.K + lane] = wk;
    if (p.ids_out) p.ids_out[(size_t)t * p.K + lane] = id;
    if (p.w_out) p.w_out[(size_t)t * p.K + lane] = wk;
  }
  __syncwarp();
  return id;
}

K3_DEVI void topk_token(const TopkParams& p, int t, float* sb, float* sr, TopkScratch& S, int lane) {
  (void)sr;
  const int P = min(p.E, p.K + REFINE_EXTRA);
  if (p.E <= 1024) topk_select<32>(p, t, S, lane, P);
  else topk_select_smem(p, t, reinterpret_cast<uint32_t*>(sb), S, lane, P);
  __syncwarp();
  // order the P candidates by (score desc, id asc) = key desc: bitonic sort in the warp
  // for P <= 32, else a selection sort by lane 0 (top-k above 24 only)
  if (P <= 32) {
    uint64_t v = (lane < P) ? (uint64_t)S.key[lane] : 0ull;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const uint64_t o = __shfl_xor_sync(0xffffffffu, v, stride);
        const bool desc = ((lane & size) == 0);
        const bool lower = ((lane & stride) == 0);
        const bool take = (lower == desc) ? (o > v) : (o < v);
        if (take) v = o;
      }
    }
    topk_finish_warp(p, t, v, lane, P);
    return;
  } else if (lane == 0) {
    for (int a2 = 0; a2 < P; ++a2) {
      int b2 = a2;
      for (int c2 = a2 + 1; c2 < P; ++c2)
        if ((uint64_t)S.key[c2] > (uint64_t)S.key[b2]) b2 = c2;
      const long long tk = S.key[a2]; S.key[a2] = S.key[b2]; S.key[b2] = tk;
    }
  }
  __syncwarp();
  for (int k = lane; k < P; k += 32) {
    const uint64_t key = (uint64_t)S.key[k];
    const int id = (int)(0xFFFFFFFFu - (uint32_t)key);
    S.cv[k] = f32_from_order((uint32_t)(key >> 32));
    S.ci[k] = id;
    S.cs[k] = sigmoidf_(__ldcg(p.logits + (size_t)t * p.E + id));
  }
  __syncwarp();
  // near-tie clusters: consecutive candidates closer than tau are linked; a cluster
  // is refined when it starts at or before position K (it can change the top K or
  // their order)
  __syncwarp();
  {
    // lane k handles candidate k (P <= 72: up to three rounds); the start of k's cluster
    // is the last unlinked position at or before k, found with a warp ballot scan
    int base_start = 0;  // cluster start carried from the previous round
    for (int k0 = 0; k0 < P; k0 += 32) {
      const int k = k0 + lane;
      const bool in = k < P;
      const bool linked_prev = in && k > 0 && (S.cv[k - 1] - S.cv[k]) < p.tau;
      const bool linked_next = in && k + 1 < P && (S.cv[k] - S.cv[k + 1]) < p.tau;
      const unsigned unl = __ballot_sync(0xffffffffu, in && !linked_prev);  // cluster starts in this round
      const unsigned le = unl & ((2u << lane) - 1u);
      const int start = le ? k0 + 31 - __clz(le) : base_start;
      if (in) {
        S.rf[k] = (linked_prev || linked_next) && start <= p.K;
        S.key[k] = order_key(f32_as_f64_bits(S.cv[k]));
      }
      base_start = __shfl_sync(0xffffffffu, start, 31);
    }
  }
  __syncwarp();
  if (lane == 0 && P < p.E && S.rf[P - 1]) flag_status(p.status, K3MOE_DEV_TIE_WINDOW);
  for (int k = 0; k < P; ++k) {
    if (!S.rf[k]) continue;  // warp-uniform
    const int e = S.ci[k];
    const double acc = refine_logit(p, t, e, lane);
    if (lane == 0) {
      const double s = 1.0 / (1.0 + exp(-acc));
      S.cs[k] = (float)s;
      S.key[k] = order_key((uint64_t)__double_as_longlong(s + (double)p.bias[e]));
    }
    __syncwarp();
  }
  // without refinements the tournament order is already the final order
  bool any_rf = false;
  for (int k = 0; k < P; ++k) any_rf |= (S.rf[k] != 0);
  if (lane == 0 && any_rf) {
    for (int a = 0; a < p.K; ++a) {  // selection sort of the first K by (key desc, id asc)
      int b = a;
      for (int c = a + 1; c < P; ++c)
        if (S.key[c] > S.key[b] || (S.key[c] == S.key[b] && S.ci[c] < S.ci[b])) b = c;
      if (b != a) {
        const long long tk = S.key[a]; S.key[a] = S.key[b]; S.key[b] = tk;
        const float ts = S.cs[a]; S.cs[a] = S.cs[b]; S.cs[b] = ts;
        const int ti = S.ci[a]; S.ci[a] = S.ci[b]; S.ci[b] = ti;
      }
    }
  }
  __syncwarp();
  {
    // the sum runs in k order (as a serial loop would), then lane k writes entry k
    float sum = 0.f;
    for (int k = 0; k < p.K; ++k) sum += S.cs[k];
    for (int k = lane; k < p.K; k += 32) {
      const int id = S.ci[k];
      const float wk = S.cs[k] / sum;
      p.ids[(size_t)t * p.K + k] = id;
      p.w[(size_t)t * p.K + k] = wk;
      if (p.ids_out) p.ids_out[(size_t)t * p.K + k] = id;
      if (p.w_out) p.w_out[(size_t)t * p.K + k] = wk;
    }
  }
  __syncwarp();
}

constexpr int TOPK_WARPS = 4;

__global__ void __launch_bounds__(TOPK_WARPS * 32) k3_topk_kernel(TopkParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ TopkScratch S[TOPK_WARPS];
  grid_dep_wait();
  grid_dep_launch();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = blockIdx.x * TOPK_WARPS + warp;
  if (t >= p.T) return;
  float* sb = reinterpret_cast<float*>(smem) + warp * (2 * p.E);
  topk_token(p, t, sb, sb + p.E, S[warp], lane);
}

// ============================================================================ permutation
// Single CTA stable counting sort of the T*K routed slots by expert (the chunk's
// expert union with per-expert position lists).  Each warp owns a contiguous range
// of slots and a private histogram; positions are handed out in slot order inside
// a warp (warp-synchronous ranking with __match_any_sync) and in warp order across
// warps, so the result is the stable sort by (expert, t*K + k).  The expert kernels'
// token batches (up to NB tokens of one expert each, with the expert's weight
// pointers) are written last.
constexpr int PERM_WARPS = 16;

struct PermParams {
  const int32_t* ids;  // [T*K], or null: every slot routes to fixed_expert
  int fixed_expert;
  int T, K, E, NB;
  k3moe_experts ex;    // pointer tables (device arrays of E pointers)
  int32_t* counts;     // [E]
  int32_t* offsets;    // [E+1]
  int32_t* slot_of;    // [T*K] sorted slot -> flat index t*K+k
  int32_t* slot_tok;   // [T*K] sorted slot -> token
  int32_t* inv;        // [T*K] flat index -> sorted slot
  int32_t* uniq;       // [E]
  int32_t* n_uniq;     // [1]
  int32_t* nb_prefix;  // [E+1] over unique experts: prefix of ceil(count/NB)
  MxBatch* batches;    // [nb_prefix[n_uniq]] token batches
  int32_t* n_batches;  // [1]
  uint32_t* status;
  int32_t* cta_cnt;    // multi-CTA path: [ceil(T*K / PERM_SPAN)][E] per-CTA expert counts
  int32_t* cta_base;   // ... and each CTA's first sorted position per expert
};

// exclusive scan of 4 values per thread over a PERM_WARPS-warp block (values in order
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

// hist: PERM_WARPS * E ints of shared memory; wsum: PERM_WARPS + 1 ints
// Expert of routed slot i: -1 for a slot pruned by top-p (id -1: no position, inv -1);
// an id outside [0, E) is reported (K3MOE_DEV_BAD_ID) and clamped.
K3_DEVI int slot_expert(const PermParams& p, int i, bool flag_bad) {
  int e = p.ids ? p.ids[i] : p.fixed_expert;
  if (e == -1) return -1;
  if (e < 0 || e >= p.E) {
    if (flag_bad) flag_status(p.status, K3MOE_DEV_BAD_ID);
    e = min(max(e, 0), p.E - 1);
  }
  return e;
}

K3_DEVI void permute_block(const PermParams& p, int32_t* hist, int* wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = p.T * p.K;
  const int chunk = (n + PERM_WARPS - 1) / PERM_WARPS;
  const int b0 = min(n, warp * chunk), b1 = min(n, b0 + chunk);

  for (int i = threadIdx.x; i < PERM_WARPS * p.E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (int i = b0 + lane; i < b1; i += 32) {
    const int e = slot_expert(p, i, true);
    if (e >= 0) atomicAdd(&hist[warp * p.E + e], 1);
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
    const int e = (i < b1) ? slot_expert(p, i, false) : -2;
    const bool valid = e >= 0;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int leader = __ffs(peers) - 1;
    if (valid) {
      const int pos = hist[warp * p.E + e] + rank;
      p.slot_of[pos] = i;
      p.slot_tok[pos] = i / p.K;
      p.inv[i] = pos;
    } else if (e == -1) {
      p.inv[i] = -1;  // pruned: no position
    }
    __syncwarp();
    if (valid && lane == leader) hist[warp * p.E + e] += __popc(peers);
    __syncwarp();
  }
  // unique experts (ascending) and their token-batch prefix
  int flag[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) flag[q] = cnt[q] > 0 ? 1 : 0;
  const int nu = block_scan4(flag, wsum);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e = threadIdx.x * 4 + q;
    if (e < p.E && cnt[q] > 0) p.uniq[flag[q]] = e;
  }
  if (threadIdx.x == 0) *p.n_uniq = nu;
  __syncthreads();
  int nbv[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int u = threadIdx.x * 4 + q;
    nbv[q] = (u < nu) ? (p.counts[p.uniq[u]] + p.NB - 1) / p.NB : 0;
  }
  int nbx[4] = {nbv[0], nbv[1], nbv[2], nbv[3]};
  const int nbt = block_scan4(nbx, wsum);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int u = threadIdx.x * 4 + q;
    if (u < nu) {
      p.nb_prefix[u] = nbx[q];
      if (!p.ex.gate_q) continue;  // permutation only: no expert tables, no batch records
      const int e = p.uniq[u];
      const int cntu = p.counts[e], offu = p.offsets[e];
      const uint8_t* wp[6] = {p.ex.gate_q[e], p.ex.gate_s[e], p.ex.up_q[e], p.ex.up_s[e], p.ex.down_q[e],
                              p.ex.down_s[e]};
      for (int b = 0; b < nbv[q]; ++b) {
        MxBatch* r = p.batches + nbx[q] + b;
#pragma unroll
        for (int k = 0; k < 6; ++k) r->w[k] = wp[k];
        const int s0 = offu + b * p.NB;
        const int nn = min(p.NB, cntu - b * p.NB);
        r->slot0 = s0;
        r->n = nn;
        for (int j = 0; j < MX_MAX_NB; ++j) r->tok[j] = (j < nn) ? p.slot_tok[s0 + j] : 0;
        r->pad[0] = r->pad[1] = 0;
      }
    }
  }
  if (threadIdx.x == 0) {
    p.nb_prefix[nu] = nbt;
    *p.n_batches = nbt;
  }
}

// The same permutation for at most 32 routed slots, by one warp: a bitonic sort of
// (expert, flat index) pairs across the lanes gives the stable order; runs of equal
// experts are the unique experts.  counts/offsets are written for the routed experts
// only (nothing downstream reads the others).
// lane_id >= 0: the caller's id of slot `lane` (instead of reading p.ids)
K3_DEVI void permute_warp(const PermParams& p, int lane, const uint8_t* const* tab_smem = nullptr, bool have_id = false,
                          int lane_id = 0) {
  const int n_all = p.T * p.K;
  int e = 0x7fffffff, f = 0x7fffffff;
  if (lane < n_all) {
    if (have_id) {
      e = lane_id;
      if (e != -1 && (e < 0 || e >= p.E)) {
        flag_status(p.status, K3MOE_DEV_BAD_ID);
        e = min(max(e, 0), p.E - 1);
      }
    } else {
      e = slot_expert(p, lane, true);
    }
    if (e == -1) {  // pruned by top-p: no position; sorts after every placed slot
      p.inv[lane] = -1;
      e = 0x7fffffff;
    } else {
      f = lane;
    }
  }
  const int n = __popc(__ballot_sync(0xffffffffu, e != 0x7fffffff));  // placed slots
  // bitonic sort ascending by (e, f)
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int oe = __shfl_xor_sync(0xffffffffu, e, stride);
      const int of = __shfl_xor_sync(0xffffffffu, f, stride);
      const bool up = ((lane & size) == 0);
      const bool lower = ((lane & stride) == 0);
      const bool other_less = (oe < e) || (oe == e && of < f);
      const bool take = (lower == up) ? other_less : !other_less;
      if (take) {
        e = oe;
        f = of;
      }
    }
  }
  const bool valid = lane < n;
  const int pe = __shfl_up_sync(0xffffffffu, e, 1);
  const bool start = valid && (lane == 0 || pe != e);
  const unsigned starts = __ballot_sync(0xffffffffu, start);
  const int u = __popc(starts & ((1u << lane) - 1u)) + (start ? 0 : -1);  // run index of this lane
  const int nu = __popc(starts);
  // run start and length of this lane's run
  const unsigned le = starts & ((2u << lane) - 1u);
  const int run0 = valid ? 31 - __clz(le) : 0;
  const unsigned after = starts & ~((2u << lane) - 1u);
  const int run1 = after ? __ffs(after) - 1 : n;
  if (valid) {
    p.slot_of[lane] = f;
    p.slot_tok[lane] = f / p.K;
    p.inv[f] = lane;
  }
  __syncwarp();  // slot_tok is read back below by other lanes
  // per run: batches of NB tokens
  const int cnt = run1 - run0;
  const int nbr = start ? (cnt + p.NB - 1) / p.NB : 0;
  int pre = nbr;  // inclusive scan over lanes
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, pre, off);
    if (lane >= off) pre += o;
  }
  const int total = __shfl_sync(0xffffffffu, pre, 31);
  // tokens of the first batch of this lane's run, taken from the sorted lanes by shuffles
  int tk0[MX_MAX_NB];
  const int tokv = valid ? f / p.K : 0;
#pragma unroll
  for (int j = 0; j < MX_MAX_NB; ++j) tk0[j] = __shfl_sync(0xffffffffu, tokv, min(run0 + j, 31));
  if (start) {
    p.counts[e] = cnt;
    p.offsets[e] = run0;
    p.uniq[u] = e;
    p.nb_prefix[u] = pre - nbr;
    if (p.ex.gate_q) {
      const uint8_t* wp[6];
      if (tab_smem) {
#pragma unroll
        for (int k = 0; k < 6; ++k) wp[k] = tab_smem[k * p.E + e];
      } else {
        wp[0] = p.ex.gate_q[e]; wp[1] = p.ex.gate_s[e]; wp[2] = p.ex.up_q[e];
        wp[3] = p.ex.up_s[e]; wp[4] = p.ex.down_q[e]; wp[5] = p.ex.down_s[e];
      }
      for (int b = 0; b < nbr; ++b) {
        MxBatch* r = p.batches + (pre - nbr) + b;
#pragma unroll
        for (int k = 0; k < 6; ++k) r->w[k] = wp[k];
        const int s0 = run0 + b * p.NB;
        const int nn = min(p.NB, cnt - b * p.NB);
        r->slot0 = s0;
        r->n = nn;
        if (b == 0) {
#pragma unroll
          for (int j = 0; j < MX_MAX_NB; ++j) r->tok[j] = (j < nn) ? tk0[j] : 0;
        } else {
          for (int j = 0; j < MX_MAX_NB; ++j) r->tok[j] = (j < nn) ? p.slot_tok[s0 + j] : 0;
        }
        r->pad[0] = r->pad[1] = 0;
      }
    }
  }
  if (lane == 0) {
    *p.n_uniq = nu;
    p.nb_prefix[nu] = total;
    *p.n_batches = total;
    p.offsets[p.E] = n;
  }
}

__global__ void __launch_bounds__(PERM_WARPS * 32) k3_permute_kernel(PermParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int wsum[PERM_WARPS + 1];
  grid_dep_wait();
  grid_dep_launch();
  permute_block(p, reinterpret_cast<int32_t*>(smem), wsum);
}

// ============================================================================ multi-CTA permutation
// The same stable counting sort for many slots, across CTAs of PERM_SPAN slots each
// (PERM_WARPS warps x 128 slots, in slot order):
//   1. k3_perm_hist_kernel     per-CTA expert counts            -> cta_cnt[c][e]
//   2. k3_perm_scan_kernel     one CTA: per expert, running sums over CTAs -> cta_base,
//                              counts; expert offsets; unique experts; batch prefix
//   3. k3_perm_scatter_kernel  per CTA: per-warp counts again, warp-major running
//                              offsets from cta_base, stable placement as permute_block
//   4. k3_perm_records_kernel  one thread per token-batch record
// Equal to permute_block: within an expert, slots keep increasing flat index.
constexpr int PERM_SPAN = PERM_WARPS * 128;

// per-warp expert histogram of this CTA's slots into hist[PERM_WARPS][E]; returns the
// warp's slot range [b0, b1)
K3_DEVI void perm_warp_hist(const PermParams& p, int32_t* hist, int& b0, int& b1, bool flag_bad) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = p.T * p.K;
  b0 = min(n, (int)blockIdx.x * PERM_SPAN + warp * 128);
  b1 = min(n, b0 + 128);
  for (int i = threadIdx.x; i < PERM_WARPS * p.E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (int i = b0 + lane; i < b1; i += 32) {
    const int e = slot_expert(p, i, flag_bad);
    if (e >= 0) atomicAdd(&hist[warp * p.E + e], 1);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(PERM_WARPS * 32) k3_perm_hist_kernel(PermParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  int32_t* hist = reinterpret_cast<int32_t*>(smem);
  grid_dep_wait();
  grid_dep_launch();
  int b0, b1;
  perm_warp_hist(p, hist, b0, b1, true);
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
    int c = 0;
    for (int w = 0; w < PERM_WARPS; ++w) c += hist[w * p.E + e];
    p.cta_cnt[(size_t)blockIdx.x * p.E + e] = c;
  }
}

__global__ void __launch_bounds__(PERM_WARPS * 32) k3_perm_scan_kernel(PermParams p, int nct) {
  __shared__ int wsum[PERM_WARPS + 1];
  grid_dep_wait();
  grid_dep_launch();
  int cnt[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e = threadIdx.x * 4 + q;
    int run = 0;
    if (e < p.E) {
      for (int c = 0; c < nct; ++c) {
        const int v = p.cta_cnt[(size_t)c * p.E + e];
        p.cta_base[(size_t)c * p.E + e] = run;
        run += v;
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
      for (int c = 0; c < nct; ++c) p.cta_base[(size_t)c * p.E + e] += off[q];
    }
  }
  if (threadIdx.x == 0) p.offsets[p.E] = tot;
  // unique experts (ascending) and their token-batch prefix
  int flag[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) flag[q] = cnt[q] > 0 ? 1 : 0;
  const int nu = block_scan4(flag, wsum);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e = threadIdx.x * 4 + q;
    if (e < p.E && cnt[q] > 0) p.uniq[flag[q]] = e;
  }
  if (threadIdx.x == 0) *p.n_uniq = nu;
  __syncthreads();
  int nbv[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int u = threadIdx.x * 4 + q;
    nbv[q] = (u < nu) ? (p.counts[p.uniq[u]] + p.NB - 1) / p.NB : 0;
  }
  int nbx[4] = {nbv[0], nbv[1], nbv[2], nbv[3]};
  const int nbt = block_scan4(nbx, wsum);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int u = threadIdx.x * 4 + q;
    if (u < nu) p.nb_prefix[u] = nbx[q];
  }
  if (threadIdx.x == 0) {
    p.nb_prefix[nu] = nbt;
    *p.n_batches = nbt;
  }
}

__global__ void __launch_bounds__(PERM_WARPS * 32) k3_perm_scatter_kernel(PermParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  int32_t* hist = reinterpret_cast<int32_t*>(smem);
  grid_dep_wait();
  grid_dep_launch();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int b0, b1;
  perm_warp_hist(p, hist, b0, b1, false);
  // warp-major running offsets, starting at this CTA's first position per expert
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
    int run = p.cta_base[(size_t)blockIdx.x * p.E + e];
    for (int w = 0; w < PERM_WARPS; ++w) {
      const int c = hist[w * p.E + e];
      hist[w * p.E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int base = b0; base < b1; base += 32) {
    const int i = base + lane;
    const int e = (i < b1) ? slot_expert(p, i, false) : -2;
    const bool valid = e >= 0;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int leader = __ffs(peers) - 1;
    if (valid) {
      const int pos = hist[warp * p.E + e] + rank;
      p.slot_of[pos] = i;
      p.slot_tok[pos] = i / p.K;
      p.inv[i] = pos;
    } else if (e == -1) {
      p.inv[i] = -1;  // pruned: no position
    }
    __syncwarp();
    if (valid && lane == leader) hist[warp * p.E + e] += __popc(peers);
    __syncwarp();
  }
}

// one thread per token-batch record: the unique expert is found by binary search of the
// batch prefix
__global__ void __launch_bounds__(256) k3_perm_records_kernel(PermParams p) {
  grid_dep_wait();
  grid_dep_launch();
  const int nu = *p.n_uniq, nbt = *p.n_batches;
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < nbt; r += gridDim.x * blockDim.x) {
    int lo = 0, hi = nu - 1;  // largest u with nb_prefix[u] <= r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.nb_prefix[mid] <= r) lo = mid;
      else hi = mid - 1;
    }
    const int u = lo, e = p.uniq[u], b = r - p.nb_prefix[u];
    const int cntu = p.counts[e], offu = p.offsets[e];
    MxBatch* rec = p.batches + r;
    rec->w[0] = p.ex.gate_q[e];
    rec->w[1] = p.ex.gate_s[e];
    rec->w[2] = p.ex.up_q[e];
    rec->w[3] = p.ex.up_s[e];
    rec->w[4] = p.ex.down_q[e];
    rec->w[5] = p.ex.down_s[e];
    const int s0 = offu + b * p.NB, nn = min(p.NB, cntu - b * p.NB);
    rec->slot0 = s0;
    rec->n = nn;
    for (int j = 0; j < MX_MAX_NB; ++j) rec->tok[j] = (j < nn) ? p.slot_tok[s0 + j] : 0;
    rec->pad[0] = rec->pad[1] = 0;
  }
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

// one warp converts one token (L a multiple of 64: 16-byte vectors); up to 16 vectors
// per lane (L <= 4096) the row is read once into registers, all loads in flight together
K3_DEVI void z16_token(const Z16Params& p, int t, int lane) {
  const uint4* zr = reinterpret_cast<const uint4*>(p.z + (size_t)t * p.L);
  uint4* o = reinterpret_cast<uint4*>(p.z16 + (size_t)t * p.L);
  const int nv = p.L / 8;
  auto exp_of = [&](uint32_t mx) {
    int pw = 0;
    if (mx != 0u && mx < 0x7F80u) {
      const int ex = (int)(mx >> 7);               // biased exponent field of the largest |z|
      const int E2 = (ex == 0) ? -127 : ex - 127;  // floor(log2) (subnormal: below -126)
      pw = 14 - E2;
    }
    return pw;
  };
  auto conv = [&](const uint4& v, int pw) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t r[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 h = __floats2half2_rn(scalbnf(bf16_bits_to_f32(w[k] & 0xFFFFu), pw),
                                          scalbnf(bf16_bits_to_f32(w[k] >> 16), pw));
      r[k] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
  };
  auto vmax = [](uint32_t mx, const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) mx = max(mx, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
    return mx;
  };
  if (nv <= 16 * 32) {
    uint4 v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = (lane + 32 * j < nv) ? __ldcg(zr + lane + 32 * j) : make_uint4(0u, 0u, 0u, 0u);
    uint32_t mx = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) mx = vmax(mx, v[j]);
    mx = __reduce_max_sync(0xffffffffu, mx);
    const int pw = exp_of(mx);
    if (lane == 0) p.pow2[t] = pw;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (lane + 32 * j < nv) o[lane + 32 * j] = conv(v[j], pw);
    return;
  }
  uint32_t mx = 0;
  for (int c = lane; c < nv; c += 32) mx = vmax(mx, __ldcg(zr + c));
  mx = __reduce_max_sync(0xffffffffu, mx);
  const int pw = exp_of(mx);
  if (lane == 0) p.pow2[t] = pw;
  for (int c = lane; c < nv; c += 32) o[c] = conv(__ldcg(zr + c), pw);
}

__global__ void k3_z16_kernel(Z16Params p) {
  grid_dep_wait();
  grid_dep_launch();
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t < p.T) z16_token(p, t, threadIdx.x & 31);
}

// ============================================================================ slot-order activation rows
// act[s] = z[slot_tok[s]] for every routed slot: the B operand rows of the tensor-core
// expert GEMM (one expert's tokens contiguous), bf16, each group of 8 elements stored in
// the interleaved order 0, 4, 1, 5, 2, 6, 3, 7 that the GEMM's weight decode produces.
__global__ void k3_gather_rows_kernel(const uint16_t* z, const int32_t* slot_tok, const int32_t* n_placed, int slots,
                                      int L, uint16_t* out) {
  grid_dep_wait();
  grid_dep_launch();
  const int per = L / 8;  // 16-byte chunks (8 elements) per row
  const int ns = min(slots, *n_placed);  // slots pruned by top-p have no position
  const size_t total = (size_t)ns * per;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int s = (int)(i / per), c = (int)(i - (size_t)s * per);
    const int t = __ldg(slot_tok + s);
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(z + (size_t)t * L) + c);  // [e0 e1] [e2 e3] [e4 e5] [e6 e7]
    reinterpret_cast<uint4*>(out + (size_t)s * L)[c] =
        make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632), __byte_perm(v.y, v.w, 0x5410),
                   __byte_perm(v.y, v.w, 0x7632));
  }
}

// One token's routing over a whole CTA (E <= TOPK_BLOCK_N, P <= 32), for the decode step.
// Every thread forms the 32-bit ranking keys of its experts (biased scores' order images),
// keeps the logits in shared memory for the weights, and copies the expert pointer tables
// to shared memory for the batch records -- one round trip to memory for all three.  The
// P-th largest key is then found by a radix select (four passes of an 8-bit digit: a
// shared histogram of the keys still matching the prefix found so far, scanned from the top
// by one warp); the keys above it and the lowest ids among the keys equal to it make the
// P candidates, which one warp sorts (key descending, id ascending) and finishes as
// topk_finish_warp does.  Short phases with all threads instead of one warp's long chain.
constexpr int TOPK_BLOCK_N = 1024;
struct RouteSmem {
  static constexpr int HIST = 0;                   // 2 x 256 uint32 digit counts
  static constexpr int CTRL = HIST + 512 * 4;      // prefix, mask, need, n_above, n_tie
  static constexpr int LG = CTRL + 64;             // E floats: logits
  static constexpr int CAND = LG + TOPK_BLOCK_N * 4;     // 64 candidate keys
  static constexpr int TIE = CAND + 64 * 8;        // E ints: ids of keys equal to the threshold
  static constexpr int TAB = TIE + TOPK_BLOCK_N * 4;     // 6 x E expert tensor pointers
  __host__ __device__ static constexpr int bytes(int E) { return TAB + 6 * E * 8; }
};

K3_DEVI void route_one_token_block(const TopkParams& p, const PermParams& pp, uint8_t* sm, int lane, int warp) {
  uint32_t* hist0 = reinterpret_cast<uint32_t*>(sm + RouteSmem::HIST);  // two buffers, alternating by pass
  int* ctrl = reinterpret_cast<int*>(sm + RouteSmem::CTRL);
  float* lgs = reinterpret_cast<float*>(sm + RouteSmem::LG);
  uint64_t* cand = reinterpret_cast<uint64_t*>(sm + RouteSmem::CAND);
  int* tie = reinterpret_cast<int*>(sm + RouteSmem::TIE);
  const uint8_t** tab = reinterpret_cast<const uint8_t**>(sm + RouteSmem::TAB);
  const int E = p.E, P = min(E, p.K + REFINE_EXTRA);
  const int nt = blockDim.x;
  // keys, logits and expert tables (all loads issued before their uses)
  uint32_t kk[TOPK_BLOCK_N / (PERM_WARPS * 32)];
#pragma unroll
  for (int r = 0; r < TOPK_BLOCK_N / (PERM_WARPS * 32); ++r) {
    const int e = threadIdx.x + r * nt;
    kk[r] = 0u;  // below every real key
    if (e < E) {
      const float l = __ldcg(p.logits + e);
      lgs[e] = l;
      const float v = __fdividef(1.0f, 1.0f + __expf(-l)) + __ldg(p.bias + e);
      kk[r] = f32_order((v == v) ? v + 0.0f : -INFINITY);
    }
  }
  if (pp.ex.gate_q) {
    const uint8_t* const* src[6] = {pp.ex.gate_q, pp.ex.gate_s, pp.ex.up_q, pp.ex.up_s, pp.ex.down_q, pp.ex.down_s};
    constexpr int R = TOPK_BLOCK_N / (PERM_WARPS * 32);
    const uint8_t* v[6][R];
#pragma unroll
    for (int k = 0; k < 6; ++k)
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int e = threadIdx.x + r * nt;
        v[k][r] = (e < E) ? reinterpret_cast<const uint8_t*>(__ldg(reinterpret_cast<const unsigned long long*>(src[k]) + e))
                          : nullptr;
      }
#pragma unroll
    for (int k = 0; k < 6; ++k)
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int e = threadIdx.x + r * nt;
        if (e < E) tab[k * E + e] = v[k][r];
      }
  }
  if (threadIdx.x < 512) hist0[threadIdx.x] = 0u;
  if (threadIdx.x == 0) {
    ctrl[0] = 0;  // prefix of the P-th largest key found so far
    ctrl[1] = 0;  // mask of the digits found
    ctrl[2] = P;  // rank of the wanted key among the keys matching the prefix
    ctrl[3] = 0;
    ctrl[4] = 0;
  }
  __syncthreads();
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    uint32_t* hist = hist0 + ((shift >> 3) & 1) * 256;
    const uint32_t prefix = (uint32_t)ctrl[0], mask = (uint32_t)ctrl[1];
#pragma unroll
    for (int r = 0; r < TOPK_BLOCK_N / (PERM_WARPS * 32); ++r) {
      const int e = threadIdx.x + r * nt;
      if (e < E && (kk[r] & mask) == prefix) atomicAdd(hist + ((kk[r] >> shift) & 255u), 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds the digits 255 - 8l down to 248 - 8l; counts scanned from the top
      uint32_t c[8], sum = 0u;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * lane - j];
        sum += c[j];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      const uint32_t excl = incl - sum, need = (uint32_t)ctrl[2];
      const unsigned own = __ballot_sync(0xffffffffu, excl < need && need <= incl);
      if (lane == __ffs(own) - 1) {
        uint32_t acc = excl;
#pragma unroll 1
        for (int j = 0; j < 8; ++j) {
          if (acc + c[j] >= need) {
            ctrl[0] = (int)(prefix | ((uint32_t)(255 - 8 * lane - j) << shift));
            ctrl[1] = (int)(mask | (255u << shift));
            ctrl[2] = (int)(need - acc);
            break;
          }
          acc += c[j];
        }
      }
    }
    // the other buffer (read two passes ago, before the barrier above) is cleared for the next pass
    if (threadIdx.x < 256) hist0[(((shift >> 3) & 1) ^ 1) * 256 + threadIdx.x] = 0u;
    __syncthreads();
  }
  // the P-th largest key is thr; `need` keys equal to it complete the P
  const uint32_t thr = (uint32_t)ctrl[0];
  const int need = ctrl[2];
#pragma unroll
  for (int r = 0; r < TOPK_BLOCK_N / (PERM_WARPS * 32); ++r) {
    const int e = threadIdx.x + r * nt;
    if (e < E && kk[r] > thr) cand[atomicAdd(ctrl + 3, 1)] = ((uint64_t)kk[r] << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)e);
    else if (e < E && kk[r] == thr) tie[atomicAdd(ctrl + 4, 1)] = e;
  }
  __syncthreads();
  if (warp == 0) {
    const int n_above = ctrl[3], n_tie = ctrl[4];
    // the `need` lowest ids among the keys equal to the threshold
    if (n_tie <= 32) {
      int id = (lane < n_tie) ? tie[lane] : 0x7fffffff;
#pragma unroll
      for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          const int o = __shfl_xor_sync(0xffffffffu, id, stride);
          const bool up = (lane & size) == 0, lower = (lane & stride) == 0;
          if ((lower == up) ? (o < id) : (o > id)) id = o;
        }
      if (lane < need) cand[n_above + lane] = ((uint64_t)thr << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)id);
    } else if (lane == 0) {  // many exactly equal scores: selection by smallest id
      int last = -1;
      for (int q = 0; q < need; ++q) {
        int best = 0x7fffffff;
        for (int i = 0; i < n_tie; ++i)
          if (tie[i] > last && tie[i] < best) best = tie[i];
        cand[n_above + q] = ((uint64_t)thr << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)best);
        last = best;
      }
    }
    __syncwarp();
    uint64_t v = (lane < P) ? cand[lane] : 0ull;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const uint64_t o = __shfl_xor_sync(0xffffffffu, v, stride);
        const bool desc = ((lane & size) == 0);
        const bool lower = ((lane & stride) == 0);
        if ((lower == desc) ? (o > v) : (o < v)) v = o;
      }
    const int id = topk_finish_warp(p, 0, v, lane, P, lgs);
    permute_warp(pp, lane, pp.ex.gate_q ? tab : nullptr, true, id);
  }
}

// ============================================================================ fused route tail
// For small token counts one CTA runs top-k, the permutation and the activation
// prep back to back (one launch instead of three).
constexpr int TAIL_MAX_T = 64;

__global__ void __launch_bounds__(PERM_WARPS * 32) k3_route_tail_kernel(TopkParams tp, PermParams pp, Z16Params zp) {
  extern __shared__ __align__(128) uint8_t smem[];  // max(PERM_WARPS * 2E floats, PERM_WARPS * E ints)
  __shared__ TopkScratch S[PERM_WARPS];
  __shared__ int wsum[PERM_WARPS + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  grid_dep_wait();
  grid_dep_launch();
  if (tp.T == 1 && tp.E <= TOPK_BLOCK_N && tp.K + REFINE_EXTRA <= 32 && blockDim.x == PERM_WARPS * 32) {
    // one token: the activation prep (one warp), then the routing over the whole CTA
    if (warp == 1 && zp.T > 0) z16_token(zp, 0, lane);
    route_one_token_block(tp, pp, smem, lane, warp);
    return;
  } else {
    // top-k of token t on warp t % 16; the activation prep (independent of routing) of
    // token t on warp (t + 8) % 16, so both run at once
    for (int t = warp; t < tp.T; t += PERM_WARPS) {
      float* sb = reinterpret_cast<float*>(smem) + warp * (2 * tp.E);
      topk_token(tp, t, sb, sb + tp.E, S[warp], lane);
    }
    for (int t = (warp + PERM_WARPS / 2) % PERM_WARPS; t < zp.T; t += PERM_WARPS) z16_token(zp, t, lane);
  }
  __syncthreads();
  if (pp.T * pp.K <= 32) {
    if (warp == 0) permute_warp(pp, lane);
  } else {
    permute_block(pp, reinterpret_cast<int32_t*>(smem), wsum);
  }
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
  float* part;         // [T, COMB_MAX_SPLIT] partial sums of squares
  uint32_t* count;     // [T] arrival counters (zero on entry; reset by the last CTA)
};

constexpr int COMB_THREADS = 256;
constexpr int COMB_MAX_SPLIT = 32;
constexpr int COMB_ROW_MAX_THREADS = 1024;  // one-column-per-thread row kernel (few tokens)

// grid T, for L <= 8 * 4 * COMB_THREADS: one CTA per token; thread i combines the float4
// columns i + j * blockDim.x (j < CPT) in k order, the K expert rows read with independent
// loads (KB at a time), and keeps them in registers; the row's sum of squares is reduced in the CTA
// (warp partials added in warp order) and y and yhat are written from registers.
template <int CPT, int MAXT = COMB_THREADS, int KB = 16>
__global__ void __launch_bounds__(MAXT) k3_combine_row_kernel(CombineParams p) {
  __shared__ float wpart[MAXT / 32];
  __shared__ const float* rows[64];
  __shared__ float wk[64];
  grid_dep_wait();
  grid_dep_launch();
  const int t = blockIdx.x;
  if ((int)threadIdx.x < p.K) {
    // a slot pruned by top-p (inv -1, weight 0) has no row: it reads the token's first
    // slot, which is always kept, and adds nothing
    int sl = p.inv[(size_t)t * p.K + threadIdx.x];
    if (sl < 0) sl = p.inv[(size_t)t * p.K];
    rows[threadIdx.x] = p.o + (size_t)sl * p.L;
    wk[threadIdx.x] = p.w[(size_t)t * p.K + threadIdx.x];
  }
  __syncthreads();
  const int L4 = p.L >> 2;
  float4 y[CPT];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c4 = threadIdx.x + j * blockDim.x;
    y[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c4 < L4) {
      for (int k0 = 0; k0 < p.K; k0 += KB) {
        float4 v[KB];
#pragma unroll
        for (int q = 0; q < KB; ++q)
          if (k0 + q < p.K) v[q] = reinterpret_cast<const float4*>(rows[k0 + q])[c4];
#pragma unroll
        for (int q = 0; q < KB; ++q) {
          if (k0 + q < p.K) {
            const float wq = wk[k0 + q];
            y[j].x = fmaf(wq, v[q].x, y[j].x);
            y[j].y = fmaf(wq, v[q].y, y[j].y);
            y[j].z = fmaf(wq, v[q].z, y[j].z);
            y[j].w = fmaf(wq, v[q].w, y[j].w);
          }
        }
      }
      ss = fmaf(y[j].x, y[j].x, ss);
      ss = fmaf(y[j].y, y[j].y, ss);
      ss = fmaf(y[j].z, y[j].z, ss);
      ss = fmaf(y[j].w, y[j].w, ss);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) wpart[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += wpart[w];
  const float r = 1.0f / sqrtf(tot / (float)p.L + p.eps);
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c4 = threadIdx.x + j * blockDim.x;
    if (c4 < L4) {
      reinterpret_cast<float4*>(p.y + (size_t)t * p.L)[c4] = y[j];
      const float4 g = __ldg(reinterpret_cast<const float4*>(p.gamma) + c4);
      const uint32_t lo = f32_to_bf16_bits(g.x * (y[j].x * r)) | (f32_to_bf16_bits(g.y * (y[j].y * r)) << 16);
      const uint32_t hi = f32_to_bf16_bits(g.z * (y[j].z * r)) | (f32_to_bf16_bits(g.w * (y[j].w * r)) << 16);
      reinterpret_cast<uint2*>(p.yhat + (size_t)t * p.L)[c4] = make_uint2(lo, hi);
    }
  }
}

// grid (T, split): CTA sp of token t combines float4 columns [sp*256, sp*256+256) in k
// order -- one column per thread, the K expert rows read with independent loads --,
// writes y and its partial sum of squares; the last CTA of the token to finish adds
// the partials in split order and writes yhat for the whole row.
__global__ void __launch_bounds__(COMB_THREADS) k3_combine_norm_kernel(CombineParams p) {
  __shared__ float wpart[COMB_THREADS / 32];
  __shared__ const float* rows[64];
  __shared__ float wk[64];
  __shared__ int last;
  __shared__ float r_sh;
  grid_dep_wait();
  grid_dep_launch();
  const int t = blockIdx.x, sp = blockIdx.y, nsplit = gridDim.y;
  if ((int)threadIdx.x < p.K) {
    // a slot pruned by top-p (inv -1, weight 0) has no row: it reads the token's first
    // slot, which is always kept, and adds nothing
    int sl = p.inv[(size_t)t * p.K + threadIdx.x];
    if (sl < 0) sl = p.inv[(size_t)t * p.K];
    rows[threadIdx.x] = p.o + (size_t)sl * p.L;
    wk[threadIdx.x] = p.w[(size_t)t * p.K + threadIdx.x];
  }
  __syncthreads();
  const int c4 = sp * COMB_THREADS + threadIdx.x;
  float ss = 0.f;
  if (c4 < p.L / 4) {
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = 0; k0 < p.K; k0 += 16) {
      float4 v[16];
#pragma unroll
      for (int q = 0; q < 16; ++q)
        if (k0 + q < p.K) v[q] = reinterpret_cast<const float4*>(rows[k0 + q])[c4];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        if (k0 + q < p.K) {
          const float wq = wk[k0 + q];
          y.x = fmaf(wq, v[q].x, y.x);
          y.y = fmaf(wq, v[q].y, y.y);
          y.z = fmaf(wq, v[q].z, y.z);
          y.w = fmaf(wq, v[q].w, y.w);
        }
      }
    }
    reinterpret_cast<float4*>(p.y + (size_t)t * p.L)[c4] = y;
    ss = fmaf(y.x, y.x, ss);
    ss = fmaf(y.y, y.y, ss);
    ss = fmaf(y.z, y.z, ss);
    ss = fmaf(y.w, y.w, ss);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) wpart[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += wpart[w];
    p.part[(size_t)t * COMB_MAX_SPLIT + sp] = tot;
    __threadfence();
    const uint32_t prev = atomicAdd(p.count + t, 1u);
    last = (prev == (uint32_t)nsplit - 1u);
    if (last) p.count[t] = 0;  // ready for the next call
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int q = 0; q < nsplit; ++q) tot += __ldcg(p.part + (size_t)t * COMB_MAX_SPLIT + q);
    r_sh = 1.0f / sqrtf(tot / (float)p.L + p.eps);
  }
  __syncthreads();
  const float r = r_sh;
  for (int c = threadIdx.x; c < p.L; c += blockDim.x) {
    const float y = __ldcg(p.y + (size_t)t * p.L + c);
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

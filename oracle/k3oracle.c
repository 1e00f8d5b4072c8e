/*
 * k3oracle.c -- fp64 reference ("oracle") for the Stable LatentMoE routed-expert
 * block on native MXFP4 expert weights.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the bench's
 * CPU-baseline leg may load this file's library.  It shares no code with the CUDA
 * path: plain C99, no SIMD intrinsics, fp64 arithmetic, optional OpenMP over
 * independent tokens / experts (work split only, the arithmetic order of every
 * sum is fixed).
 *
 * Sources (page titles and sections):
 *  [P1] colibri PR #676 "Kimi K3 engine: native-MXFP4 expert streaming, KDA + gated
 *       NoPE MLA + AttnRes + LatentMoE": architecture bullets (Stable LatentMoE,
 *       SiTU-GLU formula), the expert-streaming paragraph (896 experts, top-16),
 *       the chunked-prefill paragraph (chunk expert union, bit-identical to
 *       token-at-a-time), "What's in the commits" item 1 (MXFP4 matmul kernel).
 *  [P2] colibri PR #684 "Kimi K3: integrate coli chat, API, and Web": the quant.h
 *       MXFP4 commit message (packed [O,I/2] u8, low nibble = even column, bit3 =
 *       sign, scales [O,I/32] ue8m0, w = v*2^(s-127)); the engine commit message
 *       (sigmoid router + score-correction bias, top-16, raw-score renormalisation,
 *       latent projections, RMSNorm on the aggregate, SiTU-GLU); the chunked
 *       prefill commit message (counting-sort position lists per unique expert).
 *  [P3] llama.cpp PR #21 "Adding kimi-k3 arch test and saver fix": latent MoE with
 *       routed experts at the latent width; situ betas 4.0 / 25.0; compressed-
 *       tensors MXFP4 shares the E2M1 code assignment and E8M0 scale byte of the
 *       OCP MX format.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - E2M1 magnitudes are the OCP Microscaling (MX) v1.0 E2M1 values
 *    {0, 0.5, 1, 1.5, 2, 3, 4, 6}; code 8 is -0.  E8M0 byte 255 is NaN.
 *  - bf16 rounding points in "spec" mode: R1 z = x Wd^T, R2 h = SiTU(g, u),
 *    R3 yhat = RMSNorm(y).  "pure" mode keeps everything in fp64.
 *  - Top-K order: descending biased score, ties to the lower expert id.
 *  - The combine sums the K weighted expert outputs in that order.
 *  - Gate rows first, then up rows, when gate/up are viewed as one [2I, L] matrix.
 *  - No routed scaling factor; no grouped routing.
 *  - The low-precision-activation variant (act_mxfp8) reads the pages' per-32-group
 *    quantized activations [P1 "What's in the commits" item 7; P2 quant.h commit:
 *    matmul_mxfp4_i8] as OCP MX v1.0 MXFP8: E4M3 elements (bias 7, S.1111.111 NaN, max
 *    448) sharing one E8M0 scale per 32 consecutive elements along the contraction.  The
 *    shared exponent is floor(log2(max |x|)) - 8 (8 = the largest E4M3 exponent), the
 *    elements are x / 2^X rounded to nearest even and saturated to +-448; an all-zero
 *    group takes scale byte 0.  z (after R1) and h (after R2) are quantized before the
 *    expert contractions that read them; nothing else changes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int hidden, latent, n_experts, top_k, inter;
  double rms_eps;
  double top_p; /* K3_TOPP: 0 < p < 1 prunes the top-K to cumulative weight p; else off */
  int act_mxfp8; /* 1: the experts read MXFP8 (E4M3, 32-element groups) activations */
} k3o_dims;

/* ----------------------------------------------------------------------------------------
 * MXFP4 decode [P2 quant.h commit message; P3 E2M1/E8M0 equivalence; OCP MX v1.0 tables]
 * -------------------------------------------------------------------------------------- */
static const double k3o_e2m1_mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* value of a 4-bit E2M1 code: bit3 = sign, bits 0..2 = magnitude code */
double k3o_e2m1(unsigned code) {
  double m = k3o_e2m1_mag[code & 7u];
  return (code & 8u) ? -m : m;
}

/* value of an E8M0 (ue8m0) scale byte: 2^(s-127); 255 is NaN */
double k3o_ue8m0(unsigned s) {
  if (s == 255u) return NAN;
  return ldexp(1.0, (int)s - 127);
}

/* element (o, c) of an [O, I] MXFP4 matrix: packed [O, I/2], scales [O, I/32] */
static double k3o_mx_elem(const uint8_t* q, const uint8_t* s, int I, int o, int c) {
  uint8_t b = q[(size_t)o * (size_t)(I / 2) + (size_t)(c / 2)];
  unsigned code = (c & 1) ? (unsigned)(b >> 4) : (unsigned)(b & 15u); /* low nibble = even column */
  return k3o_e2m1(code) * k3o_ue8m0(s[(size_t)o * (size_t)(I / 32) + (size_t)(c / 32)]);
}

void k3o_dequant(const uint8_t* q, const uint8_t* s, int O, int I, double* out) {
  for (int o = 0; o < O; ++o)
    for (int c = 0; c < I; ++c) out[(size_t)o * I + c] = k3o_mx_elem(q, s, I, o, c);
}

/* ----------------------------------------------------------------------------------------
 * MXFP8 activations [P1 "What's in the commits" item 7 and P2 quant.h commit (per-32-group
 * quantized activations, the variant's idea); OCP MX v1.0 E4M3 element and E8M0 scale]
 * -------------------------------------------------------------------------------------- */
/* value of an E4M3 code: bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa;
 * exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN (no infinities) */
double k3o_e4m3(unsigned code) {
  const unsigned e = (code >> 3) & 15u, m = code & 7u;
  if (e == 15u && m == 7u) return NAN;
  const double mag = e ? ldexp(1.0 + m / 8.0, (int)e - 7) : ldexp(m / 8.0, -6);
  return (code & 0x80u) ? -mag : mag;
}

/* nearest E4M3 code to v (ties to the even code, i.e. even mantissa), saturating at
 * +-448; the sign bit follows v's sign (a negative value that rounds to zero is -0).
 * The non-negative finite codes 0..126 are increasing in value: binary search for the
 * largest code not above |v|, then compare with its successor. */
unsigned k3o_e4m3_encode(double v) {
  const unsigned sign = signbit(v) ? 0x80u : 0u;
  const double a = fabs(v);
  if (a >= 448.0) return sign | 126u;
  unsigned lo = 0, hi = 126;
  while (lo < hi) { /* invariant: value(lo) <= a */
    const unsigned mid = (lo + hi + 1) / 2;
    if (k3o_e4m3((int)mid) <= a) lo = mid;
    else hi = mid - 1;
  }
  if (k3o_e4m3(lo) == a) return sign | lo;
  const unsigned up = lo + 1;
  const double dl = a - k3o_e4m3(lo), du = k3o_e4m3(up) - a;
  const unsigned c = (dl < du) ? lo : (du < dl) ? up : ((lo & 1u) ? up : lo);
  return sign | c;
}

/* scale byte of one group from its largest magnitude: 127 + floor(log2(amax)) - 8,
 * clamped to [0, 254]; 0 for an all-zero group */
static unsigned k3o_mxfp8_scale(double amax) {
  if (amax == 0.0) return 0u;
  int ex = 0;
  frexp(amax, &ex); /* amax = f 2^ex, f in [0.5, 1): floor(log2(amax)) = ex - 1 */
  int s = 127 + (ex - 1) - 8;
  if (s < 0) s = 0;
  if (s > 254) s = 254;
  return (unsigned)s;
}

/* x [n] (n a multiple of 32) -> E4M3 codes [n] and scale bytes [n/32] */
void k3o_mxfp8_quant(int64_t n, const double* x, uint8_t* codes, uint8_t* scales) {
  for (int64_t g = 0; g < n / 32; ++g) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) amax = fmax(amax, fabs(x[g * 32 + i]));
    const unsigned s = k3o_mxfp8_scale(amax);
    scales[g] = (uint8_t)s;
    for (int i = 0; i < 32; ++i) codes[g * 32 + i] = (uint8_t)k3o_e4m3_encode(ldexp(x[g * 32 + i], 127 - (int)s));
  }
}

/* x -> the values of its MXFP8 quantization (code value times 2^(s-127)) */
void k3o_mxfp8_round(int64_t n, const double* x, double* out) {
  uint8_t* c = (uint8_t*)malloc((size_t)(n > 0 ? n : 1));
  uint8_t* s = (uint8_t*)malloc((size_t)(n / 32 > 0 ? n / 32 : 1));
  k3o_mxfp8_quant(n, x, c, s);
  for (int64_t i = 0; i < n; ++i) out[i] = ldexp(k3o_e4m3(c[i]), (int)s[i / 32] - 127);
  free(c);
  free(s);
}

/* ----------------------------------------------------------------------------------------
 * storage types
 * -------------------------------------------------------------------------------------- */
static double k3o_from_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* round to the nearest bf16 value (8 significant bits, ties to even), kept as fp64 */
double k3o_round_bf16(double v) {
  if (v == 0.0 || !isfinite(v)) return v;
  int e = ilogb(v);             /* v = m * 2^e, 1 <= |m| < 2 */
  if (e < -126) e = -126;       /* bf16 subnormal quantum is 2^-133 */
  double q = ldexp(1.0, e - 7); /* spacing of bf16 values near v */
  double r = nearbyint(v / q) * q; /* default rounding mode: nearest, ties to even */
  if (fabs(r) > 0x1.FEp127) r = copysign(INFINITY, v); /* above the largest finite bf16 */
  return r;
}

/* ----------------------------------------------------------------------------------------
 * activation and normalisation [P1 architecture bullets; P2 engine commit; P3 situ betas]
 * -------------------------------------------------------------------------------------- */
static double k3o_sigmoid(double a) { return 1.0 / (1.0 + exp(-a)); }

/* SiTU-GLU: 4 tanh(g/4) * sigmoid(g) * 25 tanh(u/25) */
double k3o_situ(double g, double u) { return 4.0 * tanh(g / 4.0) * k3o_sigmoid(g) * 25.0 * tanh(u / 25.0); }

/* RMSNorm of the aggregate: yhat = gamma * y / sqrt(mean(y^2) + eps) */
void k3o_rmsnorm(int L, const double* y, const float* gamma, double eps, int spec, double* yhat) {
  double ss = 0.0;
  for (int c = 0; c < L; ++c) ss += y[c] * y[c];
  double den = sqrt(ss / (double)L + eps);
  for (int c = 0; c < L; ++c) {
    double v = (double)gamma[c] * (y[c] / den);
    yhat[c] = spec ? k3o_round_bf16(v) : v;
  }
}

/* ----------------------------------------------------------------------------------------
 * router [P2 engine commit: sigmoid router + score-correction bias, top-16,
 *         raw-score renormalisation]
 * -------------------------------------------------------------------------------------- */
void k3o_router_logits(const k3o_dims* d, int T, const uint16_t* x, const uint16_t* wr, double* logits) {
  const int H = d->hidden, E = d->n_experts;
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < T; ++t) {
    const uint16_t* xt = x + (size_t)t * H;
    for (int e = 0; e < E; ++e) {
      const uint16_t* we = wr + (size_t)e * H;
      double acc = 0.0;
      for (int h = 0; h < H; ++h) acc += k3o_from_bf16(xt[h]) * k3o_from_bf16(we[h]);
      logits[(size_t)t * E + e] = acc;
    }
  }
}

/* Selects, per token, the top_k experts by biased score s + b (descending, ties to
 * the lower id), and renormalises their raw scores s to sum to one.
 * gap[t] (nullable) = biased score of the k-th minus the (k+1)-th selected expert;
 * mingap[t] (nullable) = smallest difference between consecutive biased scores among
 * the first k+1 (decides whether the selected order is unique). */
/* K3_TOPP [P1 K3_TOPP paragraph; P2 engine commit "drop the low-weight tail of the top-16
 * to cumulative weight p, renormalized"]: the K selected experts ordered by weight
 * (descending; equal weights keep their top-K order), the shortest prefix whose weights
 * sum to at least p kept (an expert is kept while the weight of those before it is below
 * p, so the first always is), the kept ones renormalised by their raw scores, the rest
 * marked id -1 with weight 0.  The kept experts come first, in weight order.  s: raw
 * scores of all experts; ids, w: one token's K entries, overwritten. */
static void k3o_top_p(int K, double p, const double* s, int32_t* ids, double* w) {
  int* ord = (int*)malloc(sizeof(int) * (size_t)K);
  for (int k = 0; k < K; ++k) ord[k] = k;
  for (int a = 1; a < K; ++a) { /* insertion sort: stable, descending weight */
    const int v = ord[a];
    int b = a - 1;
    while (b >= 0 && w[ord[b]] < w[v]) {
      ord[b + 1] = ord[b];
      --b;
    }
    ord[b + 1] = v;
  }
  int nkeep = 0;
  double cum = 0.0;
  for (int j = 0; j < K; ++j) {
    if (j > 0 && !(cum < p)) break;
    cum += w[ord[j]];
    ++nkeep;
  }
  int32_t* id2 = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
  double sk = 0.0;
  for (int j = 0; j < nkeep; ++j) sk += s[ids[ord[j]]];
  for (int j = 0; j < K; ++j) id2[j] = ids[ord[j]];
  for (int j = 0; j < K; ++j) {
    if (j < nkeep) {
      ids[j] = id2[j];
      w[j] = s[id2[j]] / sk;
    } else {
      ids[j] = -1;
      w[j] = 0.0;
    }
  }
  free(id2);
  free(ord);
}

void k3o_topk(const k3o_dims* d, int T, const double* logits, const float* bias, int32_t* ids, double* w,
              double* gap, double* mingap) {
  const int E = d->n_experts, K = d->top_k;
  const int P = (K < E) ? K + 1 : K;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    double* s = (double*)malloc(sizeof(double) * (size_t)E * 2);
    double* sb = s + E;
    unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
    int* sel = (int*)malloc(sizeof(int) * (size_t)P);
    for (int e = 0; e < E; ++e) {
      s[e] = k3o_sigmoid(logits[(size_t)t * E + e]);
      sb[e] = s[e] + (double)bias[e];
    }
    for (int k = 0; k < P; ++k) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || sb[e] > sb[best]) best = e; /* strict: equal scores keep the lower id */
      }
      taken[best] = 1;
      sel[k] = best;
    }
    double sum = 0.0;
    for (int k = 0; k < K; ++k) sum += s[sel[k]];
    for (int k = 0; k < K; ++k) {
      ids[(size_t)t * K + k] = sel[k];
      w[(size_t)t * K + k] = s[sel[k]] / sum;
    }
    if (d->top_p > 0.0 && d->top_p < 1.0) k3o_top_p(K, d->top_p, s, ids + (size_t)t * K, w + (size_t)t * K);
    if (gap) gap[t] = (P > K) ? sb[sel[K - 1]] - sb[sel[K]] : INFINITY;
    if (mingap) {
      double m = INFINITY;
      for (int k = 0; k + 1 < P; ++k) {
        double g = sb[sel[k]] - sb[sel[k + 1]];
        if (g < m) m = g;
      }
      mingap[t] = m;
    }
    free(sel);
    free(taken);
    free(s);
  }
}

/* ----------------------------------------------------------------------------------------
 * chunk expert union by counting sort [P1 chunked-prefill paragraph; P2 chunked
 * prefill commit: "builds the chunk's expert union per layer ... position lists via
 * counting sort"].  slot_of lists the flat (t*K + k) indices grouped by expert in
 * ascending expert id, in ascending (t, k) order inside an expert.
 * -------------------------------------------------------------------------------------- */
void k3o_permute(int T, int K, int E, const int32_t* ids, int32_t* counts, int32_t* offsets, int32_t* slot_of,
                 int32_t* uniq, int32_t* n_uniq) {
  const int n = T * K;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int i = 0; i < n; ++i)
    if (ids[i] >= 0) counts[ids[i]] += 1; /* id -1: a slot pruned by top-p, not placed */
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* pos = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
  for (int e = 0; e < E; ++e) pos[e] = offsets[e];
  for (int i = 0; i < n; ++i)
    if (ids[i] >= 0) slot_of[pos[ids[i]]++] = i;
  free(pos);
  int u = 0;
  for (int e = 0; e < E; ++e)
    if (counts[e] > 0) uniq[u++] = e;
  *n_uniq = u;
}

/* ----------------------------------------------------------------------------------------
 * latent projections [P1 "routed experts run in a 3584-dim latent space behind shared
 * down/up projections"; P3 latent MoE]
 * -------------------------------------------------------------------------------------- */
void k3o_latent_down(const k3o_dims* d, int T, const uint16_t* x, const uint16_t* wd, int spec, double* z) {
  const int H = d->hidden, L = d->latent;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t)
    for (int l = 0; l < L; ++l) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h) acc += k3o_from_bf16(x[(size_t)t * H + h]) * k3o_from_bf16(wd[(size_t)l * H + h]);
      z[(size_t)t * L + l] = spec ? k3o_round_bf16(acc) : acc;
    }
}

void k3o_latent_up(const k3o_dims* d, int T, const double* yhat, const uint16_t* wu, double* out) {
  const int H = d->hidden, L = d->latent;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int l = 0; l < L; ++l) acc += yhat[(size_t)t * L + l] * k3o_from_bf16(wu[(size_t)h * L + l]);
      out[(size_t)t * H + h] = acc;
    }
}

/* ----------------------------------------------------------------------------------------
 * one expert on one latent vector, decoding the vendor bytes on the fly
 * [P1 architecture bullets; P2 quant.h and engine commits]
 *   g_j = sum_c gate[j][c] z_c,  u_j = sum_c up[j][c] z_c,  h_j = SiTU(g_j, u_j)
 *   o_c = sum_j down[c][j] h_j
 * -------------------------------------------------------------------------------------- */
void k3o_expert(const k3o_dims* d, const double* z, const uint8_t* gq, const uint8_t* gs, const uint8_t* uq,
                const uint8_t* us, const uint8_t* dq, const uint8_t* ds, int spec, double* h_out, double* o) {
  const int L = d->latent, I = d->inter;
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  double* zq = NULL;
  if (d->act_mxfp8) { /* the variant's gate/up input: z quantized to MXFP8 */
    zq = (double*)malloc(sizeof(double) * (size_t)L);
    k3o_mxfp8_round(L, z, zq);
    z = zq;
  }
  for (int j = 0; j < I; ++j) {
    double g = 0.0, u = 0.0;
    for (int c = 0; c < L; ++c) g += k3o_mx_elem(gq, gs, L, j, c) * z[c];
    for (int c = 0; c < L; ++c) u += k3o_mx_elem(uq, us, L, j, c) * z[c];
    double v = k3o_situ(g, u);
    h[j] = spec ? k3o_round_bf16(v) : v;
  }
  if (d->act_mxfp8) k3o_mxfp8_round(I, h, h); /* the down input: h quantized to MXFP8 */
  free(zq);
  for (int c = 0; c < L; ++c) {
    double acc = 0.0;
    for (int j = 0; j < I; ++j) acc += k3o_mx_elem(dq, ds, I, c, j) * h[j];
    o[c] = acc;
  }
  if (h_out) memcpy(h_out, h, sizeof(double) * (size_t)I);
  free(h);
}

/* the same expert applied to several latent vectors from dense fp64 copies of its
 * weights (decoded once) -- the chunked path; every dot product runs over the same
 * index order with the same element values as k3o_expert */
static void k3o_expert_dense(const k3o_dims* d, int n, const double* const* zs, const double* Wg, const double* Wu,
                             const double* Wdn, int spec, double* const* os) {
  const int L = d->latent, I = d->inter;
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  double* zq = (double*)malloc(sizeof(double) * (size_t)L);
  for (int i = 0; i < n; ++i) {
    const double* z = zs[i];
    if (d->act_mxfp8) {
      k3o_mxfp8_round(L, z, zq);
      z = zq;
    }
    for (int j = 0; j < I; ++j) {
      double g = 0.0, u = 0.0;
      const double* rg = Wg + (size_t)j * L;
      const double* ru = Wu + (size_t)j * L;
      for (int c = 0; c < L; ++c) g += rg[c] * z[c];
      for (int c = 0; c < L; ++c) u += ru[c] * z[c];
      double v = k3o_situ(g, u);
      h[j] = spec ? k3o_round_bf16(v) : v;
    }
    if (d->act_mxfp8) k3o_mxfp8_round(I, h, h);
    for (int c = 0; c < L; ++c) {
      double acc = 0.0;
      const double* rd = Wdn + (size_t)c * I;
      for (int j = 0; j < I; ++j) acc += rd[j] * h[j];
      os[i][c] = acc;
    }
  }
  free(h);
  free(zq);
}

/* ----------------------------------------------------------------------------------------
 * shared experts beside the routed block [P1 architecture bullets, P2 engine commit "2
 * fused shared experts"]: SiTU-GLU experts on the hidden width whose weights are fused
 * along the intermediate dimension (gate rows 0..Is-1 and up rows Is..2Is-1 of wgu [2Is,
 * H]; wdn [H, Is]), so the fused expert computes the sum of the separate ones:
 *   g_j = sum_c wgu[j][c] x_c,  u_j = sum_c wgu[Is + j][c] x_c,  h_j = SiTU(g_j, u_j)
 *   (bf16-rounded in spec mode, as the routed h),  out_c = sum_j wdn[c][j] h_j.
 * The block's output adds it to the routed output. h_out (nullable) [T, Is], out [T, H].
 * -------------------------------------------------------------------------------------- */
void k3o_shared(const k3o_dims* d, int T, int Is, const uint16_t* x, const uint16_t* wgu, const uint16_t* wdn,
                int spec, double* h_out, double* out) {
  const int H = d->hidden;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    double* h = (double*)malloc(sizeof(double) * (size_t)Is);
    const uint16_t* xt = x + (size_t)t * H;
    for (int j = 0; j < Is; ++j) {
      double g = 0.0, u = 0.0;
      for (int c = 0; c < H; ++c) g += k3o_from_bf16(wgu[(size_t)j * H + c]) * k3o_from_bf16(xt[c]);
      for (int c = 0; c < H; ++c) u += k3o_from_bf16(wgu[(size_t)(Is + j) * H + c]) * k3o_from_bf16(xt[c]);
      const double v = k3o_situ(g, u);
      h[j] = spec ? k3o_round_bf16(v) : v;
    }
    for (int c = 0; c < H; ++c) {
      double acc = 0.0;
      for (int j = 0; j < Is; ++j) acc += k3o_from_bf16(wdn[(size_t)c * Is + j]) * h[j];
      out[(size_t)t * H + c] = acc;
    }
    if (h_out) memcpy(h_out + (size_t)t * Is, h, sizeof(double) * (size_t)Is);
    free(h);
  }
}

/* ----------------------------------------------------------------------------------------
 * whole block.  Expert e's tensors are ex[0..5][e] = gate_q, gate_s, up_q, up_s,
 * down_q, down_s; entries of experts that no token routes to may be NULL.
 * chunk = 0: token at a time (each expert decoded where it is used);
 * chunk = C > 0: tokens in chunks of C, each chunk's expert union built by counting
 * sort and every unique expert decoded once.
 * Outputs: out [T, H]; ids [T, K]; w [T, K]; z [T, L], y [T, L], yhat [T, L] (nullable).
 * Returns 0, or -(1 + e) when expert e is routed to but has NULL tensors.
 * -------------------------------------------------------------------------------------- */
int k3o_forward(const k3o_dims* d, int T, const uint16_t* x, const uint16_t* wr, const float* bias,
                const uint16_t* wd, const uint16_t* wu, const float* gamma, const uint8_t* const* const* ex, int spec,
                int chunk, double* out, int32_t* ids, double* w, double* z_out, double* y_out, double* yhat_out) {
  const int E = d->n_experts, K = d->top_k, L = d->latent, I = d->inter;
  double* logits = (double*)malloc(sizeof(double) * (size_t)T * E);
  double* z = (double*)malloc(sizeof(double) * (size_t)T * L);
  double* y = (double*)calloc((size_t)T * L, sizeof(double));
  double* yhat = (double*)malloc(sizeof(double) * (size_t)T * L);
  double* o = (double*)malloc(sizeof(double) * (size_t)T * K * L); /* per (t, k) expert output */
  int rc = 0;

  k3o_router_logits(d, T, x, wr, logits);
  k3o_topk(d, T, logits, bias, ids, w, NULL, NULL);
  k3o_latent_down(d, T, x, wd, spec, z);
  for (int i = 0; i < T * K; ++i) {
    int e = ids[i];
    if (e < 0) continue; /* pruned by top-p */
    for (int j = 0; j < 6; ++j)
      if (!ex[j][e]) rc = -(1 + e);
  }
  if (rc) goto done;
  memset(o, 0, sizeof(double) * (size_t)T * K * L);

  if (chunk <= 0) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < T * K; ++i) {
      int t = i / K, e = ids[i];
      if (e < 0) continue;
      k3o_expert(d, z + (size_t)t * L, ex[0][e], ex[1][e], ex[2][e], ex[3][e], ex[4][e], ex[5][e], spec, NULL,
                 o + (size_t)i * L);
    }
  } else {
    for (int t0 = 0; t0 < T; t0 += chunk) {
      const int C = (T - t0 < chunk) ? T - t0 : chunk;
      int32_t* counts = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
      int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
      int32_t* slot_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)C * K);
      int32_t* uniq = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
      int32_t nu = 0;
      k3o_permute(C, K, E, ids + (size_t)t0 * K, counts, offsets, slot_of, uniq, &nu);
#pragma omp parallel for schedule(dynamic, 1)
      for (int ui = 0; ui < nu; ++ui) {
        const int e = uniq[ui];
        double* Wg = (double*)malloc(sizeof(double) * (size_t)I * L);
        double* Wup = (double*)malloc(sizeof(double) * (size_t)I * L);
        double* Wdn = (double*)malloc(sizeof(double) * (size_t)L * I);
        k3o_dequant(ex[0][e], ex[1][e], I, L, Wg);
        k3o_dequant(ex[2][e], ex[3][e], I, L, Wup);
        k3o_dequant(ex[4][e], ex[5][e], L, I, Wdn);
        const int n = counts[e];
        const double** zs = (const double**)malloc(sizeof(double*) * (size_t)n);
        double** os = (double**)malloc(sizeof(double*) * (size_t)n);
        for (int p = 0; p < n; ++p) {
          const int flat = slot_of[offsets[e] + p]; /* (t - t0) * K + k */
          zs[p] = z + (size_t)(t0 + flat / K) * L;
          os[p] = o + ((size_t)t0 * K + flat) * L;
        }
        k3o_expert_dense(d, n, zs, Wg, Wup, Wdn, spec, os);
        free(zs);
        free(os);
        free(Wg);
        free(Wup);
        free(Wdn);
      }
      free(counts);
      free(offsets);
      free(slot_of);
      free(uniq);
    }
  }

  /* gate-weighted combine in k order, then RMSNorm on the aggregate, then latent up */
  for (int t = 0; t < T; ++t) {
    double* yt = y + (size_t)t * L;
    for (int k = 0; k < K; ++k) {
      if (ids[(size_t)t * K + k] < 0) continue; /* pruned by top-p */
      const double wk = w[(size_t)t * K + k];
      const double* ok = o + ((size_t)t * K + k) * L;
      for (int c = 0; c < L; ++c) yt[c] += wk * ok[c];
    }
    k3o_rmsnorm(L, yt, gamma, d->rms_eps, spec, yhat + (size_t)t * L);
  }
  k3o_latent_up(d, T, yhat, wu, out);
  if (z_out) memcpy(z_out, z, sizeof(double) * (size_t)T * L);
  if (y_out) memcpy(y_out, y, sizeof(double) * (size_t)T * L);
  if (yhat_out) memcpy(yhat_out, yhat, sizeof(double) * (size_t)T * L);
done:
  free(logits);
  free(z);
  free(y);
  free(yhat);
  free(o);
  return rc;
}

/* array helpers for the test bindings */
void k3o_round_bf16_array(int64_t n, const double* in, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = k3o_round_bf16(in[i]);
}
void k3o_situ_array(int64_t n, const double* g, const double* u, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = k3o_situ(g[i], u[i]);
}

int k3o_abi_version(void) { return 3; }

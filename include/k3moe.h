/*
 * k3moe.h -- C ABI of the GB300 (sm_103a) Stable LatentMoE routed-expert block on
 * native MXFP4 expert weights.
 *
 * What the block computes (colibri PR #684, engine commit message: "Stable
 * LatentMoE: sigmoid router + score-correction bias, top-16, raw-score
 * renormalization; latent 7168<->3584 projections around the experts; RMSNorm on
 * the aggregate; ... SiTU-GLU (4 tanh(g/4) sigmoid(g) * 25 tanh(u/25))"; colibri
 * PR #676, architecture bullets), per token t with x_t in R^H:
 *
 *   l_e   = x_t . Wr_e                     router logits, e < E
 *   s_e   = sigmoid(l_e),  s'_e = s_e + b_e
 *   ids   = the K experts with largest s' (descending, ties to the lower id)
 *   w_k   = s_ids[k] / sum_j s_ids[j]      raw-score renormalisation
 *   z     = bf16(x_t Wd^T)                 latent down, [L]
 *   g, u  = z Wgate_e^T, z Wup_e^T         per selected expert, MXFP4 weights, [I]
 *   h     = bf16(4 tanh(g/4) sigmoid(g) 25 tanh(u/25))
 *   o_k   = h Wdown_e^T                    MXFP4 weights, [L]
 *   y     = sum_k w_k o_k                  gate-weighted combine
 *   yhat  = bf16(gamma * y / sqrt(mean(y^2) + eps))   RMSNorm on the aggregate
 *   out_t = yhat Wu^T                      latent up, [H], returned in fp32
 *
 * MXFP4 vendor layout (colibri PR #684, quant.h commit message): an [O, I] matrix
 * is packed [O, I/2] u8 (low nibble = even column, bit 3 = sign, E2M1 codes) plus
 * scales [O, I/32] u8 (E8M0), value = e2m1(code) * 2^(s - 127).  The library reads
 * these bytes as they are; nothing is re-encoded.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers, row-major and densely packed, unless
 *    stated otherwise.  bf16 tensors are passed as uint16_t bit patterns.
 *  - The caller owns all memory, including the workspace; the library allocates,
 *    frees and synchronises nothing in the compute calls, and keeps no per-call
 *    global state.  Calls on different streams with different workspaces may run
 *    concurrently.
 *  - Arguments are validated on the host before anything is launched; an invalid
 *    call returns a status and launches nothing.  No call aborts or traps.
 *  - Launch errors return K3MOE_ERR_CUDA.  Conditions that only the device can see
 *    are OR-ed into a status word inside the workspace; read it with
 *    k3moe_device_status().
 *  - 16-byte alignment is required for every tensor pointer.
 */
#ifndef K3MOE_H
#define K3MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t hidden;    /* H: model width (7168 for K3); multiple of 64 */
  int32_t latent;    /* L: latent width (3584 for K3); multiple of 64 */
  int32_t n_experts; /* E: routed experts (896 for K3); 1..2048 */
  int32_t top_k;     /* K: experts per token (16 for K3); 1..min(E, 64) */
  int32_t inter;     /* I: expert intermediate width (3072 for K3); multiple of 64 */
  float rms_eps;     /* epsilon of the aggregate RMSNorm */
  float top_p;       /* cumulative-weight pruning of the top-K (K3_TOPP): for 0 < top_p < 1 the
                        K experts are ordered by weight (equal weights keep their top-K order),
                        the shortest prefix whose weights reach top_p is kept and renormalised
                        over its raw scores, and the rest are dropped (id -1, weight 0 in the
                        routing outputs; no expert work).  0 (or >= 1): off.  With pruning on,
                        K + 8 <= 32 is required */
  int32_t act_mxfp8; /* 0: the expert contractions read the bf16 activations (exact path).
                        1: the low-precision-activation variant: the tensor-core expert GEMMs
                        (T >= k3moe_tc_min_tokens) read z and h quantized to MXFP8 (OCP MX
                        E4M3 elements, one E8M0 scale per 32 consecutive elements along the
                        contraction) and run block-scaled on the MXFP4 weights as stored;
                        smaller batches run the exact path.  Lossy by about one E4M3 step
                        per activation element */
} k3moe_dims;

typedef enum {
  K3MOE_OK = 0,
  K3MOE_ERR_ARG = 1,       /* null pointer, negative count, bad enum */
  K3MOE_ERR_SHAPE = 2,     /* a width is not a supported multiple, or K > E */
  K3MOE_ERR_ALIGN = 3,     /* a pointer is not 16-byte aligned */
  K3MOE_ERR_WORKSPACE = 4, /* workspace null or smaller than k3moe_workspace_bytes() */
  K3MOE_ERR_DEVICE = 5,    /* current device is not compute capability 10.3 */
  K3MOE_ERR_CUDA = 6       /* a CUDA launch or copy failed */
} k3moe_status;

/* Bits of the device status word (k3moe_device_status). */
#define K3MOE_DEV_TIE_WINDOW 0x1u /* a near-tie cluster of biased scores reached the end of the
                                     refinement window; the selected ids may differ from an
                                     exact ranking for that token */
#define K3MOE_DEV_TIMEOUT 0x2u    /* a device-side bounded wait ran out; outputs are invalid */
#define K3MOE_DEV_BAD_ID 0x4u     /* an expert id outside [0, E) reached the permutation */
#define K3MOE_DEV_SCALE_RANGE 0x8u /* never set: every path decodes every scale byte exactly
                                      (the value is kept so that the bit stays reserved) */
#define K3MOE_DEV_ALIGN 0x10u      /* the tensor-core expert path (T >= k3moe_tc_min_tokens) met an
                                      expert weight tensor below its alignment (see k3moe_experts);
                                      the call was abandoned and its outputs are invalid */

/* The six vendor tensors of every expert, as DEVICE arrays of n_experts DEVICE
 * pointers (the pointer tables themselves live in device memory):
 *   gate_q[e] [I, L/2], gate_s[e] [I, L/32]    gate projection of expert e
 *   up_q[e]   [I, L/2], up_s[e]   [I, L/32]    up projection
 *   down_q[e] [L, I/2], down_s[e] [L, I/32]    down projection
 * A checkpoint that stores gate and up as one fused [2I, L] matrix (gate rows first)
 * passes up_q[e] = gate_q[e] + I*L/2 and up_s[e] = gate_s[e] + I*L/32.
 * Every pointer in the tables must be 16-byte aligned like any other tensor.  The
 * tensor-core path's block-scaled GEMMs (the split form and the act_mxfp8 variant) copy the
 * packed tensors gate_q, up_q and down_q with 4-bit tensor copies, which need them 32-byte
 * aligned (true of any pool whose tensors start at multiples of 32 bytes, e.g. 256-byte
 * padded); run a pool with 16- but not 32-byte aligned packed tensors on the weight-decode
 * form (k3moe_set_tc_split_max_tokens(0)).  The host cannot see the pointers, so the
 * tensor-core path checks them on the device, reports K3MOE_DEV_ALIGN and abandons the
 * call when one falls short. */
typedef struct {
  const uint8_t* const* gate_q;
  const uint8_t* const* gate_s;
  const uint8_t* const* up_q;
  const uint8_t* const* up_s;
  const uint8_t* const* down_q;
  const uint8_t* const* down_s;
} k3moe_experts;

/* Bytes of workspace that k3moe_route / k3moe_forward / k3moe_expert_forward need
 * for T tokens.  Returns 0 for invalid dims or T < 0. */
size_t k3moe_workspace_bytes(const k3moe_dims* dims, int32_t T);

/* Router only (steps l, s, s', ids, w above).
 *   x     [T, H] bf16    activations
 *   wr    [E, H] bf16    router weight
 *   bias  [E]    f32     score-correction bias (selects; does not weight)
 *   ids   [T, K] int32   out: selected experts, descending biased score
 *   w     [T, K] f32     out: renormalised raw scores
 * Logits are accumulated in fp32; candidates whose biased scores lie within 3e-5
 * of a neighbour in a cluster reaching the top K+1 get their logits recomputed from
 * the bf16 inputs in double-f32 arithmetic (error-free sums, about 48 significant
 * bits) and are re-ranked, so the ids equal an exact-arithmetic ranking unless two
 * biased scores differ by less than about 1e-12.
 * T = 0 is a valid no-op.  `stream` is a cudaStream_t (NULL = legacy default). */
k3moe_status k3moe_route(const k3moe_dims* dims, int32_t T, const uint16_t* x, const uint16_t* wr,
                         const float* bias, int32_t* ids, float* w, void* ws, size_t ws_bytes, void* stream);

/* The whole block for T tokens (the chunk's expert union is built once; each
 * selected expert's weights are streamed once per call).  From 9 tokens on (see
 * k3moe_set_tc_min_tokens) the projections and experts run on tensor-core GEMMs.
 *   x      [T, H] bf16;  wr [E, H] bf16;  bias [E] f32
 *   w_down [L, H] bf16   latent down;  w_up [H, L] bf16 latent up
 *   norm_w [L]    f32    RMSNorm weight gamma
 *   experts              pointer tables (see k3moe_experts), read on the device
 *   out    [T, H] f32    out
 *   ids_out [T, K] int32, w_out [T, K] f32   optional copies of the routing (may be NULL)
 * Numerics: bf16 operands, fp32 accumulation; z, h and yhat are rounded to bf16
 * (round-to-nearest-even) where the definition above says bf16. */
k3moe_status k3moe_forward(const k3moe_dims* dims, int32_t T, const uint16_t* x, const uint16_t* wr,
                           const float* bias, const uint16_t* w_down, const uint16_t* w_up, const float* norm_w,
                           const k3moe_experts* experts, float* out, int32_t* ids_out, float* w_out, void* ws,
                           size_t ws_bytes, void* stream);

/* k3moe_forward with per-phase timing.  `events` holds n_events (0..7) cudaEvent_t
 * handles created by the caller; event i is recorded on `stream` at the start of
 * phase i and event 6 after the last phase.  Phases: 0 router logits + latent down
 * (one pass over x), 1 top-k + permutation + activation prep, 2 expert gate/up +
 * SiTU-GLU, 3 expert down, 4 combine + RMSNorm, 5 latent up.  NULL entries are
 * skipped.  With events the kernels run strictly one after another (k3moe_forward
 * lets each kernel start while its predecessor drains); results are identical. */
k3moe_status k3moe_forward_profiled(const k3moe_dims* dims, int32_t T, const uint16_t* x, const uint16_t* wr,
                                    const float* bias, const uint16_t* w_down, const uint16_t* w_up,
                                    const float* norm_w, const k3moe_experts* experts, float* out, int32_t* ids_out,
                                    float* w_out, void* ws, size_t ws_bytes, void* stream, void* const* events,
                                    int32_t n_events);

/* Size in bytes of the fixed device scratch array that k3moe_forward_noalloc uses. */
#define K3MOE_NOALLOC_SCRATCH_BYTES (4u << 20)

/* k3moe_forward for callers that cannot allocate device memory: no workspace
 * argument, and no cudaMalloc / cudaFree or allocating library call inside.  This
 * suits code that runs where the allocator is off limits, e.g. a plugin inside a
 * host framework that owns every device allocation, or a path that must not touch
 * the allocator once it is set up.  The pages have no counterpart to this entry
 * point; it is a packaging variant of k3moe_forward.
 *  - Scratch lives in one fixed array of K3MOE_NOALLOC_SCRATCH_BYTES (4 MiB) in device
 *    memory that every GPU which loads the library holds until the process exits.  A
 *    call fits when k3moe_workspace_bytes(dims, T) is at most that size: at K3 shapes
 *    (H 7168, L 3584, E 896, K 16, I 3072) that is up to 8 tokens per call (the
 *    weight-streaming regime below k3moe_tc_min_tokens).  A call
 *    that needs more returns K3MOE_ERR_WORKSPACE and launches nothing.
 *  - The first call on a device looks up the array's device address with
 *    cudaGetSymbolAddress (with that device current); make that first call before
 *    any stream capture.  The lookup is repeated only if the device's context has
 *    changed since (e.g. after cudaDeviceReset).
 *  - Every call shares the array and leaves its contents behind (the call clears
 *    what must start at zero).  Calls that overlap on the GPU, on any stream, race
 *    on the array: serialise them.
 *  - Conditions that only the device sees go to the status word at the start of the
 *    array: read it with k3moe_device_status(NULL, ...).
 * Arguments, results and other errors are those of k3moe_forward. */
k3moe_status k3moe_forward_noalloc(const k3moe_dims* dims, int32_t T, const uint16_t* x, const uint16_t* wr,
                                   const float* bias, const uint16_t* w_down, const uint16_t* w_up,
                                   const float* norm_w, const k3moe_experts* experts, float* out, int32_t* ids_out,
                                   float* w_out, void* stream);

/* One expert applied to T latent vectors (gate/up, SiTU-GLU, down; no routing):
 *   z [T, L] bf16 in; out [T, L] f32 = h(z_t) Wdown_e^T with h rounded to bf16.
 * `expert` indexes the pointer tables.  Same workspace rule as k3moe_forward. */
k3moe_status k3moe_expert_forward(const k3moe_dims* dims, int32_t T, const uint16_t* z, int32_t expert,
                                  const k3moe_experts* experts, float* out, void* ws, size_t ws_bytes,
                                  void* stream);

/* MXFP4 -> f32 decode of an [O, I] vendor matrix (I a multiple of 32):
 *   q [O, I/2] u8, s [O, I/32] u8 -> out [O, I] f32, value e2m1(code) * 2^(s-127).
 * Exact wherever the value is a finite f32 (scale bytes 0..252 always; above that
 * large codes overflow to +-inf); scale byte 255 gives NaN; code 8 gives -0. */
k3moe_status k3moe_dequant_mxfp4(const uint8_t* q, const uint8_t* s, int32_t O, int32_t I, float* out,
                                 void* stream);

/* Counting-sort permutation of routed slots (the chunk expert union) as the
 * forward pass builds it, exposed for checking.  ids [T, K] int32 in;
 * counts [E], offsets [E+1], slot_of [T*K] (flat t*K+k indices grouped by expert
 * ascending, (t, k) ascending inside an expert), uniq [E] (experts with a nonzero
 * count, ascending; entries past n_uniq are unspecified) and n_uniq [1], all int32
 * device outputs.  Same workspace rule as k3moe_forward. */
k3moe_status k3moe_permute(const k3moe_dims* dims, int32_t T, const int32_t* ids, int32_t* counts,
                           int32_t* offsets, int32_t* slot_of, int32_t* uniq, int32_t* n_uniq, void* ws,
                           size_t ws_bytes, void* stream);

/* Reads the device status word of the last call that used `ws` (K3MOE_DEV_* bits)
 * into *host_out.  ws = NULL reads the status word of the last
 * k3moe_forward_noalloc call on the current device.  Synchronises `stream`. */
k3moe_status k3moe_device_status(const void* ws, uint32_t* host_out, void* stream);

/* ---- Shared experts beside the routed block (colibri PR #684, engine commit: "2 fused
 * shared experts"; colibri PR #676, architecture bullets: SiTU-GLU).  Two SiTU-GLU experts
 * on the hidden width H, fused along the intermediate dimension into one of width inter_s
 * (the pages give no width; at K3 shapes each is read as a routed expert's 3072, inter_s
 * = 6144):
 *   g = x . Wgu[0:Is]^T,  u = x . Wgu[Is:2Is]^T  (fp32 accumulation),
 *   h = bf16(SiTU(g, u)),  out[t] += h . Wdn^T   (fp32).
 * The block's output is the routed output plus this: call it after k3moe_forward on the
 * same stream with the same out (or on a zeroed buffer of its own).
 *   x          [T, H] bf16, device, 16-byte aligned
 *   w_gate_up  [2 inter_s, H] bf16 (gate rows first, then up rows), device
 *   w_down     [H, inter_s] bf16, device
 *   out        [T, H] f32, device, read and written (accumulated into)
 *   ws         device workspace of k3moe_shared_workspace_bytes(dims, T, inter_s) bytes
 * inter_s must be a positive multiple of 64 (ERR_SHAPE otherwise).  Below
 * k3moe_tc_min_tokens tokens the products run on the weight-streaming GEMVs, from it on
 * the tcgen05 GEMMs.  Status word at the start of ws (k3moe_device_status). */
size_t k3moe_shared_workspace_bytes(const k3moe_dims* dims, int32_t T, int32_t inter_s);
k3moe_status k3moe_shared_forward(const k3moe_dims* dims, int32_t T, int32_t inter_s, const uint16_t* x,
                                  const uint16_t* w_gate_up, const uint16_t* w_down, float* out, void* ws,
                                  size_t ws_bytes, void* stream);

/* Token count from which k3moe_forward (and k3moe_route) run the projections and the
 * experts on the tensor-core GEMMs instead of the weight-streaming GEMVs (default 9, the
 * crossover measured on GB300 at K3 shapes: 8 random tokens 523 us on the GEMVs against
 * 712 us, 9 tokens 836 us against 786 us).  Process-wide: it changes the workspace size
 * and the launch sequence of every later call, so set it before sizing workspaces and with
 * no call in flight.  Returns the previous value, or -1 for t < 1 (nothing changed).  A
 * tuning control for measuring the crossover; the pages have no counterpart. */
int32_t k3moe_set_tc_min_tokens(int32_t t);
/* The current value of that token count. */
int32_t k3moe_tc_min_tokens(void);

/* Operand form of the exact tensor-core expert GEMMs (act_mxfp8 = 0, T >=
 * k3moe_tc_min_tokens), by token count.  Below t tokens (default 2^30: every count; on
 * GB300 at K3 shapes the split form measured faster from 9 to 8192 tokens, e.g. the 4096-
 * token forward 4.85 ms against 5.78 ms) the bf16 activations z and h are each split into two
 * MXFP8 terms, x = hi + lo (hi: E4M3 at the smallest power-of-two scale per 32 elements
 * that keeps the group's largest within 448; lo: the residual x - hi at a scale 2^-4 of
 * hi's), which holds every element within 2^14 of its group's largest exactly and the rest
 * to within 2^-21 of the group's largest; two block-scaled MMAs per k-block then read the
 * E2M1 weights and E8M0 scales as stored (E2M1 x E4M3 products are exact), so no weight
 * decode runs on the SMs.  From t tokens on (and for latent or inter < 512) the SMs decode
 * the weights exactly to bf16 and the MMAs read the bf16 activations.  t = 0: never split.
 * Process-wide like k3moe_set_tc_min_tokens (it changes the workspace size): set it before
 * sizing workspaces, with no call in flight.  Returns the previous value, or -1 for t < 0
 * (nothing changed). */
int32_t k3moe_set_tc_split_max_tokens(int32_t t);
/* The current value of that token bound. */
int32_t k3moe_tc_split_max_tokens(void);

/* Self-test of the device-side bounded waits (the pages have no counterpart; it checks
 * the library's own failure reporting): one small kernel waits on an mbarrier that nothing
 * completes, once with a limit of `limit_cycles` clock cycles (1 .. 2^32) and once with the
 * kernels' own limit, left early through the abort flag that the first wait sets.  The
 * kernel returns normally and sets K3MOE_DEV_TIMEOUT in the status word at the start of
 * `ws` (>= 256 bytes, 16-byte aligned), read with k3moe_device_status(ws, ...).  Nothing
 * faults, traps or hangs; the wait lasts about limit_cycles plus up to ~0.5 ms. */
k3moe_status k3moe_selftest_wait_timeout(void* ws, size_t ws_bytes, int64_t limit_cycles, void* stream);

/* Intermediate tensors of the last k3moe_forward that used `ws`, for inspection:
 * 0 = z [T, L] bf16, 1 = yhat [T, L] bf16, 2 = y [T, L] f32 (combined, before the
 * norm), 3 = logits [T, E] f32, 4 = h [T*K, I] in expert-sorted slot order (on the
 * weight-decode tensor-core path: bf16 with the 8 elements of each group stored in the
 * order 0, 4, 1, 5, 2, 6, 3, 7; on the split form: bf16 in natural order; on the
 * weight-streaming GEMVs: f16 holding h * 2^8; on the MXFP8 variant: see 8), 5 = o
 * [T*K, L] f32 in expert-sorted slot order.  When the expert
 * GEMMs read MXFP8 rows (the act_mxfp8 variant: one term; the exact split form: two terms,
 * hi rows then lo rows), 6 = the z codes [terms][T*K][L] E4M3 in slot order, 7 = their
 * E8M0 scale bytes, 8 = the h codes [terms][T*K][I], 9 = their scale bytes; NULL
 * otherwise.  Scale bytes are stored k-block-major over the terms * T*K rows: the bytes of
 * row r for the 32-element groups 4w .. 4w+3 form 32-bit word w * rows + r.  Returns a device pointer inside ws, or NULL. */
void* k3moe_workspace_view(const k3moe_dims* dims, int32_t T, void* ws, int32_t which);

/* Static text for a status code. */
const char* k3moe_status_str(k3moe_status st);

/* ABI version of this header (increments on incompatible change). */
int32_t k3moe_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* K3MOE_H */

"""GPU parity of the low-precision-activation variant (k3moe_dims.act_mxfp8 = 1): MXFP8
activations into block-scaled tcgen05 MMAs on the stored MXFP4 weights (colibri PR #676,
"What's in the commits" item 7; colibri PR #684, quant.h commit: per-32-group quantized
activations), against the oracle's variant mode.

- The MXFP8 codes and scale bytes of z are compared bit for bit with the oracle's
  quantization of the GPU's own z (a quantized code is an integer decided in fp32 on the
  GPU and fp64 in the oracle from the same bf16 value: the scaling by a power of two is
  exact in both and the rounding to E4M3 is to nearest even in both).
- The grouped GEMMs' own outputs per slot: o against the fp64 product of the down matrix
  with the GPU's own MXFP8 h (only fp32 accumulation differs); h codes against the oracle
  quantizing its own bf16 h from the GPU's quantized z.  A bf16 rounding flip of h (fp32
  vs fp64 accumulation next to a boundary, as on the exact path) changes the E4M3 code
  only where it also crosses an E4M3 rounding boundary.
- The block output against the variant oracle.  The GPU and the oracle differ by the
  same fp32-accumulation cascade as on the exact path (bf16 rounding flips of z and h),
  but a flip now also moves the E4M3 code when it crosses an E4M3 rounding boundary:
  with 3 mantissa bits against bf16's 7, that happens for about 1 flip in 2^4, and moves
  the element by 2^4 bf16 units, i.e. 2^4 times the perturbation variance per flip of
  the exact path, about 4 times its rel-L2.  The bars are 4 times the exact path's.
"""
import dataclasses

import numpy as np
import pytest

import oracle
from datagen import configs as C
from tests._harness import REL_L2_BAR, oracle_forward, oracle_route, rel_l2
from tests.test_gpu_parity import PER_TOKEN_BAR, Layer, _slot_map, _ws_view, scales_by_row  # noqa: F401

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

MX_PREFILL = dataclasses.replace(C.PREFILL, act_mxfp8=1)
MX_BAR, MX_PER_TOKEN_BAR = 4 * REL_L2_BAR, 4 * PER_TOKEN_BAR


@pytest.fixture(scope="module")
def k3():
    import __graft_entry__ as g
    g.build()
    import mxfp4_routed_expert_latentmoe_gb300 as mod
    torch.cuda.set_device(0)
    return mod


@pytest.fixture(scope="module")
def mx_prefill(k3):
    L = Layer(k3, MX_PREFILL)
    yield L
    del L
    torch.cuda.empty_cache()


def _codes_view(k3, L, ws, which, n):
    ptr = k3.workspace_view(L.d, L.cfg.T, ws, which)
    assert ptr != 0
    off = ptr - ws.data_ptr()
    return ws[off: off + n].cpu().numpy()


E4M3 = np.array([oracle.e4m3(c) for c in range(256)])


def _mx_values(codes, scales):
    return E4M3[codes] * np.exp2(np.repeat(scales.astype(np.float64), 32, axis=-1) - 127)


def test_variant_needs_the_grouped_gemm_shapes(k3):
    import ctypes
    L = k3.lib()
    d = k3.dims(**dict(C.TINY.dims, act_mxfp8=1))  # latent 128: too short for the variant
    assert L.k3moe_workspace_bytes(ctypes.byref(d), 1) == 0
    d = k3.dims(**dict(C.PREFILL.dims, act_mxfp8=2))
    assert L.k3moe_workspace_bytes(ctypes.byref(d), 1) == 0


@pytest.mark.parametrize("T", [256, 300])
def test_variant_quantized_z_and_expert_slots(k3, mx_prefill, T):
    cfg = MX_PREFILL.with_tokens(T, x_seed=31 + T)
    L = mx_prefill.with_tokens(k3, cfg)
    got, ids, w, ws = L.forward(k3)
    assert k3.device_status(ws) == 0
    rids, rw, _, _ = oracle_route(cfg)
    assert np.array_equal(ids, rids)
    Lt, I, K = cfg.latent, cfg.inter, cfg.top_k
    slots = T * K
    z = _ws_view(k3, L, ws, 0, T, T * Lt, torch.bfloat16).reshape(T, Lt)
    zc = _codes_view(k3, L, ws, 6, slots * Lt).reshape(slots, Lt)
    zs = scales_by_row(_codes_view(k3, L, ws, 7, slots * Lt // 32), slots, Lt // 32)
    s_exp, s_tok, offs = _slot_map(ids, cfg.n_experts)
    rc, rs = oracle.mxfp8_quant(z[s_tok])
    assert np.array_equal(zs, rs)
    assert np.array_equal(zc, rc)
    # per slot, three experts: the most used, the least used and one in between
    hc = _codes_view(k3, L, ws, 8, slots * I).reshape(slots, I)
    hs = scales_by_row(_codes_view(k3, L, ws, 9, slots * I // 32), slots, I // 32)
    o_all = _ws_view(k3, L, ws, 5, T, slots * Lt, torch.float32).reshape(slots, Lt)
    counts = np.bincount(ids.ravel(), minlength=cfg.n_experts)
    used = np.nonzero(counts)[0]
    experts = [int(np.argmax(counts)), int(used[np.argmin(counts[used])]), int(used[len(used) // 2])]
    z8 = _mx_values(zc, zs)
    h8 = _mx_values(hc, hs)
    code_diff = total = 0
    worst_h = worst_o = 0.0
    for e in experts:
        t = C.expert_tensors(cfg, e)
        Wg = oracle.dequant(t["gate_q"], t["gate_s"])
        Wu = oracle.dequant(t["up_q"], t["up_s"])
        W2 = oracle.dequant(t["down_q"], t["down_s"])
        sl = np.arange(offs[e], offs[e + 1])
        zq = z8[sl]
        href = oracle.mxfp8_round(oracle.round_bf16(oracle.situ(zq @ Wg.T, zq @ Wu.T)))
        code_diff += int(np.count_nonzero(h8[sl] != href))
        total += href.size
        oref = h8[sl] @ W2.T
        for i in range(len(sl)):
            worst_h = max(worst_h, rel_l2(h8[sl[i]], href[i]))
            worst_o = max(worst_o, rel_l2(o_all[sl[i]], oref[i]))
    print(f"T={T}: h code differences {code_diff}/{total}, worst h {worst_h:.2e}, worst o {worst_o:.2e}")
    assert code_diff <= 0.002 * total, (code_diff, total)
    assert worst_h <= 2e-2, worst_h
    assert worst_o <= 1e-5, worst_o


@pytest.mark.parametrize("T,n_rows", [(256, 16), (4096, 48)])
def test_variant_forward_against_variant_oracle(k3, mx_prefill, T, n_rows):
    cfg = MX_PREFILL if T == MX_PREFILL.T else MX_PREFILL.with_tokens(T, x_seed=41)
    L = mx_prefill if T == MX_PREFILL.T else mx_prefill.with_tokens(k3, cfg)
    got, ids, w, ws = L.forward(k3)
    assert k3.device_status(ws) == 0
    rids, rw, _, _ = oracle_route(cfg)
    assert np.array_equal(ids, rids)
    rng = np.random.default_rng(T)
    rows = sorted({0, T - 1} | set(int(r) for r in rng.choice(T, n_rows - 2, replace=False)))
    ref = oracle_forward(cfg, token_rows=rows)
    pooled = rel_l2(got[rows], ref["out"])
    per = [rel_l2(got[r], ref["out"][i]) for i, r in enumerate(rows)]
    exact = oracle_forward(dataclasses.replace(cfg, act_mxfp8=0), token_rows=rows)
    cost = rel_l2(ref["out"], exact["out"])
    print(f"T={T} MXFP8 variant: rel-L2 vs variant oracle {pooled:.3e} (worst token {max(per):.3e}); "
          f"variant oracle vs exact oracle {cost:.3e}")
    assert pooled <= MX_BAR, pooled
    assert max(per) <= MX_PER_TOKEN_BAR, max(per)


def test_variant_with_top_p_pruning(k3, mx_prefill):
    """The variant on the tensor-core path with K3_TOPP pruning (slots with id -1 take no
    part in the batches): ids and weights as the oracle's, outputs within the variant's bars."""
    cfg = dataclasses.replace(MX_PREFILL.with_tokens(300, x_seed=61), top_p=0.5)
    L = mx_prefill.with_tokens(k3, cfg)
    L.d = k3.dims(**cfg.dims)
    got, ids, w, ws = L.forward(k3)
    assert k3.device_status(ws) == 0
    assert (ids == -1).any()
    rows = [0, 1, 150, 299]
    ref = oracle_forward(cfg, token_rows=rows)
    assert np.array_equal(ids[rows], ref["ids"])
    assert np.allclose(w[rows], ref["w"], rtol=0, atol=2e-6)
    pooled = rel_l2(got[rows], ref["out"])
    print(f"MXFP8 variant with top-p 0.5 at T=300: rel-L2 {pooled:.3e}")
    assert pooled <= MX_BAR

"""GPU: the exact split form of the tensor-core expert GEMMs (below
k3moe_tc_split_max_tokens tokens).  The bf16 activations z and h reach the block-scaled MMAs as two MXFP8 terms
x = hi + lo per 32-element group: hi at the smallest E8M0 scale that keeps the group's
largest magnitude within 448 (the E4M3 maximum), lo -- the residual -- at that scale times
2^-4.  Checked on the terms the library wrote, against the definitions restated here:
the two scale rules; hi + lo == x exactly for every element within 2^14 of its group's
largest and within 2^-21 of the group's largest for the others (the error bound stated in
the library's header), for z (the gather's terms) and h (the terms the pass between the two
GEMMs makes from the gate/up GEMM's bf16 h).  The products with the terms are those of the
exact path, which the parity tests check through the outputs."""
import dataclasses

import numpy as np
import pytest

from datagen import configs as C
from tests._harness import smallest_scale_within_448
from tests.test_gpu_parity import Layer, _slot_map, _ws_view, split_terms

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def k3():
    import __graft_entry__ as g
    g.build()
    import mxfp4_routed_expert_latentmoe_gb300 as mod
    torch.cuda.set_device(0)
    return mod


@pytest.fixture(scope="module")
def prefill(k3):
    L = Layer(k3, C.PREFILL)
    yield L
    del L
    torch.cuda.empty_cache()


def _check_terms(x, hi, lo, s_hi, s_lo, what):
    rows, width = x.shape
    amax = np.abs(x).reshape(rows, width // 32, 32).max(-1)
    assert np.array_equal(s_hi.astype(np.int64), smallest_scale_within_448(amax)), what
    assert np.array_equal(s_lo.astype(np.int64), np.maximum(s_hi.astype(np.int64) - 4, 0)), what
    rec = hi + lo
    A = np.repeat(amax, 32, axis=1)
    inside = np.abs(x) >= A * 2.0 ** -14
    assert np.array_equal(rec[inside], x[inside]), what
    assert np.all(np.abs(rec - x)[~inside] <= A[~inside] * 2.0 ** -21), what
    return float(np.mean(~inside))


@pytest.mark.parametrize("T", [9, 300])
def test_split_terms_hold_z_and_h(k3, prefill, T):
    """9 tokens (the smallest tensor-core batch) and 300 (ragged tiles): z's terms against
    the GPU's own z rows in slot order, h's terms against the GPU's own bf16 h (the grouped
    GEMM's h is compared with the oracle's by the parity tests)."""
    cfg = C.PREFILL.with_tokens(T, x_seed=41 + T)
    L = prefill.with_tokens(k3, cfg)
    assert k3.tc_min_tokens() <= T < k3.tc_split_max_tokens()
    got, ids, w, ws = L.forward(k3)
    assert k3.device_status(ws) == 0
    Lt, I, K = cfg.latent, cfg.inter, cfg.top_k
    slots = T * K
    z = _ws_view(k3, L, ws, 0, T, T * Lt, torch.bfloat16).reshape(T, Lt)
    _, s_tok, _ = _slot_map(ids, cfg.n_experts)
    hi, lo, s_hi, s_lo = split_terms(k3, L, ws, 6, 7, slots, Lt)
    frac_z = _check_terms(z[s_tok].astype(np.float64), hi, lo, s_hi, s_lo, "z")
    h = _ws_view(k3, L, ws, 4, T, slots * I, torch.bfloat16).reshape(slots, I).astype(np.float64)
    hi, lo, s_hi, s_lo = split_terms(k3, L, ws, 8, 9, slots, I)
    frac_h = _check_terms(h, hi, lo, s_hi, s_lo, "h")
    print(f"T={T}: elements below 2^-14 of their group's largest: z {frac_z:.1e}, h {frac_h:.1e}")


# a layer with other widths: latent 768 (gate/up contraction of 6 stages of 128, a count
# that is not a multiple of 4), inter 512 (the down contraction at the 4-stage minimum),
# hidden 1024, 32 experts, top-4
MID = C.MID


@pytest.mark.parametrize("split", [1, 0])
def test_both_forms_on_other_widths(k3, split):
    """The tensor-core expert path on a layer of other widths, in both operand forms, against
    the oracle for every token (ids bit-exact, outputs within the bars); the split form's
    terms of z and h against the GPU's own z and h as above."""
    from tests.test_gpu_parity import PER_TOKEN_BAR, _check_block, tc_form
    from tests._harness import oracle_forward, rel_l2
    L = Layer(k3, MID)
    with tc_form(k3, split):
        assert MID.T >= k3.tc_min_tokens()
        got, ids, w, ws = L.forward(k3)
        assert k3.device_status(ws) == 0
        ref = oracle_forward(MID)
        r = _check_block(got, ids, w, ref)
        worst = max(rel_l2(got[t], ref["out"][t]) for t in range(MID.T))
        assert worst <= PER_TOKEN_BAR, worst
        if split:
            T, Lt, I, K = MID.T, MID.latent, MID.inter, MID.top_k
            slots = T * K
            z = _ws_view(k3, L, ws, 0, T, T * Lt, torch.bfloat16).reshape(T, Lt)
            _, s_tok, _ = _slot_map(ids, MID.n_experts)
            hi, lo, s_hi, s_lo = split_terms(k3, L, ws, 6, 7, slots, Lt)
            _check_terms(z[s_tok].astype(np.float64), hi, lo, s_hi, s_lo, "z")
            h = _ws_view(k3, L, ws, 4, T, slots * I, torch.bfloat16).reshape(slots, I).astype(np.float64)
            hi, lo, s_hi, s_lo = split_terms(k3, L, ws, 8, 9, slots, I)
            _check_terms(h, hi, lo, s_hi, s_lo, "h")
    print(f"mid widths, split {split}: rel-L2 {r:.2e}, worst token {worst:.2e}")


def test_pool_aligned_to_16_bytes_only(k3):
    """A pool whose tensors start 16 bytes past 32-byte boundaries (the same bytes, copied
    16 bytes further on): the split form's 4-bit tensor copies need 32-byte aligned packed
    tensors, so it reports K3MOE_DEV_ALIGN and abandons the call (no copy issued); the
    weight-decode form, which needs 16, runs it and gives bit for bit what it gives on the
    aligned pool."""
    from tests.test_gpu_parity import tc_form
    L = Layer(k3, MID)
    n = L.pool.numel()
    raw = torch.zeros(n + 64, dtype=torch.uint8, device="cuda")
    start = (-raw.data_ptr()) % 32 + 16  # 16 bytes past a 32-byte boundary
    shifted = raw[start:start + n]
    shifted.copy_(L.pool)
    assert shifted.data_ptr() % 32 == 16
    S = Layer.__new__(Layer)
    S.cfg, S.d, S.t = L.cfg, L.d, L.t
    S.pool, S.eb, S.offs = shifted, L.eb, L.offs
    S.tables = k3.ExpertTables.from_pool(shifted, L.eb, L.offs)
    with tc_form(k3, 1):
        _, _, _, ws = S.forward(k3)
        assert k3.device_status(ws) & k3.DEV_ALIGN
    with tc_form(k3, 0):
        got_s, ids_s, _, ws = S.forward(k3)
        assert k3.device_status(ws) == 0
        got_a, ids_a, _, ws = L.forward(k3)
        assert k3.device_status(ws) == 0
    assert np.array_equal(ids_s, ids_a)
    assert np.array_equal(got_s.view(np.uint32), got_a.view(np.uint32))


# contractions of 6 stages (latent and inter 768) so that the small-batch layouts apply;
# 32 experts, top-4: at 200 and 300 tokens experts get ~25 and ~38 tokens, more than the
# 16- and 32-token batches of the layouts those counts use (several batches per expert)
MID768 = dataclasses.replace(C.MID, name="mid768", inter=768, seed=5)


@pytest.mark.parametrize("T", [200, 300])
def test_small_batch_layouts_split_experts_over_batches(k3, T):
    """The block-scaled GEMMs' small-batch layouts (16 tokens a batch up to 256 tokens, 32
    up to 512) on experts that receive more tokens than a batch holds: every token of the
    split form against the oracle."""
    from tests.test_gpu_parity import PER_TOKEN_BAR, _check_block
    from tests._harness import oracle_forward, rel_l2
    cfg = MID768.with_tokens(T, x_seed=50 + T)
    L = Layer(k3, cfg)
    got, ids, w, ws = L.forward(k3)
    assert k3.device_status(ws) == 0
    counts = np.bincount(ids.ravel(), minlength=cfg.n_experts)
    assert counts.max() > (16 if T <= 256 else 32)  # some expert spans several batches
    ref = oracle_forward(cfg)
    r = _check_block(got, ids, w, ref)
    worst = max(rel_l2(got[t], ref["out"][t]) for t in range(T))
    assert worst <= PER_TOKEN_BAR, worst
    print(f"T={T}: max tokens per expert {counts.max()}, rel-L2 {r:.2e}, worst token {worst:.2e}")

"""GPU parity of the shared experts beside the routed block (colibri PR #684, engine
commit: "2 fused shared experts"): k3moe_shared_forward accumulates into out, compared
with the oracle's fused shared experts.  Both the weight-streaming path (below the
tensor-core threshold) and the tcgen05 path, at the K3 hidden width with the fused width
2 x 3072; the bars are the routed block's (the same bf16 rounding of h, the same fp32 vs
fp64 accumulation)."""
import numpy as np
import pytest

import oracle
from datagen import configs as C
from tests._harness import REL_L2_BAR, rel_l2
from tests.test_gpu_parity import PER_TOKEN_BAR

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
def shared_w():
    from datagen import device as D
    W = C.shared_weights(C.DECODE)
    return W, D.bf16_tensor(W["wgu"], "cuda"), D.bf16_tensor(W["wdn"], "cuda")


@pytest.mark.parametrize("T", [1, 5, 16, 300])
def test_shared_forward_accumulates_the_fused_experts(k3, shared_w, T):
    from datagen import device as D
    W, wgu, wdn = shared_w
    cfg = C.DECODE.with_tokens(T, x_seed=51 + T)
    d = k3.dims(**cfg.dims)
    xb = C.layer_x(cfg)
    x = D.bf16_tensor(xb, "cuda")
    base = torch.randn(T, cfg.hidden, generator=torch.Generator().manual_seed(T)).to("cuda")
    out = base.clone()
    ws = torch.empty(k3.shared_workspace_bytes(d, T, C.SHARED_INTER), dtype=torch.uint8, device="cuda")
    k3.shared_forward(d, x, wgu, wdn, out, ws)
    torch.cuda.synchronize()
    assert k3.device_status(ws) == 0
    got = (out - base).double().cpu().numpy()
    rows = list(range(T)) if T <= 16 else sorted({0, 127, 128, T - 1} | set(range(5, T, 37)))
    _, ref = oracle.shared(oracle.dims(**cfg.dims), np.ascontiguousarray(xb[rows]), W["wgu"], W["wdn"], True)
    pooled = rel_l2(got[rows], ref)
    per = [rel_l2(got[r], ref[i]) for i, r in enumerate(rows)]
    path = "tensor-core" if T >= k3.tc_min_tokens() else "GEMV"
    print(f"shared experts T={T} ({path}): rel-L2 {pooled:.3e}, worst token {max(per):.3e}")
    assert pooled <= REL_L2_BAR, pooled
    assert max(per) <= PER_TOKEN_BAR, max(per)


def test_shared_forward_edge_cases(k3, shared_w):
    """Zero tokens launch nothing; two calls add the experts twice (the accumulation is exact
    in its order: out + s + s); the first tensor-core batch (T = the threshold) and the last
    weight-streaming one (T = threshold - 1) agree with the oracle."""
    from datagen import device as D
    W, wgu, wdn = shared_w
    d = k3.dims(**C.DECODE.dims)
    ws = torch.empty(k3.shared_workspace_bytes(d, 16, C.SHARED_INTER), dtype=torch.uint8, device="cuda")
    out = torch.zeros(0, C.DECODE.hidden, dtype=torch.float32, device="cuda")
    k3.shared_forward(d, torch.zeros(0, C.DECODE.hidden, dtype=torch.bfloat16, device="cuda"), wgu, wdn, out, ws)
    t0 = k3.tc_min_tokens()
    for T in (t0 - 1, t0):
        cfg = C.DECODE.with_tokens(T, x_seed=71 + T)
        xb = C.layer_x(cfg)
        x = D.bf16_tensor(xb, "cuda")
        out = torch.zeros(T, cfg.hidden, dtype=torch.float32, device="cuda")
        k3.shared_forward(d, x, wgu, wdn, out, ws)
        once = out.clone()
        k3.shared_forward(d, x, wgu, wdn, out, ws)
        torch.cuda.synchronize()
        assert k3.device_status(ws) == 0
        assert torch.equal(out, once + once)
        _, ref = oracle.shared(oracle.dims(**cfg.dims), xb, W["wgu"], W["wdn"], True)
        got = once.double().cpu().numpy()
        print(f"shared experts T={T}: rel-L2 {rel_l2(got, ref):.3e}")
        assert rel_l2(got, ref) <= REL_L2_BAR
        assert max(rel_l2(got[i], ref[i]) for i in range(T)) <= PER_TOKEN_BAR

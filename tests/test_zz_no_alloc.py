"""The allocation-free forward (k3moe_forward_noalloc) against k3moe_forward.

Some callers cannot call cudaMalloc -- for example code embedded in a host
framework that owns every device allocation -- so the library offers one entry
point that takes no workspace and uses its own fixed device scratch instead.  This
test calls it through the C ABI twice in a row (the second call reuses the scratch
the first one left behind) and checks both results against the workspace-taking
entry point on the same inputs: the two run the same kernels with the same launch
shapes, so ids, weights and outputs must be bit-identical; the device status word
of each call (read with k3moe_device_status(NULL, ...)) must be clear; and the
8-token chunk is also checked against the fp64 oracle.
It sits in its own file, collected last, so that a run stopping at the first
failure has run every other test before it.
"""
import numpy as np
import pytest

from datagen import configs as C
from tests._harness import REL_L2_BAR, oracle_forward, rel_l2

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def k3():
    import __graft_entry__ as g
    g.build()
    import mxfp4_routed_expert_latentmoe_gb300 as mod
    torch.cuda.set_device(0)
    return mod


@pytest.mark.parametrize("cfg", [C.TINY, C.DECODE, C.CHUNK.with_tokens(8)], ids=["tiny", "decode", "chunk8"])
def test_noalloc_forward_matches_workspace_forward(k3, cfg):
    from datagen import device as D
    d = k3.dims(**cfg.dims)
    t = D.layer_tensors(cfg, "cuda")
    pool, eb, offs = D.expert_pool(cfg, "cuda")
    tables = k3.ExpertTables.from_pool(pool, eb, offs)
    T = cfg.T
    args = (d, t["x"], t["wr"], t["bias"], t["wd"], t["wu"], t["gamma"], tables)

    def outputs():
        return (torch.empty(T, cfg.hidden, dtype=torch.float32, device="cuda"),
                torch.empty(T, cfg.top_k, dtype=torch.int32, device="cuda"),
                torch.empty(T, cfg.top_k, dtype=torch.float32, device="cuda"))

    ref_out, ref_ids, ref_w = outputs()
    ws = torch.empty(k3.workspace_bytes(d, T), dtype=torch.uint8, device="cuda")
    k3.forward(*args, ref_out, ws, ref_ids, ref_w)
    torch.cuda.synchronize()
    assert k3.device_status(ws) == 0
    ref = ref_out.cpu().numpy()
    for call in range(2):
        out, ids, w = outputs()
        k3.forward_noalloc(*args, out, ids, w)
        torch.cuda.synchronize()
        assert k3.device_status(None) == 0, call
        assert np.array_equal(ids.cpu().numpy(), ref_ids.cpu().numpy()), call
        assert np.array_equal(w.cpu().numpy().view(np.uint32), ref_w.cpu().numpy().view(np.uint32)), call
        assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32)), call
    if cfg.name == "chunk":
        o = oracle_forward(cfg)
        assert np.array_equal(ids.cpu().numpy(), o["ids"])
        assert rel_l2(out.cpu().numpy(), o["out"]) <= REL_L2_BAR


def test_noalloc_rejects_calls_beyond_its_scratch(k3):
    import ctypes
    d = k3.dims(**C.DECODE.dims)
    assert k3.workspace_bytes(d, 9) > k3.NOALLOC_SCRATCH_BYTES >= k3.workspace_bytes(d, 8)
    v = ctypes.c_void_p(16)
    L = k3.lib()
    ex = k3.ExpertsC(16, 16, 16, 16, 16, 16)
    for T in (9, 4096):
        rc = L.k3moe_forward_noalloc(ctypes.byref(d), T, v, v, v, v, v, v, ctypes.byref(ex), v, None, None, None)
        assert rc == 4, T  # K3MOE_ERR_WORKSPACE: needs more scratch than the fixed array holds

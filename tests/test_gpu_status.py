"""Device-detected conditions, made to happen on purpose without faulting or hanging the
GPU: a bounded wait that runs out, an expert id outside [0, E) in the permutation, exact
ties of biased scores at the top-K boundary, and a tie cluster longer than the near-tie
refinement window.  Each checks the status bit the header documents and, where the result
is still defined, the ids against the oracle (ties go to the lower id)."""
import dataclasses

import numpy as np
import pytest

import oracle
from datagen import configs as C
from tests._harness import REL_L2_BAR, oracle_dims, rel_l2

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def k3():
    import __graft_entry__ as g
    g.build()
    import mxfp4_routed_expert_latentmoe_gb300 as mod
    torch.cuda.set_device(0)
    return mod


def test_bounded_wait_runs_out_and_reports_timeout(k3):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    k3.selftest_wait_timeout(ws, 1 << 20)
    torch.cuda.synchronize()
    assert k3.device_status(ws) & k3.DEV_TIMEOUT
    # the context is still usable: a normal call afterwards succeeds and reports nothing
    from datagen import device as D
    cfg = C.TINY
    d = k3.dims(**cfg.dims)
    t = D.layer_tensors(cfg, "cuda")
    pool, eb, offs = D.expert_pool(cfg, "cuda")
    tables = k3.ExpertTables.from_pool(pool, eb, offs)
    out = torch.empty(cfg.T, cfg.hidden, dtype=torch.float32, device="cuda")
    ws2 = torch.empty(k3.workspace_bytes(d, cfg.T), dtype=torch.uint8, device="cuda")
    k3.forward(d, t["x"], t["wr"], t["bias"], t["wd"], t["wu"], t["gamma"], tables, out, ws2)
    torch.cuda.synchronize()
    assert k3.device_status(ws2) == 0


@pytest.mark.parametrize("T,K,E", [(3, 2, 8), (4096, 16, 896)])
def test_permute_reports_an_expert_id_out_of_range(k3, T, K, E):
    rng = np.random.default_rng(3)
    ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    ids[T // 2, 0] = E  # one id past the last expert
    d = k3.dims(64, 64, E, K, 64)
    dev = lambda n: torch.empty(n, dtype=torch.int32, device="cuda")
    ws = torch.empty(k3.workspace_bytes(d, T), dtype=torch.uint8, device="cuda")
    k3.permute(d, torch.from_numpy(ids).cuda(), dev(E), dev(E + 1), dev(T * K), dev(E), dev(1), ws)
    torch.cuda.synchronize()
    assert k3.device_status(ws) & k3.DEV_BAD_ID


# ------------------------------------------------------------------------------ exact ties
TIE_CFG = dataclasses.replace(C.DECODE, name="ties", n_experts=64, x_seed=5)


@pytest.fixture(scope="module")
def tie_layer(k3):
    from datagen import device as D
    cfg = TIE_CFG
    pool, eb, offs = D.expert_pool(cfg, "cuda")
    return cfg, k3.ExpertTables.from_pool(pool, eb, offs), pool


def _with_copied_rows(cfg, src, dsts):
    """Router weight and bias with the row (and bias) of expert `src` copied to `dsts`:
    those experts get exactly equal biased scores for every token."""
    W = C.layer_weights(cfg)
    wr, bias = W["wr"].copy(), W["bias"].copy()
    for e in dsts:
        wr[e] = wr[src]
        bias[e] = bias[src]
    return W, wr, bias


def _forward_ids(k3, cfg, tables, wr, bias):
    from datagen import device as D
    d = k3.dims(**cfg.dims)
    t = D.layer_tensors(cfg, "cuda")
    t["wr"] = D.bf16_tensor(wr, "cuda")
    t["bias"] = torch.from_numpy(bias).cuda()
    out = torch.empty(cfg.T, cfg.hidden, dtype=torch.float32, device="cuda")
    ids = torch.empty(cfg.T, cfg.top_k, dtype=torch.int32, device="cuda")
    w = torch.empty(cfg.T, cfg.top_k, dtype=torch.float32, device="cuda")
    ws = torch.empty(k3.workspace_bytes(d, cfg.T), dtype=torch.uint8, device="cuda")
    k3.forward(d, t["x"], t["wr"], t["bias"], t["wd"], t["wu"], t["gamma"], tables, out, ws, ids, w)
    rids = torch.empty_like(ids)
    rw = torch.empty_like(w)
    ws_r = torch.empty(k3.workspace_bytes(d, cfg.T), dtype=torch.uint8, device="cuda")
    k3.route(d, t["x"], t["wr"], t["bias"], rids, rw, ws_r)
    torch.cuda.synchronize()
    return (out.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy(), k3.device_status(ws), rids.cpu().numpy(),
            k3.device_status(ws_r))


def test_exact_tie_at_the_top_k_boundary_goes_to_the_lower_id(k3, tie_layer):
    cfg, tables, _ = tie_layer
    K = cfg.top_k
    W = C.layer_weights(cfg)
    x = C.layer_x(cfg)
    d = oracle_dims(cfg)
    ids0, _, _, _ = oracle.route(d, x, W["wr"], W["bias"])
    order = list(ids0[0])
    a = order[K - 1]  # rank K
    rest = [e for e in range(cfg.n_experts) if e not in order]
    b = min(rest)     # an unselected expert, made to tie with rank K exactly
    _, wr, bias = _with_copied_rows(cfg, a, [b])
    rids, _, _, _ = oracle.route(d, x, wr, bias)
    assert min(a, b) in rids[0] and max(a, b) not in rids[0]
    out, ids, w, st, ids_r, st_r = _forward_ids(k3, cfg, tables, wr, bias)
    assert np.array_equal(ids, rids) and np.array_equal(ids_r, rids)
    assert st == 0 and st_r == 0
    ex = {int(e): C.expert_tensors(cfg, int(e)) for e in np.unique(rids)}
    ref = oracle.forward(d, x, wr, bias, W["wd"], W["wu"], W["gamma"], ex, True, 0)
    assert rel_l2(out, ref["out"]) <= REL_L2_BAR


def test_tie_cluster_longer_than_the_refinement_window_sets_the_flag(k3, tie_layer):
    """21 experts with exactly the score of rank 10: the cluster runs past the K + 8
    candidates the top-k refines, which the status word reports; the ids are still those of
    the exact ranking here (equal scores, lower ids first)."""
    cfg, tables, _ = tie_layer
    W = C.layer_weights(cfg)
    x = C.layer_x(cfg)
    d = oracle_dims(cfg)
    ids0, _, _, _ = oracle.route(d, x, W["wr"], W["bias"])
    order = list(ids0[0])
    a = order[9]
    dsts = [e for e in range(cfg.n_experts) if e not in order[:10]][:20]
    _, wr, bias = _with_copied_rows(cfg, a, dsts)
    rids, _, _, _ = oracle.route(d, x, wr, bias)
    out, ids, w, st, ids_r, st_r = _forward_ids(k3, cfg, tables, wr, bias)
    assert st & k3.DEV_TIE_WINDOW and st_r & k3.DEV_TIE_WINDOW
    assert np.array_equal(ids, rids) and np.array_equal(ids_r, rids)

"""Pins for the oracle's router, permutation, activation, norm, projections and whole
block (CPU only).  Each check compares the oracle with something other than itself:
closed forms, limits, invariants, brute force on tiny inputs, or numpy library
primitives in a different summation order."""
import dataclasses
import math
import os

import numpy as np
import pytest

import datagen
import oracle
from datagen import configs as C

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _minifloat_e2m1(code):
    sign = -1.0 if code & 8 else 1.0
    e, m = (code >> 1) & 3, code & 1
    return sign * (m * 0.5 if e == 0 else math.ldexp(1 + m / 2, e - 1))


E2M1 = np.array([_minifloat_e2m1(c) for c in range(16)])


def np_dequant(q, s):
    """Test-side decode: nibble split with numpy, E2M1 from the field definition."""
    lo = E2M1[q & 15]
    hi = E2M1[q >> 4]
    v = np.empty((q.shape[0], q.shape[1] * 2))
    v[:, 0::2], v[:, 1::2] = lo, hi
    return v * np.repeat(np.ldexp(1.0, s.astype(np.int64) - 127), 32, axis=1)


def bf16_round_datagen(a):
    return datagen.bf16_to_f64(datagen.bf16_bits(a))


# ------------------------------------------------------------------------------ rounding
def test_round_bf16_matches_independent_roundings():
    rng = np.random.default_rng(1)
    a = rng.standard_normal(200_000) * np.exp(rng.uniform(-30, 30, 200_000))
    # exact midpoints between adjacent bf16 values: ties must go to the even neighbour
    lo = datagen.bf16_to_f64(np.arange(0x3F80, 0x3FC0, dtype=np.uint16))
    mids = (lo[:-1] + lo[1:]) / 2
    a = np.concatenate([a, mids, -mids, [0.0, -0.0, 1e-40, 3.3e38, 3.4e38]])
    ours = oracle.round_bf16(a)
    assert np.array_equal(ours, bf16_round_datagen(a))
    even = datagen.bf16_to_f64(np.arange(0x3F80, 0x3FC0, 2, dtype=np.uint16))
    assert set(oracle.round_bf16(mids)) <= set(even)
    torch = pytest.importorskip("torch")
    f32 = a.astype(np.float32).astype(np.float64)
    t = torch.from_numpy(f32.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_bf16(f32), t)


# ------------------------------------------------------------------------------ SiTU
def test_situ_reduces_to_silu_times_u_for_small_arguments():
    rng = np.random.default_rng(2)
    g = rng.uniform(-0.05, 0.05, 5000)
    u = rng.uniform(-0.05, 0.05, 5000)
    silu_u = g / (1 + np.exp(-g)) * u
    # 4 tanh(g/4) = g (1 - g^2/48 + ...), 25 tanh(u/25) = u (1 - u^2/1875 + ...)
    bound = np.abs(silu_u) * (g ** 2 / 48 + u ** 2 / 1875) * 1.01 + 1e-300
    assert np.all(np.abs(oracle.situ(g, u) - silu_u) <= bound)


def test_situ_limits_zeros_and_symmetry():
    assert oracle.situ([60.0], [1e4])[0] == pytest.approx(100.0, rel=1e-12)  # 4 * 1 * 25
    assert oracle.situ([60.0], [-1e4])[0] == pytest.approx(-100.0, rel=1e-12)
    assert abs(oracle.situ([-60.0], [1e4])[0]) < 1e-20  # sigmoid(g) -> 0
    assert oracle.situ([0.0], [3.0])[0] == 0.0 and oracle.situ([2.0], [0.0])[0] == 0.0
    rng = np.random.default_rng(3)
    g, u = rng.normal(0, 5, 1000), rng.normal(0, 30, 1000)
    assert np.array_equal(oracle.situ(g, -u), -oracle.situ(g, u))  # odd in u
    # u -> infinity: SiTU / 25 -> 4 tanh(g/4) sigmoid(g); the betas printed on the pages
    consts = dict(l.split()[:2] for l in open(os.path.join(GOLDEN, "k3_layer_constants.txt")) if l[0] != "#")
    bg, bu = float(consts["situ_beta_gate"]), float(consts["situ_beta_up"])
    gg = np.linspace(-8, 8, 33)
    lim = oracle.situ(gg, np.full_like(gg, 1e6)) / bu
    assert np.allclose(lim, bg * np.tanh(gg / bg) / (1 + np.exp(-gg)), rtol=1e-13, atol=1e-300)


# ------------------------------------------------------------------------------ RMSNorm
def test_rmsnorm_closed_form_and_scale_invariance():
    L = 64
    gamma = np.linspace(0.5, 2.0, L).astype(np.float32)
    c = 3.0
    out = oracle.rmsnorm(np.full(L, c), gamma, 1e-6, False)
    assert np.allclose(out, gamma.astype(np.float64) * c / math.sqrt(c * c + 1e-6), rtol=1e-15)
    rng = np.random.default_rng(4)
    y = rng.normal(0, 40, L)
    a, b = oracle.rmsnorm(y, gamma, 0.0, False), oracle.rmsnorm(7.5 * y, gamma, 0.0, False)
    assert np.allclose(a, b, rtol=1e-14)
    assert np.mean((a / gamma.astype(np.float64)) ** 2) == pytest.approx(1.0, rel=1e-14)  # unit mean square
    spec = oracle.rmsnorm(y, gamma, 1e-6, True)
    assert np.array_equal(spec, bf16_round_datagen(oracle.rmsnorm(y, gamma, 1e-6, False)))


# ------------------------------------------------------------------------------ router
def _small_router(T=24, H=96, E=40, K=6, seed=5):
    d = oracle.dims(H, 32, E, K, 64)
    x = datagen.bf16_bits(datagen.normal_f64(seed, 1, T * H)).reshape(T, H)
    wr = datagen.bf16_bits(datagen.normal_f64(seed, 2, E * H, 1 / math.sqrt(H))).reshape(E, H)
    b = datagen.f32(datagen.uniform_f64(seed, 3, E, -0.1, 0.1))
    return d, x, wr, b


def test_router_logits_match_numpy_matmul():
    d, x, wr, b = _small_router()
    lg = oracle.router_logits(d, x, wr)
    ref = datagen.bf16_to_f64(x) @ datagen.bf16_to_f64(wr).T
    assert np.allclose(lg, ref, rtol=1e-13, atol=1e-14)


def test_topk_against_full_sort_and_renorm():
    d, x, wr, b = _small_router()
    lg = oracle.router_logits(d, x, wr)
    ids, w, gap, mingap = oracle.topk(d, lg, b)
    s = 1 / (1 + np.exp(-lg))
    sb = s + b.astype(np.float64)
    for t in range(lg.shape[0]):
        order = sorted(range(d.n_experts), key=lambda e: (-sb[t, e], e))
        assert list(ids[t]) == order[: d.top_k]
        assert gap[t] == pytest.approx(sb[t, order[d.top_k - 1]] - sb[t, order[d.top_k]], abs=1e-15)
        sel = s[t, order[: d.top_k]]
        assert np.allclose(w[t], sel / sel.sum(), rtol=1e-14)
        assert abs(w[t].sum() - 1.0) <= 1e-15
        assert mingap[t] == pytest.approx(np.min(-np.diff(sb[t, order[: d.top_k + 1]])), abs=1e-15)


def test_topk_ties_go_to_lower_id_and_bias_only_selects():
    d = oracle.dims(8, 32, 6, 3, 64)
    lg = np.array([[0.0, 0.0, 0.0, 0.0, 0.0, 0.0]])
    ids, w, _, _ = oracle.topk(d, lg, np.zeros(6, np.float32))
    assert list(ids[0]) == [0, 1, 2]
    # the bias decides the selection, the raw score decides the weights
    bias = np.array([0, 0, 0.3, 0, 0.2, 0.1], np.float32)
    lg = np.array([[2.0, 1.0, -1.0, 0.5, -2.0, 0.0]])
    ids, w, _, _ = oracle.topk(d, lg, bias)
    sb = 1 / (1 + np.exp(-lg[0])) + bias
    assert list(ids[0]) == list(np.argsort(-sb, kind="stable")[:3])
    s = 1 / (1 + np.exp(-lg[0]))
    assert np.allclose(w[0], s[ids[0]] / s[ids[0]].sum(), rtol=1e-15)


def test_router_sigmoid_closed_form_values():
    """The sigmoid at points where it has exact closed-form values: sigma(0) = 1/2,
    sigma(ln 3) = 3/4, sigma(-ln 3) = 1/4, read through the top-K gap (a difference of
    biased scores) and the renormalised weights."""
    d = oracle.dims(8, 32, 3, 2, 64)
    ln3 = math.log(3.0)
    lg = np.array([[0.0, ln3, -ln3]])
    ids, w, gap, mingap = oracle.topk(d, lg, np.zeros(3, np.float32))
    assert list(ids[0]) == [1, 0]
    assert gap[0] == pytest.approx(0.5 - 0.25, abs=1e-15)      # sigma(0) - sigma(-ln 3)
    assert mingap[0] == pytest.approx(0.75 - 0.5, abs=1e-15)   # sigma(ln 3) - sigma(0)
    assert w[0, 0] == pytest.approx(0.75 / 1.25, abs=1e-15) and w[0, 1] == pytest.approx(0.5 / 1.25, abs=1e-15)
    # a bias shifts the ranking score only: +0.3 on expert 2 puts it first, weights from raw scores
    ids, w, gap, _ = oracle.topk(d, lg, np.array([0.0, 0.0, 0.6], np.float32))
    assert list(ids[0]) == [2, 1]
    assert w[0, 0] == pytest.approx(0.25 / 1.0, abs=1e-15)
    assert gap[0] == pytest.approx(0.75 - 0.5, abs=1e-15)
    # saturation: large logits give scores 1 and 0 (equal weights among saturated experts)
    ids, w, _, _ = oracle.topk(d, np.array([[800.0, 800.0, -800.0]]), np.zeros(3, np.float32))
    assert list(ids[0]) == [0, 1] and np.array_equal(w[0], [0.5, 0.5])


def _topk_from_scores(scores, bias, K, top_p):
    E = len(scores)
    d = oracle.dims(8, 32, E, K, 64, top_p=top_p)
    s = np.asarray(scores, dtype=np.float64)
    lg = np.log(s / (1.0 - s))[None, :]
    return oracle.topk(d, lg, np.asarray(bias, np.float32))


def test_top_p_hand_example():
    """K3_TOPP (colibri PR #676, K3_TOPP paragraph): weights 0.4, 0.3, 0.2, 0.1 of the top 4."""
    scores = [0.8, 0.6, 0.4, 0.2, 0.1, 0.05]
    ids, w, _, _ = _topk_from_scores(scores, np.zeros(6), 4, 0.65)
    assert list(ids[0]) == [0, 1, -1, -1]
    assert np.allclose(w[0], [0.8 / 1.4, 0.6 / 1.4, 0.0, 0.0], rtol=1e-14, atol=0)
    ids, w, _, _ = _topk_from_scores(scores, np.zeros(6), 4, 0.75)  # 0.7 before the third: kept
    assert list(ids[0]) == [0, 1, 2, -1]
    assert np.allclose(w[0], [0.8 / 1.8, 0.6 / 1.8, 0.4 / 1.8, 0.0], rtol=1e-14, atol=0)
    ids, w, _, _ = _topk_from_scores(scores, np.zeros(6), 4, 0.01)  # the first is always kept
    assert list(ids[0]) == [0, -1, -1, -1] and w[0, 0] == 1.0
    for off in (0.0, 1.0, 1.5):
        ids, w, _, _ = _topk_from_scores(scores, np.zeros(6), 4, off)
        assert list(ids[0]) == [0, 1, 2, 3]
    # the bias ranks expert 5 first, but the cut follows the weights (raw scores)
    ids, w, _, _ = _topk_from_scores(scores, [0, 0, 0, 0, 0, 0.9], 4, 0.7)
    assert list(ids[0]) == [0, 1, -1, -1]
    assert np.allclose(w[0, :2], [0.8 / 1.4, 0.6 / 1.4], rtol=1e-14, atol=0)


def test_top_p_invariants_on_random_routing():
    d, x, wr, b = _small_router()
    lg = oracle.router_logits(d, x, wr)
    ids_all, w_all, _, _ = oracle.topk(d, lg, b)
    s = 1 / (1 + np.exp(-lg))
    for p in (0.2, 0.5, 0.8):
        dp = oracle.dims(d.hidden, d.latent, d.n_experts, d.top_k, d.inter, top_p=p)
        ids, w, _, _ = oracle.topk(dp, lg, b)
        for t in range(lg.shape[0]):
            kept = _np_top_p(s[t, ids_all[t]], w_all[t], p)
            n = len(kept)
            assert list(ids[t, :n]) == [int(ids_all[t, k]) for k in kept]
            assert (ids[t, n:] == -1).all() and (w[t, n:] == 0).all()
            assert abs(w[t, :n].sum() - 1.0) <= 1e-14
            cw = np.cumsum(w_all[t, kept])
            assert cw[-1] >= p - 1e-15 and (n == 1 or cw[-2] < p)
            assert np.all(np.diff(w_all[t, kept]) <= 0)  # kept in descending weight order


# ------------------------------------------------------------------------------ permutation
def test_permute_matches_stable_sort():
    rng = np.random.default_rng(6)
    for T, K, E in ((1, 16, 896), (32, 16, 896), (200, 4, 37), (5, 2, 8)):
        ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
        counts, offsets, slot_of, uniq = oracle.permute(ids, E)
        flat = ids.ravel()
        assert list(slot_of) == sorted(range(T * K), key=lambda i: (flat[i], i))
        assert np.array_equal(counts, np.bincount(flat, minlength=E))
        assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
        assert list(uniq) == sorted(set(flat.tolist()))


# ------------------------------------------------------------------------------ projections
def test_latent_projections_match_numpy():
    d = oracle.dims(96, 40, 8, 2, 64)
    T = 5
    x = datagen.bf16_bits(datagen.normal_f64(7, 1, T * 96)).reshape(T, 96)
    wd = datagen.bf16_bits(datagen.normal_f64(7, 4, 40 * 96, 0.1)).reshape(40, 96)
    wu = datagen.bf16_bits(datagen.normal_f64(7, 5, 96 * 40, 0.15)).reshape(96, 40)
    z = oracle.latent_down(d, x, wd, False)
    ref = datagen.bf16_to_f64(x) @ datagen.bf16_to_f64(wd).T
    assert np.allclose(z, ref, rtol=1e-13, atol=1e-15)
    zs = oracle.latent_down(d, x, wd, True)
    assert np.max(np.abs(zs - bf16_round_datagen(ref)) / np.abs(ref)) <= 2.0 ** -8
    y = np.random.default_rng(8).normal(size=(T, 40))
    assert np.allclose(oracle.latent_up(d, y, wu), y @ datagen.bf16_to_f64(wu).T, rtol=1e-13, atol=1e-14)


# ------------------------------------------------------------------------------ one expert
def test_expert_matches_dense_numpy():
    d = oracle.dims(64, 96, 4, 2, 128)
    cfg = C.TINY
    t = {}
    I, L = 128, 96
    for which, name in enumerate(C.EXPERT_TENSORS):
        shp = {"gate": (I, L), "up": (I, L), "down": (L, I)}[name.split("_")[0]]
        if name.endswith("_q"):
            t[name] = datagen.u8(3, 40 + which, shp[0] * shp[1] // 2).reshape(shp[0], shp[1] // 2)
        else:
            t[name] = datagen.int_u8(3, 40 + which, shp[0] * shp[1] // 32, 115, 130).reshape(shp[0], shp[1] // 32)
    z = datagen.bf16_to_f64(datagen.bf16_bits(datagen.normal_f64(3, 1, L)))
    for spec in (False, True):
        h, o = oracle.expert(d, z, t, spec)
        g = np_dequant(t["gate_q"], t["gate_s"]) @ z
        u = np_dequant(t["up_q"], t["up_s"]) @ z
        href = 4 * np.tanh(g / 4) / (1 + np.exp(-g)) * 25 * np.tanh(u / 25)
        if spec:
            href = bf16_round_datagen(href)
            assert np.sum(h != href) <= 1  # a rounding-boundary flip from summation order at most
        else:
            assert np.allclose(h, href, rtol=1e-12, atol=1e-14)
        oref = np_dequant(t["down_q"], t["down_s"]) @ h
        assert np.allclose(o, oref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------------------ whole block
def _np_top_p(s_sel, w, p):
    """numpy restatement of K3_TOPP for one token: order by weight (stable), keep while the
    weight before is below p, renormalise the kept by raw score.  Returns kept positions."""
    order = sorted(range(len(w)), key=lambda k: -w[k])  # Python's sort is stable
    kept, cum = [], 0.0
    for j, k in enumerate(order):
        if j > 0 and not cum < p:
            break
        kept.append(k)
        cum += w[k]
    return kept


def _np_block(cfg, x, W, experts, spec, top_p=0.0, mx=None):
    """Brute-force numpy re-implementation of the block from the pages' definitions;
    mx (optional) rounds the experts' activations (z before gate/up, h before down)."""
    E, K, L = cfg.n_experts, cfg.top_k, cfg.latent
    xf = datagen.bf16_to_f64(x)
    lg = xf @ datagen.bf16_to_f64(W["wr"]).T
    s = 1 / (1 + np.exp(-lg))
    sb = s + W["bias"].astype(np.float64)
    rnd = bf16_round_datagen if spec else (lambda v: v)
    z = rnd(xf @ datagen.bf16_to_f64(W["wd"]).T)
    out = []
    for t in range(x.shape[0]):
        ids = np.argsort(-sb[t], kind="stable")[:K]
        w = s[t, ids] / s[t, ids].sum()
        if 0.0 < top_p < 1.0:
            kept = _np_top_p(s[t, ids], w, top_p)
            ids = ids[kept]
            w = s[t, ids] / s[t, ids].sum()
        y = np.zeros(L)
        for k, e in enumerate(ids):
            ex = experts[int(e)]
            ze = mx(z[t]) if mx else z[t]
            g = np_dequant(ex["gate_q"], ex["gate_s"]) @ ze
            u = np_dequant(ex["up_q"], ex["up_s"]) @ ze
            h = rnd(4 * np.tanh(g / 4) / (1 + np.exp(-g)) * 25 * np.tanh(u / 25))
            h = mx(h) if mx else h
            y += w[k] * (np_dequant(ex["down_q"], ex["down_s"]) @ h)
        yh = rnd(W["gamma"].astype(np.float64) * y / np.sqrt(np.mean(y * y) + cfg.rms_eps))
        out.append(yh @ datagen.bf16_to_f64(W["wu"]).T)
    return np.array(out)


@pytest.mark.parametrize("top_p", [0.3, 0.6])
def test_block_with_top_p_matches_bruteforce_on_tiny(top_p):
    cfg = dataclasses.replace(C.TINY, top_k=4, top_p=top_p)
    d = oracle.dims(**cfg.dims)
    x, W = C.layer_x(cfg), C.layer_weights(cfg)
    ex = {e: C.expert_tensors(cfg, e) for e in range(cfg.n_experts)}
    r = oracle.forward(d, x, W["wr"], W["bias"], W["wd"], W["wu"], W["gamma"], ex, False, 0)
    ref = _np_block(cfg, x, W, ex, False, top_p)
    assert np.linalg.norm(r["out"] - ref) / np.linalg.norm(ref) < 1e-12
    assert (r["ids"] == -1).any()  # something was pruned on these tokens
    # chunked execution (pruned slots take no part in the expert union) is bit-identical
    r2 = oracle.forward(d, x, W["wr"], W["bias"], W["wd"], W["wu"], W["gamma"], ex, False, 2)
    assert np.array_equal(r["out"], r2["out"])


@pytest.mark.parametrize("spec", [False, True])
def test_block_matches_bruteforce_on_tiny(spec):
    cfg = C.TINY
    d = oracle.dims(**cfg.dims)
    x, W = C.layer_x(cfg), C.layer_weights(cfg)
    ex = {e: C.expert_tensors(cfg, e) for e in range(cfg.n_experts)}
    r = oracle.forward(d, x, W["wr"], W["bias"], W["wd"], W["wu"], W["gamma"], ex, spec, 0)
    ref = _np_block(cfg, x, W, ex, spec)
    rel = np.linalg.norm(r["out"] - ref) / np.linalg.norm(ref)
    assert rel < (1e-12 if not spec else 1e-5), rel


def test_chunked_equals_token_at_a_time_bit_exact():
    cfg = C.LayerConfig("mid", T=24, hidden=128, latent=64, n_experts=12, top_k=4, inter=96, seed=9,
                        bias_range=0.1, scale_lo=115, scale_hi=128)
    d = oracle.dims(**cfg.dims)
    x, W = C.layer_x(cfg), C.layer_weights(cfg)
    ex = {e: C.expert_tensors(cfg, e) for e in range(cfg.n_experts)}
    for spec in (False, True):
        a = oracle.forward(d, x, W["wr"], W["bias"], W["wd"], W["wu"], W["gamma"], ex, spec, 0)
        for chunk in (1, 5, 24):
            b = oracle.forward(d, x, W["wr"], W["bias"], W["wd"], W["wu"], W["gamma"], ex, spec, chunk)
            for k in ("out", "ids", "w", "y", "yhat"):
                assert np.array_equal(a[k], b[k]), (k, spec, chunk)


def test_top1_block_reduces_to_single_expert():
    cfg = C.LayerConfig("k1", T=3, hidden=64, latent=64, n_experts=5, top_k=1, inter=64, seed=4,
                        bias_range=0.1, scale_lo=118, scale_hi=126)
    d = oracle.dims(**cfg.dims)
    x, W = C.layer_x(cfg), C.layer_weights(cfg)
    ex = {e: C.expert_tensors(cfg, e) for e in range(cfg.n_experts)}
    r = oracle.forward(d, x, W["wr"], W["bias"], W["wd"], W["wu"], W["gamma"], ex, True, 0)
    assert np.all(r["w"] == 1.0)
    for t in range(cfg.T):
        _, o = oracle.expert(d, r["z"][t], ex[int(r["ids"][t, 0])], True)
        assert np.array_equal(r["y"][t], o)


def test_layer_constants_match_recipes():
    consts = dict(l.split()[:2] for l in open(os.path.join(GOLDEN, "k3_layer_constants.txt")) if l[0] != "#")
    for cfg in (C.DECODE, C.CHUNK, C.PREFILL):
        assert cfg.n_experts == int(consts["n_routed_experts"]) and cfg.top_k == int(consts["top_k"])
        assert cfg.hidden == int(consts["hidden"]) and cfg.latent == int(consts["latent"])
        assert cfg.latent % int(consts["mx_group"]) == 0 and cfg.inter % int(consts["mx_group"]) == 0
    assert C.CHUNK.T == int(consts["chunk_tokens"])
    # per-expert bytes of the vendor layout: 3 matrices of 3072 x 3584 at 4.25 bits
    assert C.DECODE.expert_bytes == 17_547_264


def test_decode_seed_satisfies_gap_rule():
    cfg = C.DECODE
    d = oracle.dims(**cfg.dims)
    W = C.layer_weights(cfg)
    _, _, gap, _ = oracle.route(d, C.layer_x(cfg), W["wr"], W["bias"])
    assert gap[0] > 1e-4
    # and it is the first such seed
    for s in range(cfg.seed):
        c2 = C.LayerConfig(**{**cfg.__dict__, "seed": s})
        W2 = C.layer_weights(c2)
        assert oracle.route(d, C.layer_x(c2), W2["wr"], W2["bias"])[2][0] <= 1e-4

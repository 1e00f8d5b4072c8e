"""Pins of the oracle's shared experts (colibri PR #684, engine commit: "2 fused shared
experts"; colibri PR #676, architecture bullets: SiTU-GLU): a numpy brute force, the
fusion property (the fused expert is the sum of the two separate ones) and the reduction
to the routed expert (a shared expert whose bf16 weights are MXFP4 values computes what
the routed-expert oracle computes on the same vector)."""
import dataclasses

import numpy as np
import pytest

import datagen
import oracle
from datagen import configs as C
from tests.test_oracle_layer import np_dequant

TINY_SHARED = 128  # fused width on the tiny layer


def _np_shared(x_bits, wgu_bits, wdn_bits, spec):
    x = datagen.bf16_to_f64(x_bits)
    wgu = datagen.bf16_to_f64(wgu_bits)
    wdn = datagen.bf16_to_f64(wdn_bits)
    Is = wdn.shape[1]
    g, u = x @ wgu[:Is].T, x @ wgu[Is:].T
    h = 4 * np.tanh(g / 4) / (1 + np.exp(-g)) * 25 * np.tanh(u / 25)
    if spec:
        h = datagen.bf16_to_f64(datagen.bf16_bits(h))
    return h, h @ wdn.T


@pytest.mark.parametrize("spec", [False, True])
def test_shared_matches_bruteforce_on_tiny(spec):
    cfg = C.TINY
    d = oracle.dims(**cfg.dims)
    x = C.layer_x(cfg)
    W = C.shared_weights(cfg, TINY_SHARED)
    h, out = oracle.shared(d, x, W["wgu"], W["wdn"], spec)
    href, oref = _np_shared(x, W["wgu"], W["wdn"], spec)
    assert np.abs(out).max() > 1e-3  # non-trivial outputs
    if spec:  # fp64 sums in another order may round a bf16 h the other way at a boundary
        assert np.mean(h != href) < 0.01
        assert np.linalg.norm(out - oref) / np.linalg.norm(oref) < 1e-3
    else:
        assert np.allclose(h, href, rtol=1e-12, atol=1e-14)
        assert np.linalg.norm(out - oref) / np.linalg.norm(oref) < 1e-12


def test_fused_expert_is_the_sum_of_the_separate_ones():
    cfg = C.TINY
    d = oracle.dims(**cfg.dims)
    x = C.layer_x(cfg)
    W = C.shared_weights(cfg, TINY_SHARED)
    half = TINY_SHARED // 2
    _, fused = oracle.shared(d, x, W["wgu"], W["wdn"], False)
    parts = []
    for sl in (slice(0, half), slice(half, TINY_SHARED)):
        g = W["wgu"][:TINY_SHARED][sl]
        u = W["wgu"][TINY_SHARED:][sl]
        parts.append(oracle.shared(d, x, np.concatenate([g, u]), np.ascontiguousarray(W["wdn"][:, sl]), False)[1])
    assert np.linalg.norm(fused - parts[0] - parts[1]) / np.linalg.norm(fused) < 1e-12


def test_shared_reduces_to_the_routed_expert():
    # a routed expert of the tiny layer, its weights taken as bf16 values (every E2M1 value
    # times 2^(s - 127) with these scale bytes is a bf16 number): the shared-expert oracle on
    # the hidden width H = L computes the routed expert's h and o on the same vector
    cfg = C.TINY
    L, I = cfg.latent, cfg.inter
    t = C.expert_tensors(cfg, 5)
    Wg, Wu, Wd = (np_dequant(t[a], t[b]) for a, b in (("gate_q", "gate_s"), ("up_q", "up_s"),
                                                      ("down_q", "down_s")))
    wgu = datagen.bf16_bits(np.concatenate([Wg, Wu]))
    wdn = datagen.bf16_bits(Wd)
    assert np.array_equal(datagen.bf16_to_f64(wgu), np.concatenate([Wg, Wu]))  # exact in bf16
    z = datagen.bf16_bits(np.random.default_rng(3).standard_normal((1, L)))
    dl = oracle.dims(**dict(cfg.dims, hidden=L))
    for spec in (False, True):
        h_s, o_s = oracle.shared(dl, z, wgu, wdn, spec)
        h_r, o_r = oracle.expert(oracle.dims(**cfg.dims), datagen.bf16_to_f64(z[0]), t, spec)
        assert np.array_equal(h_s[0], h_r)
        assert np.array_equal(o_s[0], o_r)

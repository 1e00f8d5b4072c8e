"""Helpers shared by the GPU parity tests: device workloads, oracle references."""
from __future__ import annotations

import numpy as np

import datagen
import oracle
from datagen import configs as C

REL_L2_BAR = 2e-3  # output tolerance against the oracle's bf16-rounding spec mode


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def oracle_dims(cfg):
    return oracle.dims(**cfg.dims)


def oracle_route(cfg, x_bits=None):
    W = C.layer_weights(cfg)
    x = C.layer_x(cfg) if x_bits is None else x_bits
    return oracle.route(oracle_dims(cfg), x, W["wr"], W["bias"])


def oracle_forward(cfg, token_rows=None, spec=True, chunk=0):
    """Oracle forward on all tokens of cfg, or on the given subset of token rows.
    Only the experts the routed tokens need are generated."""
    W = C.layer_weights(cfg)
    x = C.layer_x(cfg)
    if token_rows is not None:
        x = np.ascontiguousarray(x[np.asarray(token_rows)])
    d = oracle_dims(cfg)
    ids, _, _, _ = oracle.route(d, x, W["wr"], W["bias"])
    ex = {int(e): C.expert_tensors(cfg, int(e)) for e in np.unique(ids) if e >= 0}
    return oracle.forward(d, x, W["wr"], W["bias"], W["wd"], W["wu"], W["gamma"], ex, spec, chunk)


def smallest_scale_within_448(amax):
    """Per group: the smallest scale byte s (0..254) with amax <= 448 * 2^(s - 127); 0 for a
    group of zeros.  Searched directly from a frexp estimate."""
    s = np.zeros(amax.shape, np.int64)
    nz = amax > 0
    _, ex = np.frexp(amax[nz])
    c = ex.astype(np.int64) + 127 - 9  # 448 < 2^9
    lim = lambda c: 448.0 * np.exp2(c.astype(np.float64) - 127)
    for _ in range(4):
        c = np.where(amax[nz] > lim(c), c + 1, c)
    for _ in range(4):
        c = np.where((c > 0) & (amax[nz] <= lim(c - 1)), c - 1, c)
    s[nz] = np.clip(c, 0, 254)
    return s

"""Pins of the oracle's MXFP8 activation quantization (the low-precision-activation
variant: colibri PR #676, "What's in the commits" item 7, and colibri PR #684's quant.h
commit, per-32-group quantized activations; read as OCP MX v1.0 MXFP8 with E4M3
elements) against PyTorch's independent float8_e4m3fn implementation, closed forms and
a brute-force numpy composition of the variant's expert and block."""
import dataclasses

import numpy as np
import pytest

import datagen
import oracle
from datagen import configs as C
from tests.test_oracle_layer import _np_block, np_dequant

torch = pytest.importorskip("torch")
if not hasattr(torch, "float8_e4m3fn"):
    pytest.skip("torch without float8_e4m3fn", allow_module_level=True)


def _bf16(a):
    return datagen.bf16_to_f64(datagen.bf16_bits(a))


def _torch_e4m3_values():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_matches_torch_for_every_code():
    ref = _torch_e4m3_values()
    got = np.array([oracle.e4m3(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))  # 0x80 is -0
    # closed forms: 1.0, the largest normal, the smallest normal and subnormal
    assert (oracle.e4m3(0x38), oracle.e4m3(0x7E), oracle.e4m3(0x08), oracle.e4m3(0x01)) == (1.0, 448.0, 2.0 ** -6,
                                                                                            2.0 ** -9)


def test_e4m3_encode_matches_torch_cast():
    vals = _torch_e4m3_values()
    fin = np.sort(np.unique(vals[np.isfinite(vals) & (vals >= 0)]))
    mids = (fin[:-1] + fin[1:]) / 2  # exact ties: round to the even code
    rng = np.random.default_rng(0)
    rnd = rng.uniform(-448, 448, 4000).astype(np.float32).astype(np.float64)
    small = (rng.standard_normal(4000) * 2.0 ** rng.integers(-12, 2, 4000)).astype(np.float32).astype(np.float64)
    for xs in (fin, -fin, mids, -mids, rnd, small):
        got = np.array([oracle.e4m3_encode(v) for v in xs], dtype=np.uint8)
        ref = torch.from_numpy(xs.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(got, ref), xs[np.nonzero(got != ref)[0][:5]]


def test_e4m3_encode_saturates_and_keeps_the_sign_of_zero():
    assert oracle.e4m3_encode(448.0) == 0x7E and oracle.e4m3_encode(500.0) == 0x7E
    assert oracle.e4m3_encode(1e30) == 0x7E and oracle.e4m3_encode(-1e30) == 0xFE
    assert oracle.e4m3_encode(0.0) == 0x00 and oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-2.0 ** -11) == 0x80  # below half the smallest subnormal
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00   # exactly half: ties to even (0)
    assert oracle.e4m3_encode(3 * 2.0 ** -11) == 0x01


def test_mxfp8_scale_rule_by_hand():
    ones = np.ones(32)
    c, s = oracle.mxfp8_quant(ones)
    assert s[0] == 119 and (c == 0x78).all()  # X = 0 - 8; 1.0 / 2^-8 = 256 = 2^8 -> E 15, M 0
    g = np.zeros(32)
    g[3] = 3.0
    g[7] = -0.25
    c, s = oracle.mxfp8_quant(g)
    assert s[0] == 120  # floor(log2 3) = 1 -> X = -7
    assert c[3] == 0x7C  # 3 * 2^7 = 384 = 1.5 * 2^8
    assert c[7] == 0xE0  # -0.25 * 2^7 = -32 = -(2^5): exponent field 12 (0x60), M 0, sign
    assert (np.delete(c, [3, 7]) == 0).all()
    g = np.full(32, 500.0)  # 500 / 2^0 saturates to 448
    c, s = oracle.mxfp8_quant(g)
    assert s[0] == 127 and (c == 0x7E).all()
    c, s = oracle.mxfp8_quant(np.zeros(32))
    assert s[0] == 0 and (c == 0).all()
    c, s = oracle.mxfp8_quant(-np.zeros(32))
    assert s[0] == 0 and (c == 0x80).all()
    # clamps: a tiny group takes byte 0, a huge one 254
    assert oracle.mxfp8_quant(np.full(32, 2.0 ** -140))[1][0] == 0
    assert oracle.mxfp8_quant(np.full(32, 2.0 ** 200))[1][0] == 254


def _mx_ref(x):
    """Independent MXFP8 rounding: numpy's frexp for the shared exponent, PyTorch's
    float8_e4m3fn cast (round to nearest even) for the elements, after clamping to the
    largest finite magnitude (saturation).  x must be exact in fp32 after scaling."""
    g = np.asarray(x, dtype=np.float64).reshape(-1, 32)
    amax = np.abs(g).max(1)
    _, ex = np.frexp(amax)
    s = np.where(amax == 0, 0, np.clip(127 + ex - 1 - 8, 0, 254))
    v = np.clip(g * np.exp2(127.0 - s)[:, None], -448, 448)
    q = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    return (q * np.exp2(s - 127.0)[:, None]).reshape(np.shape(x))


def test_mxfp8_round_matches_independent_quantizer_and_bounds():
    rng = np.random.default_rng(1)
    # bf16 values with a wide spread inside and between groups
    x = _bf16(rng.standard_normal(32 * 400) * 2.0 ** rng.integers(-20, 20, 32 * 400))
    x = x * np.repeat(2.0 ** rng.integers(-30, 30, 400), 32)
    got = oracle.mxfp8_round(x)
    assert np.array_equal(got, _mx_ref(x))
    codes, scales = oracle.mxfp8_quant(x)
    vals = np.array([oracle.e4m3(c) for c in range(256)])
    assert np.array_equal(got, vals[codes] * np.exp2(np.repeat(scales.astype(np.float64), 32) - 127))
    # error: at most half an E4M3 step of the element's binade (the steps are 2^(e-3) for
    # exponents e >= -6 of the scaled value, 2^-9 below), except the saturated range
    g = x.reshape(-1, 32)
    X = np.repeat(scales.astype(np.float64) - 127, 32).reshape(-1, 32)
    v = np.abs(g) * np.exp2(-X)
    e = np.floor(np.log2(np.where(v > 0, v, 1.0)))
    step = np.exp2(np.maximum(e, -6) - 3)
    err = np.abs(got.reshape(-1, 32) - g) * np.exp2(-X)
    sat = v > 448
    assert (err[~sat] <= step[~sat] / 2).all()
    assert (err[sat] <= 64).all()
    # idempotent
    assert np.array_equal(oracle.mxfp8_round(got), got)


def test_variant_expert_matches_numpy_composition():
    cfg = C.TINY
    d = oracle.dims(**dict(cfg.dims, act_mxfp8=1))
    d0 = oracle.dims(**cfg.dims)
    ex = C.expert_tensors(cfg, 3)
    rng = np.random.default_rng(2)
    z = _bf16(rng.standard_normal(cfg.latent))
    h, o = oracle.expert(d, z, ex, True)
    zq = _mx_ref(z)
    g = np_dequant(ex["gate_q"], ex["gate_s"]) @ zq
    u = np_dequant(ex["up_q"], ex["up_s"]) @ zq
    href = _bf16(4 * np.tanh(g / 4) / (1 + np.exp(-g)) * 25 * np.tanh(u / 25))
    hq = _mx_ref(href)
    assert np.array_equal(h, hq)  # the expert returns the quantized h it contracts
    oref = np_dequant(ex["down_q"], ex["down_s"]) @ hq
    assert np.allclose(o, oref, rtol=1e-12, atol=1e-12)
    # an input already on the MXFP8 grid with an exact-path h on it too: the variant
    # reduces to the exact expert where quantization is the identity
    h0, o0 = oracle.expert(d0, zq, ex, True)
    assert np.array_equal(oracle.expert(d, zq, ex, True)[0], _mx_ref(h0))


def test_variant_block_matches_bruteforce_on_tiny():
    cfg = dataclasses.replace(C.TINY, act_mxfp8=1)
    d = oracle.dims(**cfg.dims)
    x, W = C.layer_x(cfg), C.layer_weights(cfg)
    ex = {e: C.expert_tensors(cfg, e) for e in range(cfg.n_experts)}
    r = oracle.forward(d, x, W["wr"], W["bias"], W["wd"], W["wu"], W["gamma"], ex, True, 0)
    ref = _np_block(cfg, x, W, ex, True, mx=_mx_ref)
    assert np.linalg.norm(r["out"] - ref) / np.linalg.norm(ref) < 1e-12
    r2 = oracle.forward(d, x, W["wr"], W["bias"], W["wd"], W["wu"], W["gamma"], ex, True, 2)
    assert np.array_equal(r["out"], r2["out"])  # the chunked path quantizes the same way
    exact = oracle.forward(oracle.dims(**C.TINY.dims), x, W["wr"], W["bias"], W["wd"], W["wu"], W["gamma"], ex,
                           True, 0)
    rel = np.linalg.norm(r["out"] - exact["out"]) / np.linalg.norm(exact["out"])
    assert 1e-4 < rel < 0.1  # the variant is lossy, by about an E4M3 step per element

"""fp64 oracle for the Stable LatentMoE routed-expert block (TEST INFRASTRUCTURE ONLY).

Thin ctypes binding over ``k3oracle.c``.  Only the test suite, ``__graft_entry__.smoke``
and the bench's CPU-baseline leg may import this package; the product library never
does.  Every array crosses the boundary as a plain host pointer.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libk3oracle.so")
_lock = threading.Lock()
_lib = None
_openmp = None

EXPERT_TENSORS = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")


class Dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("latent", ctypes.c_int), ("n_experts", ctypes.c_int),
                ("top_k", ctypes.c_int), ("inter", ctypes.c_int), ("rms_eps", ctypes.c_double),
                ("top_p", ctypes.c_double), ("act_mxfp8", ctypes.c_int)]


def dims(hidden, latent, n_experts, top_k, inter, rms_eps=1e-6, top_p=0.0, act_mxfp8=0) -> Dims:
    return Dims(hidden, latent, n_experts, top_k, inter, rms_eps, top_p, int(act_mxfp8))


def build(force: bool = False) -> str:
    """Compile the oracle (plain C99; OpenMP when available)."""
    global _openmp
    os.makedirs(_BUILD, exist_ok=True)
    src = os.path.join(_HERE, "k3oracle.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
        _openmp = True
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
        _openmp = False
    os.replace(tmp, _SO)
    return _SO


def _L():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p, i, i64, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            D = ctypes.POINTER(Dims)
            sig = {
                "k3o_e2m1": ([ctypes.c_uint], d),
                "k3o_ue8m0": ([ctypes.c_uint], d),
                "k3o_e4m3": ([ctypes.c_uint], d),
                "k3o_e4m3_encode": ([d], ctypes.c_uint),
                "k3o_mxfp8_quant": ([i64, p, p, p], None),
                "k3o_mxfp8_round": ([i64, p, p], None),
                "k3o_round_bf16": ([d], d),
                "k3o_situ": ([d, d], d),
                "k3o_dequant": ([p, p, i, i, p], None),
                "k3o_rmsnorm": ([i, p, p, d, i, p], None),
                "k3o_router_logits": ([D, i, p, p, p], None),
                "k3o_topk": ([D, i, p, p, p, p, p, p], None),
                "k3o_permute": ([i, i, i, p, p, p, p, p, p], None),
                "k3o_latent_down": ([D, i, p, p, i, p], None),
                "k3o_latent_up": ([D, i, p, p, p], None),
                "k3o_expert": ([D, p, p, p, p, p, p, p, i, p, p], None),
                "k3o_forward": ([D, i, p, p, p, p, p, p, p, i, i, p, p, p, p, p, p], i),
                "k3o_shared": ([D, i, i, p, p, p, i, p, p], None),
                "k3o_round_bf16_array": ([i64, p, p], None),
                "k3o_situ_array": ([i64, p, p, p], None),
                "k3o_abi_version": ([], i),
            }
            for name, (args, res) in sig.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
        return _lib


def threads_used() -> int:
    """OpenMP threads the oracle's parallel loops use (1 when built without OpenMP)."""
    _L()
    if not _openmp and _openmp is not None:
        return 1
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


# ---------------------------------------------------------------- scalar / elementwise
def e2m1(code: int) -> float:
    return _L().k3o_e2m1(code)


def ue8m0(s: int) -> float:
    return _L().k3o_ue8m0(s)


def e4m3(code: int) -> float:
    return _L().k3o_e4m3(code)


def e4m3_encode(v: float) -> int:
    return int(_L().k3o_e4m3_encode(float(v)))


def mxfp8_quant(x):
    """x [..., n] (n a multiple of 32, groups along the last axis) -> (E4M3 codes uint8
    [..., n], scale bytes uint8 [..., n/32])."""
    x, px = _c(x, np.float64)
    assert x.shape[-1] % 32 == 0
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty(x.shape[:-1] + (x.shape[-1] // 32,), dtype=np.uint8)
    _L().k3o_mxfp8_quant(x.size, px, codes.ctypes.data, scales.ctypes.data)
    return codes, scales


def mxfp8_round(x) -> np.ndarray:
    """The values of x's MXFP8 quantization (groups of 32 along the last axis)."""
    x, px = _c(x, np.float64)
    assert x.shape[-1] % 32 == 0
    out = np.empty_like(x)
    _L().k3o_mxfp8_round(x.size, px, out.ctypes.data)
    return out


def round_bf16(a) -> np.ndarray:
    a, pa = _c(a, np.float64)
    out = np.empty_like(a)
    _L().k3o_round_bf16_array(a.size, pa, out.ctypes.data)
    return out


def situ(g, u) -> np.ndarray:
    g, pg = _c(g, np.float64)
    u, pu = _c(np.broadcast_to(u, g.shape), np.float64)
    out = np.empty_like(g)
    _L().k3o_situ_array(g.size, pg, pu, out.ctypes.data)
    return out


def dequant(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """[O, I/2] packed + [O, I/32] scales -> [O, I] fp64."""
    O, half = q.shape
    I = 2 * half
    assert s.shape == (O, I // 32)
    q, pq = _c(q, np.uint8)
    s, ps = _c(s, np.uint8)
    out = np.empty((O, I), dtype=np.float64)
    _L().k3o_dequant(pq, ps, O, I, out.ctypes.data)
    return out


def rmsnorm(y, gamma, eps: float, spec: bool) -> np.ndarray:
    y, py = _c(y, np.float64)
    gamma, pg = _c(gamma, np.float32)
    out = np.empty_like(y)
    _L().k3o_rmsnorm(y.size, py, pg, eps, int(spec), out.ctypes.data)
    return out


# ---------------------------------------------------------------- router
def router_logits(d: Dims, x_bits: np.ndarray, wr_bits: np.ndarray) -> np.ndarray:
    T = x_bits.shape[0]
    x, px = _c(x_bits, np.uint16)
    wr, pw = _c(wr_bits, np.uint16)
    out = np.empty((T, d.n_experts), dtype=np.float64)
    _L().k3o_router_logits(ctypes.byref(d), T, px, pw, out.ctypes.data)
    return out


def topk(d: Dims, logits: np.ndarray, bias: np.ndarray):
    """-> ids [T,K] int32, w [T,K] fp64, gap [T], mingap [T]."""
    T = logits.shape[0]
    lg, pl = _c(logits, np.float64)
    b, pb = _c(bias, np.float32)
    ids = np.empty((T, d.top_k), dtype=np.int32)
    w = np.empty((T, d.top_k), dtype=np.float64)
    gap = np.empty(T, dtype=np.float64)
    mingap = np.empty(T, dtype=np.float64)
    _L().k3o_topk(ctypes.byref(d), T, pl, pb, ids.ctypes.data, w.ctypes.data, gap.ctypes.data,
                  mingap.ctypes.data)
    return ids, w, gap, mingap


def permute(ids: np.ndarray, n_experts: int):
    """Counting sort of the flat (t*K+k) slots by expert -> counts, offsets, slot_of, uniq."""
    T, K = ids.shape
    ids_c, pi = _c(ids, np.int32)
    counts = np.empty(n_experts, dtype=np.int32)
    offsets = np.empty(n_experts + 1, dtype=np.int32)
    slot_of = np.empty(T * K, dtype=np.int32)
    uniq = np.empty(n_experts, dtype=np.int32)
    nu = ctypes.c_int32(0)
    _L().k3o_permute(T, K, n_experts, pi, counts.ctypes.data, offsets.ctypes.data, slot_of.ctypes.data,
                     uniq.ctypes.data, ctypes.addressof(nu))
    return counts, offsets, slot_of, uniq[: nu.value].copy()


# ---------------------------------------------------------------- projections / experts
def latent_down(d: Dims, x_bits, wd_bits, spec: bool) -> np.ndarray:
    T = x_bits.shape[0]
    x, px = _c(x_bits, np.uint16)
    wd, pw = _c(wd_bits, np.uint16)
    out = np.empty((T, d.latent), dtype=np.float64)
    _L().k3o_latent_down(ctypes.byref(d), T, px, pw, int(spec), out.ctypes.data)
    return out


def latent_up(d: Dims, yhat, wu_bits) -> np.ndarray:
    T = yhat.shape[0]
    y, py = _c(yhat, np.float64)
    wu, pw = _c(wu_bits, np.uint16)
    out = np.empty((T, d.hidden), dtype=np.float64)
    _L().k3o_latent_up(ctypes.byref(d), T, py, pw, out.ctypes.data)
    return out


def expert(d: Dims, z: np.ndarray, tensors: dict, spec: bool):
    """One expert on one latent vector z [L] (fp64 values) -> (h [I], o [L])."""
    z, pz = _c(z, np.float64)
    keep = [np.ascontiguousarray(tensors[n], dtype=np.uint8) for n in EXPERT_TENSORS]
    h = np.empty(d.inter, dtype=np.float64)
    o = np.empty(d.latent, dtype=np.float64)
    _L().k3o_expert(ctypes.byref(d), pz, *[k.ctypes.data for k in keep], int(spec), h.ctypes.data, o.ctypes.data)
    return h, o


def shared(d: Dims, x_bits, wgu_bits, wdn_bits, spec: bool = True):
    """Fused shared experts on x [T, H] (bf16 bits): wgu [2 Is, H] (gate rows, then up rows),
    wdn [H, Is] -> (h [T, Is], out [T, H]) fp64."""
    T = x_bits.shape[0]
    Is = wdn_bits.shape[1]
    assert wgu_bits.shape == (2 * Is, d.hidden) and wdn_bits.shape == (d.hidden, Is)
    x, px = _c(x_bits, np.uint16)
    wgu, pg = _c(wgu_bits, np.uint16)
    wdn, pd = _c(wdn_bits, np.uint16)
    h = np.empty((T, Is), dtype=np.float64)
    out = np.empty((T, d.hidden), dtype=np.float64)
    _L().k3o_shared(ctypes.byref(d), T, Is, px, pg, pd, int(spec), h.ctypes.data, out.ctypes.data)
    return h, out


def forward(d: Dims, x_bits, wr_bits, bias, wd_bits, wu_bits, gamma, experts: dict, spec: bool = True,
            chunk: int = 0):
    """Whole block.  ``experts`` maps expert id -> dict of the six tensors; experts no
    token routes to may be absent.  Returns dict(out, ids, w, z, y, yhat)."""
    T = x_bits.shape[0]
    E, K, L = d.n_experts, d.top_k, d.latent
    arrs = [_c(a, dt) for a, dt in ((x_bits, np.uint16), (wr_bits, np.uint16), (bias, np.float32),
                                    (wd_bits, np.uint16), (wu_bits, np.uint16), (gamma, np.float32))]
    keep = []
    tables = []
    for n in EXPERT_TENSORS:
        tab = (ctypes.c_void_p * E)()
        for e, t in experts.items():
            a = np.ascontiguousarray(t[n], dtype=np.uint8)
            keep.append(a)
            tab[e] = a.ctypes.data
        tables.append(tab)
    ex = (ctypes.c_void_p * 6)(*[ctypes.cast(t, ctypes.c_void_p) for t in tables])
    out = np.empty((T, d.hidden), dtype=np.float64)
    ids = np.empty((T, K), dtype=np.int32)
    w = np.empty((T, K), dtype=np.float64)
    z = np.empty((T, L), dtype=np.float64)
    y = np.empty((T, L), dtype=np.float64)
    yhat = np.empty((T, L), dtype=np.float64)
    rc = _L().k3o_forward(ctypes.byref(d), T, *[a[1] for a in arrs], ctypes.cast(ex, ctypes.c_void_p), int(spec),
                          int(chunk), out.ctypes.data, ids.ctypes.data, w.ctypes.data, z.ctypes.data, y.ctypes.data,
                          yhat.ctypes.data)
    if rc != 0:
        raise KeyError(f"expert {-rc - 1} is routed to but was not supplied")
    return dict(out=out, ids=ids, w=w, z=z, y=y, yhat=yhat)


def route(d: Dims, x_bits, wr_bits, bias):
    """Router only: ids, w, gap, mingap (used to find which experts a token set needs)."""
    return topk(d, router_logits(d, x_bits, wr_bits), bias)

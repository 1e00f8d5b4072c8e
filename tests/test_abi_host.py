"""Host-only checks of the C ABI: the library builds and loads, exports every
function the header declares, and validates arguments before touching a device."""
import ctypes

import pytest

import mxfp4_routed_expert_latentmoe_gb300 as k3
from datagen import configs as C

ERR_ARG, ERR_SHAPE, ERR_ALIGN, ERR_WS, ERR_DEVICE = 1, 2, 3, 4, 5


def test_library_exports_every_declared_function():
    names = k3.declared_functions()
    assert "k3moe_route" in names and "k3moe_forward" in names
    L = k3.lib()
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    assert L.k3moe_abi_version() == 3
    for code, text in k3.STATUS.items():
        assert L.k3moe_status_str(code).decode() == text


def _d(cfg=C.DECODE):
    return k3.dims(**cfg.dims)


def test_workspace_bytes_is_monotone_and_rejects_bad_dims():
    L = k3.lib()
    d = _d()
    sizes = [L.k3moe_workspace_bytes(ctypes.byref(d), T) for T in (0, 1, 32, 4096)]
    assert sizes[0] > 0 and sizes == sorted(sizes)
    # the expert intermediates dominate: T*K*(I*2 + L*4) bytes at least
    assert sizes[3] >= 4096 * 16 * (3072 * 2 + 3584 * 4)
    for bad in (dict(hidden=7000), dict(latent=100), dict(inter=96 + 16), dict(top_k=0), dict(top_k=897),
                dict(n_experts=4096)):
        kw = dict(C.DECODE.dims)
        kw.update(bad)
        assert L.k3moe_workspace_bytes(ctypes.byref(k3.dims(**kw)), 1) == 0, bad
    assert L.k3moe_workspace_bytes(ctypes.byref(d), -1) == 0


T_SPLIT_DEFAULT = 1 << 30


def test_workspace_holds_the_tensor_core_path_buffers_from_the_threshold():
    # from k3moe_tc_min_tokens tokens the grouped expert GEMM needs the slot-ordered
    # activations (bf16 rows, or two MXFP8 terms plus their scale bytes), the weight tensor
    # maps (256 CTAs x 2 blocks x 2 x 128 bytes), the split form's two terms of h (codes and
    # scale bytes) and the projections' split-K partial sums (8 x T x max(E + L, H) f32);
    # below that the workspace grows by the per-token buffers only
    L = k3.lib()
    d = _d()
    t0 = k3.tc_min_tokens()
    assert t0 == 9  # the measured GEMV / tensor-core crossover
    assert T_SPLIT_DEFAULT > t0  # the split form's buffers at the threshold
    ws = {T: L.k3moe_workspace_bytes(ctypes.byref(d), T) for T in (t0 - 2, t0 - 1, t0)}
    per_token = ws[t0 - 1] - ws[t0 - 2]
    slots = t0 * 16
    split_extra = slots * 3584 // 16 + slots * 3072 * 2 + slots * 3072 // 16
    part = 8 * t0 * max(896 + 3584, 7168) * 4
    tc_bytes = slots * 3584 * 2 + 256 * 2 * 2 * 128 + split_extra + part
    assert ws[t0] - ws[t0 - 1] >= tc_bytes
    assert ws[t0] - ws[t0 - 1] <= tc_bytes + 2 * per_token + 6 * 256


def test_split_form_token_bound():
    """k3moe_set_tc_split_max_tokens sets the token count below which the exact tensor-core
    expert GEMMs take the two-term MXFP8 split (default 2^30: every count, as measured),
    returns the previous value, rejects t < 0, and sizes the workspace: the split form adds
    z's terms' scale bytes (slots x L / 16) and h's two terms (slots x I x 2 codes and
    slots x I / 16 scale bytes) to the bf16-sized buffers; below the tensor-core threshold the
    form does not matter."""
    L = k3.lib()
    d = _d()
    assert k3.tc_split_max_tokens() == 1 << 30 == k3.SPLIT_ALWAYS
    T = 64
    slots = T * 16
    on = L.k3moe_workspace_bytes(ctypes.byref(d), T)
    below = L.k3moe_workspace_bytes(ctypes.byref(d), 8)
    prev = k3.set_tc_split_max_tokens(0)
    try:
        assert prev == 1 << 30 and k3.tc_split_max_tokens() == 0
        off = L.k3moe_workspace_bytes(ctypes.byref(d), T)
        assert 0 <= on - off - (slots * (3584 + 3072) // 16 + slots * 3072 * 2) < 3 * 256
        assert L.k3moe_workspace_bytes(ctypes.byref(d), 8) == below
        with pytest.raises(ValueError):
            k3.set_tc_split_max_tokens(-1)
        assert L.k3moe_set_tc_split_max_tokens(-5) == -1 and k3.tc_split_max_tokens() == 0
        # the bound is exclusive: T = t runs the weight-decode form
        k3.set_tc_split_max_tokens(T)
        assert L.k3moe_workspace_bytes(ctypes.byref(d), T) == off
        k3.set_tc_split_max_tokens(T + 1)
        assert L.k3moe_workspace_bytes(ctypes.byref(d), T) == on
    finally:
        k3.set_tc_split_max_tokens(prev)
    assert k3.tc_split_max_tokens() == 1 << 30
    # the MXFP8-activation variant never takes the split form
    dv = k3.dims(hidden=7168, latent=3584, n_experts=896, top_k=16, inter=3072, act_mxfp8=1)
    v = L.k3moe_workspace_bytes(ctypes.byref(dv), T)
    assert v == off

def test_device_status_bits_match_the_header():
    import re
    text = open(k3._HEADER).read()
    bits = {m.group(1): int(m.group(2), 16) for m in re.finditer(r"#define K3MOE_DEV_(\w+) (0x[0-9a-fA-F]+)u", text)}
    assert bits == {"TIE_WINDOW": k3.DEV_TIE_WINDOW, "TIMEOUT": k3.DEV_TIMEOUT, "BAD_ID": k3.DEV_BAD_ID,
                    "SCALE_RANGE": k3.DEV_SCALE_RANGE, "ALIGN": k3.DEV_ALIGN}


def _route(d, T, x=16, wr=16, bias=16, ids=16, w=16, ws=16, ws_bytes=None):
    L = k3.lib()
    nb = ws_bytes if ws_bytes is not None else L.k3moe_workspace_bytes(ctypes.byref(d), T)
    p = lambda v: None if v is None else ctypes.c_void_p(v)
    return L.k3moe_route(ctypes.byref(d), T, p(x), p(wr), p(bias), p(ids), p(w), p(ws), nb, None)


def test_route_validates_on_the_host():
    d = _d()
    assert _route(d, 0) == 0  # empty call is a no-op
    assert _route(d, -1) == ERR_ARG
    assert _route(d, 1, x=None) == ERR_ARG
    assert _route(d, 1, ws=None) == ERR_ARG
    assert _route(d, 1, x=24) == ERR_ALIGN
    assert _route(d, 1, ws_bytes=100) == ERR_WS
    bad = k3.dims(7168, 3584, 896, 0, 3072)
    assert _route(bad, 1) == ERR_SHAPE
    # a fully valid call on a machine without a compute-capability-10.3 device
    import torch
    if not torch.cuda.is_available():
        assert _route(d, 1) == ERR_DEVICE


def test_forward_and_expert_forward_validate_on_the_host():
    L = k3.lib()
    d = _d()
    ex = k3.ExpertsC(16, 16, 16, 16, 16, 16)
    nb = L.k3moe_workspace_bytes(ctypes.byref(d), 1)
    v = ctypes.c_void_p(16)
    args = [ctypes.byref(d), 1, v, v, v, v, v, v, ctypes.byref(ex), v, None, None, v, nb, None]
    import torch
    if not torch.cuda.is_available():
        assert L.k3moe_forward(*args) == ERR_DEVICE
    args2 = list(args)
    args2[8] = ctypes.byref(k3.ExpertsC(16, 16, 0, 16, 16, 16))
    assert L.k3moe_forward(*args2) == ERR_ARG
    args3 = list(args)
    args3[13] = nb - 1
    assert L.k3moe_forward(*args3) == ERR_WS
    args4 = list(args)
    args4[9] = ctypes.c_void_p(20)
    assert L.k3moe_forward(*args4) == ERR_ALIGN
    assert L.k3moe_expert_forward(ctypes.byref(d), 1, v, 896, ctypes.byref(ex), v, v, nb, None) == ERR_ARG
    assert L.k3moe_expert_forward(ctypes.byref(d), 1, v, -1, ctypes.byref(ex), v, v, nb, None) == ERR_ARG


def test_dequant_validates_shape():
    L = k3.lib()
    v = ctypes.c_void_p(16)
    assert L.k3moe_dequant_mxfp4(v, v, 4, 48, v, None) == ERR_SHAPE
    assert L.k3moe_dequant_mxfp4(v, v, -1, 64, v, None) == ERR_ARG
    assert L.k3moe_dequant_mxfp4(v, v, 0, 64, v, None) == 0
    assert L.k3moe_dequant_mxfp4(ctypes.c_void_p(8), v, 4, 64, v, None) == ERR_ALIGN


def test_noalloc_scratch_limit_is_the_workspace_size_rule():
    """k3moe_forward_noalloc refuses, before touching a device, any call whose workspace
    (k3moe_workspace_bytes) exceeds its fixed scratch array: at K3 shapes 8 tokens fit
    and 9 (the first tensor-core batch) do not."""
    import re
    L = k3.lib()
    d = _d()
    text = open(k3._HEADER).read()
    m = re.search(r"#define K3MOE_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert m and (int(m.group(1)) << int(m.group(2))) == k3.NOALLOC_SCRATCH_BYTES
    cap = k3.NOALLOC_SCRATCH_BYTES
    assert L.k3moe_workspace_bytes(ctypes.byref(d), 8) <= cap < L.k3moe_workspace_bytes(ctypes.byref(d), 9)
    v = ctypes.c_void_p(16)
    ex = k3.ExpertsC(16, 16, 16, 16, 16, 16)
    assert L.k3moe_forward_noalloc(ctypes.byref(d), 9, v, v, v, v, v, v, ctypes.byref(ex), v, None, None,
                                   None) == ERR_WS
    assert L.k3moe_forward_noalloc(ctypes.byref(d), 0, v, v, v, v, v, v, ctypes.byref(ex), v, None, None,
                                   None) == 0
    import torch
    if not torch.cuda.is_available():  # a call that fits reaches the device check
        assert L.k3moe_forward_noalloc(ctypes.byref(d), 8, v, v, v, v, v, v, ctypes.byref(ex), v, None, None,
                                       None) == ERR_DEVICE
        st = ctypes.c_uint32(0)
        assert L.k3moe_device_status(None, ctypes.byref(st), None) == ERR_DEVICE


def test_tensor_core_threshold_moves_the_workspace_step():
    """k3moe_set_tc_min_tokens moves the token count at which the workspace grows by the
    tensor-core path's buffers, returns the previous value and rejects t < 1."""
    L = k3.lib()
    d = _d()
    prev = k3.set_tc_min_tokens(64)
    try:
        assert prev == 9
        step = lambda T: L.k3moe_workspace_bytes(ctypes.byref(d), T) - L.k3moe_workspace_bytes(ctypes.byref(d), T - 1)
        tc_bytes = 64 * 16 * 3584 * 2
        assert step(64) >= tc_bytes and step(63) < tc_bytes and step(9) < tc_bytes
        with pytest.raises(ValueError):
            k3.set_tc_min_tokens(0)
        assert k3.set_tc_min_tokens(64) == 64
    finally:
        k3.set_tc_min_tokens(prev)
    assert L.k3moe_set_tc_min_tokens(9) == 9


def test_shared_forward_validates_on_the_host():
    L = k3.lib()
    d = _d()
    assert L.k3moe_shared_workspace_bytes(ctypes.byref(d), 1, 6144) > 1 * 2 * 6144 * 4
    for bad in (0, -64, 100):
        assert L.k3moe_shared_workspace_bytes(ctypes.byref(d), 1, bad) == 0
    v = ctypes.c_void_p(16)
    nb = L.k3moe_shared_workspace_bytes(ctypes.byref(d), 1, 6144)
    assert L.k3moe_shared_forward(ctypes.byref(d), 0, 6144, v, v, v, v, v, nb, None) == 0
    assert L.k3moe_shared_forward(ctypes.byref(d), 1, 100, v, v, v, v, v, nb, None) == ERR_SHAPE
    assert L.k3moe_shared_forward(ctypes.byref(d), 1, 6144, None, v, v, v, v, nb, None) == ERR_ARG
    assert L.k3moe_shared_forward(ctypes.byref(d), 1, 6144, ctypes.c_void_p(24), v, v, v, v, nb, None) == ERR_ALIGN
    assert L.k3moe_shared_forward(ctypes.byref(d), 1, 6144, v, v, v, v, v, nb - 1, None) == ERR_WS
    import torch
    if not torch.cuda.is_available():
        assert L.k3moe_shared_forward(ctypes.byref(d), 1, 6144, v, v, v, v, v, nb, None) == ERR_DEVICE

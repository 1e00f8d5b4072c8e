"""GB300 (sm_103a) Stable LatentMoE routed-expert block on native MXFP4 weights.

Thin Python binding over the C ABI declared in ``include/k3moe.h``: every function
here only marshals arguments (torch tensors -> device pointers, the current CUDA
stream) and calls the compiled library, whose kernels do all the work.  There is
no Python or CPU fallback: if the library is missing or fails to load, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libk3moe.so")
_CSRC = os.path.join(_HERE, "csrc")
_HEADER = os.path.join(_ROOT, "include", "k3moe.h")
_lock = threading.Lock()
_lib = None

NOALLOC_SCRATCH_BYTES = 4 << 20  # K3MOE_NOALLOC_SCRATCH_BYTES

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared"]

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "pointer not 16-byte aligned",
          4: "workspace too small", 5: "current device is not compute capability 10.3", 6: "CUDA launch or copy failed"}
DEV_TIE_WINDOW, DEV_TIMEOUT, DEV_BAD_ID, DEV_SCALE_RANGE, DEV_ALIGN = 0x1, 0x2, 0x4, 0x8, 0x10


class K3MoEError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)} (status {code})")
        self.code = code


def _sources():
    return [os.path.join(_CSRC, f) for f in sorted(os.listdir(_CSRC)) if f.endswith((".cu", ".cuh"))] + [_HEADER]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/ into _build/libk3moe.so for sm_103a (in-tree)."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(f) for f in _sources())
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= newest:
        return _SO
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = [nvcc, *NVCC_FLAGS, "-o", tmp, os.path.join(_CSRC, "k3moe_api.cu")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + r.stdout + r.stderr)
    if verbose:
        print(r.stdout + r.stderr)
    os.replace(tmp, _SO)
    return _SO


class Dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("latent", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("inter", ctypes.c_int32), ("rms_eps", ctypes.c_float),
                ("top_p", ctypes.c_float), ("act_mxfp8", ctypes.c_int32)]


def dims(hidden, latent, n_experts, top_k, inter, rms_eps=1e-6, top_p=0.0, act_mxfp8=0) -> Dims:
    return Dims(hidden, latent, n_experts, top_k, inter, rms_eps, top_p, int(act_mxfp8))


class ExpertsC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")]


def lib():
    """The loaded C library (built on first use if absent)."""
    global _lib
    with _lock:
        if _lib is None:
            so = _SO if os.path.exists(_SO) else build()
            L = ctypes.CDLL(so)
            p, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
            D = ctypes.POINTER(Dims)
            X = ctypes.POINTER(ExpertsC)
            sigs = {
                "k3moe_workspace_bytes": ([D, i32], sz),
                "k3moe_route": ([D, i32, p, p, p, p, p, p, sz, p], ctypes.c_int),
                "k3moe_forward": ([D, i32, p, p, p, p, p, p, X, p, p, p, p, sz, p], ctypes.c_int),
                "k3moe_forward_profiled": ([D, i32, p, p, p, p, p, p, X, p, p, p, p, sz, p, p, i32], ctypes.c_int),
                "k3moe_expert_forward": ([D, i32, p, i32, X, p, p, sz, p], ctypes.c_int),
                "k3moe_shared_workspace_bytes": ([D, i32, i32], sz),
                "k3moe_shared_forward": ([D, i32, i32, p, p, p, p, p, sz, p], ctypes.c_int),
                "k3moe_forward_noalloc": ([D, i32, p, p, p, p, p, p, X, p, p, p, p], ctypes.c_int),
                "k3moe_dequant_mxfp4": ([p, p, i32, i32, p, p], ctypes.c_int),
                "k3moe_permute": ([D, i32, p, p, p, p, p, p, p, sz, p], ctypes.c_int),
                "k3moe_device_status": ([p, ctypes.POINTER(ctypes.c_uint32), p], ctypes.c_int),
                "k3moe_workspace_view": ([D, i32, p, i32], p),
                "k3moe_selftest_wait_timeout": ([p, sz, ctypes.c_int64, p], ctypes.c_int),
                "k3moe_set_tc_min_tokens": ([i32], i32),
                "k3moe_tc_min_tokens": ([], i32),
                "k3moe_set_tc_split_max_tokens": ([i32], i32),
                "k3moe_tc_split_max_tokens": ([], i32),
                "k3moe_status_str": ([ctypes.c_int], ctypes.c_char_p),
                "k3moe_abi_version": ([], i32),
            }
            for name, (args, res) in sigs.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _lib = L
        return _lib


def declared_functions() -> list:
    """Function names declared in include/k3moe.h."""
    import re
    txt = open(_HEADER).read()
    return sorted(set(re.findall(r"\b(k3moe_[a-z0-9_]+)\s*\(", txt)))


# ------------------------------------------------------------------------------ marshalling
def _ptr(t):
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code: int, what: str):
    if code != 0:
        raise K3MoEError(code, what)


class ExpertTables:
    """Device pointer tables of the six vendor tensors of every expert (the
    k3moe_experts struct).  Built from per-expert base addresses and the offsets of
    the six tensors inside an expert's block, e.g. a pool tensor holding all
    experts back to back."""

    def __init__(self, bases, offsets, device=None):
        import torch
        bases = torch.as_tensor(bases, dtype=torch.int64)
        self.tables = [(bases + int(o)).to(device or "cuda") for o in offsets]
        self.c = ExpertsC(*[t.data_ptr() for t in self.tables])

    @classmethod
    def from_pool(cls, pool, expert_bytes: int, offsets):
        import torch
        n = pool.numel() // expert_bytes
        bases = pool.data_ptr() + torch.arange(n, dtype=torch.int64) * expert_bytes
        return cls(bases, offsets, device=pool.device)


def workspace_bytes(d: Dims, T: int) -> int:
    return int(lib().k3moe_workspace_bytes(ctypes.byref(d), T))


def route(d: Dims, x, wr, bias, ids, w, ws, stream=None):
    _check(lib().k3moe_route(ctypes.byref(d), x.shape[0], _ptr(x), _ptr(wr), _ptr(bias), _ptr(ids), _ptr(w),
                             _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "k3moe_route")


def forward(d: Dims, x, wr, bias, w_down, w_up, norm_w, experts: ExpertTables, out, ws, ids_out=None, w_out=None,
            stream=None):
    _check(lib().k3moe_forward(ctypes.byref(d), x.shape[0], _ptr(x), _ptr(wr), _ptr(bias), _ptr(w_down), _ptr(w_up),
                               _ptr(norm_w), ctypes.byref(experts.c), _ptr(out), _ptr(ids_out), _ptr(w_out), _ptr(ws),
                               ws.numel() * ws.element_size(), _stream(stream)), "k3moe_forward")


def forward_noalloc(d: Dims, x, wr, bias, w_down, w_up, norm_w, experts: ExpertTables, out, ids_out=None,
                    w_out=None, stream=None):
    """k3moe_forward_noalloc: the block without a caller workspace (the library's own
    fixed device scratch; see include/k3moe.h for its size limit and sharing rules)."""
    _check(lib().k3moe_forward_noalloc(ctypes.byref(d), x.shape[0], _ptr(x), _ptr(wr), _ptr(bias), _ptr(w_down),
                                       _ptr(w_up), _ptr(norm_w), ctypes.byref(experts.c), _ptr(out), _ptr(ids_out),
                                       _ptr(w_out), _stream(stream)), "k3moe_forward_noalloc")


PHASES = ("proj", "route", "gateup", "down", "combine", "up")


def forward_profiled(d: Dims, x, wr, bias, w_down, w_up, norm_w, experts: ExpertTables, out, ws, events,
                     ids_out=None, w_out=None, stream=None):
    """k3moe_forward recording the given CUDA event handles (up to 7, cudaEvent_t as ints or
    c_void_p) at phase boundaries."""
    arr = (ctypes.c_void_p * len(events))(*[e.value if isinstance(e, ctypes.c_void_p) else e for e in events])
    _check(lib().k3moe_forward_profiled(ctypes.byref(d), x.shape[0], _ptr(x), _ptr(wr), _ptr(bias), _ptr(w_down),
                                        _ptr(w_up), _ptr(norm_w), ctypes.byref(experts.c), _ptr(out), _ptr(ids_out),
                                        _ptr(w_out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream),
                                        ctypes.cast(arr, ctypes.c_void_p), len(events)), "k3moe_forward_profiled")


def expert_forward(d: Dims, z, expert: int, experts: ExpertTables, out, ws, stream=None):
    _check(lib().k3moe_expert_forward(ctypes.byref(d), z.shape[0], _ptr(z), expert, ctypes.byref(experts.c),
                                      _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "k3moe_expert_forward")


def shared_workspace_bytes(d: Dims, T: int, inter_s: int) -> int:
    return int(lib().k3moe_shared_workspace_bytes(ctypes.byref(d), T, inter_s))


def shared_forward(d: Dims, x, w_gate_up, w_down, out, ws, stream=None):
    """k3moe_shared_forward: out [T, H] += the fused shared experts of x [T, H];
    w_gate_up [2 Is, H] (gate rows, then up rows), w_down [H, Is], all bf16."""
    inter_s = w_down.shape[1]
    _check(lib().k3moe_shared_forward(ctypes.byref(d), x.shape[0], inter_s, _ptr(x), _ptr(w_gate_up), _ptr(w_down),
                                      _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "k3moe_shared_forward")


def dequant_mxfp4(q, s, out, stream=None):
    O, half = q.shape
    _check(lib().k3moe_dequant_mxfp4(_ptr(q), _ptr(s), O, 2 * half, _ptr(out), _stream(stream)),
           "k3moe_dequant_mxfp4")


def permute(d: Dims, ids, counts, offsets, slot_of, uniq, n_uniq, ws, stream=None):
    _check(lib().k3moe_permute(ctypes.byref(d), ids.shape[0], _ptr(ids), _ptr(counts), _ptr(offsets), _ptr(slot_of),
                               _ptr(uniq), _ptr(n_uniq), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "k3moe_permute")


def device_status(ws, stream=None) -> int:
    """K3MOE_DEV_* bits of the last call that used workspace `ws`; ws=None reads the
    status of the last k3moe_forward_noalloc call on the current device."""
    v = ctypes.c_uint32(0)
    _check(lib().k3moe_device_status(_ptr(ws), ctypes.byref(v), _stream(stream)), "k3moe_device_status")
    return int(v.value)


def set_tc_min_tokens(t: int) -> int:
    """k3moe_set_tc_min_tokens: the token count from which the tensor-core GEMMs run
    (process-wide); returns the previous value."""
    prev = int(lib().k3moe_set_tc_min_tokens(int(t)))
    if prev < 0:
        raise ValueError("token threshold must be >= 1")
    return prev


def tc_min_tokens() -> int:
    """k3moe_tc_min_tokens: the token count from which the tensor-core GEMMs run."""
    return int(lib().k3moe_tc_min_tokens())


def set_tc_split_max_tokens(t: int) -> int:
    """k3moe_set_tc_split_max_tokens: below t tokens the exact tensor-core expert GEMMs take
    the bf16 activations as two exact MXFP8 terms on block-scaled MMAs, from t on the SMs
    decode the weights to bf16 (process-wide; 0 = never split); returns the previous value."""
    prev = int(lib().k3moe_set_tc_split_max_tokens(int(t)))
    if prev < 0:
        raise ValueError("token bound must be >= 0")
    return prev


def tc_split_max_tokens() -> int:
    """k3moe_tc_split_max_tokens: the token count from which the weight-decode form runs."""
    return int(lib().k3moe_tc_split_max_tokens())


SPLIT_ALWAYS = 1 << 30  # a bound no call reaches: the split form at every token count


def selftest_wait_timeout(ws, limit_cycles: int, stream=None):
    """k3moe_selftest_wait_timeout: a bounded device wait that runs out (sets DEV_TIMEOUT)."""
    _check(lib().k3moe_selftest_wait_timeout(_ptr(ws), ws.numel() * ws.element_size(), int(limit_cycles),
                                             _stream(stream)), "k3moe_selftest_wait_timeout")


def workspace_view(d: Dims, T: int, ws, which: int) -> int:
    return int(lib().k3moe_workspace_view(ctypes.byref(d), T, _ptr(ws), which) or 0)

"""Seeded, counter-based synthetic inputs for the LatentMoE routed-expert block.

This package is the one piece of code that both the fp64 oracle's tests and the GPU
tests/bench use.  It holds none of the block's arithmetic: only the generator
defined in ``k3gen.h`` (integer hash, uniform and normal draws) and the storage
rounding of drawn reals (to bf16 / f32).  Workload recipes live in ``configs.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_HOST_SO = os.path.join(_BUILD, "libk3gen_host.so")
_CUDA_SO = os.path.join(_BUILD, "libk3gen_cuda.so")
_lock = threading.Lock()
_host = None
_cuda = None


def build_host(force: bool = False) -> str:
    """Compile the host fill library (plain C, OpenMP when the compiler has it)."""
    os.makedirs(_BUILD, exist_ok=True)
    src = os.path.join(_HERE, "k3gen_host.c")
    if not force and os.path.exists(_HOST_SO) and os.path.getmtime(_HOST_SO) >= max(
        os.path.getmtime(src), os.path.getmtime(os.path.join(_HERE, "k3gen.h"))
    ):
        return _HOST_SO
    tmp = _HOST_SO + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _HOST_SO)
    return _HOST_SO


def build_cuda(force: bool = False) -> str:
    """Compile the device fill library used to materialise large expert pools in HBM."""
    os.makedirs(_BUILD, exist_ok=True)
    src = os.path.join(_HERE, "k3gen_cuda.cu")
    if not force and os.path.exists(_CUDA_SO) and os.path.getmtime(_CUDA_SO) >= max(
        os.path.getmtime(src), os.path.getmtime(os.path.join(_HERE, "k3gen.h"))
    ):
        return _CUDA_SO
    tmp = _CUDA_SO + f".tmp{os.getpid()}"
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    subprocess.run(
        [nvcc, "-O3", "-gencode", "arch=compute_103a,code=sm_103a", "-Xcompiler", "-fPIC", "-shared",
         "-o", tmp, src],
        check=True, capture_output=True,
    )
    os.replace(tmp, _CUDA_SO)
    return _CUDA_SO


def _host_lib():
    global _host
    with _lock:
        if _host is None:
            lib = ctypes.CDLL(build_host())
            u64, u32, p = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_void_p
            lib.k3gen_fill_u8.argtypes = [u64, u64, u64, p]
            lib.k3gen_fill_int_u8.argtypes = [u64, u64, u64, u32, u32, p]
            lib.k3gen_fill_uniform_f64.argtypes = [u64, u64, u64, ctypes.c_double, ctypes.c_double, p]
            lib.k3gen_fill_normal_f64.argtypes = [u64, u64, u64, ctypes.c_double, p]
            lib.k3gen_round_bf16.argtypes = [u64, p, p]
            lib.k3gen_round_f32.argtypes = [u64, p, p]
            for f in ("k3gen_fill_u8", "k3gen_fill_int_u8", "k3gen_fill_uniform_f64",
                      "k3gen_fill_normal_f64", "k3gen_round_bf16", "k3gen_round_f32"):
                getattr(lib, f).restype = None
            _host = lib
        return _host


def cuda_lib():
    global _cuda
    with _lock:
        if _cuda is None:
            lib = ctypes.CDLL(build_cuda())
            lib.k3gen_cuda_fill_pool.argtypes = [
                ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32,
                ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint32,
                ctypes.c_void_p]
            lib.k3gen_cuda_fill_pool.restype = ctypes.c_int
            _cuda = lib
        return _cuda


def _ptr(a: np.ndarray) -> int:
    assert a.flags.c_contiguous
    return a.ctypes.data


def u8(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint8)
    _host_lib().k3gen_fill_u8(seed, stream, n, _ptr(out))
    return out


def int_u8(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    assert 0 <= lo <= hi <= 255
    out = np.empty(n, dtype=np.uint8)
    _host_lib().k3gen_fill_int_u8(seed, stream, n, lo, hi, _ptr(out))
    return out


def uniform_f64(seed: int, stream: int, n: int, lo: float, hi: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _host_lib().k3gen_fill_uniform_f64(seed, stream, n, lo, hi, _ptr(out))
    return out


def normal_f64(seed: int, stream: int, n: int, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _host_lib().k3gen_fill_normal_f64(seed, stream, n, sigma, _ptr(out))
    return out


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (nearest-even); returns the raw uint16 bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    _host_lib().k3gen_round_bf16(a.size, _ptr(a), _ptr(out))
    return out


def f32(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.float32)
    _host_lib().k3gen_round_f32(a.size, _ptr(a), _ptr(out))
    return out


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (storage conversion, used to feed fp64 inputs)."""
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


if __name__ == "__main__":  # pragma: no cover
    print(build_host(), file=sys.stderr)

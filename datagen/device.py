"""Materialise the synthetic workloads on a CUDA device (torch tensors).

Small tensors come from the host generator and are copied; the expert pool
(896 x 17.5 MB at K3 shape) is filled directly in HBM by the device generator,
which evaluates the same integer hash (bit-identical to the host fill).
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import cuda_lib
from .configs import EXPERT_TENSORS, LayerConfig, expert_stream, layer_weights, layer_x


def bf16_tensor(bits: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def layer_tensors(cfg: LayerConfig, device="cuda") -> dict:
    import torch
    W = layer_weights(cfg)
    return {
        "x": bf16_tensor(layer_x(cfg), device),
        "wr": bf16_tensor(W["wr"], device),
        "bias": torch.from_numpy(W["bias"]).to(device),
        "wd": bf16_tensor(W["wd"], device),
        "wu": bf16_tensor(W["wu"], device),
        "gamma": torch.from_numpy(W["gamma"]).to(device),
    }


def expert_pool(cfg, device="cuda", n_experts: int | None = None):
    """All experts' vendor tensors back to back in one uint8 device tensor.
    Returns (pool, expert_bytes, offsets of the six tensors inside an expert)."""
    import torch
    layout, eb = cfg.expert_layout()
    E = n_experts if n_experts is not None else cfg.n_experts
    pool = torch.empty(E * eb, dtype=torch.uint8, device=device)
    lib = cuda_lib()
    stream = torch.cuda.current_stream(pool.device).cuda_stream
    for which, (name, off, n, _shape) in enumerate(layout):
        is_int = 0 if name.endswith("_q") else 1
        rc = lib.k3gen_cuda_fill_pool(ctypes.c_void_p(pool.data_ptr()), eb, off, n, E, cfg.seed, which, is_int,
                                      cfg.scale_lo, cfg.scale_hi, ctypes.c_void_p(stream))
        if rc != 0:
            raise RuntimeError(f"device fill failed ({rc})")
    return pool, eb, [off for (_n, off, _c, _s) in layout]


def expert_from_pool(pool, cfg, e: int) -> dict:
    """Copy expert e's six tensors back to the host (for checks)."""
    layout, eb = cfg.expert_layout()
    out = {}
    for name, off, n, shape in layout:
        out[name] = pool[e * eb + off: e * eb + off + n].cpu().numpy().reshape(shape)
    return out

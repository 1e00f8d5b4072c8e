"""Synthetic workload recipes for the LatentMoE routed-expert block.

Each recipe fixes shapes, seeds and value distributions.  Tensors come from the
counter-based generator in ``k3gen.h`` so any piece (one token, one expert) can be
regenerated alone.  Shapes follow the Kimi-K3 layer described on colibri PR #676
("Stable LatentMoE": 896 routed experts, top-16, latent 3584 behind 7168-wide
projections); distributions are the synthetic stand-ins for the real checkpoint.

Recipes (names are the workloads, by size):
  tiny      T=4, H=256, L=128, E=8, K=2, I=256; x~N(0,1); Wr~N(0,1/H); b~U(-0.1,0.1);
            Wd~N(0,1/H), Wu~N(0,1/L); packed bytes U(u8); scale bytes U[117,127]; seed 0
  expert    one expert at K3 shape, z[1,3584]~N(0,1); scale bytes U[118,124]
  decode    T=1 at K3 shape; Wr~N(0,1/7168); b~U(-0.05,0.05); gamma=1; scales U[118,124];
            the seed is the first seed >= 0 whose oracle 16th/17th biased-score gap
            exceeds 1e-4 (checked by the oracle tests)
  chunk     T=32 at K3 shape, same weights as decode; x_t = base_{t//8} + 0.3 N(0,1)
            with 4 base vectors ~N(0,1) (temporal locality: neighbouring tokens share
            a base)
  prefill   T=4096 at K3 shape; x~N(0,1); b=0 (flat expert marginals); scales U[117,127]
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from . import bf16_bits, f32, int_u8, normal_f64, u8, uniform_f64

# stream ids (mirror k3gen.h)
S_X, S_WR, S_BIAS, S_WD, S_WU, S_XBASE, S_XNOISE, S_EXPERT0 = 1, 2, 3, 4, 5, 6, 7, 0x1000
S_SGU, S_SDN = 8, 9
EXPERT_TENSORS = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")


def expert_stream(e: int, which: int) -> int:
    return S_EXPERT0 + e * 8 + which


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    hidden: int
    latent: int
    n_experts: int
    top_k: int
    inter: int
    seed: int  # weights and (unless x_seed is set) activations
    bias_range: float  # b ~ U(-r, r); 0 -> b = 0
    scale_lo: int
    scale_hi: int
    x_kind: str = "normal"  # "normal" or "perturbed"
    n_bases: int = 0
    perturb_sigma: float = 0.0
    rms_eps: float = 1e-6
    x_seed: int | None = None
    top_p: float = 0.0  # K3_TOPP cumulative-weight pruning of the top-K; 0 = off
    act_mxfp8: int = 0  # 1: MXFP8 activations into the expert contractions (the low-precision variant)

    @property
    def dims(self):
        return dict(hidden=self.hidden, latent=self.latent, n_experts=self.n_experts, top_k=self.top_k,
                    inter=self.inter, rms_eps=self.rms_eps, top_p=self.top_p, act_mxfp8=self.act_mxfp8)

    def with_tokens(self, T: int, x_seed: int | None = None) -> "LayerConfig":
        return dataclasses.replace(self, T=T, x_seed=x_seed)

    # ---- bytes of one expert in the vendor layout: six tensors back to back ----
    def expert_layout(self):
        """(name, offset, nbytes, shape) of the six tensors inside one expert's block."""
        I, L = self.inter, self.latent
        shapes = [(I, L // 2), (I, L // 32), (I, L // 2), (I, L // 32), (L, I // 2), (L, I // 32)]
        out, off = [], 0
        for name, shp in zip(EXPERT_TENSORS, shapes):
            n = shp[0] * shp[1]
            out.append((name, off, n, shp))
            off += (n + 255) // 256 * 256
        return out, off

    @property
    def expert_bytes(self) -> int:
        return self.expert_layout()[1]


TINY = LayerConfig("tiny", T=4, hidden=256, latent=128, n_experts=8, top_k=2, inter=256, seed=0,
                   bias_range=0.1, scale_lo=117, scale_hi=127)
# first seed >= 0 whose 16th/17th biased-score gap exceeds 1e-4 (verified in the oracle tests)
DECODE_SEED = 0
DECODE = LayerConfig("decode", T=1, hidden=7168, latent=3584, n_experts=896, top_k=16, inter=3072,
                     seed=DECODE_SEED, bias_range=0.05, scale_lo=118, scale_hi=124)
CHUNK = dataclasses.replace(DECODE, name="chunk", T=32, x_kind="perturbed", n_bases=4, perturb_sigma=0.3)
PREFILL = LayerConfig("prefill", T=4096, hidden=7168, latent=3584, n_experts=896, top_k=16, inter=3072,
                      seed=0, bias_range=0.0, scale_lo=117, scale_hi=127)
# a small layer of other widths that runs the tensor-core path: latent 768 (a gate/up
# contraction of six 128-element stages), inter 512 (a down contraction of four), hidden
# 1024, 32 experts, top-4, 40 tokens
MID = dataclasses.replace(TINY, name="mid", T=40, hidden=1024, latent=768, n_experts=32, top_k=4, inter=512,
                          seed=3, bias_range=0.05)
LAYER_CONFIGS = {c.name: c for c in (TINY, DECODE, CHUNK, PREFILL, MID)}


@dataclasses.dataclass(frozen=True)
class ExpertConfig:
    """One expert applied to one latent token (the single-expert GEMV workload)."""
    name: str = "expert"
    latent: int = 3584
    inter: int = 3072
    seed: int = 0
    expert: int = 0
    scale_lo: int = 118
    scale_hi: int = 124


EXPERT = ExpertConfig()


# ------------------------------------------------------------------------------------------
def layer_x(cfg: LayerConfig) -> np.ndarray:
    """Activations x [T, H] as bf16 bits."""
    T, H = cfg.T, cfg.hidden
    seed = cfg.seed if cfg.x_seed is None else cfg.x_seed
    if cfg.x_kind == "normal":
        return bf16_bits(normal_f64(seed, S_X, T * H)).reshape(T, H)
    if cfg.x_kind == "perturbed":
        per = max(1, math.ceil(T / cfg.n_bases))
        base = normal_f64(seed, S_XBASE, cfg.n_bases * H).reshape(cfg.n_bases, H)
        noise = normal_f64(seed, S_XNOISE, T * H).reshape(T, H)
        idx = np.minimum(np.arange(T) // per, cfg.n_bases - 1)
        return bf16_bits(base[idx] + cfg.perturb_sigma * noise)
    raise ValueError(cfg.x_kind)


def layer_weights(cfg: LayerConfig) -> dict:
    """Dense (non-expert) tensors: wr [E,H], wd [L,H], wu [H,L] as bf16 bits; bias [E], gamma [L] f32."""
    E, H, L = cfg.n_experts, cfg.hidden, cfg.latent
    s = cfg.seed
    out = {
        "wr": bf16_bits(normal_f64(s, S_WR, E * H, 1.0 / math.sqrt(H))).reshape(E, H),
        "wd": bf16_bits(normal_f64(s, S_WD, L * H, 1.0 / math.sqrt(H))).reshape(L, H),
        "wu": bf16_bits(normal_f64(s, S_WU, H * L, 1.0 / math.sqrt(L))).reshape(H, L),
        "gamma": np.ones(L, dtype=np.float32),
    }
    if cfg.bias_range > 0:
        out["bias"] = f32(uniform_f64(s, S_BIAS, E, -cfg.bias_range, cfg.bias_range))
    else:
        out["bias"] = np.zeros(E, dtype=np.float32)
    return out


# Shared experts beside the routed block: two SiTU-GLU experts on the hidden width, fused
# along the intermediate dimension.  The pages give no width; each is read as wide as a
# routed expert (I = 3072), so the fused width is 2 x 3072.
SHARED_INTER = 6144


def shared_weights(cfg: LayerConfig, inter_s: int = SHARED_INTER) -> dict:
    """Fused shared-expert weights as bf16 bits: wgu [2 Is, H] (gate rows, then up rows) and
    wdn [H, Is]."""
    H, s = cfg.hidden, cfg.seed
    return {
        "wgu": bf16_bits(normal_f64(s, S_SGU, 2 * inter_s * H, 1.0 / math.sqrt(H))).reshape(2 * inter_s, H),
        "wdn": bf16_bits(normal_f64(s, S_SDN, H * inter_s, 1.0 / math.sqrt(inter_s))).reshape(H, inter_s),
    }


def expert_tensors(cfg, e: int) -> dict:
    """The six vendor-layout tensors of expert e (uint8 arrays)."""
    I, L = cfg.inter, cfg.latent
    shapes = {"gate_q": (I, L // 2), "gate_s": (I, L // 32), "up_q": (I, L // 2), "up_s": (I, L // 32),
              "down_q": (L, I // 2), "down_s": (L, I // 32)}
    out = {}
    for which, name in enumerate(EXPERT_TENSORS):
        shp = shapes[name]
        n = shp[0] * shp[1]
        st = expert_stream(e, which)
        if name.endswith("_q"):
            out[name] = u8(cfg.seed, st, n).reshape(shp)
        else:
            out[name] = int_u8(cfg.seed, st, n, cfg.scale_lo, cfg.scale_hi).reshape(shp)
    return out


def expert_z(cfg: ExpertConfig) -> np.ndarray:
    """Latent activation [1, L] (bf16 bits) of the single-expert workload."""
    return bf16_bits(normal_f64(cfg.seed, S_X, cfg.latent)).reshape(1, cfg.latent)

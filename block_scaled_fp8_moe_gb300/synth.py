"""Seeded synthetic inputs for the MoE layer (no arithmetic of the layer itself lives here).

Shapes and distributions of the five workloads the layer is exercised on:

  tiny        T=4      H=256  E=8   k=2 I=128   bias N(0, 0.1)              seed 0
  decode-6    T=6      H=4096 E=256 k=8 I=2048  bias N(0, 0.1)              seed 1
  decode-48   T=48     H=4096 E=256 k=8 I=2048  bias N(0, 0.1), 14 dead rows seed 2
  prefill-4k  T=4096   H=4096 E=256 k=8 I=2048  bias 0 (uniform routing)    seed 3
  prefill-32k T=32768  H=4096 E=256 k=8 I=576   Zipf(1.1) bias, gamma 0.2   seed 4

x ~ N(0, 1) rounded to bf16; router weight ~ N(0, 0.02) rounded to bf16; expert weights
W13 [E, 2I, H] and W2 [E, H, I] ~ N(0, 0.02) in fp32 (each side quantises them itself).
Zipf bias: p_e proportional to r_e^-1.1 over a seeded permutation r of 1..E, bias_e =
gamma * ln(E * p_e). Dead rows: round(0.3 * T) rows picked by a seeded permutation.

Two generators: numpy's PCG64 (`default_rng`) on the CPU -- identical on every platform, used for
small cases and stored fixtures -- and torch's CUDA generator for the full-size workloads, where
CPU generation of ~6e9 normals would take minutes.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class MoeConfig:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    seed: int
    bias: str = "normal"      # "normal" | "zero" | "zipf"
    dead_frac: float = 0.0
    zipf_s: float = 1.1
    zipf_gamma: float = 0.2


CONFIGS = {
    "tiny": MoeConfig("tiny", 4, 256, 8, 2, 128, 0),
    "decode-6": MoeConfig("decode-6", 6, 4096, 256, 8, 2048, 1),
    "decode-48": MoeConfig("decode-48", 48, 4096, 256, 8, 2048, 2, dead_frac=0.3),
    "prefill-4k": MoeConfig("prefill-4k", 4096, 4096, 256, 8, 2048, 3, bias="zero"),
    "prefill-32k": MoeConfig("prefill-32k", 32768, 4096, 256, 8, 576, 4, bias="zipf"),
}


@dataclass
class MoeInputs:
    cfg: MoeConfig
    x: torch.Tensor           # bf16 [T, H]
    w_router: torch.Tensor    # bf16 [E, H]
    bias: torch.Tensor        # fp32 [E]
    dead: torch.Tensor        # uint8 [T]
    w13: torch.Tensor         # fp32 [E, 2I, H]
    w2: torch.Tensor          # fp32 [E, H, I]
    extra: dict = field(default_factory=dict)


def zipf_bias(E: int, s: float, gamma: float, perm: np.ndarray) -> np.ndarray:
    ranks = perm.astype(np.float64) + 1.0
    p = ranks ** -s
    p /= p.sum()
    return (gamma * np.log(E * p)).astype(np.float32)


def dead_mask(T: int, frac: float, perm: np.ndarray) -> np.ndarray:
    n_dead = int(round(frac * T))
    m = np.zeros(T, dtype=np.uint8)
    m[perm[:n_dead]] = 1
    return m


def _bias_and_dead(cfg: MoeConfig, rng: np.random.Generator):
    if cfg.bias == "normal":
        bias = (rng.standard_normal(cfg.E) * 0.1).astype(np.float32)
    elif cfg.bias == "zero":
        bias = np.zeros(cfg.E, dtype=np.float32)
    elif cfg.bias == "zipf":
        bias = zipf_bias(cfg.E, cfg.zipf_s, cfg.zipf_gamma, rng.permutation(cfg.E))
    else:
        raise ValueError(cfg.bias)
    dead = dead_mask(cfg.T, cfg.dead_frac, rng.permutation(cfg.T))
    return bias, dead


def make_inputs_cpu(cfg: MoeConfig, T: int | None = None) -> MoeInputs:
    """Everything from numpy PCG64(seed); portable and exact across machines."""
    T = cfg.T if T is None else T
    rng = np.random.default_rng(cfg.seed)
    bias, dead = _bias_and_dead(cfg, rng)
    x = torch.from_numpy(rng.standard_normal((T, cfg.H), dtype=np.float32)).to(torch.bfloat16)
    wr = torch.from_numpy(rng.standard_normal((cfg.E, cfg.H), dtype=np.float32) * np.float32(0.02)
                          ).to(torch.bfloat16)
    w13 = torch.from_numpy(rng.standard_normal((cfg.E, 2 * cfg.I, cfg.H), dtype=np.float32)
                           * np.float32(0.02))
    w2 = torch.from_numpy(rng.standard_normal((cfg.E, cfg.H, cfg.I), dtype=np.float32)
                          * np.float32(0.02))
    return MoeInputs(cfg, x, wr, torch.from_numpy(bias), torch.from_numpy(dead[:T].copy()), w13, w2)


def make_inputs_cuda(cfg: MoeConfig, device="cuda", with_weights: bool = True) -> MoeInputs:
    """Full-size inputs drawn on the GPU (torch CUDA generator seeded with cfg.seed); the bias
    and dead mask still come from numpy PCG64 so they match make_inputs_cpu exactly."""
    rng = np.random.default_rng(cfg.seed)
    bias, dead = _bias_and_dead(cfg, rng)
    g = torch.Generator(device=device)
    g.manual_seed(cfg.seed)
    x = torch.randn((cfg.T, cfg.H), generator=g, device=device).to(torch.bfloat16)
    wr = (torch.randn((cfg.E, cfg.H), generator=g, device=device) * 0.02).to(torch.bfloat16)
    w13 = w2 = None
    if with_weights:
        w13 = torch.randn((cfg.E, 2 * cfg.I, cfg.H), generator=g, device=device)
        w13.mul_(0.02)
        w2 = torch.randn((cfg.E, cfg.H, cfg.I), generator=g, device=device)
        w2.mul_(0.02)
    return MoeInputs(cfg, x, wr, torch.from_numpy(bias).to(device),
                     torch.from_numpy(dead).to(device), w13, w2)


def custom(name: str, T: int, H: int, E: int, k: int, I: int, seed: int, **kw) -> MoeConfig:
    return MoeConfig(name, T, H, E, k, I, seed, **kw)


def touched_experts_estimate(cfg: MoeConfig) -> float:
    """Expected number of distinct experts hit by T*k uniform picks (context only)."""
    return cfg.E * (1.0 - (1.0 - cfg.k / cfg.E) ** cfg.T) if cfg.T < 1e6 else float(cfg.E)


"""Seeded synthetic inputs for the selective-scan workloads.

This module only draws random numbers and lays them out; it holds none of the
scan's arithmetic.  Both the CUDA path (tests, bench) and the CPU oracle take
their inputs from here, so a parity comparison always sees bit-identical
inputs on both sides.

Layouts (all contiguous, row-major):
  u / x, delta, z, y : (B, D, L)      -- one row of L per (batch, channel)
  Bm, Cm             : (B, N, L)      -- shared by every channel of a batch row
  A                  : (D, N) float32
  Dskip, delta_bias  : (D,)   float32
  conv_w             : (D, W) float32, conv_b: (D,) float32
  h0 / state         : (B, D, N) float32

Distributions (S4D-real A, inverse-softplus dt bias, unit normals for the
input-dependent tensors) follow the initialisation described in
"Mamba tutorial" (lshu.cn) sections 6.2 and 3.1 and in "SSM applications and
engineering" (pwwt.cn) section 3.3 (the [1e-3, 1e-1] range of the step size).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

__all__ = ["ScanConfig", "DecodeConfig", "SsdConfig", "SCAN_CONFIGS", "DECODE_CONFIG", "SSD_CONFIGS",
           "make_scan_inputs", "make_decode_layer", "make_decode_pool", "decode_pool_index", "make_ssd_inputs",
           "seed_for"]


@dataclass(frozen=True)
class ScanConfig:
    name: str
    batch: int
    dim: int
    dstate: int
    seqlen: int
    dtype: str               # "f32" or "bf16" for u/x, delta, z, Bm, Cm and y
    conv: bool = False       # fused causal depthwise conv1d (width 4) + SiLU ahead of the scan
    has_z: bool = True
    has_D: bool = True
    zoh: bool = True
    bias_kind: str = "std"   # "std": dt0 ~ U[1e-3, 1e-1]; "halflife": log-uniform half-lives 10..1e4
    chunk: int = 0           # >0: the workload is also run as seqlen/chunk calls with carried state
    seed: int = 1000

    @property
    def elements(self) -> int:
        return self.batch * self.dim * self.seqlen * self.dstate


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    batch: int
    dim: int
    dstate: int
    layers: int
    steps: int
    seed: int = 1004


SCAN_CONFIGS = {
    "tiny": ScanConfig("tiny", 1, 16, 4, 64, "f32", seed=1000),
    "mamba130m": ScanConfig("mamba130m", 8, 1536, 16, 2048, "bf16", seed=1001),
    "mamba1.4b_conv": ScanConfig("mamba1.4b_conv", 8, 4096, 16, 2048, "bf16", conv=True, seed=1002),
    "long2.8b": ScanConfig("long2.8b", 1, 5120, 16, 65536, "bf16", bias_kind="halflife", chunk=2048,
                           seed=1003),
}

DECODE_CONFIG = DecodeConfig("decode2.8b", 256, 5120, 16, 64, 128, seed=1004)


def seed_for(base: int, tag: str) -> int:
    """Stable per-tensor seed: base seed mixed with a small tag hash (no Python hash randomisation)."""
    h = 0
    for ch in tag.encode():
        h = (h * 131 + ch) % 1000003
    return base * 1000003 + h


def _gen(base: int, tag: str) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed_for(base, tag))
    return g


def _io_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _dt_bias(dim: int, kind: str, g: torch.Generator) -> torch.Tensor:
    """Per-channel bias b with softplus(b) = dt0, i.e. b = log(expm1(dt0))."""
    r = torch.rand(dim, generator=g, dtype=torch.float64)
    if kind == "std":
        dt0 = 1e-3 + r * (1e-1 - 1e-3)
    elif kind == "halflife":
        # n = 0 state has A = -1, so its half-life is ln2 / dt0; draw half-lives log-uniformly in [10, 1e4].
        half = torch.exp(math.log(10.0) + r * (math.log(1e4) - math.log(10.0)))
        dt0 = math.log(2.0) / half
    else:
        raise ValueError(kind)
    return torch.log(torch.expm1(dt0)).to(torch.float32)


def make_scan_inputs(cfg: ScanConfig, *, batch: Optional[int] = None, dim: Optional[int] = None,
                     seqlen: Optional[int] = None, dstate: Optional[int] = None, dtype: Optional[str] = None,
                     with_h0: bool = False, seed: Optional[int] = None,
                     params_seed: Optional[int] = None) -> dict:
    """CPU tensors for one scan workload.  Overrides shrink or reshape the workload (parity edge cases)
    while keeping the config's distributions.  ``params_seed`` (default: the data seed) draws the
    per-channel parameters (D skip, dt bias, conv filter) apart from the per-row tensors, so several
    shards of one global batch can share one layer's parameters."""
    Bsz = cfg.batch if batch is None else batch
    D = cfg.dim if dim is None else dim
    L = cfg.seqlen if seqlen is None else seqlen
    N = cfg.dstate if dstate is None else dstate
    dt = _io_dtype(cfg.dtype if dtype is None else dtype)
    base = cfg.seed if seed is None else seed
    pbase = base if params_seed is None else params_seed

    def normal(tag, shape, std=1.0, src=None):
        t = torch.randn(shape, generator=_gen(base if src is None else src, tag), dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        return t

    out = {}
    out["u"] = normal("u", (Bsz, D, L)).to(dt)                     # x when the conv front end is on
    out["delta"] = normal("delta", (Bsz, D, L), 0.5).to(dt)        # raw step, N(0, 0.5^2)
    out["z"] = normal("z", (Bsz, D, L)).to(dt) if cfg.has_z else None
    out["Bm"] = normal("B", (Bsz, N, L)).to(dt)
    out["Cm"] = normal("C", (Bsz, N, L)).to(dt)
    out["A"] = (-torch.arange(1, N + 1, dtype=torch.float32)).repeat(D, 1).contiguous()
    out["Dskip"] = normal("D", (D,), src=pbase) if cfg.has_D else None
    out["delta_bias"] = _dt_bias(D, cfg.bias_kind, _gen(pbase, "bias"))
    if cfg.conv:
        out["conv_w"] = normal("conv_w", (D, 4), 0.5, src=pbase)    # variance 1/4
        out["conv_b"] = torch.zeros(D, dtype=torch.float32)
    else:
        out["conv_w"] = None
        out["conv_b"] = None
    out["h0"] = normal("h0", (Bsz, D, N), 0.5) if with_h0 else None
    out["zoh"] = cfg.zoh
    out["delta_softplus"] = True
    return out


def make_decode_layer(cfg: DecodeConfig, layer: int, *, device="cpu", batch: Optional[int] = None) -> dict:
    """Per-layer constants of the decode workload (fp32 A, D skip, dt bias) and its initial fp32 state
    cache (B, D, N) ~ N(0, 0.5^2).  The state is drawn with a generator on ``device`` so that the
    full 64-layer cache (5.4 GB) never has to pass through host memory; tests read the sampled rows
    back from the device copy, so both sides still see identical values."""
    Bsz = cfg.batch if batch is None else batch
    base = cfg.seed * 131 + layer
    g = torch.Generator(device=device)
    g.manual_seed(seed_for(base, "state"))
    state = torch.randn((Bsz, cfg.dim, cfg.dstate), generator=g, dtype=torch.float32, device=device)
    return {
        "A": (-torch.arange(1, cfg.dstate + 1, dtype=torch.float32)).repeat(cfg.dim, 1).contiguous().to(device),
        "Dskip": torch.randn(cfg.dim, generator=_gen(base, "Dskip"), dtype=torch.float32).to(device),
        "delta_bias": _dt_bias(cfg.dim, "std", _gen(base, "bias")).to(device),
        "state": state.mul_(0.5),
    }


def make_decode_pool(cfg: DecodeConfig, pool: int, *, device="cpu", batch: Optional[int] = None) -> dict:
    """``pool`` distinct per-token input sets, stacked on a leading axis: bf16 u/delta/z (P, B, D) and
    Bm/Cm (P, B, N) with the tiny-config distributions.  Call (layer, step) reads set
    ``decode_pool_index(layer, step, pool)``; with pool * set size above the L2 size the inputs of a
    call always come from HBM."""
    Bsz = cfg.batch if batch is None else batch
    g = torch.Generator(device=device)
    g.manual_seed(seed_for(cfg.seed, "pool"))
    bf = torch.bfloat16

    def normal(shape, std=1.0):
        return torch.randn(shape, generator=g, dtype=torch.float32, device=device).mul_(std).to(bf)

    return {
        "u": normal((pool, Bsz, cfg.dim)),
        "delta": normal((pool, Bsz, cfg.dim), 0.5),
        "z": normal((pool, Bsz, cfg.dim)),
        "Bm": normal((pool, Bsz, cfg.dstate)),
        "Cm": normal((pool, Bsz, cfg.dstate)),
    }


def decode_pool_index(layer: int, step: int, pool: int) -> int:
    return (layer + step) % pool


@dataclass(frozen=True)
class SsdConfig:
    """A Mamba-2 (SSD) layer: H heads of P channels (d_inner = H * P), one scalar A per head, B and C
    shared by the H / G heads of each of G groups, state N per channel."""
    name: str
    batch: int
    nheads: int
    headdim: int
    ngroups: int
    dstate: int
    seqlen: int
    has_z: bool = False
    has_D: bool = True
    zoh: bool = False
    seed: int = 2000

    @property
    def dim(self) -> int:
        return self.nheads * self.headdim

    @property
    def elements(self) -> int:
        return self.batch * self.dim * self.seqlen * self.dstate


SSD_CONFIGS = {
    # small: several chunks of 128 steps and a ragged tail, two groups of two heads
    "ssd_small": SsdConfig("ssd_small", 2, 4, 64, 2, 128, 200, has_z=True, seed=2000),
    # a Mamba-2 2.7B layer: d_model 2560, expand 2, head dim 64 -> 80 heads, d_state 128, one group
    "mamba2_2.7b": SsdConfig("mamba2_2.7b", 8, 80, 64, 1, 128, 2048, seed=2001),
}


def make_ssd_inputs(cfg: SsdConfig, *, batch: Optional[int] = None, nheads: Optional[int] = None,
                    ngroups: Optional[int] = None, seqlen: Optional[int] = None, dstate: Optional[int] = None,
                    with_h0: bool = False, has_z: Optional[bool] = None, seed: Optional[int] = None) -> dict:
    """CPU tensors for one SSD workload (bf16 x, dt, B, C, z; fp32 A, D skip, dt bias, h0).

      x, z   (B, H * P, L)   channel d = h * P + p, contiguous in L (the Mamba-1 layout)
      dt     (B, H, L)       raw step of each head, N(0, 0.5^2)
      A      (H,)            -U[1, 16]
      Bm, Cm (B, G, L, N)    unit normals; head h reads group h // (H / G)
      Dskip, dt_bias (H,)    N(0, 1); inverse softplus of dt0 ~ U[1e-3, 1e-1]
      h0     (B, H, P, N)    N(0, 0.5^2) when asked for
    """
    Bsz = cfg.batch if batch is None else batch
    H = cfg.nheads if nheads is None else nheads
    G = cfg.ngroups if ngroups is None else ngroups
    L = cfg.seqlen if seqlen is None else seqlen
    P = cfg.headdim
    N = cfg.dstate if dstate is None else dstate
    base = cfg.seed if seed is None else seed
    bf = torch.bfloat16

    def normal(tag, shape, std=1.0):
        t = torch.randn(shape, generator=_gen(base, tag), dtype=torch.float32)
        return t.mul_(std) if std != 1.0 else t

    z_on = cfg.has_z if has_z is None else has_z
    return {
        "x": normal("x", (Bsz, H * P, L)).to(bf),
        "dt": normal("dt", (Bsz, H, L), 0.5).to(bf),
        "A": -(1.0 + 15.0 * torch.rand(H, generator=_gen(base, "A"), dtype=torch.float32)),
        "Bm": normal("B", (Bsz, G, L, N)).to(bf),
        "Cm": normal("C", (Bsz, G, L, N)).to(bf),
        "Dskip": normal("D", (H,)) if cfg.has_D else None,
        "dt_bias": _dt_bias(H, "std", _gen(base, "bias")),
        "z": normal("z", (Bsz, H * P, L)).to(bf) if z_on else None,
        "h0": normal("h0", (Bsz, H, P, N), 0.5) if with_h0 else None,
        "nheads": H,
        "ngroups": G,
        "zoh": cfg.zoh,
        "delta_softplus": True,
    }

"""Seeded synthetic inputs for the forward MoE layer.

This module only draws random tensors with the shapes, dtypes and load patterns of
the layer's workloads.  It holds no step of the layer's arithmetic, and both the
CUDA path and the oracle take their inputs from it.

Recipe (one generator per call, ``seed`` = 0 unless given):
  x        ~ N(0, 1)                  [N, H]
  W_r^T    ~ N(0, 1/H)                [E, H]     router weight, stored expert-major
  W_gate^T ~ N(0, 1/H), W_up^T ~ N(0, 1/H)  stacked as w_gate_up [E, 2I, H]
                                      (rows 0..I-1 gate, rows I..2I-1 up), K-major
  W_down^T ~ N(0, 1/I)                [E, H, I]  K-major
  bias b_e = c * log(1/rank_e)        [E] f32, only for the skewed workloads; the
                                      ranks are a seeded permutation of 1..E.
Values are drawn in FP32 and rounded once to the workload's master dtype (FP32 for
the tiny workload, BF16 otherwise).  MXFP8 operands are made from the BF16 masters
by each side's own quantiser, never stored here.

Small workloads draw on the CPU generator; the full-size ones draw on the device's
generator (expert by expert, to keep temporaries small).  A given workload always
uses the same device choice, so the two sides see identical bits.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    N: int          # tokens
    H: int          # hidden size
    I: int          # expert intermediate size
    E: int          # experts
    k: int          # experts per token
    S: int          # virtual source shards (N/S tokens each)
    dtype: str      # "f32" | "bf16" | "mxfp8"
    skew: float = 0.0   # c in b_e = c*log(1/rank_e); 0 means no router bias
    seed: int = 0

    @property
    def T(self) -> int:
        return self.N * self.k

    @property
    def rows_per_shard(self) -> int:
        return self.N // self.S

    @property
    def ffn_flops(self) -> int:
        """Algorithmic expert-FFN FLOPs: 2*H*2I (gate+up) + 2*I*H (down) per slot."""
        return 6 * self.H * self.I * self.T

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # FP32 tiny layer: every token checked against the oracle.
    "tiny_f32": Workload("tiny_f32", N=64, H=128, I=256, E=8, k=2, S=2, dtype="f32"),
    # BF16 small layer with balanced load (i.i.d. router logits).
    "small_bf16": Workload("small_bf16", N=4096, H=2048, I=1408, E=64, k=6, S=8, dtype="bf16"),
    # DeepSeek-V3-shaped layer, MXFP8 GEMM operands, BF16 in/out, balanced load.
    "dsv3_mxfp8": Workload("dsv3_mxfp8", N=8192, H=7168, I=2048, E=256, k=8, S=64, dtype="mxfp8"),
    # Same shapes with a Zipf-like router bias b_e = 3*log(1/rank_e).
    "dsv3_mxfp8_skew": Workload("dsv3_mxfp8_skew", N=8192, H=7168, I=2048, E=256, k=8, S=64,
                                dtype="mxfp8", skew=3.0),
    # The same layer at the mid skew the skewed configuration describes (hottest
    # expert about 18x the mean, a long tail of small experts, none empty): the
    # bias coefficient 0.5 instead of 3, which saturates (8 experts take every
    # token, 225 are empty).
    "dsv3_mxfp8_skew05": Workload("dsv3_mxfp8_skew05", N=8192, H=7168, I=2048, E=256, k=8, S=64,
                                  dtype="mxfp8", skew=0.5),
    # Profiling stand-in: DeepSeek-V3 shapes and per-expert load (T/E = 256 rows),
    # 32 experts, so a capture holds ~1.4 GB of weights instead of 11.6 GB.
    "dsv3_mxfp8_e32": Workload("dsv3_mxfp8_e32", N=1024, H=7168, I=2048, E=32, k=8, S=8,
                               dtype="mxfp8"),
    # The forward half of the 16384-token skewed layer (N=16384, 128 shards of 128).
    "dsv3_mxfp8_skew_16k": Workload("dsv3_mxfp8_skew_16k", N=16384, H=7168, I=2048, E=256, k=8,
                                    S=128, dtype="mxfp8", skew=3.0),
    # Profiling stand-in for the router pass: DeepSeek-V3 router shape (N=8192,
    # H=7168, E=256, top-8) with small experts (I=128), ~3 GB on the device.
    "dsv3_router_prof": Workload("dsv3_router_prof", N=8192, H=7168, I=128, E=256, k=8, S=64,
                                 dtype="mxfp8"),
    # Profiling stand-in for the hot experts of the skewed layers: DeepSeek-V3 shapes,
    # 8 experts that every token picks (k=8), so each expert's weight-gradient tiles
    # reduce over 2048 slots; ~3 GB on the device.
    "dsv3_mxfp8_hot8": Workload("dsv3_mxfp8_hot8", N=2048, H=7168, I=2048, E=8, k=8, S=16,
                                dtype="mxfp8"),
}

# Workloads whose tensors are drawn on the device generator (too large for the host).
DEVICE_DRAWN = {"dsv3_mxfp8", "dsv3_mxfp8_skew", "dsv3_mxfp8_skew05", "dsv3_mxfp8_e32",
                "dsv3_router_prof", "dsv3_mxfp8_skew_16k", "dsv3_mxfp8_hot8"}


def master_dtype(w: Workload) -> torch.dtype:
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def _normal(shape, std, gen, device, dtype):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    return (t * std).to(dtype)


def router_bias(w: Workload) -> torch.Tensor | None:
    """b_e = c * log(1/rank_e), ranks a permutation of 1..E drawn from seed+1 (CPU)."""
    if w.skew == 0.0:
        return None
    g = torch.Generator(device="cpu").manual_seed(w.seed + 1)
    ranks = torch.randperm(w.E, generator=g).to(torch.float64) + 1.0
    return (w.skew * torch.log(1.0 / ranks)).to(torch.float32)


def make_inputs(w: Workload, device: str | torch.device | None = None,
                with_weights: bool = True) -> dict:
    """Draw x, the router weight, the optional bias and the expert weights.

    Returns a dict of tensors on ``device`` (default: CPU for small workloads,
    cuda for the full-size ones).  Drawing order is fixed: x, W_r, then per expert
    gate, up, down.
    """
    if device is None:
        device = "cuda" if w.name in DEVICE_DRAWN else "cpu"
    device = torch.device(device)
    gen = torch.Generator(device=device).manual_seed(w.seed)
    dt = master_dtype(w)
    out = {
        "x": _normal((w.N, w.H), 1.0, gen, device, dt),
        "w_router": _normal((w.E, w.H), 1.0 / math.sqrt(w.H), gen, device, dt),
    }
    b = router_bias(w)
    out["bias"] = None if b is None else b.to(device)
    if with_weights:
        wgu = torch.empty((w.E, 2 * w.I, w.H), dtype=dt, device=device)
        wd = torch.empty((w.E, w.H, w.I), dtype=dt, device=device)
        for e in range(w.E):
            wgu[e, : w.I] = _normal((w.I, w.H), 1.0 / math.sqrt(w.H), gen, device, dt)
            wgu[e, w.I:] = _normal((w.I, w.H), 1.0 / math.sqrt(w.H), gen, device, dt)
            wd[e] = _normal((w.H, w.I), 1.0 / math.sqrt(w.I), gen, device, dt)
        out["w_gate_up"] = wgu
        out["w_down"] = wd
    return out

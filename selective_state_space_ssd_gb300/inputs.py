"""Seeded synthetic inputs shared by the CUDA path's tests, the oracle's tests
and the benchmark.

This module only draws random numbers; it holds none of the scan's
arithmetic.  Both implementations receive exactly the same values: bf16
inputs are rounded once here, and the oracle gets them widened to float64.

Recipe (one torch CPU generator, seed 0 unless given, draws in the fixed
order x, dt_raw, A, B, C, s0, dy, ds_final):

* x, dy, ds_final ~ N(0, 1)
* dt_raw ~ U(-4, -1)                          (Mamba-2, Mamba-1)
* A = -exp(U(0, ln 16))  per head (Mamba-2), per [D, N] (Mamba-1)
* B, C ~ N(0, 1) / sqrt(N)
* s0 ~ 0.1 * N(0, 1)
* MIMO: the x slot carries v ~ N(0, 1) [b,T,R,H,P]; the dt_raw slot carries
  the pre-combined decay da = softplus(u) * a_h with u ~ U(-4, -1) and
  a_h = -exp(U(0, ln 16)) per head, made with torch's softplus as part of the
  input recipe; A is absent.
"""
from __future__ import annotations

import math

import torch

_BF16 = torch.bfloat16


def _io(t: torch.Tensor, dtype: str) -> torch.Tensor:
    return t.to(_BF16) if dtype == "bf16" else t.contiguous()


def shapes(cfg: dict) -> dict:
    """Shapes of every input and output of ``cfg`` (library layouts)."""
    v, b, T = cfg["variant"], cfg["batch"], cfg["seqlen"]
    H, P, N, G, R = cfg["nheads"], cfg["headdim"], cfg["dstate"], cfg["ngroups"], cfg["mimo_rank"]
    if v == "mamba2":
        return dict(x=(b, T, H, P), dt_raw=(b, T, H), A=(H,), B=(b, T, G, N), C=(b, T, G, N),
                    s0=(b, H, P, N))
    if v == "mamba1":
        return dict(x=(b, T, H), dt_raw=(b, T, H), A=(H, N), B=(b, T, N), C=(b, T, N), s0=(b, H, N))
    if v == "mimo":
        return dict(x=(b, T, R, H, P), dt_raw=(b, T, H), A=None, B=(b, T, R, H, N), C=(b, T, R, H, N),
                    s0=(b, H, P, N))
    raise ValueError(v)


def make_inputs(cfg: dict, seed: int = 0, zero_s0: bool = False) -> dict:
    """Draw the inputs of ``cfg`` on the CPU.  x, B, C, dy are bf16 for bf16
    configs (fp32 otherwise); dt_raw, A, s0, ds_final are always fp32."""
    g = torch.Generator().manual_seed(seed)
    sh = shapes(cfg)
    dtype = cfg["dtype"]
    N = cfg["dstate"]
    out = {}
    out["x"] = _io(torch.randn(sh["x"], generator=g), dtype)
    if cfg["variant"] == "mimo":
        u = torch.rand(sh["dt_raw"], generator=g) * 3.0 - 4.0
        a = -torch.exp(torch.rand((cfg["nheads"],), generator=g) * math.log(16.0))
        out["dt_raw"] = (torch.nn.functional.softplus(u) * a).float().contiguous()
        out["A"] = None
    else:
        out["dt_raw"] = (torch.rand(sh["dt_raw"], generator=g) * 3.0 - 4.0).contiguous()
        out["A"] = (-torch.exp(torch.rand(sh["A"], generator=g) * math.log(16.0))).contiguous()
    out["B"] = _io(torch.randn(sh["B"], generator=g) / math.sqrt(N), dtype)
    out["C"] = _io(torch.randn(sh["C"], generator=g) / math.sqrt(N), dtype)
    s0 = 0.1 * torch.randn(sh["s0"], generator=g)
    out["s0"] = torch.zeros_like(s0) if zero_s0 else s0.contiguous()
    out["dy"] = _io(torch.randn(sh["x"], generator=g), dtype)
    out["ds_final"] = torch.randn(sh["s0"], generator=g).contiguous()
    return out


def kda_shapes(cfg: dict) -> dict:
    """Shapes of the KDA inputs (library layouts)."""
    b, T, H, HV, K, V = (cfg[n] for n in ("batch", "seqlen", "nheads", "value_heads", "key_dim", "value_dim"))
    return dict(q=(b, T, H, K), k=(b, T, H, K), v=(b, T, HV, V), g=(b, T, HV, K), beta=(b, T, HV),
                s0=(b, HV, K, V), do=(b, T, HV, V), ds_final=(b, HV, K, V))


def make_kda_inputs(cfg: dict, seed: int = 0, zero_s0: bool = False) -> dict:
    """Draw the KDA inputs on the CPU (fp32), in the fixed order q, k, v, g,
    beta, s0, do, ds_final:

    * q, v, do, ds_final ~ N(0, 1)
    * k: N(0, 1) draws scaled to unit length per (b, t, h), so that every step's
      I - beta k k^T keeps the state bounded over long sequences
    * g = -U(0.01, 0.5) per key row (exp(g) in (0.61, 0.99))
    * beta = U(0, 1)
    * s0 ~ 0.1 * N(0, 1)
    The attention scale is K^-1/2 (``kda_scale``)."""
    g = torch.Generator().manual_seed(seed)
    sh = kda_shapes(cfg)
    out = {}
    out["q"] = torch.randn(sh["q"], generator=g).contiguous()
    kr = torch.randn(sh["k"], generator=g)
    out["k"] = (kr / kr.norm(dim=-1, keepdim=True)).contiguous()
    out["v"] = torch.randn(sh["v"], generator=g).contiguous()
    out["g"] = (-(torch.rand(sh["g"], generator=g) * 0.49 + 0.01)).contiguous()
    out["beta"] = torch.rand(sh["beta"], generator=g).contiguous()
    s0 = 0.1 * torch.randn(sh["s0"], generator=g)
    out["s0"] = torch.zeros_like(s0) if zero_s0 else s0.contiguous()
    out["do"] = torch.randn(sh["do"], generator=g).contiguous()
    out["ds_final"] = torch.randn(sh["ds_final"], generator=g).contiguous()
    return out


def kda_scale(cfg: dict) -> float:
    return 1.0 / math.sqrt(cfg["key_dim"])


def as_float64(inputs: dict) -> dict:
    """The same values widened to float64 numpy arrays (for the oracle)."""
    return {k: (None if v is None else v.double().numpy()) for k, v in inputs.items()}

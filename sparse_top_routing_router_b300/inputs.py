"""Seeded synthetic inputs for the MoE-layer workloads.

Both the CUDA path and the CPU oracle are fed from here; this module holds none of the
method's arithmetic, only the input recipe:

* hidden states X ~ N(0, x_std^2), rounded to the workload dtype (bf16 round-to-nearest
  from an fp32 draw, or kept fp32);
* router weight W_g[H, E] ~ N(0, w_std^2), always fp32 (the router runs in fp32, as the
  "Mixture of Experts" study notes insist for the router softmax);
* expert weights ~ N(0, w_std^2) in the workload dtype, stored output-major:
  W_gate[e], W_up[e] are [I, H] and W_down[e] is [H, I] (the transpose of the
  [H, I] orientation in which "LLM Internals §14.2.1" writes the product, so that both
  operands of every expert GEMM are contiguous along the reduction axis);
* sigmoid workloads: a selection-only expert bias b ~ N(0, selection_bias_std^2);
* Zipf-skewed workloads: a fixed logit offset -s * ln(e + 1) per expert (expert 0 hottest).

Draw order is fixed, so one seed fixes every tensor on a given device type.  Large
weight stacks are drawn one expert at a time to bound the fp32 temporary.
"""

from __future__ import annotations

import math
from typing import Dict, Optional

import torch

from .configs import MoEConfig


def _dtype(cfg: MoEConfig) -> torch.dtype:
    return torch.bfloat16 if cfg.dtype == "bf16" else torch.float32


def _normal(g: torch.Generator, shape, std: float, device, out_dtype) -> torch.Tensor:
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(out_dtype)


def _stack(g, E, shape, std, device, dt) -> torch.Tensor:
    out = torch.empty((E,) + tuple(shape), device=device, dtype=dt)
    for e in range(E):
        out[e].copy_(_normal(g, shape, std, device, dt))
    return out


def make_inputs(cfg: MoEConfig, device="cpu", seed: Optional[int] = None,
                with_experts: bool = True) -> Dict[str, torch.Tensor]:
    """All tensors of one workload, drawn from a torch generator seeded with `seed`."""
    seed = cfg.seed if seed is None else seed
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = _dtype(cfg)
    T, H, E, I = cfg.T, cfg.H, cfg.E, cfg.I
    d: Dict[str, torch.Tensor] = {}
    d["X"] = _normal(g, (T, H), cfg.x_std, device, dt)
    d["Wg"] = _normal(g, (H, E), cfg.w_std, device, torch.float32)
    if cfg.selection_bias_std > 0:
        d["bias"] = _normal(g, (E,), cfg.selection_bias_std, device, torch.float32)
    if cfg.zipf_s > 0:
        off = [-cfg.zipf_s * math.log(e + 1.0) for e in range(E)]
        d["logit_bias"] = torch.tensor(off, dtype=torch.float64).to(torch.float32).to(device)
    if with_experts:
        d["W_gate"] = _stack(g, E, (I, H), cfg.w_std, device, dt)
        d["W_up"] = _stack(g, E, (I, H), cfg.w_std, device, dt)
        d["W_down"] = _stack(g, E, (H, I), cfg.w_std, device, dt)
        if cfg.shared:
            d["Ws_gate"] = _normal(g, (I, H), cfg.w_std, device, dt)
            d["Ws_up"] = _normal(g, (I, H), cfg.w_std, device, dt)
            d["Ws_down"] = _normal(g, (H, I), cfg.w_std, device, dt)
    return d


def token_subset(T: int, n: int, seed: int = 1) -> torch.Tensor:
    """A seeded sorted sample of n distinct token indices (all of them when n >= T)."""
    if n >= T:
        return torch.arange(T)
    g = torch.Generator()
    g.manual_seed(seed)
    return torch.randperm(T, generator=g)[:n].sort().values

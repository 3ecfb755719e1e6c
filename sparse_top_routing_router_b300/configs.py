"""The five MoE-layer workloads this library is measured and checked on.

Shapes follow the public configurations quoted in "LLM Internals §14.2 (Mixture of
Experts)": §14.2.1 (DeepSeek-V3 shapes: hidden 7168, expert width 2048, 256 routed
experts, top-8), §14.2.4 (one shared expert, same width as a routed expert) and
Table 14-5 (Mixtral 8x7B: 8 experts, top-2, width 14336). The Switch-style workload
follows the capacity discussion of §14.2.3 and the "AI Knowledge Map - MoE" capacity
worked example (C = ceil(c*N*k/E)).

This module holds data only: no arithmetic of the method.
"""

from __future__ import annotations

import dataclasses
from typing import Optional, Tuple


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int                      # tokens in the batch
    H: int                      # hidden size
    E: int                      # routed experts
    I: int                      # SwiGLU intermediate width of one expert
    k: int                      # experts per token
    score: str                  # "softmax" or "sigmoid"
    renorm: bool                # renormalise the gates over the k chosen experts
    shared: bool                # one always-on shared expert of width I
    dtype: str                  # "bf16" or "f32": hidden states and expert weights
    capacity_factors: Tuple[float, ...] = ()   # () = dropless
    selection_bias_std: float = 0.0            # sigmoid: per-expert bias for selection only
    zipf_s: float = 0.0                        # >0: logit offset -s*ln(e+1) per expert
    alpha: float = 0.0                         # balance-loss coefficient
    expert_choice: bool = False                # every expert takes its C = T*k/E best tokens
    fp8_experts: bool = False                  # expert weights as FP8 E4M3 + channel scales
    n_groups: int = 0                          # group-limited routing: expert groups
    topk_groups: int = 0                       # ... and the groups a token may use
    x_std: float = 1.0
    w_std: float = 0.02
    seed: int = 0

    @property
    def slots(self) -> int:
        return self.T * self.k

    def flops(self, kept_rows: Optional[int] = None) -> float:
        """Algorithmic FLOPs of one forward: router GEMM + routed experts + shared expert."""
        R = self.slots if kept_rows is None else kept_rows
        f = 2.0 * self.T * self.H * self.E
        f += 2.0 * R * 3 * self.H * self.I
        if self.shared:
            f += 2.0 * self.T * 3 * self.H * self.I
        return f


TINY_F32 = MoEConfig(
    name="tiny_f32", T=64, H=128, E=8, I=256, k=2, score="softmax", renorm=True,
    shared=False, dtype="f32")

MIXTRAL = MoEConfig(
    name="mixtral_bf16", T=4096, H=4096, E=8, I=14336, k=2, score="softmax",
    renorm=True, shared=False, dtype="bf16")

DSV3_PREFILL = MoEConfig(
    name="dsv3_prefill_bf16", T=8192, H=7168, E=256, I=2048, k=8, score="sigmoid",
    renorm=True, shared=True, dtype="bf16", selection_bias_std=0.1)

DSV3_DECODE = dataclasses.replace(DSV3_PREFILL, name="dsv3_decode_bf16", T=64)

SWITCH = MoEConfig(
    name="switch_capacity_bf16", T=16384, H=4096, E=64, I=8192, k=1, score="softmax",
    renorm=False, shared=False, dtype="bf16", capacity_factors=(1.0, 1.25),
    zipf_s=1.2, alpha=0.01)

ALL = (TINY_F32, MIXTRAL, DSV3_PREFILL, DSV3_DECODE, SWITCH)
BY_NAME = {c.name: c for c in ALL}


def scaled(cfg: MoEConfig, **kw) -> MoEConfig:
    """The same layer recipe at other sizes (used for the ragged/small parity cases)."""
    name = kw.pop("name", cfg.name + "_scaled")
    return dataclasses.replace(cfg, name=name, **kw)

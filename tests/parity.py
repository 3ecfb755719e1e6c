"""Shared helpers of the GPU parity tests: run the layer through the C ABI, run the
fp64 oracle on the same seeded inputs, compare."""

from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np
import torch

from oracle import moe_oracle as O
from sparse_top_routing_router_b300 import binding as B
from sparse_top_routing_router_b300.configs import MoEConfig
from sparse_top_routing_router_b300.inputs import make_inputs, token_subset
from sparse_top_routing_router_b300.layer import MoELayer

GAP_EXCLUDE = 1e-6          # rows whose k-th/(k+1)-th key margin is below this are excluded
# One fixed bound on |gate - gate_oracle| for every workload and both router paths, set
# from what the output needs, not from any kernel's error: a gate enters Y only as the
# weight of an expert output, so k gates each off by 1e-5 move Y by at most
# k * 1e-5 * max|o|, under 0.1 % of the 2e-2 * RMS(Y) output budget for k <= 8; it is also
# 200x finer than the bf16 resolution of a gate near 0.5.
GATE_ATOL = 1e-5
Y_TOL = {"bf16": 2e-2, "f32": 1e-4}   # max-abs error / RMS(Y_oracle)
# A bf16 layer stores the expert intermediate h in bf16 between its two projections.  On
# every token the output is held to the same bound against the oracle that rounds h the
# same way (O.round_bf16): against the exact oracle, that rounding alone takes the worst
# output of the Switch-shaped layer to 2.1e-2 * RMS(Y) (fp64 elsewhere), so the exact
# comparison runs on the seeded token samples, as the workloads' recipe states.


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy() if t.is_floating_point() \
        else t.detach().to("cpu").numpy()


@dataclasses.dataclass
class Run:
    cfg: MoEConfig
    inputs: Dict[str, torch.Tensor]
    layer: MoELayer
    capacity: Optional[int]
    status: int


def run_gpu(cfg: MoEConfig, capacity_factor: Optional[float] = None, seed=None,
            ctx=None) -> Run:
    d = make_inputs(cfg, device="cuda", seed=seed)
    layer = MoELayer(cfg, d, ctx=ctx, capacity_factor=capacity_factor)
    layer.forward(d["X"])
    torch.cuda.synchronize()
    st = layer.device_status()
    cap = None if capacity_factor is None else layer.capacity
    return Run(cfg, d, layer, cap, st)


def oracle_route(run: Run) -> Dict[str, np.ndarray]:
    c, d = run.cfg, run.inputs
    return O.route(to_np(d["X"]), to_np(d["Wg"]), c.k, c.score, c.renorm,
                   bias=to_np(d["bias"]) if "bias" in d else None,
                   logit_bias=to_np(d["logit_bias"]) if "logit_bias" in d else None,
                   C=run.capacity, n_groups=c.n_groups, topk_groups=c.topk_groups)


def check_routing(run: Run, ref: Dict[str, np.ndarray]) -> Dict[str, object]:
    """Bit-exact routing on every row whose oracle gap is >= GAP_EXCLUDE; on excluded rows
    the GPU's choice must still be a valid top-k of the oracle keys within the margin."""
    L = run.layer
    idx = to_np(L.idx).astype(np.int64)
    gate = to_np(L.gate)
    ok_rows = ref["gap"] >= GAP_EXCLUDE
    n_excl = int((~ok_rows).sum())
    assert np.array_equal(idx[ok_rows], ref["idx"][ok_rows]), \
        f"routing differs on {(idx[ok_rows] != ref['idx'][ok_rows]).any(1).sum()} rows"
    if n_excl:
        key = ref["key"]
        kth = -np.sort(-key, 1)[:, run.cfg.k - 1]
        chosen = np.take_along_axis(key, idx, 1).min(1)
        assert np.all(chosen[~ok_rows] >= kth[~ok_rows] - GAP_EXCLUDE)
    # ascending expert order, distinct experts
    assert np.all(np.diff(idx, axis=1) > 0)
    # gates of the agreed rows, against the fixed bound
    g_dev = np.abs(gate - ref["gate"]).max(axis=1)
    g_err = float(g_dev[ok_rows].max()) if ok_rows.any() else 0.0
    assert g_err <= GATE_ATOL, f"gate error {g_err:.3e} > {GATE_ATOL:g}"
    if run.cfg.renorm:
        np.testing.assert_allclose(gate.sum(1), 1.0, atol=1e-5)
    # the reported gap agrees with the oracle's where it is informative
    gap = to_np(L.gap)
    fin = np.isfinite(ref["gap"]) & ok_rows
    if fin.any():
        assert np.abs(gap[fin] - ref["gap"][fin]).max() <= 1e-4
    return {"excluded_rows": n_excl, "gate_max_err": float(g_err)}


def check_dispatch(run: Run, idx_np: np.ndarray) -> None:
    """The device dispatch equals the oracle's dispatch of the same routing, bit for bit."""
    L, c = run.layer, run.cfg
    ref = O.dispatch(idx_np, c.E, run.capacity)
    assert np.array_equal(to_np(L.counts), ref["counts"])
    assert np.array_equal(to_np(L.offsets), ref["offsets"])
    assert np.array_equal(to_np(L.row_of_slot), ref["row_of_slot"])
    R = int(ref["offsets"][-1])
    assert np.array_equal(to_np(L.slot_of_row)[:R], ref["slot_of_row"])
    # the gathered rows are the tokens' rows, bit for bit
    if R:
        rows = np.random.default_rng(0).choice(R, size=min(R, 256), replace=False)
        xp = L.Xperm[torch.as_tensor(rows, device=L.Xperm.device)]
        toks = torch.as_tensor(ref["slot_of_row"][rows] // c.k, device=xp.device)
        assert torch.equal(xp, run.inputs["X"][toks])


def expert_fetch(d: Dict[str, torch.Tensor]):
    def get(e: int):
        return (to_np(d["W_gate"][e]), to_np(d["W_up"][e]), to_np(d["W_down"][e]))
    return get


def check_output(run: Run, ref: Dict[str, np.ndarray], n_tokens: Optional[int] = None,
                 seed: int = 1) -> Dict[str, float]:
    """Y of a seeded token sample (every token when n_tokens is None) against the oracle."""
    c, d, L = run.cfg, run.inputs, run.layer
    tokens = token_subset(c.T, n_tokens if n_tokens else c.T, seed).numpy()
    # use tokens whose routing agrees (all of them unless a row was excluded)
    idx = to_np(L.idx).astype(np.int64)
    kept_gpu = to_np(L.row_of_slot).reshape(c.T, c.k) >= 0
    kept_ref = ref["row_of_slot"].reshape(c.T, c.k) >= 0
    agree = np.all(idx == ref["idx"], axis=1) & np.all(kept_gpu == kept_ref, axis=1)
    tokens = tokens[agree[tokens]]
    shared = None
    if c.shared:
        shared = (to_np(d["Ws_gate"]), to_np(d["Ws_up"]), to_np(d["Ws_down"]))
    X = to_np(d["X"])
    Yref = O.combine_subset(X, ref, expert_fetch(d), tokens, shared)
    Y = to_np(L.Y[torch.as_tensor(tokens, device=L.Y.device)])
    # A token whose every slot was dropped (and with no shared expert) outputs exactly 0
    # on both sides; it is checked for that and left out of RMS(Y), which is taken over
    # the tokens that pass through at least one expert.
    live = np.any(Yref != 0.0, axis=1)
    assert np.all(Y[~live] == 0.0), "a fully dropped token has a non-zero output"
    if not live.any():
        return {"max_abs_err": 0.0, "rms": 0.0, "ratio": 0.0, "tokens": int(tokens.size)}
    rms = float(np.sqrt(np.mean(Yref[live] ** 2)))
    err = float(np.abs(Y - Yref).max())
    tol = Y_TOL[c.dtype] * rms
    assert err <= tol, f"max |dY| = {err:.3e} > {tol:.3e} (RMS {rms:.3e})"
    return {"max_abs_err": err, "rms": rms, "ratio": err / rms, "tokens": int(tokens.size)}


def check_output_bf16_h(run: Run, ref: Dict[str, np.ndarray]) -> Dict[str, float]:
    """Y of every token against the oracle whose experts round h to bf16 (the layer's
    storage of the intermediate), to Y_TOL["bf16"] * RMS(Y)."""
    c, d, L = run.cfg, run.inputs, run.layer
    assert c.dtype == "bf16"
    idx = to_np(L.idx).astype(np.int64)
    kept_gpu = to_np(L.row_of_slot).reshape(c.T, c.k) >= 0
    kept_ref = ref["row_of_slot"].reshape(c.T, c.k) >= 0
    agree = np.all(idx == ref["idx"], axis=1) & np.all(kept_gpu == kept_ref, axis=1)
    tokens = np.nonzero(agree)[0]
    shared = None
    if c.shared:
        shared = (to_np(d["Ws_gate"]), to_np(d["Ws_up"]), to_np(d["Ws_down"]))
    Yref = O.combine_subset(to_np(d["X"]), ref, expert_fetch(d), tokens, shared,
                            h_round=O.round_bf16)
    Y = to_np(L.Y[torch.as_tensor(tokens, device=L.Y.device)])
    live = np.any(Yref != 0.0, axis=1)
    assert np.all(Y[~live] == 0.0), "a fully dropped token has a non-zero output"
    if not live.any():
        return {"bf16_h_ratio": 0.0, "tokens": int(tokens.size)}
    rms = float(np.sqrt(np.mean(Yref[live] ** 2)))
    err = float(np.abs(Y - Yref).max())
    tol = Y_TOL["bf16"] * rms
    assert err <= tol, f"max |dY| against the bf16-h oracle = {err:.3e} > {tol:.3e}"
    return {"bf16_h_ratio": err / rms, "tokens": int(tokens.size)}


def check_stats(run: Run, ref: Dict[str, np.ndarray]) -> Dict[str, float]:
    """f and the drop rate exact; CV and entropy (fp64 from exact counts) to 1e-12; p and
    the loss, which sum per-token fp32 probabilities, to 2e-6 relative.  Returns the
    largest relative errors of p and the loss."""
    c, L = run.cfg, run.layer
    s = O.balance_stats(ref["counts"], ref["prob_colsum"], c.T, c.k,
                        int(ref["offsets"][-1]), c.alpha)
    np.testing.assert_allclose(to_np(L.f), s["f"], rtol=0, atol=0)
    p = to_np(L.p)
    np.testing.assert_allclose(p, s["p"], rtol=2e-6, atol=1e-12)
    out = to_np(L.stats)
    np.testing.assert_allclose(out[0], s["loss"], rtol=2e-6, atol=1e-15)
    np.testing.assert_allclose(out[1], s["drop_rate"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(out[2], s["cv"], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(out[3], s["entropy"], rtol=1e-12, atol=1e-15)
    nz = s["p"] > 0
    return {"p_rel_err": float(np.max(np.abs(p[nz] - s["p"][nz]) / s["p"][nz])) if nz.any() else 0.0,
            "loss_rel_err": float(abs(out[0] - s["loss"]) / s["loss"]) if s["loss"] else 0.0}

"""GPU parity of the bias update step ("LLM Internals §14.2.3", bias-adjusted selection)
against the fp64 oracle, through the C ABI: the updated float32 bias must equal the
oracle's bit for bit, alone and inside a loop of forwards whose routing it steers."""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_top_routing_router_b300 import binding as B
from sparse_top_routing_router_b300 import configs as K

from . import parity as P

pytestmark = pytest.mark.gpu

GAMMA = 0.001


def _oracle_bias(bias_before: np.ndarray, counts: np.ndarray, T: int, k: int,
                 gamma: float) -> np.ndarray:
    g32 = float(np.float32(gamma))
    return O.bias_update(bias_before, counts, T, k, g32).astype(np.float32)


def test_bias_update_exact_mean_and_sides():
    ctx = B.Context(0)
    # T*k = 8 over E = 4: balanced load 2; counts 2, 2, 3, 1 -> keep, keep, -g, +g
    counts = torch.tensor([2, 2, 3, 1], dtype=torch.int32, device="cuda")
    bias = torch.tensor([0.1, -0.2, 0.3, -0.4], dtype=torch.float32, device="cuda")
    before = bias.cpu().numpy().astype(np.float64)
    B.moe_bias_update(ctx, 4, 2, counts, GAMMA, bias)
    torch.cuda.synchronize()
    want = _oracle_bias(before, counts.cpu().numpy(), 4, 2, GAMMA)
    np.testing.assert_array_equal(bias.cpu().numpy(), want)
    assert bias[0].item() == np.float32(0.1) and bias[1].item() == np.float32(-0.2)


@pytest.mark.parametrize("E", [8, 256, 512])
def test_bias_update_random_counts(E):
    ctx = B.Context(0)
    rng = np.random.default_rng(E)
    T, k = 1000, 4
    counts_np = rng.multinomial(T * k, np.ones(E) / E).astype(np.int32)
    bias_np = (rng.standard_normal(E) * 0.1).astype(np.float32)
    counts = torch.from_numpy(counts_np).cuda()
    bias = torch.from_numpy(bias_np.copy()).cuda()
    B.moe_bias_update(ctx, T, k, counts, GAMMA, bias)
    torch.cuda.synchronize()
    want = _oracle_bias(bias_np.astype(np.float64), counts_np, T, k, GAMMA)
    np.testing.assert_array_equal(bias.cpu().numpy(), want)


def test_bias_update_steers_routing_over_steps():
    """Five forwards of a DSV3-shaped layer, each followed by the bias update: every
    step's routing matches the oracle run with the current bias, and every update matches
    the oracle's update of that step's counts."""
    cfg = K.scaled(K.DSV3_PREFILL, name="dsv3_bias_steps", T=600, H=256, E=32, I=128)
    run = P.run_gpu(cfg)
    layer, d = run.layer, run.inputs
    cv = []
    for step in range(5):
        if step:
            layer.forward(d["X"])
            torch.cuda.synchronize()
        assert layer.device_status() == 0
        ref = P.oracle_route(run)
        P.check_routing(run, ref)
        counts = P.to_np(layer.counts).astype(np.int64)
        assert np.array_equal(counts, ref["counts"])
        cv.append(float(counts.std() / counts.mean()))
        before = P.to_np(d["bias"])
        layer.update_bias(0.05)
        torch.cuda.synchronize()
        want = _oracle_bias(before, counts, cfg.T, cfg.k, 0.05)
        np.testing.assert_array_equal(d["bias"].cpu().numpy(), want)
    print("load CV per step:", [round(c, 3) for c in cv])
    assert cv[-1] < cv[0]   # the update balances the load

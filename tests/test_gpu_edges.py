"""Edge cases of the forward through the C ABI on the GPU."""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_top_routing_router_b300 import binding as B
from sparse_top_routing_router_b300 import configs as K
from sparse_top_routing_router_b300.inputs import make_inputs
from sparse_top_routing_router_b300.layer import MoELayer

from . import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    return B.Context(0)


def _small(**kw):
    base = dict(name="edge", T=40, H=64, E=8, I=64, k=2, score="softmax", renorm=True,
                shared=False, dtype="bf16")
    base.update(kw)
    return K.MoEConfig(**base)


def test_empty_batch(ctx):
    cfg = _small(T=0, shared=True)
    d = make_inputs(cfg, device="cuda")
    layer = MoELayer(cfg, d, ctx=ctx)
    layer.forward(d["X"])
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    assert layer.offsets.tolist() == [0] * (cfg.E + 1)
    assert layer.counts.tolist() == [0] * cfg.E
    assert torch.all(layer.stats == 0)


@pytest.mark.parametrize("cfg", [
    _small(T=1),
    _small(T=33, E=4, k=4),                       # k == E: gates are the full softmax
    _small(T=50, E=1, k=1, shared=True),          # one expert: the gate is 1
    _small(T=77, E=512, k=32, H=64, I=64),        # the largest E and k
    _small(T=129, E=8, k=2, H=128, I=192, score="sigmoid", selection_bias_std=0.1,
           shared=True),
], ids=lambda c: f"T{c.T}_E{c.E}_k{c.k}")
def test_shapes_full_parity(ctx, cfg):
    run = P.run_gpu(cfg, ctx=ctx)
    assert run.status == 0
    ref = P.oracle_route(run)
    P.check_routing(run, ref)
    P.check_dispatch(run, P.to_np(run.layer.idx).astype(np.int64))
    P.check_output(run, ref)
    if cfg.k == cfg.E and cfg.score == "softmax":
        np.testing.assert_allclose(P.to_np(run.layer.gate), O.softmax_rows(ref["logits"]),
                                   atol=1e-6)


def test_capacity_zero_leaves_shared(ctx):
    cfg = _small(T=64, shared=True, alpha=0.01)
    run = P.run_gpu(cfg, capacity_factor=0.0, ctx=ctx)
    assert run.status == 0 and run.capacity == 0
    assert int(run.layer.offsets[-1]) == 0
    assert torch.all(run.layer.row_of_slot == -1)
    ref = P.oracle_route(run)
    P.check_output(run, ref)
    assert float(run.layer.stats[1]) == 1.0         # every slot dropped


def test_exact_ties_go_to_lower_index(ctx):
    cfg = _small(T=64, H=256, k=1)
    d = make_inputs(cfg, device="cuda")
    d["X"] = d["X"].abs()
    Wg = torch.randn(cfg.H, cfg.E, device="cuda") * 1e-3
    Wg[:, 2] = 0.1
    Wg[:, 5] = 0.1
    d["Wg"] = Wg
    layer = MoELayer(cfg, d, ctx=ctx)
    layer.forward(d["X"])
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    assert torch.all(layer.idx[:, 0] == 2)
    assert torch.all(layer.gap == 0)


def test_near_tie_is_decided_exactly(ctx):
    """Two experts whose logits differ by 2e-6 on every token, far below the fp32 error of
    a 4096-long reduction: the float64 re-decision must pick the larger one."""
    cfg = _small(T=256, H=4096, k=1)
    d = make_inputs(cfg, device="cuda")
    X = d["X"].float()
    X[:, 0] = 1.0
    X[:, 1] = 1.0
    d["X"] = X.to(torch.bfloat16)
    Wg = d["Wg"].clone()
    Wg[:, 3] = Wg[:, 1]
    Wg[1, 1] = 10.0
    Wg[1, 3] = 10.0
    Wg[0, 3] = Wg[0, 1] + 2e-6
    d["Wg"] = Wg
    layer = MoELayer(cfg, d, ctx=ctx)
    layer.forward(d["X"])
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    run = P.Run(cfg, d, layer, None, 0)
    ref = P.oracle_route(run)
    gap = ref["gap"]
    assert np.all((gap > 1.5e-6) & (gap < 2.5e-6))
    assert np.all(ref["idx"][:, 0] == 3)
    assert torch.all(layer.idx[:, 0] == 3)


def test_bad_routing_index_is_reported(ctx):
    T, k, E = 16, 2, 8
    idx = torch.tensor([[0, 1]] * T, dtype=torch.int32, device="cuda")
    idx[5, 1] = 99
    ws = torch.zeros(B.moe_workspace_bytes(T, 64, E, 64, k, 0, 0), dtype=torch.uint8,
                     device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    ros = torch.empty(T * k, dtype=torch.int32, device="cuda")
    sor = torch.empty(T * k, dtype=torch.int32, device="cuda")
    B.moe_dispatch(ctx, idx, E, -1, counts, offsets, ros, sor, ws, H=64)
    st = B.moe_get_device_status(ctx, ws)
    assert st == B.MOE_ERR_DEVICE_INDEX
    assert int(ros[5 * k + 1]) == -1
    assert B.moe_get_device_status(ctx, ws) == 0      # reset by the previous read


def test_repeated_expert_in_a_row_is_reported(ctx):
    # the k experts of a token must be distinct; a repeat is reported in the status word
    # (its rows are then unspecified, never out of bounds)
    T, k, E = 300, 3, 8
    idx = torch.tensor([[0, 2, 5]] * T, dtype=torch.int32, device="cuda")
    idx[260, 2] = 2
    ws = torch.zeros(B.moe_workspace_bytes(T, 64, E, 64, k, 0, 0), dtype=torch.uint8,
                     device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    ros = torch.empty(T * k, dtype=torch.int32, device="cuda")
    sor = torch.empty(T * k, dtype=torch.int32, device="cuda")
    B.moe_dispatch(ctx, idx, E, -1, counts, offsets, ros, sor, ws, H=64)
    assert B.moe_get_device_status(ctx, ws) == B.MOE_ERR_DEVICE_INDEX
    assert int(ros.max()) < T * k and int(ros.min()) >= 0
    idx[260, 2] = 5
    B.moe_dispatch(ctx, idx, E, -1, counts, offsets, ros, sor, ws, H=64)
    assert B.moe_get_device_status(ctx, ws) == 0


def test_bad_offsets_are_reported(ctx):
    cfg = _small(T=32)
    d = make_inputs(cfg, device="cuda")
    layer = MoELayer(cfg, d, ctx=ctx)
    layer.forward(d["X"])
    torch.cuda.synchronize()
    bad = layer.offsets.clone()
    bad[3] = 10 ** 6
    B.moe_grouped_swiglu(ctx, d["X"], layer.Xperm, bad, d["W_gate"], d["W_up"], d["W_down"],
                         layer.O, layer.ws, cfg.k)
    assert B.moe_get_device_status(ctx, layer.ws) == B.MOE_ERR_DEVICE_INDEX


def test_dispatch_combine_identity(ctx):
    """Identity experts (O = the gathered row in fp32) and renormalised gates: combine
    returns X exactly up to fp32 rounding of the convex combination."""
    cfg = _small(T=300, H=128, E=16, k=4)
    d = make_inputs(cfg, device="cuda")
    layer = MoELayer(cfg, d, ctx=ctx)
    layer.forward(d["X"])
    R = int(layer.offsets[-1])
    O = layer.Xperm[:R].float()
    Ofull = torch.zeros(cfg.T * cfg.k, cfg.H, device="cuda")
    Ofull[:R] = O
    Y = torch.empty(cfg.T, cfg.H, device="cuda")
    B.moe_combine(ctx, Ofull, layer.row_of_slot, layer.gate, Y)
    torch.cuda.synchronize()
    torch.testing.assert_close(Y, d["X"].float(), atol=1e-5 * 4, rtol=1e-6)


def test_bf16_copy_of_y(ctx):
    cfg = _small(T=64, H=128, shared=True)
    d = make_inputs(cfg, device="cuda")
    layer = MoELayer(cfg, d, ctx=ctx)
    layer.forward(d["X"])
    Yb = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(cfg.T, cfg.H, device="cuda")
    B.moe_combine(ctx, layer.O, layer.row_of_slot, layer.gate, Y, O_shared=layer.O_shared,
                  Y_bf16=Yb)
    torch.cuda.synchronize()
    assert torch.equal(Y, layer.Y)
    assert torch.equal(Yb, Y.to(torch.bfloat16))


def test_status_survives_and_context_reusable(ctx):
    """After a reported device error the context and workspace keep working."""
    cfg = _small(T=48, shared=True)
    run = P.run_gpu(cfg, ctx=ctx)
    assert run.status == 0
    ref = P.oracle_route(run)
    P.check_routing(run, ref)


@pytest.mark.parametrize("H", [128, 512])
def test_bounded_wait_timeout_is_reported(ctx, H):
    """A barrier that nothing completes (the test hook withholds the first operand load of
    every CTA of the tensor-core kernels): the bounded waits run out, the kernels record
    MOE_ERR_TIMEOUT, release tensor memory and return; the context keeps working.  With
    H = 512 the down GEMM runs as clusters of two CTAs, each waiting on stages that the
    other's multicast also fills."""
    cfg = _small(T=64, H=H, I=128, shared=True)
    d = make_inputs(cfg, device="cuda")
    layer = MoELayer(cfg, d, ctx=ctx)
    ctx.set_test_hook(B.MOE_TEST_HOOK_WITHHOLD_LOAD, wait_limit_ms=50)
    try:
        layer.forward(d["X"])
        torch.cuda.synchronize()
        st = layer.device_status()
    finally:
        ctx.set_test_hook(B.MOE_TEST_HOOK_NONE)
    assert st == B.MOE_ERR_TIMEOUT
    run = P.run_gpu(cfg, ctx=ctx)
    assert run.status == 0
    ref = P.oracle_route(run)
    P.check_output(run, ref)


def test_forward_host_matches_device(ctx):
    """The end-to-end call (pinned host X in, host Y out, on a side stream) returns the
    device forward's Y."""
    cfg = _small(T=96, H=128, shared=True)
    d = make_inputs(cfg, device="cuda")
    layer = MoELayer(cfg, d, ctx=ctx)
    Y_dev = layer.forward(d["X"]).clone()
    X_host = d["X"].cpu().pin_memory()
    Y_host = torch.empty(cfg.T, cfg.H, dtype=torch.float32, pin_memory=True)
    s = torch.cuda.Stream()
    layer.forward_host(X_host, Y_host, stream=s)
    s.synchronize()
    assert torch.equal(Y_host, Y_dev.cpu())
    assert layer.device_status() == 0


# ---------------------------------------------------------------- the further entry points

@pytest.mark.parametrize("kw", [dict(expert_choice=True), dict(fp8_experts=True),
                                dict(score="sigmoid", selection_bias_std=0.1, n_groups=4,
                                     topk_groups=2)],
                         ids=["expert_choice", "fp8", "groups"])
def test_empty_batch_other_paths(ctx, kw):
    cfg = _small(T=0, shared=True, **kw)
    d = make_inputs(cfg, device="cuda")
    layer = MoELayer(cfg, d, ctx=ctx)
    layer.forward(d["X"])
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    assert layer.offsets.tolist() == [0] * (cfg.E + 1)


def test_group_limited_single_token_and_whole_groups(ctx):
    # one token; k = topk_groups * (E / n_groups): every expert of the chosen groups
    cfg = _small(T=1, E=16, k=8, score="sigmoid", selection_bias_std=0.1, n_groups=4,
                 topk_groups=2)
    run = P.run_gpu(cfg, ctx=ctx)
    assert run.status == 0
    ref = P.oracle_route(run)
    assert np.array_equal(P.to_np(run.layer.idx).astype(np.int64), ref["idx"])
    groups = set((ref["idx"][0] // 4).tolist())
    assert len(groups) == 2


def test_expert_choice_ragged_shapes(ctx):
    # C = T*k/E = 3 tokens per expert out of 12; E = 8 experts of a 64-wide layer
    cfg = _small(T=12, k=2, expert_choice=True, shared=True)
    run = P.run_gpu(cfg, ctx=ctx)
    assert run.status == 0
    c, L = run.cfg, run.layer
    ref = O.route_expert_choice(P.to_np(run.inputs["X"]), P.to_np(run.inputs["Wg"]), c.k,
                                c.score)
    sor = P.to_np(L.slot_of_row).astype(np.int64)
    ok = ref["gap"] >= P.GAP_EXCLUDE
    assert np.array_equal((sor.reshape(c.E, 3) // c.E)[ok], ref["chosen"][ok])


def test_fp8_many_rows_per_expert(ctx):
    # 40 tokens, top-2 of 2 experts: 40 rows per expert, five 8-row passes each
    cfg = _small(T=40, E=2, k=2, fp8_experts=True, shared=True)
    run = P.run_gpu(cfg, ctx=ctx)
    assert run.status == 0
    d, L = run.inputs, run.layer
    ref = P.oracle_route(run)

    def fetch(e):
        return tuple(O.dequantize_fp8_rows(*O.quantize_fp8_rows(
            P.to_np(d[n][e]).astype(np.float32))) for n in ("W_gate", "W_up", "W_down"))
    shared = tuple(O.dequantize_fp8_rows(*O.quantize_fp8_rows(
        P.to_np(d[n]).astype(np.float32))) for n in ("Ws_gate", "Ws_up", "Ws_down"))
    Yref = O.combine_subset(P.to_np(d["X"]), ref, fetch, np.arange(cfg.T), shared)
    Y = P.to_np(L.Y)
    rms = float(np.sqrt(np.mean(Yref ** 2)))
    assert float(np.abs(Y - Yref).max()) <= P.Y_TOL["bf16"] * rms

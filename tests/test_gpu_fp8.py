"""GPU parity of the FP8 expert weights ("LLM Internals §14.2.5": one expert is 44 MB in
FP8) against the fp64 oracle, through the C ABI: the E4M3 codes and per-channel scales
bit for bit, and the decode-sized layer on FP8 weights within the layer tolerance of the
oracle run on the dequantized weights."""

import dataclasses

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_top_routing_router_b300 import binding as B
from sparse_top_routing_router_b300 import configs as K

from . import parity as P
from .fp8_oracle_pool import ordered_fetch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantize_fp8_bit_exact(dtype):
    ctx = B.Context(0)
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    W = (torch.randn(37, 640, generator=g, device="cuda") * 0.02).to(dtype)
    W[3] = 0                                   # an all-zero row: scale 1, codes 0
    W[4, :64] = 1e-30                          # tiny values next to a large one
    W[4, 64] = 3.0
    W[5] = torch.linspace(-1, 1, 640, device="cuda").to(dtype)
    q = torch.empty(W.shape, dtype=torch.uint8, device="cuda")
    s = torch.empty(W.shape[0], dtype=torch.float32, device="cuda")
    B.moe_quantize_fp8(ctx, W, q, s)
    torch.cuda.synchronize()
    q_ref, s_ref = O.quantize_fp8_rows(W.float().cpu().numpy())
    np.testing.assert_array_equal(s.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)


def _fp8_expert_fetch(d):
    def get(e):
        out = []
        for name in ("W_gate", "W_up", "W_down"):
            q, s = O.quantize_fp8_rows(P.to_np(d[name][e]).astype(np.float32))
            out.append(O.dequantize_fp8_rows(q, s))
        return tuple(out)
    return get


def _check_fp8_layer(cfg, n_tokens=None, pool=False):
    run = P.run_gpu(cfg)
    assert run.status == 0
    ref = P.oracle_route(run)
    info = P.check_routing(run, ref)
    P.check_dispatch(run, P.to_np(run.layer.idx).astype(np.int64))
    # the layer's codes equal the oracle's quantization of its weights (one expert)
    L, d = run.layer, run.inputs
    q_ref, s_ref = O.quantize_fp8_rows(P.to_np(d["W_down"][1]).astype(np.float32))
    np.testing.assert_array_equal(L.fp8["Q_down"][1].cpu().numpy(), q_ref)
    np.testing.assert_array_equal(L.fp8["S_down"][1].cpu().numpy(), s_ref)
    # outputs against the oracle on the dequantized weights
    c = cfg
    from sparse_top_routing_router_b300.inputs import token_subset
    tokens = token_subset(c.T, n_tokens if n_tokens else c.T, 1).numpy()
    shared = None
    if c.shared:
        shared = tuple(O.dequantize_fp8_rows(*O.quantize_fp8_rows(
            P.to_np(d[n]).astype(np.float32))) for n in ("Ws_gate", "Ws_up", "Ws_down"))
    if pool:
        idx, ros = ref["idx"], ref["row_of_slot"].reshape(c.T, c.k)
        need = sorted({int(idx[t, j]) for t in tokens for j in range(c.k) if ros[t, j] >= 0})
        fetch, close = ordered_fetch(
            need, lambda e: tuple(P.to_np(d[n][e]).astype(np.float32)
                                  for n in ("W_gate", "W_up", "W_down")))
        try:
            Yref = O.combine_subset(P.to_np(d["X"]), ref, fetch, tokens, shared)
        finally:
            close()
    else:
        Yref = O.combine_subset(P.to_np(d["X"]), ref, _fp8_expert_fetch(d), tokens, shared)
    Y = P.to_np(L.Y[torch.as_tensor(tokens, device=L.Y.device)])
    rms = float(np.sqrt(np.mean(Yref ** 2)))
    err = float(np.abs(Y - Yref).max())
    assert err <= P.Y_TOL["bf16"] * rms, f"max |dY| = {err:.3e}, RMS {rms:.3e}"
    return {"excluded_rows": info["excluded_rows"], "ratio": err / rms}


FP8_SMALL = [
    # decode-sized: a few rows per expert plus a 64-row shared expert (8 passes)
    K.scaled(K.DSV3_DECODE, name="dsv3_small_decode_fp8", H=256, E=64, I=128,
             fp8_experts=True),
    # 64 rows per expert on average: several 8-row passes per expert, no shared expert
    K.scaled(K.MIXTRAL, name="mixtral_small_fp8", T=256, H=192, I=320, fp8_experts=True),
]


@pytest.mark.parametrize("cfg", FP8_SMALL, ids=lambda c: c.name)
def test_fp8_layer_small(cfg):
    print(cfg.name, _check_fp8_layer(cfg))


def test_fp8_layer_full_size_decode():
    cfg = dataclasses.replace(K.DSV3_DECODE, name="dsv3_decode_bf16_fp8", fp8_experts=True)
    # every one of the 64 tokens, their experts quantized by the oracle in a process pool
    print(cfg.name, _check_fp8_layer(cfg, pool=True))

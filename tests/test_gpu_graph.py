"""The whole forward captured into one CUDA graph and replayed: the same results as the
eager forward, bit for bit, for the input the graph was captured with and for new
contents of the same input buffer."""

import pytest
import torch

from sparse_top_routing_router_b300 import configs as K
from sparse_top_routing_router_b300.inputs import make_inputs
from sparse_top_routing_router_b300.layer import MoELayer

pytestmark = pytest.mark.gpu

CASES = [
    K.TINY_F32,                                                         # CUDA-core paths
    K.scaled(K.DSV3_PREFILL, name="dsv3_graph", T=300, H=256, E=32, I=128),   # side stream
    K.scaled(K.MIXTRAL, name="mixtral_graph", T=1100, H=256, E=4, I=384),     # CTA pairs
    K.scaled(K.SWITCH, name="switch_graph", T=1000, H=256, E=16, I=256),      # capacity
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_graph_replay_matches_eager(cfg):
    d = make_inputs(cfg, device="cuda")
    cf = cfg.capacity_factors[0] if cfg.capacity_factors else None
    layer = MoELayer(cfg, d, capacity_factor=cf)
    X = d["X"]
    Y0 = layer.forward(X).clone()
    idx0, gate0, stats0 = layer.idx.clone(), layer.gate.clone(), layer.stats.clone()
    g = layer.capture(X)
    layer.Y.zero_()
    layer.idx.fill_(-1)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(layer.Y, Y0)
    assert torch.equal(layer.idx, idx0) and torch.equal(layer.gate, gate0)
    torch.testing.assert_close(layer.stats, stats0, rtol=1e-12, atol=0)

    # new token values in the captured buffer: replay == eager forward on them
    X.copy_(make_inputs(cfg, device="cuda", seed=cfg.seed + 1, with_experts=False)["X"])
    g.replay()
    torch.cuda.synchronize()
    Yg = layer.Y.clone()
    assert not torch.equal(Yg, Y0)
    Ye = layer.forward(X)
    torch.cuda.synchronize()
    assert torch.equal(Yg, Ye)
    assert layer.device_status() == 0

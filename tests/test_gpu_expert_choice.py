"""GPU parity of expert-choice routing ("LLM Internals §14.2", the two selection
paradigms; "MoE 03: efficiency frontiers", Expert Choice Routing) against the fp64 oracle,
through the C ABI: every expert's C = T*k/E tokens bit-exact (columns whose oracle margin
is below 1e-6 excluded and counted, and checked for validity), gates within the fixed
bound of the token-choice tests (1e-5), and Y within the layer tolerance."""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_top_routing_router_b300 import configs as K
from sparse_top_routing_router_b300.inputs import token_subset

from . import parity as P

pytestmark = pytest.mark.gpu


def _ref(run):
    c, d = run.cfg, run.inputs
    return O.route_expert_choice(
        P.to_np(d["X"]), P.to_np(d["Wg"]), c.k, c.score,
        logit_bias=P.to_np(d["logit_bias"]) if "logit_bias" in d else None)


def check_expert_choice(run, ref, all_columns=False, n_tokens=None):
    c, L = run.cfg, run.layer
    T, E, C = c.T, c.E, c.T * c.k // c.E
    assert np.array_equal(P.to_np(L.offsets), ref["offsets"])
    sor = P.to_np(L.slot_of_row).astype(np.int64)
    ros = P.to_np(L.row_of_slot).astype(np.int64)
    chosen = (sor.reshape(E, C) // E)
    ok = np.ones(E, bool) if all_columns else ref["gap"] >= P.GAP_EXCLUDE
    assert np.array_equal(chosen[ok], ref["chosen"][ok]), \
        f"{(chosen[ok] != ref['chosen'][ok]).any(1).sum()} experts differ"
    # every expert's rows hold distinct tokens in ascending order, and its column agrees
    assert np.all(np.diff(chosen, axis=1) > 0)
    assert np.all(sor.reshape(E, C) % E == np.arange(E)[:, None])
    assert np.array_equal(ros[sor], np.arange(E * C))
    assert (ros >= 0).sum() == E * C
    if not ok.all():   # an excluded column still takes C tokens within the margin
        S = ref["S"]
        for e in np.nonzero(~ok)[0]:
            kth = np.sort(S[:, e])[::-1][C - 1]
            assert np.all(S[chosen[e], e] >= kth - P.GAP_EXCLUDE)
    gate = P.to_np(L.gate)
    taken = ros.reshape(T, E) >= 0
    both = taken & (ref["row_of_slot"].reshape(T, E) >= 0)
    g_err = float(np.abs(gate - ref["gate"])[both].max()) if both.any() else 0.0
    print(f"{c.name}: max gate error {g_err:.3e}")
    assert g_err <= P.GATE_ATOL
    assert np.all(gate[~taken] == 0)
    # outputs of tokens whose expert set agrees with the oracle's
    tokens = token_subset(T, n_tokens if n_tokens else T, 1).numpy()
    agree = np.all(taken == (ref["row_of_slot"].reshape(T, E) >= 0), axis=1)
    tokens = tokens[agree[tokens]]
    d = run.inputs
    shared = (P.to_np(d["Ws_gate"]), P.to_np(d["Ws_up"]), P.to_np(d["Ws_down"])) \
        if c.shared else None
    Yref = O.combine_subset(P.to_np(d["X"]), ref, P.expert_fetch(d), tokens, shared)
    Y = P.to_np(L.Y[torch.as_tensor(tokens, device=L.Y.device)])
    live = np.any(Yref != 0.0, axis=1)
    assert np.all(Y[~live] == 0.0)   # a token no expert took outputs exactly 0
    rms = float(np.sqrt(np.mean(Yref[live] ** 2)))
    err = float(np.abs(Y - Yref).max())
    assert err <= P.Y_TOL[c.dtype] * rms, f"max |dY| = {err:.3e}, RMS {rms:.3e}"
    untaken = int((~taken.any(1)).sum())
    return {"excluded_columns": int((~ok).sum()), "ratio": err / rms,
            "tokens_untaken": untaken,
            "redecided_experts": int(run.layer.ws[4:8].view(torch.int32))}


SMALL = [
    # softmax, tensor-core logits, 8 experts of C = 128
    K.scaled(K.MIXTRAL, name="mixtral_small_ec", T=512, H=256, I=256, expert_choice=True),
    # sigmoid, 64 experts of C = 40, a shared expert
    K.scaled(K.DSV3_PREFILL, name="dsv3_small_ec", T=320, H=256, E=64, I=128,
             expert_choice=True),
    # CUDA-core logits (T < 256), C = 24
    K.scaled(K.MIXTRAL, name="cuda_core_ec", T=96, H=128, I=128, expert_choice=True),
    # fp32 layer
    K.scaled(K.TINY_F32, name="tiny_f32_ec", expert_choice=True),
    # C = T: every expert takes every token (k = E)
    K.scaled(K.MIXTRAL, name="all_tokens_ec", T=64, H=128, E=4, I=128, k=4,
             expert_choice=True),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_expert_choice_small(cfg):
    run = P.run_gpu(cfg)
    assert run.status == 0
    info = check_expert_choice(run, _ref(run))
    print(cfg.name, info)


def test_expert_choice_exact_ties():
    """Tokens 1 and 0 (and 3 and 2) carry the same row of X, so their affinities tie in
    every column; where a tie straddles an expert's C-th place the lower token must win.
    400 all-zero tokens have the uniform affinity 1/8 in every column, below the best of
    the other tokens and above the rest, so each expert fills its last places from that
    block: the lowest indices of it.  Every column must match the oracle."""
    cfg = K.scaled(K.MIXTRAL, name="tie_ec", T=512, H=256, I=128, expert_choice=True)
    from sparse_top_routing_router_b300.inputs import make_inputs
    from sparse_top_routing_router_b300.layer import MoELayer
    d = make_inputs(cfg, device="cuda")
    d["X"][1] = d["X"][0]
    d["X"][3] = d["X"][2]
    d["X"][100:500] = 0   # 400 tied tokens: every expert's C-th place falls among them
    layer = MoELayer(cfg, d)
    layer.forward(d["X"])
    torch.cuda.synchronize()
    run = P.Run(cfg, d, layer, None, layer.device_status())
    assert run.status == 0
    ref = _ref(run)
    assert (ref["gap"] == 0).any()
    info = check_expert_choice(run, ref, all_columns=True)
    assert info["redecided_experts"] >= int((ref["gap"] == 0).sum())
    print("tie_ec", info)


def test_expert_choice_full_size_mixtral():
    cfg = dataclasses_replace(K.MIXTRAL, name="mixtral_bf16_ec", expert_choice=True)
    run = P.run_gpu(cfg)
    assert run.status == 0
    info = check_expert_choice(run, _ref(run), n_tokens=48)
    print(cfg.name, info)


def dataclasses_replace(cfg, **kw):
    import dataclasses
    return dataclasses.replace(cfg, **kw)

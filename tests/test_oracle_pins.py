"""Pins of the fp64 oracle to what the pages and the mathematics fix (CPU only).

Each test checks the oracle against something other than itself: a value printed in a
worked example of the pages (fixtures under tests/golden/, each naming its source), a
closed form, brute force on tiny inputs, or an invariant the definition implies.
"""

import itertools
import math

import numpy as np
import pytest

from oracle import moe_oracle as O


# ---------------------------------------------------------------- parameter accounting

def test_param_accounting(golden):
    g = golden("param_accounting.json")
    H, I = g["hidden_size"], g["moe_intermediate_size"]
    pe = O.expert_params(H, I)
    assert pe == g["params_per_expert"] == 44_040_192
    layer = O.layer_params(H, I, g["routed"], g["shared"])
    assert round(layer / 1e9, 2) == g["layer_params_approx_B"]
    assert round(g["moe_layers"] * layer / 1e9, 1) == g["all_moe_layers_approx_B"]
    act = O.active_params(H, I, g["top_k"], g["shared"])
    assert round(act / 1e6, 1) == g["active_per_token_layer_approx_M"]
    assert round(g["moe_layers"] * act / 1e9, 2) == g["active_all_layers_approx_B"]
    assert round(100 * act / layer, 1) == g["active_fraction_percent_approx"]
    assert math.comb(256, 8) == g["comb_256_8"]
    assert math.comb(8, 2) == g["comb_8_2"]
    assert abs(g["comb_256_8"] / g["comb_8_2"] / g["comb_ratio_approx"] - 1) < 0.05


# ---------------------------------------------------------------- balance loss

def test_balance_loss_worked_example(golden):
    g = golden("balance_loss_example.json")
    f, p = np.array(g["f"]), np.array(g["p"])
    np.testing.assert_allclose(f * p, g["f_times_p"], atol=1e-15)
    assert abs(O.balance_loss(f, p, 1.0) / g["N_experts"] - g["sum_f_p"]) < 1e-15
    assert abs(O.balance_loss(f, p, 1.0) - g["N_sum_f_p"]) < 1e-14
    b = g["balanced"]
    assert abs(O.balance_loss(b["f"], b["p"], 1.0) - b["N_sum_f_p"]) < 1e-15
    one_hot = [1.0, 0.0, 0.0, 0.0]
    assert abs(O.balance_loss(one_hot, one_hot, 1.0) - g["collapsed_N_sum_f_p"]) < 1e-15
    # alpha scales linearly
    assert abs(O.balance_loss(f, p, 0.01) - 0.01 * g["N_sum_f_p"]) < 1e-15


def test_balance_stats_from_counts(golden):
    g = golden("balance_loss_example.json")
    # 10 tokens, top-1: counts 7,1,1,1 give f = [.7,.1,.1,.1]; column sums of p give p
    counts = np.array([7, 1, 1, 1])
    colsum = np.array(g["p"]) * 10
    s = O.balance_stats(counts, colsum, T=10, k=1, n_kept=10, alpha=1.0)
    np.testing.assert_allclose(s["f"], g["f"], atol=1e-15)
    assert abs(s["loss"] - g["N_sum_f_p"]) < 1e-14
    assert s["drop_rate"] == 0.0
    # CV = population std / mean of [7,1,1,1]: mean 2.5, var = (20.25+3*2.25)/4 = 6.75
    assert abs(s["cv"] - math.sqrt(6.75) / 2.5) < 1e-15
    ent = -(0.7 * math.log(0.7) + 3 * 0.1 * math.log(0.1))
    assert abs(s["entropy"] - ent) < 1e-15
    # uniform load: CV 0, entropy ln E, loss alpha
    s = O.balance_stats(np.array([5, 5, 5, 5]), np.full(4, 5.0), T=20, k=1, n_kept=15,
                        alpha=0.01)
    assert s["cv"] == 0.0 and abs(s["entropy"] - math.log(4)) < 1e-15
    assert abs(s["loss"] - 0.01) < 1e-17 and s["drop_rate"] == 0.25


# ---------------------------------------------------------------- capacity

def test_capacity_worked_examples(golden):
    g = golden("capacity_examples.json")
    km = g["knowledge_map"]
    assert km["T"] * km["k"] == km["requests"]
    assert O.capacity(1.0, km["T"], km["k"], km["E"]) == km["C_at_c_1.0"]
    assert O.capacity(2.0, km["T"], km["k"], km["E"]) == km["C_at_c_2.0"]
    li = g["llm_internals"]
    C = O.capacity(li["capacity_factor"], li["T"], li["k"], li["E"])
    assert C == li["slots_per_expert"]
    assert li["T"] * li["k"] // li["E"] == li["average_per_expert"]
    assert li["hot_expert_received"] - C == li["hot_expert_dropped"]
    assert li["E"] * C == li["total_slots"]
    assert li["E"] * C - li["T"] * li["k"] == li["idle_slots_if_uniform"]
    # ceil, not floor or round: 7 requests over 2 experts at c=1 -> 4
    assert O.capacity(1.0, 7, 1, 2) == 4
    assert O.capacity(1.0, 6, 1, 4) == 2
    assert O.capacity(0.0, 6, 2, 4) == 0
    # the Switch workload: T=16384, E=64, top-1
    assert O.capacity(1.0, 16384, 1, 64) == 256
    assert O.capacity(1.25, 16384, 1, 64) == 320


@pytest.mark.parametrize("c", ["c_1.0", "c_2.0"])
def test_dispatch_six_token_example(golden, c):
    g = golden("six_token_routing.json")
    idx = np.array(g["idx"])
    exp = g[c]
    d = O.dispatch(idx, g["E"], exp["C"])
    assert d["counts"].tolist() == g["counts"]
    assert d["kept"].tolist() == exp["kept"]
    assert d["offsets"].tolist() == exp["offsets"]
    assert d["row_of_slot"].tolist() == exp["row_of_slot"]
    assert d["slot_of_row"].tolist() == exp["slot_of_row"]
    assert np.nonzero(d["row_of_slot"] < 0)[0].tolist() == exp["dropped_slots"]


def test_dispatch_invariants():
    rng = np.random.default_rng(3)
    T, E, k = 50, 7, 3
    idx = np.sort(np.stack([rng.choice(E, k, replace=False) for _ in range(T)]), 1)
    for C in (None, 0, 5, 21, 1000):
        d = O.dispatch(idx, E, C)
        ros, sor, off = d["row_of_slot"], d["slot_of_row"], d["offsets"]
        kept = ros >= 0
        # mutual inverses
        assert np.all(sor[ros[kept]] == np.nonzero(kept)[0])
        assert np.all(ros[sor] == np.arange(sor.size))
        # rows sorted by (expert, token) and grouped at offsets
        ex = idx.reshape(-1)[sor]
        tok = sor // k
        assert np.all(np.diff(ex) >= 0)
        for e in range(E):
            seg = slice(off[e], off[e + 1])
            assert np.all(ex[seg] == e)
            assert np.all(np.diff(tok[seg]) > 0)
        # capacity keeps the lowest token indices, sum kept = sum min(m, C)
        cap = np.inf if C is None else C
        assert off[-1] == sum(min(m, cap) for m in d["counts"])
        for e in range(E):
            toks = np.nonzero((idx == e).any(1))[0]
            kept_toks = tok[off[e]:off[e + 1]]
            assert kept_toks.tolist() == toks[: len(kept_toks)].tolist()
        # dropless reproduces the counts
        if C is None:
            assert np.all(d["kept"] == d["counts"]) and kept.all()
    # gather by slot_of_row then scatter by row_of_slot returns the kept rows unchanged
    X = rng.standard_normal((T, 4))
    d = O.dispatch(idx, E, 5)
    Xperm = X[d["slot_of_row"] // k]
    back = np.zeros((T * k, 4))
    back[d["slot_of_row"]] = Xperm
    kept = d["row_of_slot"] >= 0
    assert np.array_equal(back[kept], X[np.nonzero(kept)[0] // k])


# ---------------------------------------------------------------- scoring and top-k

def test_router_logits_one_hot_and_offset():
    rng = np.random.default_rng(0)
    H, E = 5, 3
    Wg = rng.standard_normal((H, E))
    X = np.eye(H)[[2, 0, 4]]            # one-hot rows pick rows of W_g
    l = O.router_logits(X, Wg)
    assert np.array_equal(l, Wg[[2, 0, 4]])
    off = np.array([0.5, -1.0, 0.0])
    assert np.array_equal(O.router_logits(X, Wg, off), Wg[[2, 0, 4]] + off)
    # a wrong orientation (W_g^T) would not even have these shapes
    assert l.shape == (3, E)


def test_softmax_two_experts_closed_form():
    l = np.array([[0.3, -1.2], [5.0, 5.0], [-40.0, 2.0]])
    p = O.softmax_rows(l)
    for r in range(3):
        d = l[r, 0] - l[r, 1]
        assert abs(p[r, 0] - 1.0 / (1.0 + math.exp(-d))) < 1e-15
    np.testing.assert_allclose(p.sum(1), 1.0, atol=1e-15)
    # shift invariance and strict monotonicity
    assert np.allclose(O.softmax_rows(l + 7.0), p, atol=1e-15)


def test_sigmoid_closed_form():
    l = np.array([[0.0, math.log(3.0), -math.log(3.0)]])
    np.testing.assert_allclose(O.sigmoid(l), [[0.5, 0.75, 0.25]], atol=1e-15)
    assert O.sigmoid(np.array([[-1000.0]]))[0, 0] == 0.0


def test_topk_brute_force():
    rng = np.random.default_rng(7)
    for E in (2, 3, 5, 8):
        for k in range(1, E + 1):
            key = rng.standard_normal((12, E))
            idx, gap = O.select_topk(key, k)
            for t in range(12):
                best = max(itertools.combinations(range(E), k),
                           key=lambda S: sum(key[t, list(S)]))
                assert idx[t].tolist() == sorted(best)
                srt = sorted(key[t], reverse=True)
                want_gap = srt[k - 1] - srt[k] if k < E else math.inf
                assert gap[t] == want_gap


def test_topk_ties_lower_index():
    key = np.array([[1.0, 2.0, 2.0, 2.0, 0.0]])
    idx, gap = O.select_topk(key, 2)
    assert idx.tolist() == [[1, 2]] and gap[0] == 0.0


def test_renorm_two_page_forms_agree():
    """[KM] renormalises the full softmax over S; [SN] takes softmax of the k chosen
    scores.  The full denominator cancels, so the two must agree."""
    rng = np.random.default_rng(1)
    l = rng.standard_normal((20, 8)) * 2
    for k in (1, 2, 3, 8):
        idx, _ = O.select_topk(l, k)
        g = O.gates_for(l, idx, "softmax", True)
        chosen = np.take_along_axis(l, idx, 1)
        z = np.exp(chosen - chosen.max(1, keepdims=True))
        np.testing.assert_allclose(g, z / z.sum(1, keepdims=True), rtol=1e-14, atol=1e-16)
        np.testing.assert_allclose(g.sum(1), 1.0, atol=1e-14)
        if k == 8:
            np.testing.assert_allclose(g, O.softmax_rows(l), rtol=1e-14)
    # without renorm, the gate is the plain probability and gates sum to < 1
    idx, _ = O.select_topk(l, 2)
    g = O.gates_for(l, idx, "softmax", False)
    assert np.all(g.sum(1) < 1.0)
    np.testing.assert_allclose(g, np.take_along_axis(O.softmax_rows(l), idx, 1))


def test_sigmoid_bias_selects_but_does_not_weigh():
    """[LI §14.2.3 eq. 16]: the bias enters the top-k comparison only."""
    l = np.array([[0.0, math.log(3.0), -math.log(3.0)]])   # s = .5, .75, .25
    bias = np.array([0.0, 0.0, 0.6])                        # keys .5, .75, .85
    key = O.selection_keys(l, "sigmoid", bias)
    idx, gap = O.select_topk(key, 2)
    assert idx.tolist() == [[1, 2]]
    assert abs(gap[0] - (0.75 - 0.5)) < 1e-15
    g = O.gates_for(l, idx, "sigmoid", True)
    np.testing.assert_allclose(g, [[0.75, 0.25]], atol=1e-15)
    idx0, _ = O.select_topk(O.selection_keys(l, "sigmoid", None), 2)
    assert idx0.tolist() == [[0, 1]]
    np.testing.assert_allclose(O.gates_for(l, idx0, "sigmoid", True), [[0.4, 0.6]],
                               atol=1e-15)


# ---------------------------------------------------------------- expert and layer

def _silu(z):
    return z / (1.0 + math.exp(-z))


def test_swiglu_scalar_closed_form():
    # H = I = 1: y = w_d * silu(w_g x) * (w_u x)
    y = O.swiglu_expert(np.array([[1.0]]), np.array([[2.0]]), np.array([[3.0]]),
                        np.array([[5.0]]))
    assert abs(y[0, 0] - 5.0 * _silu(2.0) * 3.0) < 1e-13
    # swapping gate and up gives a different value: the pin catches a swap
    assert abs(5.0 * _silu(3.0) * 2.0 - 5.0 * _silu(2.0) * 3.0) > 1.0
    assert O.swiglu_expert(np.zeros((1, 1)), np.ones((1, 1)), np.ones((1, 1)),
                           np.ones((1, 1)))[0, 0] == 0.0


def test_swiglu_one_hot_orientation():
    """Non-square weights with one-hot inputs: each output is a scalar expression."""
    rng = np.random.default_rng(5)
    H, I = 3, 4
    Wg, Wu, Wd = rng.standard_normal((I, H)), rng.standard_normal((I, H)), \
        rng.standard_normal((H, I))
    for hsel in range(H):
        x = np.zeros((1, H))
        x[0, hsel] = 1.0
        y = O.swiglu_expert(x, Wg, Wu, Wd)[0]
        for o in range(H):
            want = sum(Wd[o, i] * _silu(Wg[i, hsel]) * Wu[i, hsel] for i in range(I))
            assert abs(y[o] - want) < 1e-13


def test_round_bf16_matches_torch_and_ties_go_to_even():
    """The oracle's bf16 rounding against torch's bf16 conversion (round to nearest even),
    on random values over many binades and on exact halfway cases."""
    import torch
    rng = np.random.default_rng(11)
    v = rng.standard_normal(200000) * np.exp2(rng.integers(-30, 30, 200000))
    want = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(O.round_bf16(v.astype(np.float32)), want)
    # bf16 keeps 8 significant bits: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7
    assert O.round_bf16(np.array([1.0 + 2.0 ** -8]))[0] == 1.0              # to even
    assert O.round_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6  # to even
    assert O.round_bf16(np.array([1.0 + 2.0 ** -8 + 2.0 ** -20]))[0] == 1.0 + 2.0 ** -7
    assert O.round_bf16(np.array([-(1.0 + 2.0 ** -8)]))[0] == -1.0
    assert O.round_bf16(np.array([0.0, 3.0, -0.15625]))[2] == -0.15625   # exact values stay


def test_swiglu_rounds_the_intermediate_only_when_asked():
    """h_round acts on h between the projections: with H = I = 1 the output is
    w_d * round(silu(w_g x) * (w_u x)); without it the output is exact."""
    x, wg, wu, wd = np.array([[1.0]]), np.array([[0.7]]), np.array([[1.3]]), np.array([[3.0]])
    h = _silu(0.7) * 1.3
    y = O.swiglu_expert(x, wg, wu, wd, h_round=O.round_bf16)[0, 0]
    assert y == 3.0 * O.round_bf16(np.array([h]))[0]
    assert O.round_bf16(np.array([h]))[0] != h
    assert abs(O.swiglu_expert(x, wg, wu, wd)[0, 0] - 3.0 * h) < 1e-14


def test_layer_single_expert_is_dense_swiglu():
    """E = 1, k = 1: the gate is 1 and the layer is the one expert."""
    X = np.array([[1.0], [-0.5]])
    Wg = np.array([[0.3]])
    Y, r = O.moe_layer(X, Wg, np.array([[[2.0]]]), np.array([[[3.0]]]),
                       np.array([[[5.0]]]), k=1, score="softmax", renorm=True)
    assert r["gate"].tolist() == [[1.0], [1.0]]
    for t, x in enumerate([1.0, -0.5]):
        assert abs(Y[t, 0] - 5.0 * _silu(2.0 * x) * 3.0 * x) < 1e-13


def test_layer_combine_weights_and_shared():
    """Two scalar experts, top-2 softmax renorm: Y = g0*E0(x) + g1*E1(x) + shared(x)."""
    X = np.array([[1.0]])
    Wg = np.array([[0.0, math.log(3.0)]])          # logits 0, ln3 -> gates 1/4, 3/4
    Wgt = np.array([[[2.0]], [[1.0]]])
    Wup = np.array([[[3.0]], [[1.0]]])
    Wdn = np.array([[[5.0]], [[4.0]]])
    sh = (np.array([[1.0]]), np.array([[2.0]]), np.array([[-1.0]]))
    Y, r = O.moe_layer(X, Wg, Wgt, Wup, Wdn, k=2, score="softmax", renorm=True,
                       shared=sh)
    np.testing.assert_allclose(r["gate"], [[0.25, 0.75]], atol=1e-15)
    e0 = 5.0 * _silu(2.0) * 3.0
    e1 = 4.0 * _silu(1.0) * 1.0
    s = -1.0 * _silu(1.0) * 2.0
    assert abs(Y[0, 0] - (0.25 * e0 + 0.75 * e1 + s)) < 1e-13


def test_layer_drop_contributes_nothing():
    """Capacity 0 drops every slot: only the shared expert remains; with capacity 1 the
    second token loses its slot and its gate is not renormalised onto anything."""
    X = np.array([[1.0], [2.0]])
    Wg = np.array([[1.0]])
    W = np.array([[[1.0]]])
    sh = (np.array([[1.0]]), np.array([[1.0]]), np.array([[1.0]]))
    Y, r = O.moe_layer(X, Wg, W, W, W, k=1, score="softmax", renorm=True, C=0,
                       shared=sh)
    for t, x in enumerate([1.0, 2.0]):
        assert abs(Y[t, 0] - _silu(x) * x) < 1e-13
    Y, r = O.moe_layer(X, Wg, W, W, W, k=1, score="softmax", renorm=True, C=1)
    assert r["row_of_slot"].tolist() == [0, -1]
    assert abs(Y[0, 0] - _silu(1.0)) < 1e-13 and Y[1, 0] == 0.0


def test_identity_experts_round_trip():
    """Dispatch then combine with identity experts and renormalised gates returns X:
    the gates of a token sum to 1 [KM], and the permutation pair is inverse [LI 14.2.1]."""
    rng = np.random.default_rng(11)
    T, H, E, k = 30, 6, 5, 3
    X = rng.standard_normal((T, H))
    l = rng.standard_normal((T, E))
    idx, _ = O.select_topk(l, k)
    g = O.gates_for(l, idx, "softmax", True)
    d = O.dispatch(idx, E)
    Xperm = X[d["slot_of_row"] // k]            # step 4: gather
    Operm = Xperm.copy()                        # identity experts
    Y = np.zeros_like(X)
    for s in range(T * k):                      # step 6: weighted scatter back
        Y[s // k] += g[s // k, s % k] * Operm[d["row_of_slot"][s]]
    np.testing.assert_allclose(Y, X, atol=1e-14)


def test_route_probabilities_and_gap():
    rng = np.random.default_rng(2)
    X = rng.standard_normal((10, 6))
    Wg = rng.standard_normal((6, 4)) * 0.5
    r = O.route(X, Wg, 2, "softmax", True)
    np.testing.assert_allclose(r["prob_colsum"].sum(), 10.0, atol=1e-12)
    srt = -np.sort(-r["logits"], 1)
    np.testing.assert_allclose(r["gap"], srt[:, 1] - srt[:, 2], atol=0)
    r = O.route(X, Wg, 2, "sigmoid", True, bias=np.zeros(4))
    np.testing.assert_allclose(r["prob_colsum"].sum(), 10.0, atol=1e-12)


# ---------------------------------------------------------------- group-limited routing

def _group_limited_brute(key, aff, k, G, M):
    """Group-limited top-k of one row as maxima over subsets: a group's score is the
    largest sum of k/M of its affinities; the groups used are the M-subset with the
    largest total score; the experts are the k-subset of the allowed ones with the
    largest total key.  (Distinct random values: every maximiser is unique.)"""
    E = len(key)
    gs, n = E // G, k // M
    score = [max(sum(c) for c in itertools.combinations(aff[g * gs:(g + 1) * gs], n))
             for g in range(G)]
    groups = max(itertools.combinations(range(G), M), key=lambda c: sum(score[g] for g in c))
    allowed = [e for e in range(E) if e // gs in groups]
    chosen = max(itertools.combinations(allowed, k), key=lambda c: sum(key[e] for e in c))
    others_g = [score[g] for g in range(G) if g not in groups]
    g_gap = min(score[g] for g in groups) - max(others_g) if others_g else math.inf
    others_e = [key[e] for e in allowed if e not in chosen]
    k_gap = min(key[e] for e in chosen) - max(others_e) if others_e else math.inf
    return sorted(chosen), min(g_gap, k_gap)


@pytest.mark.parametrize("E,G,M,k", [(12, 4, 2, 4), (12, 3, 1, 2), (16, 4, 2, 2),
                                     (12, 6, 3, 3), (8, 4, 2, 4)])
def test_group_limited_brute_force(E, G, M, k):
    rng = np.random.default_rng(E * 100 + G * 10 + M)
    T = 25
    aff = rng.random((T, E))
    key = aff + rng.standard_normal((T, E)) * 0.3     # a selection bias reorders the keys
    idx, gap = O.group_limited_topk(key, aff, k, G, M)
    for t in range(T):
        want, want_gap = _group_limited_brute(key[t], aff[t], k, G, M)
        assert idx[t].tolist() == want
        assert gap[t] == pytest.approx(want_gap, abs=1e-12) if math.isfinite(want_gap) \
            else gap[t] == math.inf


def test_group_limited_reduces_to_plain_topk():
    rng = np.random.default_rng(5)
    l = rng.standard_normal((40, 16))
    key = O.selection_keys(l, "sigmoid", rng.standard_normal(16) * 0.1)
    aff = O.routing_affinity(l, "sigmoid")
    plain_idx, plain_gap = O.select_topk(key, 4)
    for G, M in [(1, 1), (4, 4), (2, 2)]:     # every group allowed
        idx, gap = O.group_limited_topk(key, aff, 4, G, M)
        assert np.array_equal(idx, plain_idx)
        np.testing.assert_array_equal(gap, plain_gap)


def test_group_limited_hand_example():
    # 8 experts in 4 groups of 2, affinities s; k = 2 over M = 2 groups: each group
    # is scored by its single best affinity (k/M = 1):
    #   g0 = {0.90, 0.85} -> 0.90, g1 = {0.10, 0.20} -> 0.20,
    #   g2 = {0.80, 0.05} -> 0.80, g3 = {0.30, 0.40} -> 0.40.
    # Groups g0 and g2 are used; the top two keys among experts 0, 1, 4, 5 are 0 and 1.
    # Group margin 0.80 - 0.40, key margin 0.85 - 0.80.
    s = np.array([[0.90, 0.85, 0.10, 0.20, 0.80, 0.05, 0.30, 0.40]])
    idx, gap = O.group_limited_topk(s, s, 2, 4, 2)
    assert idx.tolist() == [[0, 1]]
    assert gap[0] == pytest.approx(0.05, abs=1e-15)
    # a bias that makes expert 7 the largest key does not rescue its group: the group
    # score uses the unbiased affinity (0.40 < 0.80)
    key = s + np.array([0, 0, 0, 0, 0, 0, 0, 1.0])
    idx, _ = O.group_limited_topk(key, s, 2, 4, 2)
    assert idx.tolist() == [[0, 1]]
    assert O.select_topk(key, 2)[0].tolist() == [[0, 7]]
    # k = 4 over M = 2 groups: the two best affinities of a group are summed:
    #   g0 1.75, g1 0.30, g2 0.85, g3 0.70 -> g0, g2; all four allowed experts are chosen
    idx, gap = O.group_limited_topk(s, s, 4, 4, 2)
    assert idx.tolist() == [[0, 1, 4, 5]]
    assert gap[0] == pytest.approx(0.85 - 0.70, abs=1e-15)


def test_group_limited_route_softmax_affinity_is_probability():
    # for softmax scoring the group score sums probabilities: with 2 experts per group
    # and k/M = 2 a group's score is the probability mass of the group
    rng = np.random.default_rng(9)
    X = rng.standard_normal((30, 8))
    Wg = rng.standard_normal((8, 8))
    r = O.route(X, Wg, 4, "softmax", True, n_groups=4, topk_groups=2)
    p = O.softmax_rows(r["logits"]).reshape(30, 4, 2).sum(2)
    best2 = np.sort(np.argsort(-p, 1, kind="stable")[:, :2], 1)
    assert np.array_equal(r["idx"] // 2, np.repeat(best2, 2, axis=1))


def test_group_limited_rejects_bad_shapes():
    key = np.zeros((1, 8))
    for G, M, k in [(3, 1, 2), (4, 3, 4), (4, 2, 3), (4, 1, 4), (4, 5, 5)]:
        with pytest.raises(ValueError):
            O.group_limited_topk(key, key, k, G, M)


# ---------------------------------------------------------------- bias update step

def test_bias_update_hand_example():
    # T*k = 8 slots over E = 4 experts: balanced load 2.  Counts 5, 1, 2, 0: expert 0 is
    # overloaded (-gamma), experts 1 and 3 underloaded (+gamma), expert 2 unchanged.
    b = np.array([0.5, -0.25, 0.125, 0.0])
    out = O.bias_update(b, [5, 1, 2, 0], T=4, k=2, gamma=0.001)
    np.testing.assert_array_equal(out, [0.5 - 0.001, -0.25 + 0.001, 0.125, 0.001])


def test_bias_update_mean_compared_exactly():
    # T*k/E = 10/3: counts 3 and 4 sit below and above it; no count equals it
    out = O.bias_update(np.zeros(3), [3, 4, 3], T=10, k=1, gamma=0.5)
    np.testing.assert_array_equal(out, [0.5, -0.5, 0.5])
    # gamma = 0 (the rate of the last phase of training on the page) changes nothing
    b = np.random.default_rng(0).standard_normal(16)
    np.testing.assert_array_equal(O.bias_update(b, np.arange(16), 30, 4, 0.0), b)


def test_bias_update_float32_rounding_is_single():
    # float32 bias and gamma: the float64 result is the exact sum, so one rounding to
    # float32 equals a float32 addition (correctly rounded)
    rng = np.random.default_rng(3)
    b = (rng.standard_normal(64) * 0.1).astype(np.float32)
    g = np.float32(0.001)
    counts = rng.integers(0, 9, 64)
    out = O.bias_update(b, counts, T=128, k=2, gamma=float(g)).astype(np.float32)
    over = 64 * counts > 256
    under = 64 * counts < 256
    want = np.where(over, b - g, np.where(under, b + g, b)).astype(np.float32)
    np.testing.assert_array_equal(out, want)


# ---------------------------------------------------------------- expert-choice routing

def test_expert_choice_brute_force():
    rng = np.random.default_rng(11)
    T, E, C = 8, 3, 3
    S = rng.random((T, E))
    r = O.expert_choice(S, C)
    for e in range(E):
        col = S[:, e]
        best = max(itertools.combinations(range(T), C), key=lambda c: sum(col[t] for t in c))
        assert r["chosen"][e].tolist() == list(best)
        rest = [col[t] for t in range(T) if t not in best]
        assert r["gap"][e] == pytest.approx(min(col[list(best)]) - max(rest), abs=1e-15)


def test_expert_choice_hand_examples():
    # T = 4 tokens, E = 2 experts, k = 1: C = T*k/E = 2 tokens per expert
    S = np.array([[0.9, 0.1], [0.6, 0.4], [0.3, 0.7], [0.2, 0.8]])
    r = O.expert_choice(S, 2)
    assert r["chosen"].tolist() == [[0, 1], [2, 3]]
    np.testing.assert_allclose(r["gap"], [0.6 - 0.3, 0.7 - 0.4], atol=1e-15)
    # tokens 0 and 1 are taken twice, tokens 2 and 3 by nobody (the page's caveat)
    S = np.array([[0.9, 0.8], [0.6, 0.7], [0.1, 0.2], [0.3, 0.05]])
    r = O.expert_choice(S, 2)
    assert r["chosen"].tolist() == [[0, 1], [0, 1]]
    assert r["row_of_slot"].tolist() == [0, 2, 1, 3, -1, -1, -1, -1]
    assert r["slot_of_row"].tolist() == [0, 2, 1, 3]
    np.testing.assert_array_equal(r["gate"], [[0.9, 0.8], [0.6, 0.7], [0, 0], [0, 0]])


def test_expert_choice_ties_and_balance():
    S = np.full((6, 3), 0.5)
    r = O.expert_choice(S, 4)
    assert r["chosen"].tolist() == [[0, 1, 2, 3]] * 3      # ties: lowest token indices
    assert np.all(r["gap"] == 0)
    rng = np.random.default_rng(4)
    S = rng.random((40, 5))
    r = O.expert_choice(S, 16)
    # every expert takes exactly C; the rows are the inverse permutation of their slots
    assert np.all((r["row_of_slot"].reshape(40, 5) >= 0).sum(0) == 16)
    assert np.array_equal(r["row_of_slot"][r["slot_of_row"]], np.arange(80))
    assert np.array_equal(r["slot_of_row"] % 5, np.repeat(np.arange(5), 16))


def test_expert_choice_single_expert_is_dense():
    # E = 1, k = 1: the expert takes every token with softmax affinity 1
    rng = np.random.default_rng(6)
    X = rng.standard_normal((7, 4))
    Wg = rng.standard_normal((4, 1))
    r = O.route_expert_choice(X, Wg, 1, "softmax")
    assert r["chosen"].tolist() == [list(range(7))]
    np.testing.assert_array_equal(r["gate"], np.ones((7, 1)))
    Wgt, Wup, Wdn = (rng.standard_normal((3, 4)), rng.standard_normal((3, 4)),
                     rng.standard_normal((4, 3)))
    Y = O.combine_subset(X, r, lambda e: (Wgt, Wup, Wdn), np.arange(7))
    np.testing.assert_allclose(Y, O.swiglu_expert(X, Wgt, Wup, Wdn), rtol=1e-14)


def test_expert_choice_needs_integer_capacity():
    with pytest.raises(ValueError):
        O.route_expert_choice(np.zeros((5, 2)), np.zeros((2, 2)), 1, "softmax")


# ---------------------------------------------------------------- FP8 (E4M3) weights

def test_e4m3_codes_from_the_format():
    # 1.0 = 2^0: e = 7, m = 0; 448 = 2^8 * 1.75: e = 15, m = 6; 2^-6 smallest normal;
    # 2^-9 smallest subnormal; -0 keeps its sign
    v = [1.0, 448.0, 2.0 ** -6, 2.0 ** -9, 7 * 2.0 ** -9, -0.0, -2.5, 0.0]
    assert O.e4m3_encode(np.array(v)).tolist() == [0x38, 0x7E, 0x08, 0x01, 0x07, 0x80,
                                                   0xC2, 0x00]
    # ties to even: 1.0625 lies between 1.0 (m = 0) and 1.125 (m = 1) -> 1.0; 1.1875
    # between 1.125 and 1.25 (m = 2) -> 1.25; 2^-10 between 0 and 2^-9 -> 0
    assert O.e4m3_encode(np.array([1.0625, 1.1875, 2.0 ** -10])).tolist() == [0x38, 0x3A, 0]
    # saturation above the largest finite value
    assert O.e4m3_encode(np.array([464.0, 1e6, -500.0])).tolist() == [0x7E, 0x7E, 0xFE]


def test_e4m3_round_trip_and_library_cast():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = O.e4m3_decode(codes)
    back = O.e4m3_encode(vals)
    assert np.array_equal(back[vals != 0], codes[vals != 0])
    # in range, the codes equal torch's round-to-nearest-even float8_e4m3fn cast
    import torch
    rng = np.random.default_rng(8)
    x = (rng.standard_normal(4000) * 40).astype(np.float32)
    x = x[np.abs(x) <= 448]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(x.astype(np.float64)), want)


def test_quantize_fp8_rows_scale_and_error():
    rng = np.random.default_rng(12)
    W = (rng.standard_normal((6, 300)) * 0.02).astype(np.float32)
    W[2] = 0.0
    q, s = O.quantize_fp8_rows(W)
    assert q.dtype == np.uint8 and s.dtype == np.float32
    assert s[2] == 1.0 and np.all(q[2] == 0)
    # the largest magnitude of every non-zero row maps to +-448
    for r in (0, 1, 3, 4, 5):
        assert np.abs(O.e4m3_decode(q[r])).max() == 448.0
    D = O.dequantize_fp8_rows(q, s)
    # relative error at most half a step: 2^-4 of the magnitude for normals, plus the
    # subnormal step 2^-9 * scale near zero
    err = np.abs(D - W)
    # (plus the rounding of w / scale in float32)
    assert np.all(err <= np.abs(W) * (2.0 ** -4 + 2.0 ** -20) + s[:, None] * 2.0 ** -10)

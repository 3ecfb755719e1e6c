"""Plain fp64 CPU oracle for the sparse top-k routed MoE layer forward.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline leg may import or call this module.  It shares no code with the CUDA path and
imports nothing from the library package: it takes numpy arrays and returns numpy
arrays.

Every function writes out the plain definition the pages give, in float64, with no
blocking, fusion or reordering beyond what the definition states.  Library primitives
used as steps: numpy matmul (a dot product over the hidden axis), numpy stable argsort,
numpy exp.  Inputs that arrive as bf16/fp32 widen to float64 exactly.

Sources (page title and section):
  [KM]  AI Knowledge Map, "MoE: each token activates only a few FFNs" - router in four
        steps (score, softmax, top-k hard selection, renormalise and combine); capacity
        C = ceil(c*N*k/E) with the 6-token / 4-expert / top-2 worked example; overflow
        handling (drop, reroute, larger c); load CV = std/mean.
  [LI]  LLM Internals §14.2 "Mixture of experts" - §14.2.1 six steps and shapes
        (input, router scoring, top-k + normalisation, dispatch permutation, grouped
        GEMM, combine + shared expert); §14.2.2 parameter accounting; §14.2.3 balance
        loss L = alpha*N*sum f_i p_i with worked example, bias-adjusted selection
        (tech-report eq. 16), capacity factor with worked example; §14.2.4 shared
        expert.
  [SN]  "Mixture of Experts (MoE)" study notes, Case 1: top-k pseudo-code (softmax over
        the k chosen values).
  [P1]  "MoE 03: efficiency frontiers", DeepSeek's hardware-aware design: each token
        goes to at most 4 of the 8 nodes that hold the experts.

Readings where the pages are silent:
  * ties in top-k go to the lower expert index; the chosen set is written in ascending
    expert order (the pages define S as a set);
  * capacity keeps the lowest token indices of each expert;
  * a dropped slot contributes nothing; the other gates are not renormalised;
  * f_i counts router choices before capacity, f_i = m_i / (T*k);
  * for sigmoid scoring, p_i averages the row-normalised affinities s / sum_e s;
  * group-limited routing scores a group by its k/M largest UNBIASED affinities, and
    its groups are runs of consecutive expert indices;
  * SwiGLU expert: h = SiLU(x W_gate) * (x W_up), y = h W_down, SiLU(z) = z*sigmoid(z),
    no biases;
  * a bf16 layer may store the intermediate h in bf16 between its two projections (it is
    a GEMM operand like the inputs); `round_bf16` gives that variant of the expert
    (`h_round`), the default stays exact.

Parity is pinned for every function here (tests/test_oracle_pins.py); none is unpinned.
"""

from __future__ import annotations

from fractions import Fraction
from typing import Callable, Dict, Optional, Sequence, Tuple

import numpy as np

f64 = np.float64


# ---------------------------------------------------------------------------
# Step 2: router scoring                                          [LI §14.2.1 step 2]
# ---------------------------------------------------------------------------

def router_logits(X: np.ndarray, Wg: np.ndarray,
                  logit_bias: Optional[np.ndarray] = None) -> np.ndarray:
    """l[t, e] = sum_h X[t, h] * W_g[h, e]  (+ a fixed per-expert logit offset).

    [LI §14.2.1 step 2]: X[T, H] x W_g[H, E] -> s[T, E].  [KM] step one: W_r x.
    Products of a bf16 or fp32 value by an fp32 value are exact in float64.
    """
    l = np.asarray(X, dtype=f64) @ np.asarray(Wg, dtype=f64)
    if logit_bias is not None:
        l = l + np.asarray(logit_bias, dtype=f64)[None, :]
    return l


def softmax_rows(l: np.ndarray) -> np.ndarray:
    """g_e = exp(l_e) / sum_j exp(l_j) per row  [KM step two].

    The row maximum is subtracted first; that leaves the quotient unchanged.
    """
    m = l.max(axis=1, keepdims=True)
    z = np.exp(l - m)
    return z / z.sum(axis=1, keepdims=True)


def sigmoid(l: np.ndarray) -> np.ndarray:
    """Per-cell affinity s = 1 / (1 + exp(-l))  [LI §14.2.1 step 2, DeepSeek-V3]."""
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-l))


def selection_keys(l: np.ndarray, score: str,
                   bias: Optional[np.ndarray] = None) -> np.ndarray:
    """The value the top-k compares.

    softmax: the logit itself (softmax is strictly increasing in each logit of a row,
    so top-k on logits equals top-k on probabilities - [SN] Case 1 takes top-k on the
    raw router scores, [KM] on the probabilities).
    sigmoid: s + b, the bias taking part in selection only  [LI §14.2.3, eq. 16].
    """
    if score == "softmax":
        return l.copy()
    if score == "sigmoid":
        s = sigmoid(l)
        return s + (0.0 if bias is None else np.asarray(bias, dtype=f64)[None, :])
    raise ValueError(score)


# ---------------------------------------------------------------------------
# Step 3: top-k hard selection and renormalisation     [LI §14.2.1 step 3; KM steps 3-4]
# ---------------------------------------------------------------------------

def select_topk(key: np.ndarray, k: int) -> Tuple[np.ndarray, np.ndarray]:
    """The k largest keys of each row  [LI §14.2.1 step 3; KM step three; SN Case 1].

    Returns idx[T, k] (the chosen experts, ascending expert index) and gap[T] =
    key_(k) - key_(k+1), the margin between the k-th and (k+1)-th largest key
    (+inf when k == E).  Ties go to the lower expert index (stable sort).
    """
    T, E = key.shape
    order = np.argsort(-key, axis=1, kind="stable")
    rows = np.arange(T)
    if k < E:
        gap = key[rows, order[:, k - 1]] - key[rows, order[:, k]]
    else:
        gap = np.full(T, np.inf)
    idx = np.sort(order[:, :k], axis=1)
    return idx.astype(np.int64), gap


def routing_affinity(l: np.ndarray, score: str) -> np.ndarray:
    """The affinity of token t for expert e, unbiased: softmax(l)_e for softmax scoring,
    s = sigmoid(l_e) for sigmoid scoring  [LI §14.2.1 step 2; §14.2.3 eq. 16, where the
    bias enters only the top-k comparison]."""
    if score == "softmax":
        return softmax_rows(l)
    if score == "sigmoid":
        return sigmoid(l)
    raise ValueError(score)


def group_limited_topk(key: np.ndarray, affinity: np.ndarray, k: int, n_groups: int,
                       topk_groups: int) -> Tuple[np.ndarray, np.ndarray]:
    """Node-limited (group-limited) routing  [LI §14.2.3, node-limited routing; P1].

    The E experts sit in n_groups equal groups of consecutive indices (the experts of
    one node).  A group's score is the sum of its k / topk_groups largest affinities.
    Each token may use only the experts of its topk_groups best groups (ties to the
    lower group index); among those it takes the k largest keys (ties to the lower
    expert index).  The affinity is the unbiased one (routing_affinity): the page
    scores a node by its experts' affinities, and the selection bias enters only the
    top-k comparison of experts.

    Returns idx[T, k] (ascending expert index) and gap[T] = the smaller of the group
    margin S_(M) - S_(M+1) and the key margin key_(k) - key_(k+1) among the allowed
    experts (a margin that does not exist counts as +inf).
    """
    T, E = key.shape
    G, M = n_groups, topk_groups
    if G < 1 or E % G or not 1 <= M <= G or k % M or k // M > E // G or M * (E // G) < k:
        raise ValueError("unsupported group-limited routing shape")
    gs, n = E // G, k // M
    rows = np.arange(T)
    per_group = np.asarray(affinity, dtype=f64).reshape(T, G, gs)
    top_n = -np.sort(-per_group, axis=2)[:, :, :n]          # descending
    S = top_n.sum(axis=2)                                   # [T, G] group scores
    g_order = np.argsort(-S, axis=1, kind="stable")
    if M < G:
        g_gap = S[rows, g_order[:, M - 1]] - S[rows, g_order[:, M]]
    else:
        g_gap = np.full(T, np.inf)
    allowed_g = np.zeros((T, G), dtype=bool)
    allowed_g[rows[:, None], g_order[:, :M]] = True
    allowed = np.repeat(allowed_g, gs, axis=1)
    masked = np.where(allowed, key, -np.inf)
    order = np.argsort(-masked, axis=1, kind="stable")
    if M * gs > k:
        k_gap = key[rows, order[:, k - 1]] - key[rows, order[:, k]]
    else:
        k_gap = np.full(T, np.inf)
    idx = np.sort(order[:, :k], axis=1)
    return idx.astype(np.int64), np.minimum(g_gap, k_gap)


def gates_for(l: np.ndarray, idx: np.ndarray, score: str, renorm: bool) -> np.ndarray:
    """Gate weights of the chosen experts.

    softmax: g_e = softmax(l)_e; with renorm, g_e / sum_{e' in S} g_{e'}  [KM step four].
    sigmoid: s_e = sigmoid(l_e) of the UNBIASED logit; with renorm, s_e / sum_S s
             [LI §14.2.3 eq. 16: the gate keeps the original affinity; §14.2.1 step 3
             normalises among the k chosen].
    """
    rows = np.arange(l.shape[0])[:, None]
    if score == "softmax":
        g = softmax_rows(l)[rows, idx]
    elif score == "sigmoid":
        g = sigmoid(l)[rows, idx]
    else:
        raise ValueError(score)
    if renorm:
        g = g / g.sum(axis=1, keepdims=True)
    return g


def row_probabilities(l: np.ndarray, score: str) -> np.ndarray:
    """p[t, e] used by the balance statistics  [LI §14.2.3]: the softmax row, or for
    sigmoid scoring the affinities normalised over the row (an extension: the pages
    define p_i only as the router's mean probability for expert i)."""
    if score == "softmax":
        return softmax_rows(l)
    s = sigmoid(l)
    return s / s.sum(axis=1, keepdims=True)


# ---------------------------------------------------------------------------
# Capacity and step 4: dispatch permutation                  [KM capacity; LI §14.2.1]
# ---------------------------------------------------------------------------

def capacity(c: float, T: int, k: int, E: int) -> int:
    """C = ceil(c * N * k / E) with N the token count  [KM capacity formula].

    Evaluated exactly: the float c is the dyadic rational it stores.
    """
    q = Fraction(c) * T * k / E
    return int(-((-q.numerator) // q.denominator))


def dispatch(idx: np.ndarray, E: int, C: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Group the (token, choice) slots by expert  [LI §14.2.1 step 4].

    Slot s = t*k + j is the j-th choice of token t.  m_e counts the slots routed to e
    (before capacity).  With a capacity C, expert e keeps its C slots of lowest token
    index and drops the rest  [KM overflow: drop].  Rows of the permuted batch are
    ordered by (expert ascending, token ascending); offsets[e] is the first row of e.
    row_of_slot[s] = permuted row of slot s, or -1 when the slot was dropped;
    slot_of_row is its inverse on the kept rows.
    """
    T, k = idx.shape
    flat = idx.reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    kept = counts.copy() if C is None else np.minimum(counts, C)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(kept)
    R = int(offsets[-1])
    row_of_slot = np.full(T * k, -1, dtype=np.int64)
    slot_of_row = np.full(R, -1, dtype=np.int64)
    for e in range(E):
        # a token routes to e at most once, so ascending slot = ascending token
        slots = np.nonzero(flat == e)[0]
        keep = slots[: kept[e]]
        rows = offsets[e] + np.arange(keep.size)
        row_of_slot[keep] = rows
        slot_of_row[rows] = keep
    return dict(counts=counts, kept=kept, offsets=offsets,
                row_of_slot=row_of_slot, slot_of_row=slot_of_row)


# ---------------------------------------------------------------------------
# FP8 expert weights                        [LI §14.2.5: one expert = 44 MB in FP8]
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """FP8 E4M3 codes of float values: 1 sign bit, 4 exponent bits (bias 7) and 3
    mantissa bits; normals 2^(e-7) * (1 + m/8) for e = 1..15 (e = 15 with m = 7 is NaN,
    so 448 is the largest finite value), subnormals 2^-6 * m/8.  Round to nearest, ties
    to even; magnitudes above 448 saturate to 448.  The page states the FP8 size of an
    expert and no format details: E4M3 is the FP8 format whose range holds weights."""
    v = np.asarray(v, dtype=f64)
    neg = np.signbit(v)
    a = np.abs(v)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))       # a = f * 2^ex, f in [0.5, 1)
    E = np.clip(ex - 1, -6, 8)                      # binade; below 2^-6 the subnormal step
    step = np.ldexp(1.0, E - 3)                     # spacing of E4M3 values in the binade
    r = np.round(a / step) * step                   # a / step is exact; ties to even
    r = np.minimum(r, E4M3_MAX)
    _, rex = np.frexp(np.where(r > 0, r, 1.0))
    rE = rex - 1
    normal = r >= 2.0 ** -6
    e = np.where(normal, rE + 7, 0)
    m = np.where(normal, r / np.ldexp(1.0, rE) * 8 - 8, r / 2.0 ** -9)
    code = (neg.astype(np.int64) << 7) | (e.astype(np.int64) << 3) | m.astype(np.int64)
    return code.astype(np.uint8)


def e4m3_decode(code: np.ndarray) -> np.ndarray:
    """The value of every finite E4M3 code (see e4m3_encode), in float64."""
    c = np.asarray(code, dtype=np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 7
    return s * np.where(e > 0, np.ldexp(1.0 + m / 8.0, e - 7), m * 2.0 ** -9)


def quantize_fp8_rows(W: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per-output-channel FP8 weights: W[..., r, :] ~= scale[..., r] * e4m3(q[..., r, :]).

    The page gives one byte per parameter and no scale convention; this takes one fp32
    scale per row of the output-major weight (per output channel), scale = amax / 448
    (1 for an all-zero row), and q = E4M3(w / scale), every step in float32 (division
    correctly rounded), so that the codes are a deterministic function of the weights.
    """
    W32 = np.asarray(W, dtype=np.float32)
    amax = np.abs(W32).max(axis=-1)
    scale = np.where(amax > 0, (amax / np.float32(E4M3_MAX)).astype(np.float32),
                     np.float32(1.0)).astype(np.float32)
    v = (W32 / scale[..., None]).astype(np.float32)
    return e4m3_encode(v.astype(f64)), scale


def dequantize_fp8_rows(q: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """scale[r] * value(q[r, :]) in float64 (exact: a 4-bit significand times an fp32);
    the weights an FP8 expert computes with  [LI §14.2.5]."""
    return np.asarray(scale, dtype=f64)[..., None] * e4m3_decode(q)


# ---------------------------------------------------------------------------
# Step 5: one SwiGLU expert                                  [LI §14.2.1 step 5, §14.2.2]
# ---------------------------------------------------------------------------

def round_bf16(v: np.ndarray) -> np.ndarray:
    """The bf16 value nearest to each (finite) v, ties to even, as float64.

    bf16 is the upper half of an fp32 bit pattern, so v is first rounded to fp32 (numpy's
    correctly rounded conversion) and then the lower 16 bits of that pattern are rounded
    off: adding 0x7FFF plus the lowest kept bit carries into the kept half exactly when
    the dropped half exceeds one half ulp, or equals it with the kept half odd.
    """
    v32 = np.ascontiguousarray(np.asarray(v, dtype=f64).astype(np.float32))
    bits = v32.view(np.uint32).astype(np.uint64)
    bits = (bits + 0x7FFF + ((bits >> 16) & 1)) & 0xFFFF0000
    return bits.astype(np.uint32).view(np.float32).astype(f64)


def swiglu_expert(x: np.ndarray, W_gate: np.ndarray, W_up: np.ndarray,
                  W_down: np.ndarray,
                  h_round: Optional[Callable[[np.ndarray], np.ndarray]] = None) -> np.ndarray:
    """y = (SiLU(x W_gate^T) * (x W_up^T)) W_down^T for a batch of rows x[m, H].

    Weights are stored output-major: W_gate, W_up [I, H]; W_down [H, I].  The expert is
    the three-matrix SwiGLU of [LI §14.2.2]; [LI §14.2.1 step 5] projects [m, H] to
    [m, I] and back to H.  `h_round`, if given, is applied to the [m, I] intermediate
    before the second projection (e.g. round_bf16 for a layer that stores it in bf16).
    """
    x = np.asarray(x, dtype=f64)
    a = x @ np.asarray(W_gate, dtype=f64).T
    u = x @ np.asarray(W_up, dtype=f64).T
    h = a * sigmoid(a) * u
    if h_round is not None:
        h = h_round(h)
    return h @ np.asarray(W_down, dtype=f64).T


# ---------------------------------------------------------------------------
# Balance statistics                             [LI §14.2.3; KM monitoring, CV]
# ---------------------------------------------------------------------------

def balance_loss(f: Sequence[float], p: Sequence[float], alpha: float) -> float:
    """L = alpha * N * sum_i f_i p_i with N the number of experts  [LI §14.2.3]."""
    f = np.asarray(f, dtype=f64)
    p = np.asarray(p, dtype=f64)
    return float(alpha * f.size * np.sum(f * p))


def balance_stats(counts: np.ndarray, prob_colsum: np.ndarray, T: int, k: int,
                  n_kept: int, alpha: float) -> Dict[str, object]:
    """f_i = m_i/(T k) (router choices before capacity), p_i = mean_t p[t, i],
    loss = alpha*E*sum f p, drop rate = dropped slots / (T k),
    CV = population std / mean of m_i  [KM monitoring], routing entropy -sum f ln f
    [LI §14.2.3 monitoring: routing entropy, per-expert load, drop rate]."""
    counts = np.asarray(counts, dtype=f64)
    E = counts.size
    f = counts / (T * k)
    p = np.asarray(prob_colsum, dtype=f64) / T
    loss = balance_loss(f, p, alpha)
    drop_rate = (T * k - n_kept) / (T * k)
    mean = counts.mean()
    cv = float(np.sqrt(np.mean((counts - mean) ** 2)) / mean) if mean > 0 else 0.0
    nz = f[f > 0]
    entropy = float(-np.sum(nz * np.log(nz)))
    return dict(f=f, p=p, loss=loss, drop_rate=drop_rate, cv=cv, entropy=entropy)


def bias_update(bias: np.ndarray, counts: np.ndarray, T: int, k: int,
                gamma: float) -> np.ndarray:
    """The auxiliary-loss-free balancing step  [LI §14.2.3, bias-adjusted selection]:
    after a step, the load of every expert over the whole batch is compared with the
    balanced load; an overloaded expert's bias drops by gamma, an underloaded one's
    rises by gamma, and the bias is not learned by backpropagation.

    Load = m_e, the router's choices before capacity; the balanced load is the mean
    T*k/E (the page names no threshold), compared exactly as E*m_e against T*k.  An
    expert at exactly the mean keeps its bias.  Returns the new bias in float64; the
    inputs are float32 values, so b +- gamma is exact here and rounding it to float32
    gives the correctly rounded float32 sum.
    """
    m = np.asarray(counts, dtype=np.int64)
    E = m.size
    b = np.asarray(bias, dtype=f64)
    g = f64(gamma)
    over = E * m > T * k
    under = E * m < T * k
    return np.where(over, b - g, np.where(under, b + g, b))


# ---------------------------------------------------------------------------
# The whole layer                                  [LI §14.2.1 steps 1-6; KM combine]
# ---------------------------------------------------------------------------

def route(X, Wg, k: int, score: str, renorm: bool, bias=None, logit_bias=None,
          C: Optional[int] = None, n_groups: int = 0,
          topk_groups: int = 0) -> Dict[str, np.ndarray]:
    """Steps 2-4 on every token  [LI §14.2.1 steps 2-4; KM capacity] (capacity is a
    property of the whole batch).  With n_groups > 1 the selection is group-limited
    (group_limited_topk)."""
    l = router_logits(X, Wg, logit_bias)
    key = selection_keys(l, score, bias)
    if n_groups > 1:
        idx, gap = group_limited_topk(key, routing_affinity(l, score), k, n_groups,
                                      topk_groups)
    else:
        idx, gap = select_topk(key, k)
    g = gates_for(l, idx, score, renorm)
    d = dispatch(idx, Wg.shape[1], C)
    d.update(logits=l, key=key, idx=idx, gap=gap, gate=g,
             prob_colsum=row_probabilities(l, score).sum(axis=0))
    return d


def expert_choice(S: np.ndarray, C: int) -> Dict[str, np.ndarray]:
    """Expert-choice routing  [LI §14.2, the two selection paradigms: expert-choice; P1,
    "Expert Choice Routing"]: every expert takes the C tokens of the batch with the
    largest affinity S[t, e]; ties go to the lower token index.  A token may be taken
    by several experts or by none.

    In the slot layout of token-choice routing with k = E: slot s = t*E + e is the pair
    (token t, expert e).  Returns chosen[E, C] (each expert's tokens, ascending), the
    rows ordered by (expert, token) - offsets[e] = e*C, row_of_slot[T*E] (-1 = not
    taken), slot_of_row[E*C] - the gates gate[T, E] (S where taken, 0 elsewhere), idx[T, E]
    = e in slot (t, e), and gap[E] = S_(C) - S_(C+1) down each expert's column (+inf
    when C == T).
    """
    S = np.asarray(S, dtype=f64)
    T, E = S.shape
    if not 0 <= C <= T:
        raise ValueError("expert-choice capacity outside [0, T]")
    order = np.argsort(-S, axis=0, kind="stable")          # per column: descending
    chosen = np.sort(order[:C, :].T, axis=1)
    cols = np.arange(E)
    if 0 < C < T:
        gap = S[order[C - 1, cols], cols] - S[order[C, cols], cols]
    else:
        gap = np.full(E, np.inf)
    row_of_slot = np.full(T * E, -1, dtype=np.int64)
    slot_of_row = np.zeros(E * C, dtype=np.int64)
    gate = np.zeros((T, E), dtype=f64)
    for e in range(E):
        rows = e * C + np.arange(C)
        slots = chosen[e] * E + e
        row_of_slot[slots] = rows
        slot_of_row[rows] = slots
        gate[chosen[e], e] = S[chosen[e], e]
    return dict(chosen=chosen, offsets=np.arange(E + 1, dtype=np.int64) * C,
                row_of_slot=row_of_slot, slot_of_row=slot_of_row, gate=gate,
                idx=np.tile(np.arange(E, dtype=np.int64), (T, 1)), gap=gap)


def route_expert_choice(X, Wg, k: int, score: str, logit_bias=None) -> Dict[str, np.ndarray]:
    """Scoring and expert-choice selection on every token  [LI §14.2, the two selection
    paradigms: expert-choice].  Each expert takes the balanced load C = T*k/E (the
    average number of experts per token is k), which must be an integer; S is the
    unbiased affinity (routing_affinity), since a per-expert selection bias would shift
    a whole column and change no expert's choice."""
    l = router_logits(X, Wg, logit_bias)
    T, E = l.shape
    if (T * k) % E:
        raise ValueError("expert-choice needs E to divide T*k")
    S = routing_affinity(l, score)
    d = expert_choice(S, T * k // E)
    d.update(logits=l, S=S)
    return d


ExpertFn = Callable[[int], Tuple[np.ndarray, np.ndarray, np.ndarray]]


def combine_subset(X, routing: Dict[str, np.ndarray], expert: ExpertFn, tokens,
                   shared: Optional[Tuple[np.ndarray, np.ndarray, np.ndarray]] = None,
                   h_round: Optional[Callable[[np.ndarray], np.ndarray]] = None
                   ) -> np.ndarray:
    """Steps 5-6 for the given tokens: Y[t] = sum over kept j of g_j * E_{idx_j}(x_t)
    plus the shared expert's output  [LI §14.2.1 step 6; KM final weighted sum].

    `expert(e)` returns (W_gate[e], W_up[e], W_down[e]); experts are fetched one at a
    time, and only those that a kept slot of the given tokens uses.  `h_round` is passed
    to every expert (swiglu_expert).
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    X = np.asarray(X)
    idx, gate, ros = routing["idx"], routing["gate"], routing["row_of_slot"]
    T, k = idx.shape
    H = X.shape[1]
    Y = np.zeros((tokens.size, H), dtype=f64)
    uses: Dict[int, list] = {}
    for n, t in enumerate(tokens):
        for j in range(k):
            if ros[t * k + j] >= 0:
                uses.setdefault(int(idx[t, j]), []).append((n, j))
    for e in sorted(uses):
        Wgt, Wup, Wdn = expert(e)
        sel = np.asarray(uses[e], dtype=np.int64)
        sel_t, sel_j = sel[:, 0], sel[:, 1]
        o = swiglu_expert(X[tokens[sel_t]], Wgt, Wup, Wdn, h_round)
        Y[sel_t] += gate[tokens[sel_t], sel_j][:, None] * o
    if shared is not None:
        Y += swiglu_expert(X[tokens], *shared, h_round=h_round)
    return Y


def moe_layer(X, Wg, W_gate, W_up, W_down, k: int, score: str, renorm: bool,
              bias=None, logit_bias=None, C: Optional[int] = None,
              shared=None, tokens=None) -> Tuple[np.ndarray, Dict[str, np.ndarray]]:
    """The full forward on in-memory weights (small workloads)  [LI §14.2.1 steps 1-6]."""
    routing = route(X, Wg, k, score, renorm, bias, logit_bias, C)
    if tokens is None:
        tokens = np.arange(np.asarray(X).shape[0])
    Y = combine_subset(X, routing, lambda e: (W_gate[e], W_up[e], W_down[e]), tokens,
                       shared)
    return Y, routing


# ---------------------------------------------------------------------------
# Parameter accounting                                           [LI §14.2.2]
# ---------------------------------------------------------------------------

def expert_params(H: int, I: int) -> int:
    """One SwiGLU expert is three [H, I] matrices: 3*H*I parameters  [LI §14.2.2]."""
    return 3 * H * I


def layer_params(H: int, I: int, routed: int, shared: int) -> int:
    """Parameters of one MoE layer: every routed and shared expert  [LI §14.2.2]."""
    return (routed + shared) * expert_params(H, I)


def active_params(H: int, I: int, k: int, shared: int) -> int:
    """Expert parameters one token uses in a layer: k routed + the shared  [LI §14.2.2]."""
    return (k + shared) * expert_params(H, I)

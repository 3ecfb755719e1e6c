"""GPU parity of the whole forward against the fp64 oracle, through the C ABI.

Small cases (several tiles and ragged tails) and the full-size workloads alike compare the
routing, dispatch and gates of every token, and the output of every token against the
oracle that stores the expert intermediate in bf16 as the layer does; the output is also
compared with the exact oracle on every token of the small cases and on a seeded sample
of the full-size ones.
"""

import gc

import numpy as np
import pytest
import torch

from sparse_top_routing_router_b300 import configs as K

from . import parity as P

pytestmark = pytest.mark.gpu

SMALL = [
    K.TINY_F32,
    K.scaled(K.MIXTRAL, name="mixtral_small", T=300, H=256, I=512),
    K.scaled(K.DSV3_PREFILL, name="dsv3_small", T=200, H=512, E=64, I=256),
    K.scaled(K.DSV3_PREFILL, name="dsv3_small_noshared", T=130, H=256, E=32, I=192,
             shared=False, k=4),
    K.scaled(K.SWITCH, name="switch_small", T=1000, H=256, E=16, I=256),
    # E = 40: tensor-core router logits with N = 48 and a partial 32-column epilogue chunk
    K.scaled(K.DSV3_PREFILL, name="dsv3_small_e40", T=300, H=256, E=40, I=128, k=6),
    # E = 320 experts: tensor-core router logits over two 256-wide expert tiles
    K.scaled(K.DSV3_PREFILL, name="dsv3_small_e320", T=400, H=256, E=320, I=128, k=6),
    # decode-sized: a few rows per expert (operand-swapped tiny tiles) plus the shared expert
    K.scaled(K.DSV3_PREFILL, name="dsv3_small_decode", T=24, H=256, E=64, I=128),
    # uneven group sizes (0 to 583 rows of 2400) beside a 600-row shared expert
    K.scaled(K.DSV3_PREFILL, name="dsv3_small_uneven", T=600, H=256, E=16, I=256, k=4),
    # >= 512 rows per expert on average: the CTA-pair (256-row) tensor-core tiles
    K.scaled(K.MIXTRAL, name="mixtral_small_pairs", T=1100, H=256, E=4, I=384),
    K.scaled(K.DSV3_PREFILL, name="dsv3_small_pairs", T=1100, H=256, E=2, I=256, k=1),
    # group-limited routing: 8 groups of 8 experts, 4 groups per token
    K.scaled(K.DSV3_PREFILL, name="dsv3_small_groups", T=300, H=256, E=64, I=128,
             n_groups=8, topk_groups=4),
    K.scaled(K.SWITCH, name="switch_small_pairs", T=4200, H=128, E=8, I=128),
]


def _cleanup():
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_small_full_parity(cfg):
    cfs = cfg.capacity_factors or (None,)
    for cf in cfs:
        run = P.run_gpu(cfg, capacity_factor=cf)
        assert run.status == 0
        ref = P.oracle_route(run)
        info = P.check_routing(run, ref)
        P.check_dispatch(run, P.to_np(run.layer.idx).astype(np.int64))
        out = P.check_output(run, ref)
        st = P.check_stats(run, ref)
        assert out["tokens"] >= cfg.T - info["excluded_rows"]
        if cfg.dtype == "bf16":
            out.update(P.check_output_bf16_h(run, ref))
        print(cfg.name, cf, info, out, st)
    _cleanup()


# (workload, capacity factor, seeded token sample compared with the exact oracle to the
# 2e-2 * RMS(Y) bound); routing, dispatch and gates are compared on every token, and so
# is Y, to the same bound, against the oracle that stores h in bf16 as the layer does.
# (Against the exact oracle the bound does not hold for every token of every layer:
# rounding h to bf16 alone moves the Switch-shaped layer's worst output by 2.1e-2 *
# RMS(Y).)  The oracle's expert stage over a whole DSV3-shaped batch takes about 15 s on
# 16 host cores.
FULL = [(K.MIXTRAL, None, 512), (K.DSV3_DECODE, None, 64), (K.DSV3_PREFILL, None, 512),
        (K.SWITCH, 1.0, 512), (K.SWITCH, 1.25, 512)]


@pytest.mark.parametrize("cfg,cf,n_tok", FULL,
                         ids=lambda v: v.name if hasattr(v, "name") else str(v))
def test_full_size_parity(cfg, cf, n_tok):
    run = P.run_gpu(cfg, capacity_factor=cf)
    assert run.status == 0
    ref = P.oracle_route(run)
    info = P.check_routing(run, ref)
    P.check_dispatch(run, P.to_np(run.layer.idx).astype(np.int64))
    out = P.check_output(run, ref, n_tokens=n_tok)
    full = P.check_output_bf16_h(run, ref)
    assert full["tokens"] >= cfg.T - info["excluded_rows"]
    out["bf16_h"] = full
    st = P.check_stats(run, ref) if cfg.alpha else {}
    print(cfg.name, cf, info, out, st)
    del run
    _cleanup()

"""The oracle's FP8 weights of many experts, quantized in parallel on the host cores.

Quantizing one DSV3-shaped expert with the oracle's E4M3 encoder takes seconds, and the
full-size decode check touches about a hundred experts, so the experts are quantized and
dequantized by a pool of spawned worker processes (spawn, not fork: the parent holds a CUDA
context).  Each worker runs only the oracle's own functions on the expert's weights as the
layer holds them; the parent consumes the results in ascending expert order, the order in
which the oracle's combine asks for them.  Test infrastructure only.
"""

from __future__ import annotations

import multiprocessing as mp
import os
from typing import Callable, Dict, Iterable, Tuple

import numpy as np


def _init_worker():
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"


def _dequantized(mats: Tuple[np.ndarray, ...]) -> Tuple[np.ndarray, ...]:
    from oracle import moe_oracle as O
    return tuple(O.dequantize_fp8_rows(*O.quantize_fp8_rows(m)) for m in mats)


def ordered_fetch(experts: Iterable[int], weights: Callable[[int], Tuple[np.ndarray, ...]],
                  workers: int = 0, timeout: float = 600.0):
    """A fetch(e) for the oracle's combine_subset that returns the dequantized FP8 weights
    of expert e, computed ahead by a spawned pool.  `experts` must be the ascending list of
    experts the combine will ask for; `weights(e)` gives expert e's float32 matrices.
    Returns (fetch, close)."""
    order = sorted(set(int(e) for e in experts))
    n = workers or max(1, min(16, (os.cpu_count() or 2) - 1))
    ctx = mp.get_context("spawn")
    pool = ctx.Pool(n, initializer=_init_worker)
    it = pool.imap(_dequantized, (weights(e) for e in order))
    pos = {"i": 0}
    cache: Dict[int, Tuple[np.ndarray, ...]] = {}

    def fetch(e: int):
        if e in cache:
            return cache[e]
        assert pos["i"] < len(order) and order[pos["i"]] == e, \
            f"expert {e} requested out of order"
        pos["i"] += 1
        cache.clear()
        cache[e] = it.next(timeout)      # a pool that broke raises instead of hanging
        return cache[e]

    def close():
        pool.terminate()
        pool.join()
    return fetch, close

"""The process pool that quantizes experts for the full-size FP8 parity test returns the
oracle's own FP8 weights, in the order the oracle's combine asks for them (CPU only)."""

import numpy as np
import pytest

from oracle import moe_oracle as O

from .fp8_oracle_pool import ordered_fetch


def test_pool_returns_the_oracles_dequantized_weights_in_order():
    W = {e: tuple((np.random.RandomState(e).randn(8, 32) * 0.02).astype(np.float32)
                  for _ in range(3)) for e in range(6)}
    fetch, close = ordered_fetch([4, 1, 3, 1], lambda e: W[e], workers=2, timeout=120)
    try:
        for e in [1, 1, 3, 4]:          # the combine may ask for an expert twice in a row
            got = fetch(e)
            ref = tuple(O.dequantize_fp8_rows(*O.quantize_fp8_rows(m)) for m in W[e])
            assert all(np.array_equal(a, b) for a, b in zip(got, ref))
        with pytest.raises(AssertionError):
            fetch(0)                   # not in the announced order
    finally:
        close()

"""The allocation-free dispatch entry point, moe_dispatch_static.

Some callers may not allocate device memory at the moment they need the dispatch: an
engine or host runtime that plans every device buffer up front and forbids the allocator
from growing afterwards, or a latency-bound loop that cannot afford the device-wide
synchronisation a cudaMalloc may cause.  moe_dispatch_static serves them: it takes only
inputs and outputs and keeps its scratch in a static device array inside the library.
This test calls it through the C ABI and checks it against moe_dispatch (the
workspace-based entry point) and against the oracle's dispatch of the same routing, on two
calls in a row, so the second call runs on the scratch contents the first one left
behind.  Dispatch is integer work, so the comparison is exact.  This file is named to be
collected last.
"""

import ctypes as C

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_top_routing_router_b300 import binding as B

pytestmark = pytest.mark.gpu


def _routing(T, E, k, gen):
    scores = torch.rand(T, E, generator=gen, device="cuda")
    return scores.argsort(dim=1)[:, :k].sort(dim=1).values.to(torch.int32).contiguous()


def _outputs(T, E, k, H):
    dev = "cuda"
    return (torch.full((E,), -7, dtype=torch.int32, device=dev),
            torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
            torch.full((T * k,), -7, dtype=torch.int32, device=dev),
            torch.full((T * k,), -7, dtype=torch.int32, device=dev),
            torch.zeros(T * k, H, dtype=torch.bfloat16, device=dev))


def test_static_dispatch_matches_workspace_dispatch():
    L = B.lib()
    ctx = B.Context(0)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(123)
    stream = torch.cuda.current_stream()
    # (T, E, k, capacity): the second call is smaller and capacity-limited
    for T, E, k, cap in [(3000, 64, 6, -1), (1000, 16, 2, 90)]:
        H = 128
        idx = _routing(T, E, k, gen)
        X = torch.randn(T, H, generator=gen, device="cuda").to(torch.bfloat16)

        ref = _outputs(T, E, k, H)
        ws = torch.zeros(B.moe_workspace_bytes(T, H, E, 64, k, B.MOE_DTYPE_BF16, 0),
                         dtype=torch.uint8, device="cuda")
        B.moe_dispatch(ctx, idx, E, cap, ref[0], ref[1], ref[2], ref[3], ws, X=X,
                       Xperm=ref[4])

        out = _outputs(T, E, k, H)
        r = L.moe_dispatch_static(T, k, E, H, B.MOE_DTYPE_BF16, cap,
                                  C.c_void_p(idx.data_ptr()), C.c_void_p(X.data_ptr()),
                                  *[C.c_void_p(t.data_ptr()) for t in out],
                                  C.c_void_p(stream.cuda_stream))
        assert r == B.MOE_OK
        torch.cuda.synchronize()
        R = int(ref[1][-1])
        assert torch.equal(out[0], ref[0])            # counts
        assert torch.equal(out[1], ref[1])            # offsets
        assert torch.equal(out[2], ref[2])            # row_of_slot
        assert torch.equal(out[3][:R], ref[3][:R])    # slot_of_row
        assert torch.equal(out[4][:R], ref[4][:R])    # gathered rows
        assert B.moe_get_device_status(ctx, ws) == 0
        # and directly against the oracle's dispatch of the same routing
        o = O.dispatch(idx.cpu().numpy().astype(np.int64), E, None if cap < 0 else cap)
        assert np.array_equal(out[0].cpu().numpy(), o["counts"])
        assert np.array_equal(out[1].cpu().numpy(), o["offsets"])
        assert np.array_equal(out[2].cpu().numpy(), o["row_of_slot"])
        assert np.array_equal(out[3][:R].cpu().numpy(), o["slot_of_row"])
        toks = torch.as_tensor(o["slot_of_row"] // k, device="cuda")
        assert torch.equal(out[4][:R], X[toks])


def test_static_dispatch_rejects_too_many_tokens():
    L = B.lib()
    r = L.moe_dispatch_static(65537, 1, 8, 0, B.MOE_DTYPE_BF16, -1, C.c_void_p(16), None,
                              C.c_void_p(16), C.c_void_p(16), C.c_void_p(16), C.c_void_p(16),
                              None, None)
    assert r == B.MOE_ERR_UNSUPPORTED
    assert b"65537" in L.moe_last_error_detail()

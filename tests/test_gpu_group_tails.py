"""Grouped expert GEMM at the tile boundaries, through the C ABI: groups of 1, 16, 17, 63,
64, 65, 127, 128, 129, 255, 256, 257 and 2177 rows (and, with a shared expert, its own) so
that every tail shape of the tensor-core kernel runs - M = 64 tails with 64-row A boxes,
full 128-row tiles, multi-tile groups, groups taller than the 2048-row m-block - and every
output row is compared with the oracle's SwiGLU expert ("LLM Internals §14.2.1" step 5,
§14.2.2 three matrices) on the same rows.  H = 512 gives the down GEMM two 256-column
n-tiles, so its tiles run as clusters of two CTAs that multicast the shared A rows; with
H = 128 they run as plain single CTAs."""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_top_routing_router_b300 import binding as B

from . import parity as P

pytestmark = pytest.mark.gpu

SIZES = [1, 16, 17, 63, 64, 65, 127, 128, 129, 255, 256, 257, 2177]


@pytest.mark.parametrize("H", [128, 512])
@pytest.mark.parametrize("shared", [False, True])
def test_every_row_at_tile_boundaries(shared, H):
    ctx = B.Context(0)
    E, I, k = len(SIZES), 192, 1
    T = sum(SIZES)
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    # expert e takes SIZES[e] tokens, spread over the batch by a seeded permutation
    owner = torch.repeat_interleave(torch.arange(E), torch.tensor(SIZES))
    owner = owner[torch.randperm(T, generator=torch.Generator().manual_seed(3))]
    idx = owner.to(torch.int32).view(T, 1).cuda()
    X = torch.randn(T, H, generator=g, device="cuda").to(torch.bfloat16)
    W = [(torch.randn(E, I, H, generator=g, device="cuda") * 0.02).to(torch.bfloat16),
         (torch.randn(E, I, H, generator=g, device="cuda") * 0.02).to(torch.bfloat16),
         (torch.randn(E, H, I, generator=g, device="cuda") * 0.02).to(torch.bfloat16)]
    Ws = [(torch.randn(I, H, generator=g, device="cuda") * 0.02).to(torch.bfloat16),
          (torch.randn(I, H, generator=g, device="cuda") * 0.02).to(torch.bfloat16),
          (torch.randn(H, I, generator=g, device="cuda") * 0.02).to(torch.bfloat16)]
    ws = torch.zeros(B.moe_workspace_bytes(T, H, E, I, k, B.MOE_DTYPE_BF16, int(shared)),
                     dtype=torch.uint8, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    ros = torch.empty(T * k, dtype=torch.int32, device="cuda")
    sor = torch.empty(T * k, dtype=torch.int32, device="cuda")
    Xperm = torch.empty(T * k, H, dtype=torch.bfloat16, device="cuda")
    B.moe_dispatch(ctx, idx, E, -1, counts, offsets, ros, sor, ws, X=X, Xperm=Xperm)
    Out = torch.full((T * k, H), float("nan"), device="cuda")
    Osh = torch.full((T, H), float("nan"), device="cuda") if shared else None
    kw = dict(Ws_gate=Ws[0], Ws_up=Ws[1], Ws_down=Ws[2], O_shared=Osh) if shared else {}
    B.moe_grouped_swiglu(ctx, X, Xperm, offsets, W[0], W[1], W[2], Out, ws, k, **kw)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ctx, ws) == 0
    assert P.to_np(counts).tolist() == SIZES
    off = P.to_np(offsets)
    Xd, sor_np = P.to_np(X), P.to_np(sor)
    for e, m in enumerate(SIZES):
        rows = np.arange(off[e], off[e + 1])
        x = Xd[sor_np[rows] // k]
        ref = O.swiglu_expert(x, P.to_np(W[0][e]), P.to_np(W[1][e]), P.to_np(W[2][e]))
        got = P.to_np(Out[torch.as_tensor(rows, device="cuda")])
        rms = float(np.sqrt(np.mean(ref ** 2)))
        err = float(np.abs(got - ref).max())
        assert err <= P.Y_TOL["bf16"] * rms, f"expert {e} ({m} rows): {err:.3e} vs RMS {rms:.3e}"
    if shared:
        ref = O.swiglu_expert(Xd, *(P.to_np(w) for w in Ws))
        got = P.to_np(Osh)
        rms = float(np.sqrt(np.mean(ref ** 2)))
        assert float(np.abs(got - ref).max()) <= P.Y_TOL["bf16"] * rms

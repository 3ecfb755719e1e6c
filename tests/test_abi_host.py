"""Host-side checks of the C ABI (no GPU needed): the library loads and exports every
symbol include/moe.h declares; host helpers (capacity, workspace sizes, status strings);
argument validation rejects bad calls before anything touches a device."""

import ctypes as C
import math
import os
import re

import pytest

from oracle import moe_oracle as O
from sparse_top_routing_router_b300 import binding as B
from sparse_top_routing_router_b300 import build as BUILD

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    BUILD.build()
    return B.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", src)))


def test_exports_match_header(L):
    names = header_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n
    assert sorted(B.EXPORTS) == names


def test_version_and_strings(L):
    assert L.moe_version() == 10400
    assert B.status_string(0) == "ok"
    assert B.status_string(-4) == "device wait timed out"
    for i, n in enumerate(B.KERNEL_NAMES):
        assert L.moe_kernel_name(i).decode() == n
    assert L.moe_kernel_name(99).decode() == "unknown"


@pytest.mark.parametrize("c,T,k,E", [(1.0, 6, 2, 4), (2.0, 6, 2, 4), (1.25, 8192, 2, 64),
                                     (1.0, 16384, 1, 64), (1.25, 16384, 1, 64),
                                     (0.1, 7, 3, 5), (1.1, 1000, 2, 7), (0.0, 10, 1, 2),
                                     (3.0, 0, 1, 2), (1e-300, 5, 1, 1), (0.7, 1, 1, 3)])
def test_capacity_matches_oracle(L, c, T, k, E):
    assert B.moe_capacity(c, T, k, E) == O.capacity(c, T, k, E)


def test_capacity_rejects(L):
    for bad in [(-1.0, 4, 1, 2), (math.inf, 4, 1, 2), (math.nan, 4, 1, 2), (1.0, -1, 1, 2),
                (1.0, 4, 0, 2), (1.0, 4, 1, 0), (1e30, 4, 1, 1),
                # c * T * k = 2^128 exactly: must not wrap to a capacity of 0
                (2.0 ** 82, 2 ** 23, 2 ** 23, 1), (2.0 ** 60, 2 ** 31 - 1, 2 ** 31 - 1, 2 ** 30)]:
        with pytest.raises(B.MoEError):
            B.moe_capacity(*bad)


def test_workspace_bytes(L):
    ws = B.moe_workspace_bytes(8192, 7168, 256, 2048, 8, B.MOE_DTYPE_BF16, 1)
    h = (8192 * 8 + 8192) * 2048 * 2
    logits = 7 * 8192 * 256 * 8          # up to 7 split-K slices of (hi, lo) partial logits
    wsplit = 256 * 3 * 7168 * 2          # W_g as bf16 pieces for the tensor-core router
    refine = 8192 * 16                   # rows listed for exact re-decision
    ec = 8192 * 256 * 12 + 8192 * 8 + 256 * 20   # expert-choice columns and exact rows
    assert h + wsplit + ec < ws < h + wsplit + ec + logits + refine + 2 * 32 * 256 * 4 + 8192
    assert B.moe_workspace_bytes(-1, 1, 1, 1, 1, 0, 0) == 0
    assert B.moe_workspace_bytes(0, 64, 8, 64, 2, 0, 0) >= 256


def test_validation_before_device(L):
    """Bad requests fail with the right code and never reach the (absent) device."""
    vp = C.c_void_p
    fake = vp(4096)   # never dereferenced: validation fails first
    d = B.RouterDesc(16, 64, 600, 2, 0, 1, 0)
    r = L.moe_router_topk(None, C.byref(d), fake, fake, None, None, fake, fake, None, None,
                          fake, 1 << 20, None)
    assert r == B.MOE_ERR_UNSUPPORTED and "E = 600" in B.last_error_detail()
    d = B.RouterDesc(16, 64, 8, 9, 0, 1, 0)
    r = L.moe_router_topk(None, C.byref(d), fake, fake, None, None, fake, fake, None, None,
                          fake, 1 << 20, None)
    assert r == B.MOE_ERR_UNSUPPORTED and "k = 9" in B.last_error_detail()
    d = B.RouterDesc(16, 64, 8, 2, 7, 1, 0)
    r = L.moe_router_topk(None, C.byref(d), fake, fake, None, None, fake, fake, None, None,
                          fake, 1 << 20, None)
    assert r == B.MOE_ERR_INVALID_ARG and "score" in B.last_error_detail()
    d = B.RouterDesc(16, 64, 8, 2, 0, 1, 0)
    r = L.moe_router_topk(None, C.byref(d), vp(4097), fake, None, None, fake, fake, None,
                          None, fake, 1 << 20, None)
    assert r == B.MOE_ERR_INVALID_ARG and "aligned" in B.last_error_detail()
    r = L.moe_router_topk(None, C.byref(d), fake, fake, None, None, fake, fake, None, None,
                          fake, 64, None)
    assert r == B.MOE_ERR_INVALID_ARG and "workspace" in B.last_error_detail()
    r = L.moe_router_topk(None, C.byref(d), fake, fake, None, None, fake, fake, None, None,
                          fake, 1 << 20, None)
    assert r == B.MOE_ERR_INVALID_ARG and "ctx" in B.last_error_detail()
    # group-limited routing shapes
    for G, M, k, code, text in [(3, 1, 2, B.MOE_ERR_UNSUPPORTED, "n_groups = 3"),
                                (64, 1, 2, B.MOE_ERR_UNSUPPORTED, "n_groups = 64"),
                                (4, 3, 4, B.MOE_ERR_INVALID_ARG, "topk_groups = 3"),
                                (4, 5, 5, B.MOE_ERR_INVALID_ARG, "topk_groups = 5"),
                                (8, 1, 2, B.MOE_ERR_INVALID_ARG, "topk_groups = 1"),
                                (-1, 0, 2, B.MOE_ERR_INVALID_ARG, "n_groups = -1")]:
        d = B.RouterDesc(16, 64, 8, k, 0, 1, 0, G, M)
        r = L.moe_router_topk(None, C.byref(d), fake, fake, None, None, fake, fake, None,
                              None, fake, 1 << 20, None)
        assert r == code and text in B.last_error_detail(), (G, M, k, r)
    # a valid group shape passes the shape checks (and stops at the missing context)
    d = B.RouterDesc(16, 64, 8, 4, 1, 1, 0, 4, 2)
    r = L.moe_router_topk(None, C.byref(d), fake, fake, None, None, fake, fake, None, None,
                          fake, 1 << 20, None)
    assert r == B.MOE_ERR_INVALID_ARG and "ctx" in B.last_error_detail()
    # bias update: gamma must be finite; null pointers rejected
    r = L.moe_bias_update(None, 16, 2, 8, fake, float("nan"), fake, None)
    assert r == B.MOE_ERR_INVALID_ARG and "gamma" in B.last_error_detail()
    r = L.moe_bias_update(None, 16, 2, 8, fake, float("inf"), fake, None)
    assert r == B.MOE_ERR_INVALID_ARG and "gamma" in B.last_error_detail()
    r = L.moe_bias_update(None, 16, 2, 8, None, 0.001, fake, None)
    assert r == B.MOE_ERR_INVALID_ARG and "required" in B.last_error_detail()
    r = L.moe_bias_update(None, 16, 2, 8, fake, 0.001, fake, None)
    assert r == B.MOE_ERR_INVALID_ARG and "ctx" in B.last_error_detail()
    # expert choice: E must divide T*k; at most 32768 tokens; no expert groups
    d = B.RouterDesc(10, 64, 4, 1, 0, 0, 0)
    r = L.moe_expert_choice(None, C.byref(d), fake, fake, None, fake, fake, fake, fake, None,
                            fake, 1 << 30, None)
    assert r == B.MOE_ERR_INVALID_ARG and "divide" in B.last_error_detail()
    d = B.RouterDesc(40000, 64, 8, 2, 0, 0, 0)
    r = L.moe_expert_choice(None, C.byref(d), fake, fake, None, fake, fake, fake, fake, None,
                            fake, 1 << 30, None)
    assert r == B.MOE_ERR_UNSUPPORTED and "32768" in B.last_error_detail()
    d = B.RouterDesc(16, 64, 8, 2, 0, 0, 0, 4, 2)
    r = L.moe_expert_choice(None, C.byref(d), fake, fake, None, fake, fake, fake, fake, None,
                            fake, 1 << 30, None)
    assert r == B.MOE_ERR_UNSUPPORTED and "groups" in B.last_error_detail()
    d = B.RouterDesc(16, 64, 8, 2, 0, 0, 0)
    r = L.moe_expert_choice(None, C.byref(d), fake, fake, None, fake, fake, fake, fake, None,
                            fake, 1 << 30, None)
    assert r == B.MOE_ERR_INVALID_ARG and "ctx" in B.last_error_detail()
    r = L.moe_gather_rows(None, 8, 4, 100, 0, fake, fake, 4, fake, fake, None)
    assert r == B.MOE_ERR_UNSUPPORTED and "16 B" in B.last_error_detail()
    r = L.moe_gather_rows(None, 8, 4, 64, 0, fake, fake, 4, fake, fake, None)
    assert r == B.MOE_ERR_INVALID_ARG and "ctx" in B.last_error_detail()
    # FP8 weights: odd column counts, fp32 activations
    r = L.moe_quantize_fp8(None, 4, 63, 0, fake, fake, fake, None)
    assert r == B.MOE_ERR_INVALID_ARG and "cols" in B.last_error_detail()
    e8 = B.ExpertDesc(16, 128, 8, 128, 2, B.MOE_DTYPE_F32, 0)
    r = L.moe_grouped_swiglu_fp8(None, C.byref(e8), *([fake] * 18), 1 << 30, None)
    assert r == B.MOE_ERR_UNSUPPORTED and "bf16" in B.last_error_detail()
    # dispatch: X without Xperm
    r = L.moe_dispatch(None, 16, 2, 8, 64, 0, -1, fake, fake, fake, fake, fake, fake, None,
                       fake, 1 << 20, None)
    assert r == B.MOE_ERR_INVALID_ARG and "together" in B.last_error_detail()
    # expert stage: H not a multiple of 64 for bf16
    e = B.ExpertDesc(16, 96, 8, 128, 2, 0, 0)
    args = [fake] * 12
    r = L.moe_grouped_swiglu(None, C.byref(e), *args, 1 << 30, None)
    assert r == B.MOE_ERR_UNSUPPORTED and "64" in B.last_error_detail()
    e = B.ExpertDesc(16, 128, 8, 128, 2, 0, 1)
    args = [fake, fake, fake, fake, fake, fake, None, None, None, fake, None, fake]
    r = L.moe_grouped_swiglu(None, C.byref(e), *args, 1 << 30, None)
    assert r == B.MOE_ERR_INVALID_ARG and "shared" in B.last_error_detail()
    # combine: H not a multiple of 4
    r = L.moe_combine(None, 4, 2, 6, fake, None, fake, fake, fake, None, None)
    assert r == B.MOE_ERR_UNSUPPORTED
    # stats: missing outputs
    r = L.moe_balance_stats(None, 4, 1, 4, fake, None, fake, 0.01, None, fake, fake, None)
    assert r == B.MOE_ERR_INVALID_ARG


def test_test_hook_validation(L):
    assert L.moe_ctx_set_test_hook(None, 1, 10) == B.MOE_ERR_INVALID_ARG
    assert L.moe_ctx_set_tracing(None, 1) == B.MOE_ERR_INVALID_ARG


def test_capacity_huge_factor_exact(L):
    # factors of 2^52 and above (an integer mantissa shifted left) still evaluate exactly
    assert B.moe_capacity(2.0 ** 52, 1, 1, 2 ** 30) == 2 ** 22
    assert B.moe_capacity(2.0 ** 60, 1, 1, 2 ** 30 + 1) == -(-(2 ** 60) // (2 ** 30 + 1))
    assert B.moe_capacity(3.0 * 2.0 ** 55, 5, 1, 2 ** 31 - 1) == \
        -(-(15 * 2 ** 55) // (2 ** 31 - 1))


C_CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "moe.h"

int main(void) {
  /* host-only calls: no device is touched */
  if (moe_version() != 10400) return 1;
  if (strcmp(moe_status_string(MOE_ERR_TIMEOUT), "device wait timed out") != 0) return 2;
  if (moe_capacity(1.0, 6, 2, 4) != 3 || moe_capacity(2.0, 6, 2, 4) != 6) return 3;
  if (moe_capacity(-1.0, 6, 2, 4) != MOE_ERR_INVALID_ARG) return 4;
  if (strlen(moe_last_error_detail()) == 0) return 5;
  if (moe_workspace_bytes(64, 128, 8, 256, 2, MOE_DTYPE_F32, 0) == 0) return 6;
  if (strcmp(moe_kernel_name(MOE_K_EXPERT_GATE_UP), "expert_gate_up") != 0) return 7;
  /* argument checks run before any device work */
  moe_router_desc d;
  memset(&d, 0, sizeof d);
  d.T = 4; d.H = 64; d.E = 8; d.k = 9;
  if (moe_router_topk(NULL, &d, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0,
                      NULL) != MOE_ERR_UNSUPPORTED) return 8;
  printf("ok %d\n", moe_capacity(1.25, 16384, 1, 64));
  return 0;
}
"""


def test_header_is_plain_c_and_links(L, tmp_path):
    """include/moe.h compiles as C99 with warnings as errors, and a C program linked
    against libmoe.so calls its host-only entry points."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(B.LIB_PATH)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                        "-L", libdir, "-lmoe", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stderr)
    assert r.stdout.strip() == "ok 320"


def test_binding_refuses_host_and_strided_tensors(L):
    """A host tensor or a strided view never reaches the library as a device pointer."""
    import torch

    class _Ctx:
        handle = None
    O = torch.zeros(8, 4)
    ros = torch.zeros(4, dtype=torch.int32)
    gate = torch.ones(4, 1)
    with pytest.raises(TypeError, match="CUDA tensor"):
        B.moe_combine(_Ctx(), O, ros, gate, torch.zeros(4, 4))
    with pytest.raises(TypeError, match="CUDA tensor"):
        B.moe_bias_update(_Ctx(), 4, 1, ros, 0.001, torch.zeros(4))
    if torch.cuda.is_available():
        strided = torch.zeros(4, 8, device="cuda")[:, ::2]
        with pytest.raises(ValueError, match="contiguous"):
            B.moe_combine(_Ctx(), O.cuda(), ros.cuda(), gate.cuda(), strided)
    assert B._p(None) is None


def test_binding_checks_dtypes_and_sizes(L):
    """The library sizes every buffer from the shapes passed beside the pointers, so the
    binding refuses buffers of the wrong element type or too few elements first."""
    import torch

    class _Ctx:
        handle = None
    T, H, E, I, k = 4, 64, 2, 64, 1
    X = torch.zeros(T, H)                                   # fp32 activations
    W = torch.zeros(E, I, H, dtype=torch.bfloat16)          # ... with bf16 weights
    Wd = torch.zeros(E, H, I, dtype=torch.bfloat16)
    O = torch.zeros(T * k, H)
    off = torch.zeros(E + 1, dtype=torch.int32)
    ws = torch.zeros(256, dtype=torch.uint8)
    with pytest.raises(TypeError, match="W_gate"):
        B.moe_grouped_swiglu(_Ctx(), X, X.clone(), off, W, W, Wd, O, ws, k)
    with pytest.raises(ValueError, match="O: 128 elements"):
        B.moe_grouped_swiglu(_Ctx(), X, X.clone(), off, W.float(), W.float(), Wd.float(),
                             O[:2], ws, k)
    idx = torch.zeros(T, k, dtype=torch.int64)              # int64 routing indices
    cnt = torch.zeros(E, dtype=torch.int32)
    with pytest.raises(TypeError, match="topk_idx"):
        B.moe_dispatch(_Ctx(), idx, E, -1, cnt, off, cnt, cnt, ws, H=H)
    with pytest.raises(TypeError, match="prob_colsum"):
        B.moe_balance_stats(_Ctx(), T, k, cnt, torch.zeros(E), 0.01, torch.zeros(E),
                            torch.zeros(E), torch.zeros(4))

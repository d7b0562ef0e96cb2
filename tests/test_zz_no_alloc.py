"""The allocation-free gated-RMSNorm backward, gdn_gated_rmsnorm_bwd_noalloc.

Some callers cannot give the library a workspace: a serving runtime that has
handed all device memory to its own pool and forbids new device allocations
once it is running, a plugin that holds no allocator, or a hot loop that must
not call cudaMalloc/cudaFree (cudaFree synchronises the whole device).  For
them this entry point keeps its scratch -- the per-CTA partial sums of the
norm-weight gradient -- in an array built into the library.  These tests call
it through the C ABI and hold it to what the workspace-taking entry point,
gdn_gated_rmsnorm_bwd, returns for the same inputs, on two calls in a row (the
second after the first has left its partials in the shared array).

This file is named to be collected last.
"""
import ctypes
import os
import re

import pytest
import torch

import oracle
from gated_deltanet_layer_causal_gb300 import _abi
from gdn_testutil import Checker, f64

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "gdn.h")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _both(T, H, dtype, seed):
    """Run the workspace entry point and the allocation-free one on the same inputs."""
    g = torch.Generator().manual_seed(seed)
    o, z, dy = (torch.randn(T, H, 128, generator=g).to(dtype) for _ in range(3))
    w = torch.randn(128, generator=g) * 0.02
    host = (o, z, w, dy)
    o, z, dy, w = o.cuda(), z.cuda(), dy.cuda(), w.cuda()
    d = _abi.dims(1, T, 1, H, dtype == torch.bfloat16)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    n = ctypes.c_size_t(0)
    _abi.call("gdn_workspace_size", ctypes.byref(d), None, _abi.GDN_WS_NORM_BWD,
              ctypes.byref(n))
    ws = torch.empty(max(n.value, 16), dtype=torch.uint8, device="cuda")
    ref = (torch.empty_like(o), torch.empty_like(z), torch.empty_like(w))
    _abi.call("gdn_gated_rmsnorm_bwd", ctypes.byref(d), _ptr(o), _ptr(z), _ptr(w), _ptr(dy),
              *map(_ptr, ref), _ptr(ws), ws.numel(), stream)
    out = (torch.full_like(o, float("nan")), torch.full_like(z, float("nan")),
           torch.full_like(w, float("nan")))
    _abi.call("gdn_gated_rmsnorm_bwd_noalloc", ctypes.byref(d), _ptr(o), _ptr(z), _ptr(w),
              _ptr(dy), *map(_ptr, out), stream)
    torch.cuda.synchronize()
    return out, ref, host


def _check(T, H, dtype, seed, tag):
    """The allocation-free result against the workspace entry point's and against
    the fp64 oracle's gated-norm backward."""
    out, ref, (o, z, w, dy) = _both(T, H, dtype, seed)
    rdo, rdz, rdw = oracle.gated_rmsnorm_bwd(f64(o), f64(z), f64(w), f64(dy), 1e-6)
    c = Checker(tag)
    for name, a, b, r in zip(("do", "dz", "dnorm_w"), out, ref, (rdo, rdz, rdw)):
        c.add(f"{name} vs workspace entry point", f64(a), f64(b), blocks=name != "dnorm_w")
        c.add(f"{name} vs oracle", f64(a), r, blocks=name != "dnorm_w")
    c.check()


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    # first call: 700 tokens x 5 heads (55 partial rows) in bf16
    _check(700, 5, torch.bfloat16, 1, "first call")
    # second call, smaller (16 partial rows) and fp32: it must not pick up the
    # first call's leftovers in the shared scratch
    _check(333, 3, torch.float32, 2, "second call")


@pytest.mark.gpu
def test_noalloc_at_its_row_limit():
    """Exactly GDN_NOALLOC_NORM_BWD_MAX_ROWS rows: every partial row of the array
    in use (131072 tokens x 4 heads), then a small call after it."""
    rows = _abi.GDN_NOALLOC_NORM_BWD_MAX_ROWS
    _check(rows // 4, 4, torch.bfloat16, 3, "at the limit")
    _check(100, 2, torch.bfloat16, 4, "after the limit case")


def test_noalloc_limit_is_the_headers():
    """The binding's limit is the one the header states (the library checks its
    array's capacity against the same macro at compile time)."""
    m = re.search(r"#define\s+GDN_NOALLOC_NORM_BWD_MAX_ROWS\s+(\d+)", open(HEADER).read())
    assert m and int(m.group(1)) == _abi.GDN_NOALLOC_NORM_BWD_MAX_ROWS


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """Over GDN_NOALLOC_NORM_BWD_MAX_ROWS rows it returns GDN_ERR_WORKSPACE
    before touching the GPU (so this runs without one)."""
    lib = _abi.load()
    P = ctypes.c_void_p(16)   # aligned placeholders: nothing is dereferenced
    rows = _abi.GDN_NOALLOC_NORM_BWD_MAX_ROWS
    for T, H in ((rows // 4 + 1, 4), (rows + 1, 1), (rows // 2, 3)):
        too_big = _abi.dims(1, T, 1, H, True)
        st = lib.gdn_gated_rmsnorm_bwd_noalloc(ctypes.byref(too_big), P, P, P, P, P, P, P, None)
        assert st == _abi.GDN_ERR_WORKSPACE, (T, H)
    assert lib.gdn_status_string(st).decode() == "GDN_ERR_WORKSPACE"

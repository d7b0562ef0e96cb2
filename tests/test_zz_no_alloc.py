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

import pytest
import torch

from gated_deltanet_layer_causal_gb300 import _abi
from gdn_testutil import TOL, f64, rel


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _both(T, H, dtype, seed):
    """Run the workspace entry point and the allocation-free one on the same inputs."""
    g = torch.Generator().manual_seed(seed)
    o, z, dy = (torch.randn(T, H, 128, generator=g).to(dtype).cuda() for _ in range(3))
    w = (torch.randn(128, generator=g) * 0.02).cuda()
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
    return out, ref


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    # first call: 700 tokens x 5 heads (55 partial rows) in bf16
    out, ref = _both(700, 5, torch.bfloat16, seed=1)
    for name, a, b in zip(("do", "dz", "dnorm_w"), out, ref):
        assert rel(f64(a), f64(b)) <= TOL, name
    # second call, smaller (16 partial rows) and fp32: it must not pick up the
    # first call's leftovers in the shared scratch
    out, ref = _both(333, 3, torch.float32, seed=2)
    for name, a, b in zip(("do", "dz", "dnorm_w"), out, ref):
        assert rel(f64(a), f64(b)) <= TOL, name


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """Over GDN_NOALLOC_NORM_BWD_MAX_ROWS rows it returns GDN_ERR_WORKSPACE
    before touching the GPU (so this runs without one)."""
    lib = _abi.load()
    P = ctypes.c_void_p(16)   # aligned placeholders: nothing is dereferenced
    rows = _abi.GDN_NOALLOC_NORM_BWD_MAX_ROWS
    ok = _abi.dims(1, rows // 4, 1, 4, True)
    too_big = _abi.dims(1, rows // 4 + 1, 1, 4, True)
    st = lib.gdn_gated_rmsnorm_bwd_noalloc(ctypes.byref(too_big), P, P, P, P, P, P, P, None)
    assert st == _abi.GDN_ERR_WORKSPACE
    assert lib.gdn_status_string(st).decode() == "GDN_ERR_WORKSPACE"
    # at the limit the size check passes (validated up to the launch; not launched here)
    assert ok.total_tokens * ok.h_v == rows

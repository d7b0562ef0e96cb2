"""Torch-facing binding of the GDN C ABI.

Each function here allocates its outputs (and the workspaces the C ABI asks
for) as torch tensors on the input's device, then calls the matching
``gdn_*`` entry point on torch's current stream.  Every step of the method runs
in the CUDA library; this module only moves pointers.
"""
from __future__ import annotations

import ctypes

import torch

from . import _abi

_IO = (torch.float32, torch.bfloat16)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _cu_host(cu_seqlens, cu_host):
    if cu_host is None:
        cu_host = cu_seqlens.to("cpu")
    cu_host = cu_host.to(torch.int32).contiguous()
    return cu_host, ctypes.c_void_p(cu_host.data_ptr())


def _check(t, name, dtype=None, device=None):
    if t is None:
        return
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}")


def _dims(x_or_T, N, h_k, h_v, io_dtype, l2_eps=1e-6, norm_eps=1e-6, qkv_tf32=False,
          gate="silu", layout="flat"):
    if io_dtype not in _IO:
        raise ValueError(f"io dtype must be fp32 or bf16, got {io_dtype}")
    return _abi.dims(N, x_or_T, h_k, h_v, io_dtype == torch.bfloat16, l2_eps, norm_eps,
                     qkv_tf32=qkv_tf32, gate=gate, layout=layout)


def workspace_size(kind, T, N, h_k, h_v, cu_host, io_dtype=torch.bfloat16) -> int:
    d = _dims(T, N, h_k, h_v, io_dtype)
    n = ctypes.c_size_t(0)
    cu = cu_host.to(torch.int32).contiguous() if cu_host is not None else None
    _abi.call("gdn_workspace_size", ctypes.byref(d), _ptr(cu), kind, ctypes.byref(n))
    return int(n.value)


def _workspace(kind, T, N, h_k, h_v, cu_host, io_dtype, device):
    n = workspace_size(kind, T, N, h_k, h_v, cu_host, io_dtype)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ conv
def conv1d_silu(x, conv_w, cu_seqlens, h_k, h_v, conv_state=None, output_conv_state=False,
                cu_host=None, l2_eps=1e-6, qkv_tf32=False, layout="flat"):
    """Causal conv1d + SiLU + L2(q, k) -> (qkv fp32 [T, C], conv_state_out or None).

    qkv_tf32: round qkv to nearest tf32 (for chunk_fwd / chunk_bwd called with
    qkv_tf32=True, which then skip their own rounding of the q / k / v tiles).
    layout: "flat" or "group" (group-major) channel order of x, conv_w and the
    conv states; qkv is always flat."""
    T, C = x.shape
    N = cu_seqlens.numel() - 1
    _check(x, "x", device=x.device)
    _check(conv_w, "conv_w", torch.float32, x.device)
    _check(conv_state, "conv_state", x.dtype, x.device)
    cu_host, cup = _cu_host(cu_seqlens, cu_host)
    d = _dims(T, N, h_k, h_v, x.dtype, l2_eps, qkv_tf32=qkv_tf32, layout=layout)
    qkv = torch.empty(T, C, dtype=torch.float32, device=x.device)
    cs_out = torch.empty(N, C, 3, dtype=x.dtype, device=x.device) if output_conv_state else None
    _abi.call("gdn_conv1d_silu", ctypes.byref(d), _ptr(cu_seqlens), cup, _ptr(x), _ptr(conv_w),
              _ptr(conv_state), _ptr(qkv), _ptr(cs_out), _stream())
    return qkv, cs_out


def conv1d_silu_bwd(x, conv_w, cu_seqlens, h_k, h_v, dqkv, conv_state=None,
                    want_dconv_state=False, cu_host=None, l2_eps=1e-6, dconv_state_out=None,
                    layout="flat"):
    """-> (dx [T, C] io dtype, dconv_w [C, 4] fp32, dconv_state fp32 or None).

    dconv_state_out: gradient of the forward's conv_state_out [N, C, 3] fp32
    (e.g. the next segment's dconv_state), added where those inputs came from."""
    T, C = x.shape
    N = cu_seqlens.numel() - 1
    _check(dqkv, "dqkv", torch.float32, x.device)
    _check(dconv_state_out, "dconv_state_out", torch.float32, x.device)
    cu_host, cup = _cu_host(cu_seqlens, cu_host)
    d = _dims(T, N, h_k, h_v, x.dtype, l2_eps, layout=layout)
    dx = torch.empty_like(x)
    dw = torch.empty_like(conv_w)
    dcs = (torch.empty(N, C, 3, dtype=torch.float32, device=x.device)
           if want_dconv_state and conv_state is not None else None)
    ws = _workspace(_abi.GDN_WS_CONV_BWD, T, N, h_k, h_v, cu_host, x.dtype, x.device)
    _abi.call("gdn_conv1d_silu_bwd", ctypes.byref(d), _ptr(cu_seqlens), cup, _ptr(x),
              _ptr(conv_w), _ptr(conv_state), _ptr(dqkv), _ptr(dconv_state_out), _ptr(dx),
              _ptr(dw), _ptr(dcs), _ptr(ws), ws.numel(), _stream())
    return dx, dw, dcs


# ------------------------------------------------------------------ chunked rule
def chunk_fwd(qkv, a, b, A_log, dt_bias, cu_seqlens, h_k, h_v, initial_state=None, z=None,
              norm_w=None, output_final_state=False, return_o=False, cu_host=None,
              norm_eps=1e-6, fwd_ws=None, qkv_tf32=False, gate="silu"):
    """Gated delta rule (+ fused gated norm when z is given, output gate "silu" or
    "sigmoid").  qkv_tf32: qkv holds tf32 values (conv1d_silu(..., qkv_tf32=True)).

    Returns dict(y, o, final_state, fwd_ws); fwd_ws must be kept for chunk_bwd."""
    T = qkv.shape[0]
    N = cu_seqlens.numel() - 1
    io = a.dtype
    dev = qkv.device
    _check(qkv, "qkv", torch.float32, dev)
    for t, n in ((a, "a"), (b, "b"), (z, "z")):
        _check(t, n, io, dev)
    for t, n in ((A_log, "A_log"), (dt_bias, "dt_bias"), (norm_w, "norm_w"),
                 (initial_state, "initial_state")):
        _check(t, n, torch.float32, dev)
    cu_host, cup = _cu_host(cu_seqlens, cu_host)
    d = _dims(T, N, h_k, h_v, io, norm_eps=norm_eps, qkv_tf32=qkv_tf32, gate=gate)
    if fwd_ws is None:
        fwd_ws = _workspace(_abi.GDN_WS_FWD, T, N, h_k, h_v, cu_host, io, dev)
    y = torch.empty(T, h_v, 128, dtype=io, device=dev) if z is not None else None
    o = torch.empty(T, h_v, 128, dtype=io, device=dev) if (return_o or z is None) else None
    fs = torch.empty(N, h_v, 128, 128, dtype=torch.float32, device=dev) \
        if output_final_state else None
    _abi.call("gdn_chunk_fwd", ctypes.byref(d), _ptr(cu_seqlens), cup, _ptr(qkv), _ptr(a), _ptr(b),
              _ptr(A_log), _ptr(dt_bias), _ptr(initial_state), _ptr(z), _ptr(norm_w), _ptr(o),
              _ptr(y), _ptr(fs), _ptr(fwd_ws), fwd_ws.numel(), _stream())
    return dict(y=y, o=o, final_state=fs, fwd_ws=fwd_ws)


def chunk_bwd(qkv, a, b, A_log, dt_bias, cu_seqlens, h_k, h_v, fwd_ws, dy, initial_state=None,
              z=None, norm_w=None, dfinal_state=None, want_dinitial_state=False, cu_host=None,
              norm_eps=1e-6, bwd_ws=None, qkv_tf32=False, gate="silu"):
    """Backward of chunk_fwd -> dict(dqkv, da, db, dA_log, ddt_bias, dz, dnorm_w, dinitial_state)."""
    T = qkv.shape[0]
    N = cu_seqlens.numel() - 1
    io = a.dtype
    dev = qkv.device
    _check(dy, "dy", io, dev)
    _check(dfinal_state, "dfinal_state", torch.float32, dev)
    cu_host, cup = _cu_host(cu_seqlens, cu_host)
    d = _dims(T, N, h_k, h_v, io, norm_eps=norm_eps, qkv_tf32=qkv_tf32, gate=gate)
    if bwd_ws is None:
        bwd_ws = _workspace(_abi.GDN_WS_BWD, T, N, h_k, h_v, cu_host, io, dev)
    dqkv = torch.empty_like(qkv)
    da = torch.empty_like(a)
    db = torch.empty_like(b)
    dA = torch.empty_like(A_log)
    ddt = torch.empty_like(dt_bias)
    dz = torch.empty_like(z) if z is not None else None
    dnw = torch.empty_like(norm_w) if z is not None else None
    dS0 = (torch.empty(N, h_v, 128, 128, dtype=torch.float32, device=dev)
           if want_dinitial_state else None)
    _abi.call("gdn_chunk_bwd", ctypes.byref(d), _ptr(cu_seqlens), cup, _ptr(qkv), _ptr(a), _ptr(b),
              _ptr(A_log), _ptr(dt_bias), _ptr(initial_state), _ptr(z), _ptr(norm_w), _ptr(fwd_ws),
              fwd_ws.numel(), _ptr(dy), _ptr(dfinal_state), _ptr(dqkv), _ptr(da), _ptr(db),
              _ptr(dA), _ptr(ddt), _ptr(dz), _ptr(dnw), _ptr(dS0), _ptr(bwd_ws), bwd_ws.numel(),
              _stream())
    return dict(dqkv=dqkv, da=da, db=db, dA_log=dA, ddt_bias=ddt, dz=dz, dnorm_w=dnw,
                dinitial_state=dS0)


def read_status(ws) -> int:
    """Device status word of a workspace (0 = OK); clears it."""
    code = ctypes.c_int32(0)
    _abi.call("gdn_read_status", _ptr(ws), ctypes.byref(code), _stream())
    return int(code.value)


# ------------------------------------------------------------------ norm, decode
def gated_rmsnorm(o, z, norm_w, eps=1e-6, return_rstd=False, gate="silu"):
    T, H, D = o.shape
    d = _dims(T, 1, 1, H, o.dtype, norm_eps=eps, gate=gate)
    y = torch.empty_like(o)
    rstd = torch.empty(T, H, dtype=torch.float32, device=o.device) if return_rstd else None
    _abi.call("gdn_gated_rmsnorm", ctypes.byref(d), _ptr(o), _ptr(z), _ptr(norm_w), _ptr(y),
              _ptr(rstd), _stream())
    return (y, rstd) if return_rstd else y


def gated_rmsnorm_bwd(o, z, norm_w, dy, eps=1e-6, gate="silu"):
    T, H, D = o.shape
    d = _dims(T, 1, 1, H, o.dtype, norm_eps=eps, gate=gate)
    d_o, dz, dw = torch.empty_like(o), torch.empty_like(z), torch.empty_like(norm_w)
    ws = _workspace(_abi.GDN_WS_NORM_BWD, T, 1, 1, H, None, o.dtype, o.device)
    _abi.call("gdn_gated_rmsnorm_bwd", ctypes.byref(d), _ptr(o), _ptr(z), _ptr(norm_w), _ptr(dy),
              _ptr(d_o), _ptr(dz), _ptr(dw), _ptr(ws), ws.numel(), _stream())
    return d_o, dz, dw


def recurrent_step(x_t, conv_w, conv_state, a_t, b_t, A_log, dt_bias, z_t, norm_w, state, h_k,
                   h_v, return_o=False, l2_eps=1e-6, norm_eps=1e-6, gate="silu", layout="flat"):
    """One decode step; updates conv_state and state in place; returns y_t (and o_t)."""
    N = x_t.shape[0]
    for t, n in ((conv_state, "conv_state"), (state, "state")):
        _check(t, n, None, x_t.device)
    d = _dims(N, N, h_k, h_v, x_t.dtype, l2_eps, norm_eps, gate=gate, layout=layout)
    y = torch.empty(N, h_v, 128, dtype=x_t.dtype, device=x_t.device)
    o = torch.empty_like(y) if return_o else None
    _abi.call("gdn_recurrent_step", ctypes.byref(d), _ptr(x_t), _ptr(conv_w), _ptr(conv_state),
              _ptr(a_t), _ptr(b_t), _ptr(A_log), _ptr(dt_bias), _ptr(z_t), _ptr(norm_w),
              _ptr(state), _ptr(o), _ptr(y), _stream())
    return (y, o) if return_o else y


# ------------------------------------------------------------------ whole core
class GDNCore(torch.autograd.Function):
    """conv1d+SiLU -> L2 -> gated delta rule -> gated RMSNorm, with backward.

    apply(x, conv_w, a, b, A_log, dt_bias, z, norm_w, cu_seqlens, h_k, h_v,
          initial_state, output_final_state, cu_host, conv_state,
          output_conv_state, gate, layout)
    returns (y, final_state or None, conv_state_out or None).  Mirrors the
    fla-style chunk call with cu_seqlens / initial_state / output_final_state
    keyword arguments; conv_state [N, C, 3] (the inputs before each sequence
    start) and conv_state_out resume a sequence across calls, and gradients
    flow through all four, so a sequence split across calls trains like one.
    gate: "silu" | "sigmoid"; layout: "flat" | "group" (channel order of x)."""

    @staticmethod
    def forward(ctx, x, conv_w, a, b, A_log, dt_bias, z, norm_w, cu_seqlens, h_k, h_v,
                initial_state=None, output_final_state=False, cu_host=None, conv_state=None,
                output_conv_state=False, gate="silu", layout="flat"):
        cu_host = cu_seqlens.to("cpu") if cu_host is None else cu_host
        qkv, cs_out = conv1d_silu(x, conv_w, cu_seqlens, h_k, h_v, conv_state=conv_state,
                                  output_conv_state=output_conv_state, cu_host=cu_host,
                                  layout=layout)
        r = chunk_fwd(qkv, a, b, A_log, dt_bias, cu_seqlens, h_k, h_v, initial_state, z, norm_w,
                      output_final_state, cu_host=cu_host, gate=gate)
        ctx.save_for_backward(x, conv_w, a, b, A_log, dt_bias, z, norm_w, cu_seqlens, qkv,
                              r["fwd_ws"], initial_state, conv_state)
        ctx.meta = (h_k, h_v, cu_host, gate, layout)
        return r["y"], r["final_state"], cs_out

    @staticmethod
    def backward(ctx, dy, dfs, dcs_out):
        x, conv_w, a, b, A_log, dt_bias, z, norm_w, cu, qkv, fws, s0, cs = ctx.saved_tensors
        h_k, h_v, cu_host, gate, layout = ctx.meta
        g = chunk_bwd(qkv, a, b, A_log, dt_bias, cu, h_k, h_v, fws, dy.contiguous(), s0, z,
                      norm_w, None if dfs is None else dfs.contiguous(),
                      want_dinitial_state=s0 is not None and ctx.needs_input_grad[11],
                      cu_host=cu_host, gate=gate)
        want_dcs = cs is not None and ctx.needs_input_grad[14]
        dcs_in = None if dcs_out is None else dcs_out.float().contiguous()
        dx, dw, dcs = conv1d_silu_bwd(x, conv_w, cu, h_k, h_v, g["dqkv"], conv_state=cs,
                                      want_dconv_state=want_dcs, cu_host=cu_host,
                                      dconv_state_out=dcs_in, layout=layout)
        if dcs is not None:
            dcs = dcs.to(cs.dtype)
        return (dx, dw, g["da"], g["db"], g["dA_log"], g["ddt_bias"], g["dz"], g["dnorm_w"],
                None, None, None, g["dinitial_state"], None, None, dcs, None, None, None)


def gdn_core(x, conv_w, a, b, A_log, dt_bias, z, norm_w, cu_seqlens, h_k, h_v,
             initial_state=None, output_final_state=False, cu_host=None, conv_state=None,
             output_conv_state=False, gate="silu", layout="flat"):
    """Differentiable GDN core; see :class:`GDNCore`.  Returns (y, final_state),
    or (y, final_state, conv_state_out) when output_conv_state is set."""
    y, fs, cs = GDNCore.apply(x, conv_w, a, b, A_log, dt_bias, z, norm_w, cu_seqlens, h_k, h_v,
                              initial_state, output_final_state, cu_host, conv_state,
                              output_conv_state, gate, layout)
    return (y, fs, cs) if output_conv_state else (y, fs)

"""fp64 CPU oracle of the Gated DeltaNet causal core -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never loads it and
shares no code with it.

The arithmetic lives in ``gdn_oracle.c`` (one function per stage, each citing
the page section it follows).  This module compiles that file with the host C
compiler on first use and composes the stages into the layer's forward and
backward:

    x --conv1d+SiLU--> [q | k | v] --L2 (q scaled by d_k^-1/2)--> q^, k^, v
    a, b --gates--> g, beta
    (q^, k^, v, g, beta, S0) --gated delta rule--> o, S_final
    (o, z, w) --zero-centred gated RMSNorm--> y

Channel order of x is the flat [q (H_k*d_k) | k (H_k*d_k) | v (H_v*d_v)] layout
("HF's flat layout" in "[6/8] feat(models): port Qwen3.5 / Qwen3-Next GDN to the
head-sharded layer", section "What").  All arrays are float64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I32 = ctypes.POINTER(ctypes.c_int32)
_U8 = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into _build/libgdn_oracle.so (portable flags only)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    i, i64, d = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    sig = {
        "gdn_ref_num_threads": (i, []),
        "gdn_ref_conv_silu": (None, [i, _I32, i, i, _D, _D, _D, _D, _D, _D]),
        "gdn_ref_conv_silu_bwd": (None, [i, _I32, i, i, _D, _D, _D, _D, _D, _D, _D]),
        "gdn_ref_l2norm": (None, [i64, i, d, d, _D, _D]),
        "gdn_ref_l2norm_bwd": (None, [i64, i, d, d, _D, _D, _D]),
        "gdn_ref_gates": (None, [i64, i, _D, _D, _D, _D, _D, _D]),
        "gdn_ref_gates_bwd": (None, [i64, i, _D, _D, _D, _D, _D, _D, _D, _D, _D, _D]),
        "gdn_ref_delta_rule_fwd": (None, [i, _I32, i, i, i, i, _D, _D, _D, _D, _D, _D, _U8,
                                          _D, _D]),
        "gdn_ref_delta_rule_bwd": (None, [i, _I32, i, i, i, i, _D, _D, _D, _D, _D, _D, _D, _D,
                                          _U8, _D, _D, _D, _D, _D, _D]),
        "gdn_ref_chunked_fwd": (None, [i, _I32, i, i, i, i, i, _D, _D, _D, _D, _D, _D, _D,
                                       _D]),
        "gdn_ref_gated_rmsnorm": (None, [i64, i, d, i, _D, _D, _D, _D, _D]),
        "gdn_ref_gated_rmsnorm_bwd": (None, [i64, i, d, i, _D, _D, _D, _D, _D, _D, _D]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    return int(_load().gdn_ref_num_threads())


def _p(a):
    """Pointer to a C-contiguous float64 array (None -> NULL)."""
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"], (a.dtype, a.flags)
    return a.ctypes.data_as(_D)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _cu(cu):
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    return cu, cu.ctypes.data_as(_I32)


def _mask(heads, hv):
    if heads is None:
        return None, None
    m = np.zeros(hv, dtype=np.uint8)
    m[list(heads)] = 1
    return m, m.ctypes.data_as(_U8)


# --------------------------------------------------------------------------- stages
def conv_silu(x, w, cu, conv_state=None):
    """Causal depthwise conv1d + SiLU with cu_seqlens resets.

    Returns (pre, out, conv_state_out); conv_state_* is [N, C, K-1]."""
    x, w, cs = _f64(x), _f64(w), _f64(conv_state)
    cu, cup = _cu(cu)
    T, C = x.shape
    K = w.shape[1]
    N = len(cu) - 1
    pre = np.empty_like(x)
    out = np.empty_like(x)
    cso = np.empty((N, C, K - 1))
    _load().gdn_ref_conv_silu(N, cup, C, K, _p(x), _p(w), _p(cs), _p(pre), _p(out), _p(cso))
    return pre, out, cso


def conv_silu_bwd(x, w, cu, dout, conv_state=None):
    x, w, cs, dout = _f64(x), _f64(w), _f64(conv_state), _f64(dout)
    cu, cup = _cu(cu)
    T, C = x.shape
    K = w.shape[1]
    N = len(cu) - 1
    dx = np.empty_like(x)
    dw = np.empty_like(w)
    dcs = np.empty((N, C, K - 1)) if cs is not None else None
    _load().gdn_ref_conv_silu_bwd(N, cup, C, K, _p(x), _p(w), _p(cs), _p(dout), _p(dx), _p(dw),
                                  _p(dcs))
    return dx, dw, dcs


def l2norm(x, eps, scale):
    """Row-wise x / sqrt(|x|^2 + eps) * scale over the last axis."""
    x = _f64(x)
    out = np.empty_like(x)
    d = x.shape[-1]
    _load().gdn_ref_l2norm(x.size // d, d, eps, scale, _p(x), _p(out))
    return out


def l2norm_bwd(x, dout, eps, scale):
    x, dout = _f64(x), _f64(dout)
    dx = np.empty_like(x)
    d = x.shape[-1]
    _load().gdn_ref_l2norm_bwd(x.size // d, d, eps, scale, _p(x), _p(dout), _p(dx))
    return dx


def gates(a, b, A_log, dt_bias):
    """g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b); a, b [T, H]."""
    a, b, A_log, dt_bias = _f64(a), _f64(b), _f64(A_log), _f64(dt_bias)
    T, H = a.shape
    g = np.empty_like(a)
    beta = np.empty_like(a)
    _load().gdn_ref_gates(T, H, _p(a), _p(b), _p(A_log), _p(dt_bias), _p(g), _p(beta))
    return g, beta


def gates_bwd(a, b, A_log, dt_bias, dg, dbeta):
    a, b, A_log, dt_bias, dg, dbeta = map(_f64, (a, b, A_log, dt_bias, dg, dbeta))
    T, H = a.shape
    da, db = np.empty_like(a), np.empty_like(a)
    dA, ddt = np.empty(H), np.empty(H)
    _load().gdn_ref_gates_bwd(T, H, _p(a), _p(b), _p(A_log), _p(dt_bias), _p(dg), _p(dbeta),
                              _p(da), _p(db), _p(dA), _p(ddt))
    return da, db, dA, ddt


def delta_rule(qh, kh, v, g, beta, cu, S0=None, heads=None):
    """Token-by-token gated delta rule.

    qh, kh [T, H_k, d_k]; v [T, H_v, d_v]; g, beta [T, H_v]; S0 [N, H_v, d_v, d_k].
    Returns (o [T, H_v, d_v], S_final [N, H_v, d_v, d_k]).  With ``heads`` only
    those v-heads are computed (the others are left zero)."""
    qh, kh, v, g, beta, S0 = map(_f64, (qh, kh, v, g, beta, S0))
    cu, cup = _cu(cu)
    T, hk, dk = kh.shape
    hv, dv = v.shape[1], v.shape[2]
    N = len(cu) - 1
    m, mp = _mask(heads, hv)
    o = np.zeros((T, hv, dv))
    Sf = np.zeros((N, hv, dv, dk))
    _load().gdn_ref_delta_rule_fwd(N, cup, hk, hv, dk, dv, _p(qh), _p(kh), _p(v), _p(g),
                                   _p(beta), _p(S0), mp, _p(o), _p(Sf))
    return o, Sf


def delta_rule_bwd(qh, kh, v, g, beta, cu, do, S0=None, dS_final=None, heads=None):
    """Reverse mode of :func:`delta_rule`.

    Returns dq, dk ([T, H_k, d_k], summed over the v-heads that share each
    k-head), dv [T, H_v, d_v], dg, dbeta [T, H_v] and dS0 [N, H_v, d_v, d_k]."""
    qh, kh, v, g, beta, S0, do, dS_final = map(_f64, (qh, kh, v, g, beta, S0, do, dS_final))
    cu, cup = _cu(cu)
    T, hk, dk = kh.shape
    hv, dv = v.shape[1], v.shape[2]
    N = len(cu) - 1
    m, mp = _mask(heads, hv)
    dq_v = np.zeros((T, hv, dk))
    dk_v = np.zeros((T, hv, dk))
    dvv = np.zeros((T, hv, dv))
    dg = np.zeros((T, hv))
    dbeta = np.zeros((T, hv))
    dS0 = np.zeros((N, hv, dv, dk))
    _load().gdn_ref_delta_rule_bwd(N, cup, hk, hv, dk, dv, _p(qh), _p(kh), _p(v), _p(g),
                                   _p(beta), _p(S0), _p(do), _p(dS_final), mp, _p(dq_v),
                                   _p(dk_v), _p(dvv), _p(dg), _p(dbeta), _p(dS0))
    G = hv // hk
    # grouped-value accumulation: v-heads h = kh*G .. kh*G+G-1 share k-head kh
    dq = dq_v.reshape(T, hk, G, dk).sum(axis=2)
    dkk = dk_v.reshape(T, hk, G, dk).sum(axis=2)
    return dq, dkk, dvv, dg, dbeta, dS0


def chunked_delta_rule(qh, kh, v, g, beta, cu, S0=None, chunk=64):
    """Naive chunked WY form of the same rule (check-only second method)."""
    qh, kh, v, g, beta, S0 = map(_f64, (qh, kh, v, g, beta, S0))
    cu, cup = _cu(cu)
    T, hk, dk = kh.shape
    hv, dv = v.shape[1], v.shape[2]
    N = len(cu) - 1
    o = np.zeros((T, hv, dv))
    Sf = np.zeros((N, hv, dv, dk))
    _load().gdn_ref_chunked_fwd(N, cup, hk, hv, dk, dv, chunk, _p(qh), _p(kh), _p(v), _p(g),
                                _p(beta), _p(S0), _p(o), _p(Sf))
    return o, Sf


GATES = {"silu": 0, "sigmoid": 1}


def gated_rmsnorm(o, z, w, eps, gate="silu"):
    """y = o / sqrt(mean(o^2) + eps) * (1 + w) * gate(z) over the last axis, gate
    silu or sigmoid ("prime-rl #3860", "Summary": output_gate_type)."""
    o, z, w = _f64(o), _f64(z), _f64(w)
    d = o.shape[-1]
    y = np.empty_like(o)
    rstd = np.empty(o.shape[:-1])
    _load().gdn_ref_gated_rmsnorm(o.size // d, d, eps, GATES[gate], _p(o), _p(z), _p(w), _p(y),
                                  _p(rstd))
    return y, rstd


def gated_rmsnorm_bwd(o, z, w, dy, eps, gate="silu"):
    o, z, w, dy = map(_f64, (o, z, w, dy))
    d = o.shape[-1]
    do, dz, dw = np.empty_like(o), np.empty_like(o), np.empty(d)
    _load().gdn_ref_gated_rmsnorm_bwd(o.size // d, d, eps, GATES[gate], _p(o), _p(z), _p(w),
                                      _p(dy), _p(do), _p(dz), _p(dw))
    return do, dz, dw


def conv_state_out_bwd(cu, dcso, dx, dcs=None):
    """Gradient of conv_state_out, which copies each sequence's last K-1 conv
    inputs: the input at position e-(K-1)+m of sequence [s, e) receives
    dcso[n, :, m] -- in dx when it is a token of the sequence, else in dcs, the
    gradient of the conv cache it came from (cache slot (K-1) + (p - s)).
    Adds into dx [T, C] and dcs [N, C, K-1] (nullable) in place."""
    K1 = dcso.shape[2]
    for n in range(len(cu) - 1):
        s, e = int(cu[n]), int(cu[n + 1])
        for m in range(K1):
            p = e - K1 + m
            if p >= s:
                dx[p] += dcso[n, :, m]
            elif dcs is not None:
                dcs[n, :, K1 + (p - s)] += dcso[n, :, m]


def group_major_order(hk, hv, dk=128, dv=128):
    """Flat channel of each group-major channel: x_group[:, j] = x_flat[:, order[j]].

    Flat x is [q (H_k d_k) | k (H_k d_k) | v (H_v d_v)] ("HF's flat layout");
    group-major puts each k-head group's channels together, [q_kh | k_kh |
    v_{kh G} .. v_{kh G + G - 1}] for kh = 0 .. H_k - 1 ("[6/8] feat(models): port
    Qwen3.5 / Qwen3-Next GDN to the head-sharded layer", "What": q/k/v and the
    conv change layout to group-major)."""
    G = hv // hk
    order = []
    for kh in range(hk):
        order += range(kh * dk, (kh + 1) * dk)
        order += range(hk * dk + kh * dk, hk * dk + (kh + 1) * dk)
        for h in range(kh * G, (kh + 1) * G):
            order += range(2 * hk * dk + h * dv, 2 * hk * dk + (h + 1) * dv)
    return np.array(order)


def _to_flat(a, order, axis):
    """Group-major -> flat along `axis` (None passes through)."""
    if a is None:
        return None
    a = np.asarray(a)
    out = np.empty_like(a)
    idx = [slice(None)] * a.ndim
    idx[axis] = order
    out[tuple(idx)] = a
    return out


def _to_group(a, order, axis):
    if a is None:
        return None
    return np.ascontiguousarray(np.take(a, order, axis=axis))


# --------------------------------------------------------------------------- layer
def _split(xc, hk, hv, dk, dv):
    T = xc.shape[0]
    q = xc[:, : hk * dk].reshape(T, hk, dk)
    k = xc[:, hk * dk: 2 * hk * dk].reshape(T, hk, dk)
    v = xc[:, 2 * hk * dk:].reshape(T, hv, dv)
    return np.ascontiguousarray(q), np.ascontiguousarray(k), np.ascontiguousarray(v)


def forward(x, conv_w, a, b, A_log, dt_bias, z, norm_w, cu, hk, hv, dk=128, dv=128,
            S0=None, conv_state=None, l2_eps=1e-6, norm_eps=1e-6, heads=None, gate="silu",
            layout="flat"):
    """GDN core forward.  Returns a dict with every intermediate.

    x [T, C]; conv_w [C, K]; a, b [T, H_v]; A_log, dt_bias [H_v]; z [T, H_v, d_v];
    norm_w [d_v]; cu int32 [N+1]; S0 [N, H_v, d_v, d_k]; conv_state [N, C, K-1].
    gate: "silu" | "sigmoid"; layout: "flat" | "group" -- the channel order of x,
    conv_w and the conv states (the intermediates pre / xc are always flat)."""
    if layout == "group":
        order = group_major_order(hk, hv, dk, dv)
        f = forward(_to_flat(x, order, 1), _to_flat(conv_w, order, 0), a, b, A_log, dt_bias, z,
                    norm_w, cu, hk, hv, dk, dv, S0, _to_flat(conv_state, order, 1), l2_eps,
                    norm_eps, heads, gate)
        f["conv_state_out"] = _to_group(f["conv_state_out"], order, 1)
        return f
    pre, xc, cso = conv_silu(x, conv_w, cu, conv_state)
    q, k, v = _split(xc, hk, hv, dk, dv)
    qh = l2norm(q, l2_eps, dk ** -0.5)
    kh = l2norm(k, l2_eps, 1.0)
    g, beta = gates(a, b, A_log, dt_bias)
    o, Sf = delta_rule(qh, kh, v, g, beta, cu, S0, heads)
    y, rstd = gated_rmsnorm(o, z, norm_w, norm_eps, gate)
    return dict(pre=pre, xc=xc, qh=qh, kh=kh, v=v, g=g, beta=beta, o=o, y=y, S_final=Sf,
                conv_state_out=cso, rstd=rstd)


def backward(x, conv_w, a, b, A_log, dt_bias, z, norm_w, cu, hk, hv, dy, dk=128, dv=128,
             S0=None, conv_state=None, dS_final=None, l2_eps=1e-6, norm_eps=1e-6, heads=None,
             norm=True, gate="silu", layout="flat", dconv_state_out=None):
    """GDN core backward (reverse mode through :func:`forward`).

    Returns dx, dconv_w, da, db, dA_log, ddt_bias, dz, dnorm_w, dS0, dconv_state
    and the intermediate gradients dq^, dk^, dv, dg, dbeta, do.  With ``heads``
    (whole k-head groups) only those heads' gradients are exact; dnorm_w and the
    channels of other heads are then partial.  ``norm=False``: the core without
    the gated norm -- dy is the gradient of o itself (z and norm_w unused; dz and
    dnorm_w are None).  dconv_state_out: gradient of the conv_state_out output
    [N, C, K-1] (nullable).  layout / gate as in :func:`forward`."""
    if layout == "group":
        order = group_major_order(hk, hv, dk, dv)
        r = backward(_to_flat(x, order, 1), _to_flat(conv_w, order, 0), a, b, A_log, dt_bias, z,
                     norm_w, cu, hk, hv, dy, dk, dv, S0, _to_flat(conv_state, order, 1),
                     dS_final, l2_eps, norm_eps, heads, norm, gate,
                     dconv_state_out=_to_flat(dconv_state_out, order, 1))
        r["dx"] = _to_group(r["dx"], order, 1)
        r["dconv_w"] = _to_group(r["dconv_w"], order, 0)
        r["dconv_state"] = _to_group(r["dconv_state"], order, 1)
        r["fwd"]["conv_state_out"] = _to_group(r["fwd"]["conv_state_out"], order, 1)
        return r
    if not norm:   # the norm stage is computed but receives no gradient
        z = np.zeros((x.shape[0], hv, dv)) if z is None else z
        norm_w = np.zeros(dv) if norm_w is None else norm_w
    f = forward(x, conv_w, a, b, A_log, dt_bias, z, norm_w, cu, hk, hv, dk, dv, S0, conv_state,
                l2_eps, norm_eps, heads, gate)
    if norm:
        do, dz, dnw = gated_rmsnorm_bwd(f["o"], z, norm_w, dy, norm_eps, gate)
    else:
        do, dz, dnw = _f64(dy), None, None
    dqh, dkh, dvv, dg, dbeta, dS0 = delta_rule_bwd(f["qh"], f["kh"], f["v"], f["g"], f["beta"],
                                                   cu, do, S0, dS_final, heads)
    q, k, _ = _split(f["xc"], hk, hv, dk, dv)
    dq = l2norm_bwd(q, dqh, l2_eps, dk ** -0.5)
    dkk = l2norm_bwd(k, dkh, l2_eps, 1.0)
    T = x.shape[0]
    dxc = np.concatenate([dq.reshape(T, -1), dkk.reshape(T, -1), dvv.reshape(T, -1)], axis=1)
    dx, dcw, dcs = conv_silu_bwd(x, conv_w, cu, dxc, conv_state)
    if dconv_state_out is not None:
        conv_state_out_bwd(cu, _f64(dconv_state_out), dx, dcs)
    da, db, dA, ddt = gates_bwd(a, b, A_log, dt_bias, dg, dbeta)
    return dict(dx=dx, dconv_w=dcw, da=da, db=db, dA_log=dA, ddt_bias=ddt, dz=dz, dnorm_w=dnw,
                dS0=dS0, dconv_state=dcs, dqh=dqh, dkh=dkh, dv=dvv, dg=dg, dbeta=dbeta, do=do,
                fwd=f)


def decode_step(x_t, conv_w, conv_state, a_t, b_t, A_log, dt_bias, z_t, norm_w, S, hk, hv,
                dk=128, dv=128, l2_eps=1e-6, norm_eps=1e-6, gate="silu", layout="flat"):
    """One recurrent decode step for a batch of N independent sequences.

    It is the forward of N sequences of length 1 that start from the given
    conv cache [N, C, K-1] and state [N, H_v, d_v, d_k].  Returns (y [N, H_v,
    d_v], o, S_new, conv_state_new)."""
    N = x_t.shape[0]
    cu = np.arange(N + 1, dtype=np.int32)
    f = forward(x_t, conv_w, a_t, b_t, A_log, dt_bias, z_t, norm_w, cu, hk, hv, dk, dv, S,
                conv_state, l2_eps, norm_eps, gate=gate, layout=layout)
    return f["y"], f["o"], f["S_final"], f["conv_state_out"]


# --------------------------------------------------------------------------- whole layer
def layer_backward(hidden, W_qkv, W_z, W_b, W_a, W_out, conv_w, A_log, dt_bias, norm_w, cu, hk,
                   hv, dout, d=128, gate="silu", layout="flat", act=None):
    """The GDN layer around the core: four input projections, the core, one output
    projection (library matmuls in fp64), forward and reverse mode.

    hidden [T, D_h]; W_qkv [C, D_h]; W_z [H_v d, D_h]; W_b, W_a [H_v, D_h];
    W_out [D_h, H_v d]; dout [T, D_h].  act (nullable): the layer's activation
    storage, applied to each projection's output (e.g. rounding to bf16 when the
    layer keeps its activations in bf16).  Returns the output and the gradients
    of hidden and of every weight."""
    hidden, dout = _f64(hidden), _f64(dout)
    W_qkv, W_z, W_b, W_a, W_out = map(_f64, (W_qkv, W_z, W_b, W_a, W_out))
    act = act or (lambda v: v)
    T = hidden.shape[0]
    x = act(hidden @ W_qkv.T)
    z = act(hidden @ W_z.T).reshape(T, hv, d)
    b = act(hidden @ W_b.T)
    a = act(hidden @ W_a.T)
    dy = (dout @ W_out).reshape(T, hv, d)
    r = backward(x, conv_w, a, b, A_log, dt_bias, z, norm_w, cu, hk, hv, dy, d, d, gate=gate,
                 layout=layout)
    y = r["fwd"]["y"].reshape(T, hv * d)
    dz = r["dz"].reshape(T, hv * d)
    return dict(out=y @ W_out.T, dhidden=r["dx"] @ W_qkv + dz @ W_z + r["db"] @ W_b
                + r["da"] @ W_a, dW_qkv=r["dx"].T @ hidden, dW_z=dz.T @ hidden,
                dW_b=r["db"].T @ hidden, dW_a=r["da"].T @ hidden, dW_out=dout.T @ y,
                dconv_w=r["dconv_w"], dA_log=r["dA_log"], ddt_bias=r["ddt_bias"],
                dnorm_w=r["dnorm_w"])

"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
run the fp64 oracle on the same (rounded) inputs, compare norm-wise.

Tolerances: relative error ||x - x_ref||_2 / ||x_ref||_2 of at most 5e-3 for
every output and gradient (bf16, or fp32 for the fp32 workload) and 1e-3 for
the fp32 final state.  Element-wise relative error is not used: rounding an
output to bf16 alone reaches 3.9e-3 per element and is unbounded near zero.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from gated_deltanet_layer_causal_gb300 import core, synth

TOL = 5e-3
TOL_STATE = 1e-3
D = 128


def rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / max(nb, 1e-30))


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def group_channels(w: synth.Workload, kh: int):
    """Conv channels and v-heads of k-head kh: q, k of kh and v of its G v-heads."""
    G = w.h_v // w.h_k
    heads = [kh * G + j for j in range(G)]
    ch = list(range(kh * D, (kh + 1) * D))
    ch += list(range(w.h_k * D + kh * D, w.h_k * D + (kh + 1) * D))
    for h in heads:
        ch += list(range(2 * w.h_k * D + h * D, 2 * w.h_k * D + (h + 1) * D))
    return np.array(ch), heads


def oracle_group(inp: dict, w: synth.Workload, kh: int, backward: bool, S0=None, dS=None,
                 conv_state=None, tokens=None):
    """Oracle on the sub-problem of one k-head group (H_k = 1, H_v = G).

    Heads of different groups never interact, so this is exactly the full
    problem restricted to those channels and heads (dnorm_w aside, which sums
    over all heads)."""
    ch, heads = group_channels(w, kh)
    G = len(heads)
    sl = slice(None) if tokens is None else slice(0, tokens)
    cu = inp["cu_seqlens"].numpy() if tokens is None else np.array([0, tokens], np.int32)
    args = dict(x=synth.to_f64(inp["x"][sl])[:, ch], conv_w=synth.to_f64(inp["conv_w"])[ch],
                a=synth.to_f64(inp["a"][sl])[:, heads], b=synth.to_f64(inp["b"][sl])[:, heads],
                A_log=synth.to_f64(inp["A_log"])[heads],
                dt_bias=synth.to_f64(inp["dt_bias"])[heads],
                z=synth.to_f64(inp["z"][sl])[:, heads], norm_w=synth.to_f64(inp["norm_w"]),
                cu=cu, hk=1, hv=G)
    if S0 is not None:
        args["S0"] = synth.to_f64(S0)[:, heads]
    if conv_state is not None:
        args["conv_state"] = synth.to_f64(conv_state)[:, ch]
    if not backward:
        return oracle.forward(**args), ch, heads
    dSf = None if dS is None else synth.to_f64(dS)[:, heads]
    g = oracle.backward(**args, dy=synth.to_f64(inp["dy"][sl])[:, heads], dS_final=dSf)
    return g, ch, heads


def gpu_run(inp: dict, w: synth.Workload, backward: bool, S0=None, dS=None, conv_state=None,
            dev="cuda", qkv_tf32=True):
    """Whole core through the C ABI: conv -> chunk fwd (fused norm) [-> chunk bwd -> conv bwd].
    qkv_tf32=True is the setting bench.py runs (qkv stored at tf32 precision)."""
    g = lambda k: inp[k].to(dev)
    x, cw, a, b = g("x"), g("conv_w"), g("a"), g("b")
    A_log, dtb, z, nw = g("A_log"), g("dt_bias"), g("z"), g("norm_w")
    cu, cu_host = g("cu_seqlens"), inp["cu_seqlens"]
    s0 = None if S0 is None else S0.to(dev)
    cs = None if conv_state is None else conv_state.to(dev)
    qkv, cs_out = core.conv1d_silu(x, cw, cu, w.h_k, w.h_v, conv_state=cs,
                                   output_conv_state=True, cu_host=cu_host, qkv_tf32=qkv_tf32)
    r = core.chunk_fwd(qkv, a, b, A_log, dtb, cu, w.h_k, w.h_v, s0, z, nw,
                       output_final_state=True, return_o=True, cu_host=cu_host, qkv_tf32=qkv_tf32)
    out = dict(qkv=qkv, y=r["y"], o=r["o"], S=r["final_state"], conv_state=cs_out)
    out["status_fwd"] = core.read_status(r["fwd_ws"])
    if backward:
        dS_d = None if dS is None else dS.to(dev)
        gr = core.chunk_bwd(qkv, a, b, A_log, dtb, cu, w.h_k, w.h_v, r["fwd_ws"], g("dy"), s0, z,
                            nw, dfinal_state=dS_d, want_dinitial_state=s0 is not None,
                            cu_host=cu_host, qkv_tf32=qkv_tf32)
        dx, dw, dcs = core.conv1d_silu_bwd(x, cw, cu, w.h_k, w.h_v, gr["dqkv"], conv_state=cs,
                                           want_dconv_state=cs is not None, cu_host=cu_host)
        out.update(gr)
        out.update(dx=dx, dconv_w=dw, dconv_state=dcs)
    torch.cuda.synchronize()
    return out

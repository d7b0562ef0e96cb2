"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
run the fp64 oracle on the same (rounded) inputs, compare.

Three measures per tensor, each with its bound:
  norm   ||x - x_ref||_2 / ||x_ref||_2 over the whole tensor: <= 5e-3 for every
         output and gradient (bf16, or fp32 for the fp32 workload), <= 1e-3 for
         the fp32 final state (the stated tolerances);
  max    max|x - x_ref| / max|x_ref|: <= 1e-2 (<= 5e-3 for the final state).
         Rounding one bf16 value costs at most 2^-9 ~ 2.0e-3 of it, and the
         tf32 operands of the products (10 fraction bits, ~4.9e-4 per operand)
         add a few times that on the largest elements; 1e-2 is that sum with
         about 2x to spare;
  block  the norm-wise error of every 64-token block of packed rows (all heads
         and channels of the block), the worst block: <= 1e-2.  A fault confined
         to one chunk, one sequence's tail or one head moves a block's error to
         O(1) while it can hide in the whole tensor's norm (one chunk is 1/1024
         of the 64k workload).
Element-wise relative error is not used: rounding an output to bf16 alone
reaches 3.9e-3 per element and is unbounded near zero.

dA_log and ddt_bias are sums over a head's tokens (of dg g and of da).  Where
those terms cancel, the sum is small against the terms and its relative error
grows by the cancellation factor sum|term| / |sum term| whatever the precision
of each term; so their error is measured against sum|term| per head (the scale
a sum's rounding error follows), the same bounds.  Without cancellation (every
term of one sign) this is the plain relative error.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from gated_deltanet_layer_causal_gb300 import core, synth

TOL = 5e-3
TOL_STATE = 1e-3
TOL_MAX = 1e-2
TOL_MAX_STATE = 5e-3
TOL_BLOCK = 1e-2
D = 128


def rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / max(nb, 1e-30))


def max_rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.size == 0:
        return 0.0
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def block_rel(a, b, rows=64) -> float:
    """Worst norm-wise error over blocks of `rows` leading-axis rows (blocks whose
    reference is exactly zero are skipped)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    T = a.shape[0]
    if T == 0:
        return 0.0
    e = ((a - b) ** 2).reshape(T, -1).sum(axis=1)
    r = (b ** 2).reshape(T, -1).sum(axis=1)
    starts = np.arange(0, T, rows)
    eb, rb = np.add.reduceat(e, starts), np.add.reduceat(r, starts)
    keep = rb > 0
    return float(np.sqrt(eb[keep] / rb[keep]).max()) if keep.any() else 0.0


def measures(a, b, blocks=True, scale=None) -> dict:
    """scale (same shape as b, >= |b|): measure the error against it instead of b."""
    if scale is None:
        m = {"norm": rel(a, b), "max": max_rel(a, b)}
    else:
        e = np.asarray(a, np.float64) - np.asarray(b, np.float64)
        sc = np.asarray(scale, np.float64)
        m = {"norm": float(np.linalg.norm(e) / max(np.linalg.norm(sc), 1e-30)),
             "max": float(np.abs(e).max() / max(np.abs(sc).max(), 1e-30))}
    if blocks:
        m["block"] = block_rel(a, b)
    return m


class Checker:
    """Collects the measures of several tensors, prints them, then asserts all
    bounds at once (so one run shows every margin)."""

    def __init__(self, tag=""):
        self.tag = tag
        self.rows = {}

    def add(self, name, a, b, state=False, blocks=True, scale=None):
        self.rows[name] = (measures(a, b, blocks and not state, scale), state)

    def check(self):
        bad = []
        lines = []
        for name, (m, state) in self.rows.items():
            bounds = {"norm": TOL_STATE if state else TOL,
                      "max": TOL_MAX_STATE if state else TOL_MAX, "block": TOL_BLOCK}
            lines.append(f"{name}: " + " ".join(f"{k}={v:.2e}" for k, v in m.items()))
            bad += [f"{name}.{k}={v:.3e}>{bounds[k]:.0e}" for k, v in m.items() if v > bounds[k]]
        print(f"\n{self.tag} " + "; ".join(lines))
        assert not bad, f"{self.tag}: " + ", ".join(bad)
        return self.rows


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
    chi = torch.as_tensor(ch)
    hi = torch.as_tensor(heads)
    # select the group's channels / heads first, then widen (the whole 64k x in
    # fp64 alone would be 5.4 GB)
    args = dict(x=synth.to_f64(inp["x"][sl].index_select(1, chi)),
                conv_w=synth.to_f64(inp["conv_w"])[ch],
                a=synth.to_f64(inp["a"][sl].index_select(1, hi)),
                b=synth.to_f64(inp["b"][sl].index_select(1, hi)),
                A_log=synth.to_f64(inp["A_log"])[heads],
                dt_bias=synth.to_f64(inp["dt_bias"])[heads],
                z=synth.to_f64(inp["z"][sl].index_select(1, hi)),
                norm_w=synth.to_f64(inp["norm_w"]), cu=cu, hk=1, hv=G)
    if S0 is not None:
        args["S0"] = synth.to_f64(S0)[:, heads]
    if conv_state is not None:
        args["conv_state"] = synth.to_f64(conv_state)[:, ch]
    if not backward:
        return oracle.forward(**args), ch, heads
    dSf = None if dS is None else synth.to_f64(dS)[:, heads]
    g = oracle.backward(**args, dy=synth.to_f64(inp["dy"][sl].index_select(1, hi)),
                        dS_final=dSf)
    return g, ch, heads


def gpu_run(inp: dict, w: synth.Workload, backward: bool, S0=None, dS=None, conv_state=None,
            dev="cuda", qkv_tf32=True, norm=True, gate="silu", layout="flat"):
    """Whole core through the C ABI: conv -> chunk fwd (fused norm) [-> chunk bwd -> conv bwd].
    qkv_tf32=True is the setting bench.py runs (qkv stored at tf32 precision).
    norm=False: the chunk entry points get z = NULL (no fused norm; they return o
    and take dy as the gradient of o).  gate / layout: the output gate and the
    channel order of x (inputs are taken as given in that order)."""
    g = lambda k: inp[k].to(dev)
    x, cw, a, b = g("x"), g("conv_w"), g("a"), g("b")
    A_log, dtb, z, nw = g("A_log"), g("dt_bias"), g("z"), g("norm_w")
    if not norm:
        z = nw = None
    cu, cu_host = g("cu_seqlens"), inp["cu_seqlens"]
    s0 = None if S0 is None else S0.to(dev)
    cs = None if conv_state is None else conv_state.to(dev)
    qkv, cs_out = core.conv1d_silu(x, cw, cu, w.h_k, w.h_v, conv_state=cs,
                                   output_conv_state=True, cu_host=cu_host, qkv_tf32=qkv_tf32,
                                   layout=layout)
    r = core.chunk_fwd(qkv, a, b, A_log, dtb, cu, w.h_k, w.h_v, s0, z, nw,
                       output_final_state=True, return_o=True, cu_host=cu_host, qkv_tf32=qkv_tf32,
                       gate=gate)
    out = dict(qkv=qkv, y=r["y"], o=r["o"], S=r["final_state"], conv_state=cs_out)
    out["status_fwd"] = core.read_status(r["fwd_ws"])
    if backward:
        dS_d = None if dS is None else dS.to(dev)
        gr = core.chunk_bwd(qkv, a, b, A_log, dtb, cu, w.h_k, w.h_v, r["fwd_ws"], g("dy"), s0, z,
                            nw, dfinal_state=dS_d, want_dinitial_state=s0 is not None,
                            cu_host=cu_host, qkv_tf32=qkv_tf32, gate=gate)
        dx, dw, dcs = core.conv1d_silu_bwd(x, cw, cu, w.h_k, w.h_v, gr["dqkv"], conv_state=cs,
                                           want_dconv_state=cs is not None, cu_host=cu_host,
                                           layout=layout)
        out.update(gr)
        out.update(dx=dx, dconv_w=dw, dconv_state=dcs)
    torch.cuda.synchronize()
    return out


def full_args(inp, w, S0=None, cs=None):
    """The whole problem's oracle arguments (fp64) from the rounded inputs."""
    d = {k: synth.to_f64(inp[k]) for k in ("x", "conv_w", "a", "b", "A_log", "dt_bias", "z",
                                            "norm_w")}
    d.update(cu=inp["cu_seqlens"].numpy(), hk=w.h_k, hv=w.h_v)
    if S0 is not None:
        d["S0"] = synth.to_f64(S0)
    if cs is not None:
        d["conv_state"] = synth.to_f64(cs)
    return d


_KEEP = ("y", "o", "S_final", "dx", "dconv_w", "dz", "da", "db", "dA_log", "ddt_bias",
         "dnorm_w", "dg", "g")


def token_sum_scales(ref):
    """Per head, sum over tokens of |dg g| (dA_log's terms) and of |da| (ddt_bias's)."""
    g = ref["fwd"]["g"]
    return np.abs(ref["dg"] * g).sum(axis=0), np.abs(ref["da"]).sum(axis=0)


def oracle_groups(inp: dict, w: synth.Workload, groups, backward: bool, workers: int = 4):
    """Yield (kh, ref, ch, heads) for each k-head group, the oracle running on up to
    `workers` groups at once (host threads; the C oracle releases the GIL).  Each
    ref keeps only the tensors the checks compare, so memory stays per group."""
    from concurrent.futures import ThreadPoolExecutor

    def one(kh):
        ref, ch, heads = oracle_group(inp, w, kh, backward)
        if backward:
            fw = ref["fwd"]
            ref = {k: v for k, v in ref.items() if k in _KEEP}
            ref["fwd"] = {k: v for k, v in fw.items() if k in _KEEP}
        else:
            ref = {k: v for k, v in ref.items() if k in _KEEP}
        return ref, ch, heads

    groups = list(groups)
    with ThreadPoolExecutor(max_workers=min(workers, len(groups))) as ex:
        futs = [ex.submit(one, kh) for kh in groups]
        for kh, fu in zip(groups, futs):
            ref, ch, heads = fu.result()
            yield kh, ref, ch, heads


def check_against(out, ref, backward, ch=None, heads=None, tag="", o=True, norm=True):
    """Every output of a gpu_run against the oracle's (``ref`` from oracle.forward or
    oracle.backward), restricted to conv channels ``ch`` and v-heads ``heads`` when
    the oracle ran on one k-head group (the slices are taken on the device)."""
    fw = ref["fwd"] if backward else ref
    if heads is None:
        hsel = f64
    else:
        hsel = lambda t: f64(t[:, list(heads)])
    if ch is None:
        csel = f64
    else:
        idx = torch.as_tensor(np.asarray(ch), device=out["y" if norm else "o"].device)
        csel = lambda t: f64(t.index_select(1, idx))
    c = Checker(tag)
    if norm:
        c.add("y", hsel(out["y"]), fw["y"])
    if o or not norm:
        c.add("o", hsel(out["o"]), fw["o"])
    c.add("S_final", hsel(out["S"]), fw["S_final"], state=True)
    if backward:
        c.add("dx", csel(out["dx"]), ref["dx"])
        c.add("dconv_w", f64(out["dconv_w"]) if ch is None else csel(out["dconv_w"].t()).T,
              ref["dconv_w"], blocks=False)
        if norm:
            c.add("dz", hsel(out["dz"]), ref["dz"])
        c.add("da", hsel(out["da"]), ref["da"])
        c.add("db", hsel(out["db"]), ref["db"])
        hv = f64 if heads is None else (lambda t: f64(t[list(heads)]))
        sA, sdt = token_sum_scales(ref)
        c.add("dA_log", hv(out["dA_log"]), ref["dA_log"], blocks=False, scale=sA)
        c.add("ddt_bias", hv(out["ddt_bias"]), ref["ddt_bias"], blocks=False, scale=sdt)
        if norm and heads is None:   # sums over every head: whole-problem oracle only
            c.add("dnorm_w", f64(out["dnorm_w"]), ref["dnorm_w"], blocks=False)
    return c.check()

"""Model variants and sequence-split chaining on the GPU, against the oracle.

- The sigmoid output gate of the gated norm (prime-rl #3860, "Summary": the
  shared GatedDeltaNet takes output_gate_type, "sigmoid" for Qwen3.8) and the
  group-major q/k/v/conv channel layout ("[6/8] feat(models): port Qwen3.5 /
  Qwen3-Next GDN to the head-sharded layer", "What"): whole core forward +
  backward, the standalone norm and the decode step.
- One sequence split into segments, run as separate calls whose inputs and
  outputs are pointer offsets into one packed buffer (no copies), with the
  state and conv cache handed forward and their gradients (dS, dconv_state)
  handed back: equal to one call, and to the oracle on the whole sequence
  (the context-parallel arithmetic of "[6/8] ...", "Note on CP", on one GPU).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_layer_causal_gb300 import _abi, core, gdn_core, synth
from gdn_testutil import Checker, check_against, f64, full_args, gpu_run

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("gate,layout,lens,hk,hv,io", [
    ("sigmoid", "flat", (200, 71), 2, 4, "bf16"),
    ("silu", "group", (1, 63, 130, 2), 2, 6, "bf16"),
    ("sigmoid", "group", (129,), 3, 3, "fp32"),
])
def test_gate_and_layout_variants(gate, layout, lens, hk, hv, io):
    w = synth.Workload("var", lens, hk, hv, io=io, backward=True, seed=sum(lens) + hk,
                       dt_bias=-4.0)
    inp = synth.make_inputs(w)   # x, conv_w drawn as given: read in `layout` order
    S0 = synth.make_state(w.N, hv, 128, seed=3, scale=0.2)
    cs = synth.make_conv_state(w.N, w.C, 4, seed=4, dtype=w.torch_dtype)
    out = gpu_run(inp, w, backward=True, S0=S0, conv_state=cs, gate=gate, layout=layout)
    assert out["status_fwd"] == 0
    ref = oracle.backward(**full_args(inp, w, S0, cs), dy=synth.to_f64(inp["dy"]), gate=gate,
                          layout=layout)
    np.testing.assert_array_equal(f64(out["conv_state"]), ref["fwd"]["conv_state_out"])
    check_against(out, ref, True, tag=f"{gate} {layout}")
    c = Checker(f"{gate} {layout} state grads")
    c.add("dinitial_state", f64(out["dinitial_state"]), ref["dS0"], blocks=False)
    c.add("dconv_state", f64(out["dconv_state"]), ref["dconv_state"], blocks=False)
    c.check()


@pytest.mark.parametrize("layout", ["flat", "group"])
def test_decode_step_variants(layout):
    w = synth.Workload("dec", (1,) * 17, 2, 6, io="bf16", seed=9, dt_bias=-2.0)
    inp = synth.make_inputs(w, with_grad=False)
    S = synth.make_state(w.N, w.h_v, 128, seed=10, scale=0.1)
    cs = synth.make_conv_state(w.N, w.C, 4, seed=11, dtype=torch.bfloat16)
    Sd, csd = S.cuda(), cs.cuda()
    d = lambda k: inp[k].cuda()
    y, o = core.recurrent_step(d("x"), d("conv_w"), csd, d("a"), d("b"), d("A_log"),
                               d("dt_bias"), d("z"), d("norm_w"), Sd, w.h_k, w.h_v,
                               return_o=True, gate="sigmoid", layout=layout)
    torch.cuda.synchronize()
    f = synth.to_f64
    ry, ro, rS, rcs = oracle.decode_step(f(inp["x"]), f(inp["conv_w"]), f(cs), f(inp["a"]),
                                         f(inp["b"]), f(inp["A_log"]), f(inp["dt_bias"]),
                                         f(inp["z"]), f(inp["norm_w"]), f(S), w.h_k, w.h_v,
                                         gate="sigmoid", layout=layout)
    c = Checker(f"decode sigmoid {layout}")
    c.add("y", f64(y), ry, blocks=False)
    c.add("o", f64(o), ro, blocks=False)
    c.add("S", f64(Sd), rS, state=True)
    c.check()
    np.testing.assert_array_equal(f64(csd), rcs)


def test_standalone_norm_sigmoid_gate():
    g = torch.Generator().manual_seed(5)
    o, z, dy = (torch.randn(300, 4, 128, generator=g).to(torch.bfloat16) for _ in range(3))
    w_ = torch.randn(128, generator=g) * 0.02
    y = core.gated_rmsnorm(o.cuda(), z.cuda(), w_.cuda(), gate="sigmoid")
    d_o, dz, dw = core.gated_rmsnorm_bwd(o.cuda(), z.cuda(), w_.cuda(), dy.cuda(), gate="sigmoid")
    ry, _ = oracle.gated_rmsnorm(f64(o), f64(z), f64(w_), 1e-6, "sigmoid")
    rdo, rdz, rdw = oracle.gated_rmsnorm_bwd(f64(o), f64(z), f64(w_), f64(dy), 1e-6, "sigmoid")
    c = Checker("standalone sigmoid")
    c.add("y", f64(y), ry)
    c.add("do", f64(d_o), rdo)
    c.add("dz", f64(dz), rdz)
    c.add("dnorm_w", f64(dw), rdw, blocks=False)
    c.check()


# ------------------------------------------------------------------ segment chaining
def _P(t, row=0):
    """Device address of row `row` of a contiguous tensor: a segment's view into
    the packed buffer is just this pointer."""
    return ctypes.c_void_p(t.data_ptr() + row * (t.numel() // t.shape[0]) * t.element_size())


def _segments_through_the_abi(inp, w, cuts, layout):
    """Run the sequence as len(cuts)+1 calls on pointer offsets into packed
    buffers: forward in order (state and conv cache handed on), backward in
    reverse (dS and dconv_state handed back).  Returns the packed results."""
    dev = "cuda"
    T, C, H = w.T, w.C, w.h_v
    io = w.torch_dtype
    t = {k: v.to(dev) for k, v in inp.items()}
    qkv, dqkv = (torch.empty(T, C, device=dev) for _ in range(2))
    y, dz, dx = torch.empty(T, H, 128, dtype=io, device=dev), \
        torch.empty(T, H, 128, dtype=io, device=dev), torch.empty(T, C, dtype=io, device=dev)
    da, db = (torch.empty(T, H, dtype=io, device=dev) for _ in range(2))
    bounds = [0, *cuts, T]
    segs = list(zip(bounds[:-1], bounds[1:]))
    n = len(segs)
    S = [torch.empty(1, H, 128, 128, device=dev) for _ in range(n)]       # final states
    CS = [torch.empty(1, C, 3, dtype=io, device=dev) for _ in range(n)]   # conv caches out
    st = lambda: ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P0 = lambda x: None if x is None else ctypes.c_void_p(x.data_ptr())
    keep = []
    ws_f = []
    for i, (s0, s1) in enumerate(segs):
        L = s1 - s0
        d = _abi.dims(1, L, w.h_k, w.h_v, io == torch.bfloat16, qkv_tf32=True, layout=layout)
        cu_h = torch.tensor([0, L], dtype=torch.int32)
        cu_d = cu_h.to(dev)
        keep += [cu_h, cu_d]
        sz = ctypes.c_size_t(0)
        _abi.call("gdn_workspace_size", ctypes.byref(d), P0(cu_h), _abi.GDN_WS_FWD,
                  ctypes.byref(sz))
        fws = torch.empty(sz.value, dtype=torch.uint8, device=dev)
        ws_f.append((d, cu_h, cu_d, fws))
        _abi.call("gdn_conv1d_silu", ctypes.byref(d), P0(cu_d), P0(cu_h), _P(t["x"], s0),
                  P0(t["conv_w"]), P0(CS[i - 1]) if i else None, _P(qkv, s0), P0(CS[i]), st())
        _abi.call("gdn_chunk_fwd", ctypes.byref(d), P0(cu_d), P0(cu_h), _P(qkv, s0),
                  _P(t["a"], s0), _P(t["b"], s0), P0(t["A_log"]), P0(t["dt_bias"]),
                  P0(S[i - 1]) if i else None, _P(t["z"], s0), P0(t["norm_w"]), None,
                  _P(y, s0), P0(S[i]), P0(fws), fws.numel(), st())
    dS_next, dcs_next = None, None
    par = {k: [] for k in ("dconv_w", "dA_log", "ddt_bias", "dnorm_w")}
    for i in reversed(range(n)):
        s0, s1 = segs[i]
        d, cu_h, cu_d, fws = ws_f[i]
        sz = ctypes.c_size_t(0)
        _abi.call("gdn_workspace_size", ctypes.byref(d), P0(cu_h), _abi.GDN_WS_BWD,
                  ctypes.byref(sz))
        bws = torch.empty(sz.value, dtype=torch.uint8, device=dev)
        _abi.call("gdn_workspace_size", ctypes.byref(d), P0(cu_h), _abi.GDN_WS_CONV_BWD,
                  ctypes.byref(sz))
        cws = torch.empty(sz.value, dtype=torch.uint8, device=dev)
        dS0 = torch.empty(1, H, 128, 128, device=dev) if i else None
        dcs0 = torch.empty(1, C, 3, device=dev) if i else None
        g = {k: torch.empty(H if k in ("dA_log", "ddt_bias") else 128, device=dev)
             for k in ("dA_log", "ddt_bias", "dnorm_w")}
        dcw = torch.empty(C, 4, device=dev)
        _abi.call("gdn_chunk_bwd", ctypes.byref(d), P0(cu_d), P0(cu_h), _P(qkv, s0),
                  _P(t["a"], s0), _P(t["b"], s0), P0(t["A_log"]), P0(t["dt_bias"]),
                  P0(S[i - 1]) if i else None, _P(t["z"], s0), P0(t["norm_w"]), P0(fws),
                  fws.numel(), _P(t["dy"], s0), P0(dS_next), _P(dqkv, s0), _P(da, s0),
                  _P(db, s0), P0(g["dA_log"]), P0(g["ddt_bias"]), _P(dz, s0), P0(g["dnorm_w"]),
                  P0(dS0), P0(bws), bws.numel(), st())
        _abi.call("gdn_conv1d_silu_bwd", ctypes.byref(d), P0(cu_d), P0(cu_h), _P(t["x"], s0),
                  P0(t["conv_w"]), P0(CS[i - 1]) if i else None, _P(dqkv, s0), P0(dcs_next),
                  _P(dx, s0), P0(dcw), P0(dcs0), P0(cws), cws.numel(), st())
        for k in ("dA_log", "ddt_bias", "dnorm_w"):
            par[k].append(g[k])
        par["dconv_w"].append(dcw)
        keep += [bws, cws]
        dS_next, dcs_next = dS0, dcs0
    torch.cuda.synchronize()
    out = dict(y=y, S=S[-1], dx=dx, dz=dz, da=da, db=db)
    for k, v in par.items():
        out[k] = torch.stack(v).sum(0)
    return out


@pytest.mark.parametrize("cuts,layout", [((100, 233), "flat"), ((64, 65, 192), "group"),
                                         ((2,), "flat")])
def test_segments_chain_forward_and_backward(cuts, layout):
    """Segments as pointer offsets into one packed buffer, state / conv cache
    forward and dS / dconv_state backward: the whole sequence's outputs and
    gradients, against one call and against the oracle."""
    w = synth.Workload("seg", (300,), 2, 4, io="bf16", backward=True, seed=77, dt_bias=-4.0)
    inp = synth.make_inputs(w)
    seg = _segments_through_the_abi(inp, w, cuts, layout)
    one = gpu_run(inp, w, backward=True, layout=layout)
    ref = oracle.backward(**full_args(inp, w), dy=synth.to_f64(inp["dy"]), layout=layout)
    c = Checker(f"segments {cuts} vs oracle")
    c.add("y", f64(seg["y"]), ref["fwd"]["y"])
    c.add("S_final", f64(seg["S"]), ref["fwd"]["S_final"], state=True)
    for k in ("dx", "dz", "da", "db"):
        c.add(k, f64(seg[k]), ref[k])
    for k in ("dconv_w", "dA_log", "ddt_bias", "dnorm_w"):
        c.add(k, f64(seg[k]), ref[k], blocks=False)
    c.check()
    # the split moves chunk boundaries (tf32 rounding differs): held to the one
    # call at the same bars
    c = Checker(f"segments {cuts} vs one call")
    for k in ("y", "dx", "dz", "da", "db"):
        c.add(k, f64(seg[k]), f64(one[k]))
    c.add("S_final", f64(seg["S"]), f64(one["S"]), state=True)
    c.check()


def test_autograd_resumes_a_sequence_across_calls():
    """GDNCore: (y1, S1, cache1) = core(x[:s]); y2 = core(x[s:], S1, cache1); one
    backward through both gives the whole sequence's gradients (through the
    state and through the conv cache) -- against the oracle."""
    w = synth.Workload("ag", (150,), 1, 2, io="bf16", backward=True, seed=81, dt_bias=-4.0)
    inp = synth.make_inputs(w)
    dev = "cuda"
    t = {k: v.to(dev) for k, v in inp.items()}
    leaves = ["x", "conv_w", "a", "b", "A_log", "dt_bias", "z", "norm_w"]
    for k in leaves:
        t[k] = t[k].detach().clone().requires_grad_(True)
    s = 70
    cu1 = torch.tensor([0, s], dtype=torch.int32)
    cu2 = torch.tensor([0, w.T - s], dtype=torch.int32)
    cut = lambda k, a, b: t[k][a:b]
    args = lambda a, b: [cut("x", a, b), t["conv_w"], cut("a", a, b), cut("b", a, b),
                         t["A_log"], t["dt_bias"], cut("z", a, b), t["norm_w"]]
    y1, S1, cs1 = gdn_core(*args(0, s), cu1.to(dev), 1, 2, output_final_state=True,
                           cu_host=cu1, output_conv_state=True)
    y2, _ = gdn_core(*args(s, w.T), cu2.to(dev), 1, 2, initial_state=S1, conv_state=cs1,
                     cu_host=cu2)
    dy = t["dy"]
    ((y1.float() * dy[:s].float()).sum() + (y2.float() * dy[s:].float()).sum()).backward()
    torch.cuda.synchronize()
    ref = oracle.backward(**full_args(inp, w), dy=synth.to_f64(inp["dy"]))
    names = {"x": "dx", "conv_w": "dconv_w", "a": "da", "b": "db", "A_log": "dA_log",
             "dt_bias": "ddt_bias", "z": "dz", "norm_w": "dnorm_w"}
    c = Checker("autograd across calls")
    c.add("y", f64(torch.cat([y1, y2])), ref["fwd"]["y"])
    for k, g in names.items():
        c.add(g, f64(t[k].grad), ref[g], blocks=t[k].dim() > 1 and k != "conv_w")
    c.check()

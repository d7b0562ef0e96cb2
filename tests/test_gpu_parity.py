"""CUDA path vs the fp64 oracle, element by element (norm-wise, max-relative and
per-64-token-block measures), on small shapes that span several chunks and a
ragged tail, varlen batches, GVA groups of 1-3, initial state / conv cache
handoff, the entry points without the fused norm, and the fp32 workload."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_layer_causal_gb300 import core, synth
from gdn_testutil import (TOL, TOL_STATE, Checker, check_against, f64, full_args, gpu_run,
                          oracle_group, rel)

pytestmark = pytest.mark.gpu


SMALL = [
    # lens, h_k, h_v, io, dt_bias
    ((200,), 1, 1, "fp32", 0.0),
    ((200,), 2, 4, "bf16", 0.0),
    ((200,), 2, 4, "bf16", -6.0),
    ((1, 63, 64, 65, 130, 7), 1, 3, "bf16", -6.0),
    ((300, 5, 129), 2, 6, "fp32", -6.0),
    ((0, 77, 0, 64), 1, 2, "bf16", -3.0),
]


@pytest.mark.parametrize("qkv_tf32", [False, True])
@pytest.mark.parametrize("lens,hk,hv,io,dtb", SMALL)
def test_forward_backward_small(lens, hk, hv, io, dtb, qkv_tf32):
    """Both qkv precisions: exact fp32 (the chunk kernels round each q / k / v
    tile they feed to the tensor cores) and tf32 (the conv rounds once)."""
    w = synth.Workload("small", lens, hk, hv, io=io, backward=True, seed=sum(lens) + hv,
                       dt_bias=dtb)
    inp = synth.make_inputs(w)
    out = gpu_run(inp, w, backward=True, qkv_tf32=qkv_tf32)
    assert out["status_fwd"] == 0
    for kh in range(hk):
        ref, ch, heads = oracle_group(inp, w, kh, backward=True)
        check_against(out, ref, True, ch, heads, tag=f"kh={kh}")
    # the whole problem in one call: o, dnorm_w (a sum over every head) and the rest
    full = oracle.backward(**full_args(inp, w), dy=synth.to_f64(inp["dy"]))
    check_against(out, full, True, tag="whole problem")
    # post-conv activations: fp32 within 1e-5; tf32 values (the low 13 of the
    # 23 fraction bits zero) within half a tf32 unit (2^-11) more
    q = f64(out["qkv"])
    T = w.T
    tol_act = 1e-5 + (2.0 ** -11 if qkv_tf32 else 0.0)
    assert rel(q[:, :hk * 128].reshape(T, hk, 128), full["fwd"]["qh"]) <= tol_act
    assert rel(q[:, hk * 128:2 * hk * 128].reshape(T, hk, 128), full["fwd"]["kh"]) <= tol_act
    assert rel(q[:, 2 * hk * 128:].reshape(T, hv, 128), full["fwd"]["v"]) <= tol_act
    if qkv_tf32:
        bits = out["qkv"].contiguous().view(torch.int32)
        assert int((bits & 0x1FFF).count_nonzero()) == 0


def test_initial_state_conv_cache_and_state_grads():
    """initial_state / conv cache in, final state / conv cache out, dS_final
    in, dS_init and dconv_state out."""
    w = synth.Workload("s0", (150, 40), 1, 2, io="bf16", backward=True, seed=5, dt_bias=-6.0)
    inp = synth.make_inputs(w)
    S0 = synth.make_state(2, 2, 128, seed=6, scale=0.3)
    dS = synth.make_state(2, 2, 128, seed=7, scale=1.0)
    cs = synth.make_conv_state(2, w.C, 4, seed=8, dtype=torch.bfloat16)
    out = gpu_run(inp, w, backward=True, S0=S0, dS=dS, conv_state=cs)
    args = full_args(inp, w, S0, cs)
    ref = oracle.backward(**args, dy=synth.to_f64(inp["dy"]), dS_final=synth.to_f64(dS))
    np.testing.assert_array_equal(f64(out["conv_state"]), ref["fwd"]["conv_state_out"])
    check_against(out, ref, True, tag="S0 + conv cache")
    c = Checker("state grads")
    c.add("dinitial_state", f64(out["dinitial_state"]), ref["dS0"], blocks=False)
    c.add("dconv_state", f64(out["dconv_state"]), ref["dconv_state"], blocks=False)
    c.check()


@pytest.mark.parametrize("lens,hk,hv,io,dtb", [((200,), 2, 4, "bf16", -6.0),
                                                ((1, 63, 64, 65, 130, 7), 1, 3, "fp32", -6.0),
                                                ((0, 77, 0, 64), 1, 2, "bf16", 0.0)])
def test_chunk_entry_points_without_norm(lens, hk, hv, io, dtb):
    """z == NULL: gdn_chunk_fwd returns o (no fused norm) and gdn_chunk_bwd takes
    dy as the gradient of o; against the oracle's core without the norm stage."""
    w = synth.Workload("nonorm", lens, hk, hv, io=io, backward=True, seed=sum(lens) + 3 * hv,
                       dt_bias=dtb)
    inp = synth.make_inputs(w)
    S0 = synth.make_state(w.N, hv, 128, seed=29, scale=0.2)
    dS = synth.make_state(w.N, hv, 128, seed=31, scale=1.0)
    out = gpu_run(inp, w, backward=True, S0=S0, dS=dS, norm=False)
    assert out["status_fwd"] == 0 and out["y"] is None and out["dz"] is None
    ref = oracle.backward(**full_args(inp, w, S0), dy=synth.to_f64(inp["dy"]),
                          dS_final=synth.to_f64(dS), norm=False)
    check_against(out, ref, True, tag="no norm", norm=False)
    c = Checker("no norm, state grad")
    c.add("dinitial_state", f64(out["dinitial_state"]), ref["dS0"], blocks=False)
    c.check()


@pytest.mark.parametrize("split", [1, 37, 64, 100])
def test_split_sequence_handoff_equals_one_call(split):
    """Two calls with state + conv-cache handoff equal one call (on the GPU)."""
    w = synth.Workload("h", (160,), 2, 4, io="bf16", seed=11, dt_bias=-6.0)
    inp = synth.make_inputs(w)
    one = gpu_run(inp, w, backward=False)
    w1 = w.replace(seq_lens=(split,))
    w2 = w.replace(seq_lens=(160 - split,))
    cut = lambda d, s: {k: (v[s] if k not in ("conv_w", "A_log", "dt_bias", "norm_w",
                                              "cu_seqlens") else v) for k, v in d.items()}
    i1 = cut(inp, slice(0, split))
    i1["cu_seqlens"] = torch.tensor([0, split], dtype=torch.int32)
    i2 = cut(inp, slice(split, 160))
    i2["cu_seqlens"] = torch.tensor([0, 160 - split], dtype=torch.int32)
    o1 = gpu_run(i1, w1, backward=False)
    o2 = gpu_run(i2, w2, backward=False, S0=o1["S"].cpu(), conv_state=o1["conv_state"].cpu())
    y = torch.cat([o1["y"], o2["y"]]).float()
    # The split moves the chunk boundaries, so tf32 operand rounding differs
    # between the two runs: both are held to the oracle, and to each other at
    # the same bars.
    ref = oracle.forward(**full_args(inp, w))
    assert rel(f64(y), ref["y"]) <= TOL
    assert rel(f64(o2["S"]), ref["S_final"]) <= TOL_STATE
    assert rel(f64(y), f64(one["y"])) <= TOL
    assert rel(f64(o2["S"]), f64(one["S"])) <= TOL_STATE


def test_gva_equals_repeated_heads():
    """H_v = 3 H_k reading k-heads in place equals H_k = H_v with q/k repeated."""
    w = synth.Workload("g", (130,), 1, 3, io="fp32", seed=13, dt_bias=-6.0)
    inp = synth.make_inputs(w)
    out = gpu_run(inp, w, backward=False)
    x = inp["x"]
    q, k, v = x[:, :128], x[:, 128:256], x[:, 256:]
    x_rep = torch.cat([q.repeat(1, 3), k.repeat(1, 3), v], dim=1).contiguous()
    cw = inp["conv_w"]
    cw_rep = torch.cat([cw[:128].repeat(3, 1), cw[128:256].repeat(3, 1), cw[256:]]).contiguous()
    w3 = w.replace(h_k=3)
    inp3 = dict(inp, x=x_rep, conv_w=cw_rep)
    out3 = gpu_run(inp3, w3, backward=False)
    assert rel(f64(out3["y"]), f64(out["y"])) <= 1e-5
    assert rel(f64(out3["S"]), f64(out["S"])) <= 1e-5


def test_backward_is_deterministic():
    w = synth.Workload("det", (70, 200), 2, 6, io="bf16", backward=True, seed=17, dt_bias=-4.0)
    inp = synth.make_inputs(w)
    o1 = gpu_run(inp, w, backward=True)
    o2 = gpu_run(inp, w, backward=True)
    for k in ("y", "S", "dx", "dconv_w", "da", "db", "dz", "dnorm_w", "dA_log", "ddt_bias"):
        assert torch.equal(o1[k], o2[k]), k


def test_standalone_gated_rmsnorm():
    torch.manual_seed(0)
    for dt in (torch.float32, torch.bfloat16):
        o = torch.randn(333, 5, 128).to(dt)
        z = torch.randn(333, 5, 128).to(dt)
        w_ = (torch.randn(128) * 0.02).float()
        dy = torch.randn(333, 5, 128).to(dt)
        y, rstd = core.gated_rmsnorm(o.cuda(), z.cuda(), w_.cuda(), return_rstd=True)
        ry, rr = oracle.gated_rmsnorm(f64(o), f64(z), f64(w_), 1e-6)
        d_o, dz, dw = core.gated_rmsnorm_bwd(o.cuda(), z.cuda(), w_.cuda(), dy.cuda())
        rdo, rdz, rdw = oracle.gated_rmsnorm_bwd(f64(o), f64(z), f64(w_), f64(dy), 1e-6)
        c = Checker(f"standalone norm {dt}")
        c.add("y", f64(y), ry)
        c.add("do", f64(d_o), rdo)
        c.add("dz", f64(dz), rdz)
        c.add("dnorm_w", f64(dw), rdw, blocks=False)
        c.check()
        assert rel(f64(rstd), rr) <= 1e-5


@pytest.mark.parametrize("io", ["fp32", "bf16"])
def test_decode_step_matches_oracle_and_chunk_path(io):
    """gdn_recurrent_step on the last token after a chunked prefix equals the
    chunked run over all tokens and the oracle."""
    w = synth.Workload("dec", (70, 129, 5), 2, 4, io=io, seed=19, dt_bias=-6.0)
    inp = synth.make_inputs(w)
    full = gpu_run(inp, w, backward=False)
    cu = inp["cu_seqlens"].numpy()
    last = cu[1:] - 1
    keep = np.setdiff1d(np.arange(w.T), last)
    pre = {k: (v[keep] if k in ("x", "a", "b", "z") else v) for k, v in inp.items()}
    pre["cu_seqlens"] = torch.from_numpy((cu - np.arange(len(cu))).astype(np.int32))
    wp = w.replace(seq_lens=tuple(int(l) - 1 for l in w.seq_lens))
    head = gpu_run(pre, wp, backward=False)
    state = head["S"].clone()
    cs = head["conv_state"].clone()
    dv = lambda k: inp[k][last].cuda().contiguous()
    y = core.recurrent_step(dv("x"), inp["conv_w"].cuda(), cs, dv("a"), dv("b"),
                            inp["A_log"].cuda(), inp["dt_bias"].cuda(), dv("z"),
                            inp["norm_w"].cuda(), state, w.h_k, w.h_v)
    torch.cuda.synchronize()
    assert rel(f64(y), f64(full["y"])[last]) <= TOL
    assert rel(f64(state), f64(full["S"])) <= TOL_STATE
    np.testing.assert_array_equal(f64(cs), f64(full["conv_state"]))
    ry, _, rS, rcs = oracle.decode_step(
        synth.to_f64(inp["x"][last]), synth.to_f64(inp["conv_w"]), f64(head["conv_state"]),
        synth.to_f64(inp["a"][last]), synth.to_f64(inp["b"][last]), synth.to_f64(inp["A_log"]),
        synth.to_f64(inp["dt_bias"]), synth.to_f64(inp["z"][last]),
        synth.to_f64(inp["norm_w"]), f64(head["S"]), w.h_k, w.h_v)
    c = Checker(f"decode step {io}")
    c.add("y", f64(y), ry, blocks=False)
    c.add("S", f64(state), rS, state=True)
    c.check()


def test_device_check_of_cu_seqlens_sets_status():
    """A device cu_seqlens that disagrees with the host copy is caught by the
    planning kernel: status word = GDN_ERR_DEVICE_CHECK, no chunk processed."""
    w = synth.Workload("bad", (64, 64), 1, 1, io="fp32", seed=23)
    inp = synth.make_inputs(w)
    dev = "cuda"
    qkv, _ = core.conv1d_silu(inp["x"].to(dev), inp["conv_w"].to(dev),
                              inp["cu_seqlens"].to(dev), 1, 1)
    bad_dev = torch.tensor([0, 100, 128], dtype=torch.int32, device=dev)  # 2 + 1 chunks != 2
    r = core.chunk_fwd(qkv, inp["a"].to(dev), inp["b"].to(dev), inp["A_log"].to(dev),
                       inp["dt_bias"].to(dev), bad_dev, 1, 1, None, inp["z"].to(dev),
                       inp["norm_w"].to(dev), cu_host=inp["cu_seqlens"])
    assert core.read_status(r["fwd_ws"]) == 6
    assert core.read_status(r["fwd_ws"]) == 0   # read clears it

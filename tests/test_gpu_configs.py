"""The five workloads at full size, in the launch configuration bench.py uses
(the same C-ABI calls).  The oracle checks whole k-head groups one by one: heads
of different groups never interact, so a group's sub-problem (H_k = 1,
H_v = G, its conv channels) is exactly the full problem restricted to it.
Each forward workload also runs an extra dt_bias = -6 variant (not one of the
five): at dt_bias = 0 the state forgets within a token or two, so only the
variant exercises the state carried across chunks."""
import gc

import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_layer_causal_gb300 import core, synth
from gdn_testutil import TOL, TOL_STATE, f64, gpu_run, oracle_group, rel

pytestmark = pytest.mark.gpu


def _free():
    gc.collect()
    torch.cuda.empty_cache()


def _check_group(out, ref, ch, heads, backward):
    fw = ref["fwd"] if backward else ref
    errs = {"y": rel(f64(out["y"][:, heads]), fw["y"]),
            "S_final": rel(f64(out["S"][:, heads]), fw["S_final"])}
    if backward:
        idx = torch.as_tensor(ch, device=out["dx"].device)
        errs["dx"] = rel(f64(out["dx"].index_select(1, idx)), ref["dx"])
        errs["dconv_w"] = rel(f64(out["dconv_w"][idx]), ref["dconv_w"])
        errs["dz"] = rel(f64(out["dz"][:, heads]), ref["dz"])
        errs["da"] = rel(f64(out["da"][:, heads]), ref["da"])
        errs["db"] = rel(f64(out["db"][:, heads]), ref["db"])
        errs["dA_log"] = rel(f64(out["dA_log"][heads]), ref["dA_log"])
        errs["ddt_bias"] = rel(f64(out["ddt_bias"][heads]), ref["ddt_bias"])
    print("\nerrors: " + ", ".join(f"{k}={v:.2e}" for k, v in errs.items()))
    bad = {k: e for k, e in errs.items() if e > (TOL_STATE if k == "S_final" else TOL)}
    assert not bad, f"{bad} (all: {errs})"
    return errs


CASES = [
    ("tiny_fp32", 0.0, None), ("tiny_fp32", -6.0, None),
    ("qwen35_9b_16k", 0.0, (0, 15)), ("qwen35_9b_16k", -6.0, (7,)),
    ("qwen38_flash_64k", 0.0, (0, 15)), ("qwen38_flash_64k", -6.0, (5,)),
    ("varlen64_128k", 0.0, (0,)), ("varlen64_128k", -6.0, (11,)),
    ("long_128k", 0.0, (0,)), ("long_128k", -6.0, (9,)),
]


@pytest.mark.parametrize("name,dtb,groups", CASES)
def test_workload(name, dtb, groups):
    w = synth.WORKLOADS[name].replace(dt_bias=dtb)
    backward = w.backward or name == "tiny_fp32"
    inp = synth.make_inputs(w, with_grad=backward)
    out = gpu_run(inp, w, backward=backward)
    assert out["status_fwd"] == 0
    if groups is None:   # whole problem
        groups = tuple(range(w.h_k))
    for kh in groups:
        ref, ch, heads = oracle_group(inp, w, kh, backward)
        _check_group(out, ref, ch, heads, backward)
    if name == "tiny_fp32":   # o itself (the workload's stated output) and dnorm_w
        full = oracle.backward(
            **{k: synth.to_f64(inp[k]) for k in ("x", "conv_w", "a", "b", "A_log", "dt_bias",
                                                   "z", "norm_w")},
            cu=inp["cu_seqlens"].numpy(), hk=w.h_k, hv=w.h_v, dy=synth.to_f64(inp["dy"]))
        assert rel(f64(out["o"]), full["fwd"]["o"]) <= TOL
        assert rel(f64(out["dnorm_w"]), full["dnorm_w"]) <= TOL
    del out
    _free()


@pytest.mark.parametrize("dtb", [0.0, -6.0])
def test_decode_batch_256(dtb):
    """gdn_recurrent_step over [256, 48, 128, 128] fp32 states and their conv
    caches, against the oracle's decode step for every head."""
    w = synth.WORKLOADS["long_128k"].replace(seq_lens=(1,) * synth.DECODE_BATCH, dt_bias=dtb,
                                             seed=40)
    inp = synth.make_inputs(w, with_grad=False)
    N = synth.DECODE_BATCH
    S = synth.make_state(N, w.h_v, 128, seed=41, scale=0.05)
    cs = synth.make_conv_state(N, w.C, 4, seed=42, dtype=torch.bfloat16)
    dev = "cuda"
    Sd, csd = S.to(dev), cs.to(dev)
    y, o = core.recurrent_step(inp["x"].to(dev), inp["conv_w"].to(dev), csd, inp["a"].to(dev),
                               inp["b"].to(dev), inp["A_log"].to(dev), inp["dt_bias"].to(dev),
                               inp["z"].to(dev), inp["norm_w"].to(dev), Sd, w.h_k, w.h_v,
                               return_o=True)
    torch.cuda.synchronize()
    f = synth.to_f64
    ry, ro, rS, rcs = oracle.decode_step(f(inp["x"]), f(inp["conv_w"]), f(cs), f(inp["a"]),
                                         f(inp["b"]), f(inp["A_log"]), f(inp["dt_bias"]),
                                         f(inp["z"]), f(inp["norm_w"]), f(S), w.h_k, w.h_v)
    assert rel(f64(y), ry) <= TOL
    assert rel(f64(o), ro) <= TOL
    assert rel(f64(Sd), rS) <= TOL_STATE
    np.testing.assert_array_equal(f64(csd), rcs)
    del Sd, csd
    _free()

"""The five workloads at full size, in the launch configuration bench.py uses
(the same C-ABI calls).  The Qwen3.5-9B-shaped 16k forward and the 64k
forward + backward (the benchmark) are held to the oracle on the whole problem:
every head, o, the final state and every gradient including dnorm_w.  The 128k
workloads check whole k-head groups: heads of different groups never interact,
so a group's sub-problem (H_k = 1, H_v = G, its conv channels) is exactly the
full problem restricted to it.  Every comparison applies the norm-wise,
max-relative and per-64-token-block measures of gdn_testutil.  Each workload
also runs an extra dt_bias = -6 variant (not one of the five): at dt_bias = 0
the state forgets within a token or two, so only the variant exercises the
state carried across chunks."""
import gc

import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_layer_causal_gb300 import core, synth
from gdn_testutil import (Checker, check_against, f64, full_args, gpu_run, oracle_groups)

pytestmark = pytest.mark.gpu


def _free():
    gc.collect()
    torch.cuda.empty_cache()


# (workload, dt_bias, groups): "all" = the whole-problem oracle in one call;
# "every" = every k-head group, one oracle call per group (the 64k backward's
# fp64 intermediates for all heads at once would need ~75 GB of host memory),
# with dnorm_w, a sum over all heads, checked as the sum of the groups' parts
CASES = [
    ("tiny_fp32", 0.0, "all"), ("tiny_fp32", -6.0, "all"),
    ("qwen35_9b_16k", 0.0, "all"), ("qwen35_9b_16k", -6.0, (7,)),
    ("qwen38_flash_64k", 0.0, "every"), ("qwen38_flash_64k", -6.0, (5, 10)),
    ("varlen64_128k", 0.0, (0, 8)), ("varlen64_128k", -6.0, (11,)),
    ("long_128k", 0.0, (0, 15)), ("long_128k", -6.0, (9,)),
]


@pytest.mark.parametrize("name,dtb,groups", CASES)
def test_workload(name, dtb, groups):
    w = synth.WORKLOADS[name].replace(dt_bias=dtb)
    backward = w.backward or name == "tiny_fp32"
    inp = synth.make_inputs(w, with_grad=backward)
    out = gpu_run(inp, w, backward=backward)
    assert out["status_fwd"] == 0
    tag = f"{name} dt_bias={dtb}"
    if groups == "all":
        args = full_args(inp, w)
        ref = (oracle.backward(**args, dy=synth.to_f64(inp["dy"])) if backward
               else oracle.forward(**args))
        check_against(out, ref, backward, tag=tag)
    else:
        every = groups == "every"
        groups = range(w.h_k) if every else groups
        dnw = np.zeros(128)
        for kh, ref, ch, heads in oracle_groups(inp, w, groups, backward):
            check_against(out, ref, backward, ch, heads, tag=f"{tag} kh={kh}")
            if backward:
                dnw += ref["dnorm_w"]   # this group's heads' share of the sum
        if every and backward:
            c = Checker(f"{tag} all groups")
            c.add("dnorm_w", f64(out["dnorm_w"]), dnw, blocks=False)
            c.check()
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
    c = Checker(f"decode batch {N} dt_bias={dtb}")
    c.add("y", f64(y), ry)
    c.add("o", f64(o), ro)
    c.add("S", f64(Sd), rS, state=True)
    c.check()
    np.testing.assert_array_equal(f64(csd), rcs)
    del Sd, csd
    _free()

"""The whole GDN layer (projections around the core, GDNLayer) forward +
backward on the GPU against the fp64 oracle of the same layer.  The layer
keeps its activations (the projections' outputs, the core's inputs) in bf16;
the oracle rounds them at the same points."""
import pytest
import torch

import oracle
from gated_deltanet_layer_causal_gb300 import GDNLayer, synth
from gdn_testutil import Checker, f64

pytestmark = pytest.mark.gpu


def _bf16(v):
    """Round fp64 values to the nearest bf16 (the layer's activation storage)."""
    return torch.from_numpy(v).to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("gate,layout", [("silu", "flat"), ("sigmoid", "group")])
def test_layer_forward_backward(gate, layout):
    g = torch.Generator().manual_seed(3)
    hidden, hk, hv, lens = 256, 2, 4, (170, 130)
    layer = GDNLayer(hidden, hk, hv, gate=gate, layout=layout, device="cuda")
    layer.reset_parameters(generator=g)
    with torch.no_grad():
        layer.dt_bias.fill_(-4.0)   # the state carries across chunks
    T = sum(lens)
    h = torch.randn(T, hidden, generator=g).to(torch.bfloat16).cuda().requires_grad_(True)
    dout = torch.randn(T, hidden, generator=g).to(torch.bfloat16).cuda()
    cu_h = torch.tensor([0, lens[0], T], dtype=torch.int32)
    out, _ = layer(h, cu_h.cuda(), cu_host=cu_h)
    out.backward(dout)
    torch.cuda.synchronize()
    P = {k: f64(v) for k, v in layer.named_parameters()}
    ref = oracle.layer_backward(f64(h), P["W_qkv"], P["W_z"], P["W_b"], P["W_a"], P["W_out"],
                                P["conv_w"], P["A_log"], P["dt_bias"], P["norm_w"], cu_h.numpy(),
                                hk, hv, f64(dout), gate=gate, layout=layout, act=_bf16)
    c = Checker(f"layer {gate} {layout}")
    c.add("out", f64(out), ref["out"])
    c.add("dhidden", f64(h.grad), ref["dhidden"])
    for k, p in layer.named_parameters():
        c.add("d" + k, f64(p.grad), ref["d" + k], blocks=False)
    c.check()

"""The workload shapes and the library's fixed dims agree with the GDN
arguments the pages print (tests/golden/megatron_gdn_args.txt)."""
import os

from gated_deltanet_layer_causal_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def _args():
    out = {}
    for line in open(os.path.join(HERE, "golden", "megatron_gdn_args.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            out[k] = v
    return out


def test_printed_gdn_args_match_the_workloads():
    a = _args()
    assert a["linear-attention-type"] == "gated_delta_net"
    assert int(a["linear-conv-kernel-dim"]) == 4
    for w in synth.WORKLOADS.values():
        assert w.conv_k == int(a["linear-conv-kernel-dim"])
        assert w.d == int(a["linear-key-head-dim"]) == int(a["linear-value-head-dim"])
    q35 = synth.WORKLOADS["qwen35_9b_16k"]
    assert (q35.h_k, q35.h_v) == (int(a["linear-num-key-heads"]), int(a["linear-num-value-heads"]))
    for w in synth.WORKLOADS.values():
        assert w.h_v % w.h_k == 0


def test_varlen_lengths_recipe():
    w = synth.WORKLOADS["varlen64_128k"]
    assert w.N == 64 and w.T == 131072
    assert any(L % 64 for L in w.seq_lens)            # a boundary falls mid-chunk
    assert min(w.seq_lens) >= 200 and max(w.seq_lens) <= 9000

"""bench.py's stored DRAM traffic (one ncu capture of the first 8192 tokens,
times 8) names kernels its algorithmic-byte model knows, and each figure is a
plausible multiple of that kernel's algorithmic bytes: a stale, mistyped or
mis-scaled entry fails here.  CPU only."""
import bench
from gated_deltanet_layer_causal_gb300 import synth

W = synth.WORKLOADS["qwen38_flash_64k"]
NT = sum((L + 63) // 64 for L in W.seq_lens)


def test_traffic_entries_are_known_kernels_with_plausible_ratios():
    assert bench.TRAFFIC_64K, "no traffic figures"
    for name, traffic in bench.TRAFFIC_64K.items():
        bound, alg, unit = bench.kernel_cost(name, W, NT)
        assert alg, f"{name}: no algorithmic bytes"
        assert bound == "hbm" and unit == "B"
        ratio = traffic / alg
        # the gates kernel's outputs are still in L2 when it ends (no DRAM write
        # of its own); everything else moves its interface tensors about once
        lo = 0.25 if name == "gates" else 0.85
        assert lo <= ratio <= 1.2, f"{name}: traffic / algorithmic = {ratio:.3f}"


def test_every_chunk_kernel_has_a_cost():
    for name in ("conv_fwd", "gates", "chunk_prep", "chunk_state_fwd", "chunk_out_fwd",
                 "chunk_norm_bwd", "chunk_bwd_local", "chunk_bwd_state", "chunk_bwd_dp",
                 "chunk_bwd_sfacing", "chunk_bwd_wy", "gva_sum", "conv_bwd"):
        assert bench.kernel_cost(name, W, NT)[1] > 0, name

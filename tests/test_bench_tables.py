"""bench.py's cost tables.  The stored DRAM traffic (one ncu capture of the
first 8192 tokens, times 8) names kernels its interface-byte model knows, and
each figure is a plausible multiple of that kernel's interface bytes: a stale,
mistyped or mis-scaled entry fails here.  The path-level algorithmic cost is
the 123.5 kB and about 1.7 TFLOP per 64k step of the method's accounting, and
every chunk kernel has a tensor-pipe FLOP count.  CPU only."""
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
        # of its own); in the combined reverse-pass launch the state pass and the
        # P / dP groups walk the chunks in the same order and read the same q / k /
        # dO tiles, one of the two reads from L2; everything else moves its
        # interface tensors about once
        lo = {"gates": 0.25, "chunk_bwd_state_dp": 0.75}.get(name, 0.85)
        assert lo <= ratio <= 1.2, f"{name}: traffic / algorithmic = {ratio:.3f}"


def test_every_chunk_kernel_has_a_cost():
    for name in ("conv_fwd", "gates", "chunk_prep", "chunk_state_fwd", "chunk_out_fwd",
                 "chunk_norm_bwd", "chunk_bwd_local", "chunk_bwd_state_dp",
                 "chunk_bwd_sfacing", "chunk_bwd_wy", "gva_sum", "conv_bwd"):
        assert bench.kernel_cost(name, W, NT)[1] > 0, name


def test_path_cost_is_the_method_accounting():
    b, f = bench.path_cost(W)
    assert b == W.T * 123456          # 45.2 kB forward + 78.2 kB backward per token
    assert 1.6e12 < f < 1.8e12        # ~1.7 TFLOP of products per 64k fwd+bwd step
    fw = synth.WORKLOADS["qwen35_9b_16k"]
    b1, _ = bench.path_cost(fw)
    assert b1 == fw.T * 2 * (fw.C + 2 * fw.h_v + 2 * fw.h_v * 128)   # x, a, b, z in; y out


def test_chunk_kernels_have_tensor_flops():
    total = 0
    for name in bench.MMAS:
        f = bench.kernel_flops(name, NT, W.h_v, W.h_k)
        assert f and f % (NT * W.h_k) == 0, name
        total += f
    # every product the kernels issue, recomputed ones included (the forward
    # state pass builds each chunk's d_k x d_k transition in both row slices,
    # and the output kernel's stacked products carry an unused W K^T and a zero
    # half): ~2.5 TFLOP
    assert 2.3e12 < total < 2.6e12
    assert bench.kernel_flops("conv_fwd", NT, W.h_v, W.h_k) is None

#!/usr/bin/env python
"""GDN core forward + backward throughput on GB300.

One step = the whole hot path over one batch of synthetic input:
conv1d+SiLU+L2 -> chunked gated delta rule with the fused gated RMSNorm ->
its backward -> conv backward, each through the library's C ABI on device
buffers allocated once.  The default workload is the Qwen3.8-Flash-shaped
core at 64k tokens (T = 65536, 16 k-heads, 48 v-heads, d = 128, bf16 I/O,
fp32 state).  Prints one JSON line (rank 0).

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]
    python bench.py --workload qwen35_9b_16k      # forward-only workload
    python bench.py --decode                      # decode step, batch 256

The headline steps run with the library's per-kernel timing off; a separate
profiled pass afterwards times every kernel with CUDA events on its own stream
(the roofline of the dominant kernel and the per-kernel table come from it).

--impl reference times the fp64 CPU oracle (the only other implementation
of this method here) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from gated_deltanet_layer_causal_gb300 import _abi, synth  # noqa: E402

D = 128
METRIC = "GDN core fwd+bwd tokens/s per layer at 64k on 1 GB300; % of tensor/HBM roofline"
UNIT = "tokens/s"
# the tensor cores run tf32 (kind::tf32 operands, fp32 accumulation); the measured
# denominator is a bf16 GEMM, and dense tf32 runs at half the bf16 rate
TF32_PER_BF16 = 0.5


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="qwen38_flash_64k", choices=sorted(synth.WORKLOADS))
    p.add_argument("--tokens", type=int, default=0,
                   help="profiling case: only the first TOKENS tokens of the workload, as one "
                        "sequence (0 = the whole workload)")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-tokens", type=int, default=4096,
                   help="tokens of the oracle sample (cpu_baseline)")
    p.add_argument("--ref-tokens", type=int, default=1024,
                   help="tokens per reference-arm step")
    p.add_argument("--prof-steps", type=int, default=3,
                   help="steps of the separate per-kernel profiling pass")
    p.add_argument("--decode", action="store_true",
                   help="time the recurrent decode step (batch 256) instead")
    p.add_argument("--layer", type=int, default=0, metavar="HIDDEN",
                   help="time the whole layer (projections from / to HIDDEN around the core) "
                        "forward + backward instead, e.g. 2560")
    return p.parse_args()


# ------------------------------------------------------------------ clocks
class Clocks:
    """Samples nvidia-smi every 200 ms while the timed region runs."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index: int):
        self.rows = []
        self.proc = None
        sel = str(device_index)
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        self.sel = sel

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.sel, "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [s.strip() for s in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        reasons = sorted({n for r in self.rows for n, v in zip(self.NAMES, r[3:])
                          if v.lower().startswith("active")})
        pw = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w_max": max(pw) if pw else None, "samples": len(self.rows)}


# ------------------------------------------------------------------ our arm
class Step:
    """Device buffers for one workload and the C-ABI calls of one step: conv,
    chunk forward (fused norm) and, for a forward + backward workload, the
    chunk backward and the conv backward."""

    def __init__(self, w: synth.Workload, inp: dict, dev):
        self.w = w
        T, C, H, N = w.T, w.C, w.h_v, w.N
        t = {k: v.to(dev) for k, v in inp.items()}
        self.t = t
        io = w.torch_dtype
        f32 = torch.float32
        self.bwd = w.backward
        self.cu_host = inp["cu_seqlens"].contiguous()
        self.dims = _abi.dims(N, T, w.h_k, w.h_v, io == torch.bfloat16, qkv_tf32=True)
        ws = {}
        for kind in (_abi.GDN_WS_FWD, _abi.GDN_WS_BWD, _abi.GDN_WS_CONV_BWD):
            if kind != _abi.GDN_WS_FWD and not self.bwd:
                continue
            n = ctypes.c_size_t(0)
            _abi.call("gdn_workspace_size", ctypes.byref(self.dims),
                      ctypes.c_void_p(self.cu_host.data_ptr()), kind, ctypes.byref(n))
            ws[kind] = torch.empty(n.value, dtype=torch.uint8, device=dev)
        self.ws = ws
        e = lambda *s, dt=f32: torch.empty(*s, dtype=dt, device=dev)
        self.qkv = e(T, C)
        self.y = e(T, H, D, dt=io)
        if self.bwd:
            self.dqkv = e(T, C)
            self.dz = e(T, H, D, dt=io)
            self.da, self.db = e(T, H, dt=io), e(T, H, dt=io)
            self.dA, self.ddt, self.dnw = e(H), e(H), e(D)
            self.dx, self.dw = e(T, C, dt=io), e(C, 4)

    def p(self, x):
        return None if x is None else ctypes.c_void_p(x.data_ptr())

    def __call__(self):
        t, p, d = self.t, self.p, ctypes.byref(self.dims)
        s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        cu, cuh = p(t["cu_seqlens"]), p(self.cu_host)
        fw = self.ws[_abi.GDN_WS_FWD]
        _abi.call("gdn_conv1d_silu", d, cu, cuh, p(t["x"]), p(t["conv_w"]), None, p(self.qkv),
                  None, s)
        _abi.call("gdn_chunk_fwd", d, cu, cuh, p(self.qkv), p(t["a"]), p(t["b"]), p(t["A_log"]),
                  p(t["dt_bias"]), None, p(t["z"]), p(t["norm_w"]), None, p(self.y), None, p(fw),
                  fw.numel(), s)
        if not self.bwd:
            return
        bw, cw = self.ws[_abi.GDN_WS_BWD], self.ws[_abi.GDN_WS_CONV_BWD]
        _abi.call("gdn_chunk_bwd", d, cu, cuh, p(self.qkv), p(t["a"]), p(t["b"]), p(t["A_log"]),
                  p(t["dt_bias"]), None, p(t["z"]), p(t["norm_w"]), p(fw), fw.numel(),
                  p(t["dy"]), None, p(self.dqkv), p(self.da), p(self.db), p(self.dA),
                  p(self.ddt), p(self.dz), p(self.dnw), None, p(bw), bw.numel(), s)
        _abi.call("gdn_conv1d_silu_bwd", d, cu, cuh, p(t["x"]), p(t["conv_w"]), None,
                  p(self.dqkv), None, p(self.dx), p(self.dw), None, p(cw), cw.numel(), s)

    def outputs(self):
        if not self.bwd:
            return [self.y]
        return [self.y, self.dx, self.dw, self.da, self.db, self.dA, self.ddt, self.dz, self.dnw]

    def inputs(self):
        return ["x", "conv_w", "a", "b", "A_log", "dt_bias", "z", "norm_w", "cu_seqlens"] + \
            (["dy"] if self.bwd else [])


class DecodeStep:
    """One gdn_recurrent_step over a batch of N sequences: conv caches [N, C, 3]
    and fp32 states [N, H_v, 128, 128] updated in place."""

    def __init__(self, w: synth.Workload, N: int, dev):
        self.w = w
        self.N = N
        wd = w.replace(seq_lens=(1,) * N)
        inp = synth.make_inputs(wd, with_grad=False)
        self.host = {k: inp[k] for k in ("x", "conv_w", "a", "b", "A_log", "dt_bias", "z",
                                         "norm_w")}
        self.t = {k: v.to(dev) for k, v in self.host.items()}
        self.S = synth.make_state(N, w.h_v, D, seed=w.seed + 7, scale=0.05).to(dev)
        self.cs = synth.make_conv_state(N, w.C, 4, seed=w.seed + 8, dtype=w.torch_dtype).to(dev)
        self.y = torch.empty(N, w.h_v, D, dtype=w.torch_dtype, device=dev)
        self.dims = _abi.dims(N, N, w.h_k, w.h_v, w.io == "bf16")

    def __call__(self):
        t = self.t
        p = lambda x: None if x is None else ctypes.c_void_p(x.data_ptr())
        s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        _abi.call("gdn_recurrent_step", ctypes.byref(self.dims), p(t["x"]), p(t["conv_w"]),
                  p(self.cs), p(t["a"]), p(t["b"]), p(t["A_log"]), p(t["dt_bias"]), p(t["z"]),
                  p(t["norm_w"]), p(self.S), None, p(self.y), s)

    def alg_bytes(self):
        """State read + written, conv caches read + written, x, a, b, z read, y written."""
        w, N = self.w, self.N
        io = 2 if w.io == "bf16" else 4
        return N * (2 * w.h_v * D * D * 4 + 2 * w.C * 3 * io + w.C * io + 2 * w.h_v * io +
                    2 * w.h_v * D * io)


# Measured DRAM bytes (read + write) per launch on the 64k-token workload:
# dram__bytes_read.sum + dram__bytes_write.sum of each kernel from one ncu
# capture of the first 8192 tokens, times 8 (every kernel's work is
# proportional to the chunks it processes).  Valid for the kernels as captured;
# a kernel changed since then is left out (its traffic reports null).
TRAFFIC_64K = {
    "conv_fwd": 3626989568,
    "gates": 12656640,
    "chunk_prep": 6499026944,
    "chunk_state_fwd": 6636810240,
    "chunk_out_fwd": 12034592768,
    "chunk_norm_bwd": 5311037440,
    "chunk_bwd_local": 3956418560,
    "chunk_bwd_state_dp": 13553457152,
    "chunk_bwd_sfacing": 14881130496,
    "chunk_bwd_wy": 9024550912,
    "gva_sum": 3439785984,
    "conv_bwd": 5371553792,
}

# tcgen05 / mma.sync products each chunk kernel issues per (chunk, v-head) tile,
# as (M, N, K) -- the per-unit figure of its tensor-pipe roofline:
MMAS = {
    "chunk_prep": [(64, 64, 128), (64, 128, 64), (64, 128, 64)],        # K K^T, W, U~
    # per 64-row slice (2): the chain M^T S^T, B^T = (fk K)^T U~, -M^T = (fk K)^T W
    "chunk_state_fwd": [(128, 64, 128), (128, 64, 64), (128, 128, 64)] * 2,
    # [Q; W] [K; S0]^T (Q K^T, Q S0^T, W S0^T and an unused W K^T), [P; 0] U
    "chunk_out_fwd": [(128, 192, 128), (128, 128, 64)],
    "chunk_bwd_local": [(64, 128, 64)],                                 # P^T dO
    # reverse state pass (2 row slices: K dS^T; B'^T = Q^T e^gam dO - W^T dU_local;
    # W^T Ub) and the P / dP groups' per-v-head dO U^T, one launch
    "chunk_bwd_state_dp": [(64, 64, 128), (128, 64, 64), (128, 64, 64), (128, 64, 64)] * 2 +
                          [(64, 64, 128)],
    "chunk_bwd_sfacing": [(128, 128, 128), (64, 128, 128)],            # [dO; dU] S0, U dS
    "chunk_bwd_wy": [(64, 64, 128)] * 3 + [(64, 256, 64), (64, 64, 64), (64, 64, 64),
                                           (64, 128, 64)],   # ..., (dKK + dKK^T) K
}


# products issued once per (chunk, k-head) group: the local backward's K Q^T, the
# P / dP groups' Q K^T and D_dq = dPs K, D_dk = dPs^T Q (q, k and so these are
# shared by the group's v-heads)
MMAS_KH = {
    "chunk_bwd_local": [(64, 64, 128)],                                 # K Q^T
    "chunk_bwd_state_dp": [(64, 64, 128), (64, 128, 64), (64, 128, 64)],
}


def kernel_flops(name: str, NT: int, hv: int, hk: int):
    """Tensor-core FLOPs of one launch: the kernel's products per (chunk, v-head)
    tile x tiles, plus those per (chunk, k-head) group x groups."""
    if name not in MMAS:
        return None
    return (sum(2 * m * n * k for m, n, k in MMAS[name]) * NT * hv +
            sum(2 * m * n * k for m, n, k in MMAS_KH.get(name, [])) * NT * hk)


def kernel_cost(name: str, w: synth.Workload, NT: int):
    """Interface bytes of one launch of a kernel: the tensors its interface must
    read and write, each once (the design's intermediates included).  Notation:
    io = bytes per activation, tk = one [T, H_k, d] fp32 tensor, tv = one
    [T, H_v, d] fp32 tensor (or the same bytes as per-chunk tiles), S = per-chunk
    states [NT, H_v, d, d] fp32, Tt = per-chunk 64 x 64 tiles [NT, H_v] fp32,
    g = [T, H_v] fp32, act = [T, H_v, d] in the I/O dtype."""
    T, C, H, Hk = w.T, w.C, w.h_v, w.h_k
    io = 2 if w.io == "bf16" else 4
    tk, tv = T * Hk * D * 4, T * H * D * 4
    S, Tt, g, act = NT * H * D * D * 4, NT * H * 64 * 64 * 4, T * H * 4, T * H * D * io
    gates = 2 * T * H * io
    table = {
        "conv_fwd": T * C * io + T * C * 4,
        "conv_bwd": 2 * T * C * io + T * C * 4,
        "gates": gates + 2 * g,
        "chunk_prep": tk + tv + 2 * g + 2 * tv + 2 * Tt,
        "chunk_state_fwd": 2 * tv + tk + g + S,
        "chunk_out_fwd": 2 * tk + 2 * tv + S + g + act + act + 2 * tv + g,
        "chunk_norm_bwd": tv + 2 * act + tv + act,
        "chunk_bwd_local": 2 * tk + tv + g + tv,
        "chunk_bwd_state_dp": (2 * tk + 3 * tv + g + tv + S) +     # state pass
                              (2 * tk + 2 * tv + g + 2 * tk + 2 * g),  # P / dP groups
        "chunk_bwd_sfacing": 2 * S + 3 * tv + 2 * tk + g + tv + 2 * tk + g,
        "chunk_bwd_wy": tk + tv + 2 * tv + 2 * Tt + 3 * g + gates + tv + tk + gates + g,
        "gva_sum": 7 * tk,
    }
    return "hbm", table.get(name), "B"


def path_cost(w: synth.Workload):
    """Algorithmic bytes and FLOPs of one step of the whole path (the method's
    minimum: inputs read and outputs written once, saved activations free;
    MMA FLOPs only, no recompute).  Per token, bf16, c = 64, d = 128:
      fwd bytes: x 2C + a, b 2*2H + z 2Hd + y 2Hd
      bwd bytes: dy, z 2*2Hd + x 2C + a, b 2*2H read; dx 2C, dz 2Hd, da, db 2*2H
      fwd FLOPs: H (6d^2 + 6cd + 0.7c^2) + H_k 4cd;  bwd FLOPs: H (12d^2 + 20cd + 4c^2)."""
    io = 2 if w.io == "bf16" else 4
    c, d, H, C = 64, D, w.h_v, w.C
    fwd_b = io * (C + 2 * H + 2 * H * d)
    bwd_b = io * (2 * H * d + C + 2 * H) + io * (C + H * d + 2 * H)
    fwd_f = H * (6 * d * d + 6 * c * d + 0.7 * c * c) + w.h_k * 4 * c * d
    bwd_f = H * (12 * d * d + 20 * c * d + 4 * c * c)
    if not w.backward:
        return w.T * fwd_b, w.T * fwd_f
    return w.T * (fwd_b + bwd_b), w.T * (fwd_f + bwd_f)


def _peaks():
    try:
        pk = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return pk["hbm_gbs"], pk["bf16_tflops"], "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def _sync_all(world):
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()


def _max_over_ranks(v, world, dev):
    if world == 1:
        return v
    t = torch.tensor([v], device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _timed(step, steps, world, dev):
    """K steps between CUDA events on the launching stream (torch's current stream,
    the one the library launches on), barrier + synchronize on both sides."""
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _sync_all(world)
    launches0 = _abi.launch_count()
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    e1.synchronize()
    launches = _abi.launch_count() - launches0
    _sync_all(world)
    ms = _max_over_ranks(e0.elapsed_time(e1) / steps, world, dev)
    return ms, launches


def _profile(step, steps):
    """Per-kernel device time from the library's own events (a separate pass)."""
    _abi.profile_report()
    _abi.profile_enable(True)
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    _abi.profile_enable(False)
    return _abi.profile_report()


def run_ours(args, rank, world, dev):
    if args.decode:
        return run_decode(args, rank, world, dev)
    if args.layer:
        return run_layer(args, rank, world, dev)
    w = synth.WORKLOADS[args.workload]
    w = w.replace(seed=w.seed + 1000 * rank)
    if args.tokens:
        w = w.replace(name=f"{w.name}[first {args.tokens} tokens]", seq_lens=(args.tokens,))
    inp = synth.make_inputs(w, with_grad=w.backward)
    step = Step(w, inp, dev)
    NT = sum((L + 63) // 64 for L in w.seq_lens)
    for _ in range(args.warmup):
        step()
    with Clocks(dev.index if dev.index is not None else 0) as clk:
        ms, launches = _timed(step, args.steps, world, dev)
    value = world * w.T / (ms / 1e3)
    prof = _profile(step, args.prof_steps)
    psteps = args.prof_steps

    hbm_peak, bf16_peak, peak_src = _peaks()
    tf32_peak = bf16_peak * TF32_PER_BF16
    # dominant kernel (largest share of the profiled step) and its roofline
    name, (nl, tot_ms) = max(prof.items(), key=lambda kv: kv[1][1])
    avg_ms = tot_ms / nl
    _, ibytes, _ = kernel_cost(name, w, NT)
    flops = kernel_flops(name, NT, w.h_v, w.h_k)
    traffic = (TRAFFIC_64K.get(name) if args.workload == "qwen38_flash_64k" and not args.tokens
               else None)
    if flops is not None:   # a chunk kernel: tensor pipe
        ach = flops / (avg_ms / 1e3) / 1e12
        roof = {"kernel": name, "bound": "tensor", "achieved": ach, "peak": tf32_peak,
                "unit": "TFLOP/s", "frac": ach / tf32_peak, "traffic": traffic,
                "flops_per_launch": flops,
                "peak_note": f"tf32 = {TF32_PER_BF16} x {peak_src} bf16 burst {bf16_peak}",
                "interface_bytes_per_launch": ibytes,
                "interface_gbs": ibytes / (avg_ms / 1e3) / 1e9 if ibytes else None,
                "interface_frac_of_hbm": (ibytes / (avg_ms / 1e3) / 1e9 / hbm_peak
                                          if ibytes else None)}
    else:
        ach = ibytes / (avg_ms / 1e3) / 1e9 if ibytes else None
        roof = {"kernel": name, "bound": "hbm", "achieved": ach, "peak": hbm_peak,
                "unit": "GB/s", "frac": ach / hbm_peak if ach else None, "traffic": traffic,
                "bytes_per_launch": ibytes, "peak_note": f"{peak_src} copy"}
    roof.update(traffic_unit="B per launch (ncu dram__bytes_read + write)",
                avg_launch_ms=avg_ms, step_share=tot_ms / sum(v[1] for v in prof.values()))
    pb, pf = path_cost(w)
    t_b, t_f = pb / (hbm_peak * 1e9) * 1e3, pf / (tf32_peak * 1e12) * 1e3
    path = {"bound": "tensor" if t_f >= t_b else "hbm",
            "algorithmic_bytes_per_step": pb, "algorithmic_flops_per_step": pf,
            "t_roof_ms": max(t_b, t_f), "t_hbm_ms": t_b, "t_tensor_ms": t_f,
            "frac": max(t_b, t_f) / ms, "hbm_frac": t_b / ms,
            "peaks": {"hbm_gbs": hbm_peak, "tf32_tflops": tf32_peak, "source": peak_src}}
    kernels = {k: {"launches_per_step": v[0] / psteps, "ms_per_step": v[1] / psteps}
               for k, v in prof.items()}

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(step, args.e2e_steps, w, world, dev, inp)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_tokens)

    if rank == 0:
        metric = METRIC if args.workload == "qwen38_flash_64k" and not args.tokens else \
            f"GDN core {'fwd+bwd' if w.backward else 'fwd'} tokens/s per layer, {w.name}, 1 GB300"
        line = {
            "metric": metric, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "tf32", "data": "synthetic",
            "config": {"workload": w.name, "tokens": w.T, "seqs": w.N, "h_k": w.h_k,
                       "h_v": w.h_v, "d_k": D, "d_v": D, "chunk": 64, "conv_k": 4,
                       "io": w.io, "state": "fp32",
                       "mma": "tf32 operands, fp32 accumulation, tcgen05 (every product)",
                       "qkv": "conv output stored at tf32 precision",
                       "passes": ("fwd+bwd" if w.backward else "fwd") +
                                 " (conv, chunk rule, fused gated norm)",
                       "l2": "inputs larger than L2 (x alone is %.2f GB)" % (
                           w.T * w.C * (2 if w.io == "bf16" else 4) / 1e9),
                       "timing": "headline with per-kernel events off; kernels from a "
                                 f"separate {psteps}-step profiled pass",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": roof,
            "path_roofline": path,
            "kernels": kernels,
            "gpu_launches": launches,
            "clocks": clk.summary(),
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def run_e2e(step, steps, w, world, dev, inp):
    """The same step through the C ABI with pinned host buffers: every step's
    inputs copied in and all of its results copied back inside the timed region.
    Two sets of device buffers alternate, so step i + 1's inputs go in (one copy
    stream) and step i - 1's results come out (another) while step i computes, as
    a training loop feeding the layer would overlap them; a set is refilled only
    once its previous step has finished and its results are out.  One untimed pass
    over both sets first."""
    sets = [step, Step(w, inp, dev)]
    main = torch.cuda.current_stream()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    host_in = {k: inp[k].pin_memory() for k in step.inputs()}
    host_out = [[torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in st.outputs()]
                for st in sets]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(o.numel() * o.element_size() for o in host_out[0])
    ev_in = [torch.cuda.Event() for _ in sets]     # a set's inputs are in
    ev_done = [torch.cuda.Event() for _ in sets]   # a set's step has finished
    ev_out = [torch.cuda.Event() for _ in sets]    # a set's results are out

    def pipeline(n):
        cin.wait_stream(main)
        cout.wait_stream(main)
        for i in range(n):
            b = i % 2
            st = sets[b]
            with torch.cuda.stream(cin):
                if i >= 2:
                    cin.wait_event(ev_done[b])
                for k, v in host_in.items():
                    st.t[k].copy_(v, non_blocking=True)
                ev_in[b].record(cin)
            main.wait_event(ev_in[b])
            if i >= 2:
                main.wait_event(ev_out[b])
            st()
            ev_done[b].record(main)
            with torch.cuda.stream(cout):
                cout.wait_event(ev_done[b])
                for h, o in zip(host_out[b], st.outputs()):
                    h.copy_(o, non_blocking=True)
                ev_out[b].record(cout)
        main.wait_stream(cout)

    # untimed: both sets once, so every pinned buffer has been through a copy
    pipeline(len(sets))
    _sync_all(world)
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(main)
    pipeline(steps)
    e3.record(main)
    e3.synchronize()
    e2e_ms = _max_over_ranks(e2.elapsed_time(e3) / steps, world, dev)
    return {"value": world * w.T / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "overlap": "two buffer sets"}


# the pages' whole-layer figure on GB300 (fla's kernels, projections included,
# bf16 training stack), forward + backward at 64k tokens, Qwen3.8-Flash shape
PAGES_LAYER_MS_64K = 43.5


def run_layer(args, rank, world, dev):
    """GDNLayer forward + backward (input gradient and every weight gradient)."""
    from gated_deltanet_layer_causal_gb300 import GDNLayer
    w = synth.WORKLOADS[args.workload]
    g = torch.Generator().manual_seed(w.seed + 1000 * rank)
    layer = GDNLayer(args.layer, w.h_k, w.h_v, device=dev)
    layer.reset_parameters(generator=g)
    cu_h = torch.from_numpy(w.cu_seqlens())
    cu = cu_h.to(dev)
    h = torch.randn(w.T, args.layer, generator=g).to(torch.bfloat16).to(dev).requires_grad_(True)
    dout = torch.randn(w.T, args.layer, generator=g).to(torch.bfloat16).to(dev)
    params = [h] + list(layer.parameters())

    def step():
        out, _ = layer(h, cu, cu_host=cu_h)
        torch.autograd.grad(out, params, dout)

    for _ in range(args.warmup):
        step()
    with Clocks(dev.index if dev.index is not None else 0) as clk:
        ms, launches = _timed(step, args.steps, world, dev)
    if rank == 0:
        line = {
            "metric": f"GDN layer (projections + core) fwd+bwd tokens/s, {w.name}, hidden "
                      f"{args.layer}, 1 GB300",
            "value": world * w.T / (ms / 1e3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "tf32",
            "data": "synthetic",
            "config": {"workload": w.name, "hidden": args.layer, "tokens": w.T, "h_k": w.h_k,
                       "h_v": w.h_v, "io": "bf16", "projections": "cuBLAS bf16 GEMMs (torch)",
                       "core": "libgdn.so"},
            "pages_context": {"ms_per_layer": PAGES_LAYER_MS_64K,
                              "what": "fla GDN layer incl. projections, GB300, 64k tokens, "
                                      "fwd+bwd (another stack: context, not the target)"},
            "gpu_launches": launches,
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)


def run_decode(args, rank, world, dev):
    """Decode step over the long-context workload's heads, batch DECODE_BATCH."""
    w = synth.WORKLOADS["long_128k"]
    w = w.replace(seed=w.seed + 1000 * rank)
    N = synth.DECODE_BATCH
    step = DecodeStep(w, N, dev)
    for _ in range(args.warmup):
        step()
    # one step is ~0.3 ms: time enough of them (>= 0.5 s) for the clock sampler
    args.steps = max(args.steps, 2000)
    # the states (805 MB) are larger than L2: every step reads them from HBM
    with Clocks(dev.index if dev.index is not None else 0) as clk:
        ms, launches = _timed(step, args.steps, world, dev)
    hbm_peak, _, peak_src = _peaks()
    ab = step.alg_bytes()
    gbs = ab / (ms / 1e3) / 1e9
    e2e = None
    if not args.no_e2e:
        # host copies of the step's inputs and its output (the states stay resident)
        stream = torch.cuda.current_stream()
        hin = {k: v.pin_memory() for k, v in step.host.items()}
        hy = torch.empty(step.y.shape, dtype=step.y.dtype, pin_memory=True)
        h2d = sum(v.numel() * v.element_size() for v in hin.values())
        _sync_all(world)
        e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2.record(stream)
        for _ in range(args.steps):
            for k, v in hin.items():
                step.t[k].copy_(v, non_blocking=True)
            step()
            hy.copy_(step.y, non_blocking=True)
        e3.record(stream)
        e3.synchronize()
        e_ms = _max_over_ranks(e2.elapsed_time(e3) / args.steps, world, dev)
        e2e = {"value": world * N / (e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": hy.numel() * hy.element_size(), "ms_per_step": e_ms}
    if rank == 0:
        line = {
            "metric": f"GDN decode step tokens/s, batch {N}, 1 GB300", "value": world * N / (ms / 1e3),
            "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"decode batch {N} ({w.h_k} k-heads, {w.h_v} v-heads, fp32 "
                                   f"states [{N},{w.h_v},128,128])", "io": w.io,
                       "l2": "states larger than L2 (%.0f MB)" % (N * w.h_v * D * D * 4 / 1e6)},
            "roofline": {"kernel": "recurrent_step", "bound": "hbm", "achieved": gbs,
                         "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                         "traffic": None, "bytes_per_launch": ab, "peak_note": peak_src},
            "steps_per_s": 1e3 / ms,
            "gpu_launches": launches,
            "clocks": clk.summary(),
            "e2e": e2e,
        }
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ oracle legs
def _oracle_sample(w: synth.Workload, tokens: int):
    """Inputs of the first `tokens` tokens of the workload (one sequence) as fp64."""
    ws = w.replace(seq_lens=(tokens,))
    inp = synth.make_inputs(ws, with_grad=True)
    f = synth.to_f64
    args = {k: f(inp[k]) for k in ("x", "conv_w", "a", "b", "A_log", "dt_bias", "z", "norm_w")}
    args.update(cu=inp["cu_seqlens"].numpy(), hk=w.h_k, hv=w.h_v)
    return args, f(inp["dy"])


def cpu_baseline(w: synth.Workload, tokens: int):
    import oracle
    args, dy = _oracle_sample(w, tokens)
    t0 = time.perf_counter()
    if w.backward:
        oracle.backward(**args, dy=dy)
    else:
        oracle.forward(**args)
    dt = time.perf_counter() - t0
    passes = "fwd+bwd" if w.backward else "fwd"
    return {"value": tokens / dt, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"fp64 oracle {passes} of all {w.h_v} v-heads over the first {tokens} "
                      f"tokens of {w.name}; {dt:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    w = synth.WORKLOADS[args.workload]
    args_o, dy = _oracle_sample(w, args.ref_tokens)
    for _ in range(args.warmup):
        oracle.backward(**args_o, dy=dy)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.backward(**args_o, dy=dy)
    dt = (time.perf_counter() - t0) / args.steps
    value = args.ref_tokens / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "tokens": w.T, "h_k": w.h_k, "h_v": w.h_v, "d_k": D,
                   "d_v": D, "io": w.io, "passes": "fwd+bwd",
                   "sample_tokens_per_step": args.ref_tokens},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"fp64 oracle fwd+bwd of all {w.h_v} v-heads over the "
                                   f"first {args.ref_tokens} tokens of {w.name} per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    try:
        run_ours(args, rank, world, dev)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

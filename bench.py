#!/usr/bin/env python
"""GDN core forward + backward throughput on GB300.

One step = the whole hot path over one batch of synthetic input:
conv1d+SiLU+L2 -> chunked gated delta rule with the fused gated RMSNorm ->
its backward -> conv backward, each through the library's C ABI on device
buffers allocated once.  The default workload is the Qwen3.8-Flash-shaped
core at 64k tokens (T = 65536, 16 k-heads, 48 v-heads, d = 128, bf16 I/O,
fp32 state).  Prints one JSON line (rank 0).

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]

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
METRIC = "GDN core fwd+bwd tokens/s per layer at 64k on 1 GB300"
UNIT = "tokens/s"


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
    p.add_argument("--e2e-steps", type=int, default=2)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-tokens", type=int, default=4096,
                   help="tokens of the oracle sample (cpu_baseline)")
    p.add_argument("--ref-tokens", type=int, default=1024,
                   help="tokens per reference-arm step")
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
    """Device buffers for one workload and the four C-ABI calls of one step."""

    def __init__(self, w: synth.Workload, inp: dict, dev):
        self.w = w
        T, C, H, N = w.T, w.C, w.h_v, w.N
        t = {k: v.to(dev) for k, v in inp.items()}
        self.t = t
        io = w.torch_dtype
        f32 = torch.float32
        self.cu_host = inp["cu_seqlens"].contiguous()
        self.dims = _abi.dims(N, T, w.h_k, w.h_v, io == torch.bfloat16, qkv_tf32=True)
        ws = {}
        for kind in (_abi.GDN_WS_FWD, _abi.GDN_WS_BWD, _abi.GDN_WS_CONV_BWD):
            n = ctypes.c_size_t(0)
            _abi.call("gdn_workspace_size", ctypes.byref(self.dims),
                      ctypes.c_void_p(self.cu_host.data_ptr()), kind, ctypes.byref(n))
            ws[kind] = torch.empty(n.value, dtype=torch.uint8, device=dev)
        self.ws = ws
        e = lambda *s, dt=f32: torch.empty(*s, dtype=dt, device=dev)
        self.qkv, self.dqkv = e(T, C), e(T, C)
        self.y, self.dz = e(T, H, D, dt=io), e(T, H, D, dt=io)
        self.da, self.db = e(T, H, dt=io), e(T, H, dt=io)
        self.dA, self.ddt, self.dnw = e(H), e(H), e(D)
        self.dx, self.dw = e(T, C, dt=io), e(C, 4)

    def p(self, x):
        return None if x is None else ctypes.c_void_p(x.data_ptr())

    def __call__(self):
        t, p, d = self.t, self.p, ctypes.byref(self.dims)
        s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        cu, cuh = p(t["cu_seqlens"]), p(self.cu_host)
        fw, bw, cw = self.ws[_abi.GDN_WS_FWD], self.ws[_abi.GDN_WS_BWD], \
            self.ws[_abi.GDN_WS_CONV_BWD]
        _abi.call("gdn_conv1d_silu", d, cu, cuh, p(t["x"]), p(t["conv_w"]), None, p(self.qkv),
                  None, s)
        _abi.call("gdn_chunk_fwd", d, cu, cuh, p(self.qkv), p(t["a"]), p(t["b"]), p(t["A_log"]),
                  p(t["dt_bias"]), None, p(t["z"]), p(t["norm_w"]), None, p(self.y), None, p(fw),
                  fw.numel(), s)
        _abi.call("gdn_chunk_bwd", d, cu, cuh, p(self.qkv), p(t["a"]), p(t["b"]), p(t["A_log"]),
                  p(t["dt_bias"]), None, p(t["z"]), p(t["norm_w"]), p(fw), fw.numel(),
                  p(t["dy"]), None, p(self.dqkv), p(self.da), p(self.db), p(self.dA),
                  p(self.ddt), p(self.dz), p(self.dnw), None, p(bw), bw.numel(), s)
        _abi.call("gdn_conv1d_silu_bwd", d, cu, cuh, p(t["x"]), p(t["conv_w"]), None,
                  p(self.dqkv), p(self.dx), p(self.dw), None, p(cw), cw.numel(), s)

    def outputs(self):
        return [self.y, self.dx, self.dw, self.da, self.db, self.dA, self.ddt, self.dz, self.dnw]

    INPUTS = ["x", "conv_w", "a", "b", "A_log", "dt_bias", "z", "norm_w", "dy", "cu_seqlens"]


# Measured DRAM bytes (read + write) per launch on the 64k-token workload:
# dram__bytes_read.sum + dram__bytes_write.sum of each kernel from one ncu
# capture of the first 8192 tokens, times 8 (every kernel's work is
# proportional to the chunks it processes).  Valid for the kernels as captured;
# a kernel changed since then reports null.
TRAFFIC_64K = {
    "conv_fwd": 3618197504,
    "gates": 12664832,
    "chunk_prep": 6525761536,
    "chunk_state_fwd": 13307377664,
    "chunk_out_fwd": 8944007168,
    "chunk_norm_bwd": 5314086912,
    "chunk_bwd_local": 4016205824,
    "chunk_bwd_state": 10369161216,
    "chunk_bwd_dp": 7217242112,
    "chunk_bwd_sfacing": 17421240320,
    "chunk_bwd_wy": 10134188032,
    "gva_sum": 9022685184,
    "conv_bwd": 5592219648,
}


def kernel_cost(name: str, w: synth.Workload, NT: int):
    """Algorithmic bytes of one launch of a kernel: the tensors its interface
    must read and write, each once.  Notation: io = bytes per activation,
    tk = one [T, H_k, d] fp32 tensor, tv = one [T, H_v, d] fp32 tensor (or the
    same bytes as per-chunk tiles), S = per-chunk states [NT, H_v, d, d] fp32,
    Tt = per-chunk 64 x 64 tiles [NT, H_v] fp32, g = [T, H_v] fp32,
    act = [T, H_v, d] in the I/O dtype."""
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
        "chunk_state_fwd": 2 * tv + tk + g + tv + 2 * S,
        "chunk_out_fwd": 2 * tk + tv + S + g + act + act + tv + g,
        "chunk_norm_bwd": tv + 2 * act + tv + act,
        "chunk_bwd_local": 2 * tk + tv + g + tv,
        "chunk_bwd_state": 2 * tk + 3 * tv + g + tv + S,
        "chunk_bwd_sfacing": 2 * S + 3 * tv + 2 * tk + g + 3 * tv + g,
        "chunk_bwd_dp": 2 * tk + 2 * tv + g + 2 * tv + 2 * g,
        "chunk_bwd_wy": tk + tv + 2 * tv + 2 * Tt + 3 * g + gates + 2 * tv + gates + g,
        "gva_sum": 5 * tv + 2 * tk,
    }
    return "hbm", table.get(name), "B"


def run_ours(args, rank, world, dev):
    w = synth.WORKLOADS[args.workload]
    w = w.replace(seed=w.seed + 1000 * rank)
    if args.tokens:
        w = w.replace(name=f"{w.name}[first {args.tokens} tokens]", seq_lens=(args.tokens,))
    inp = synth.make_inputs(w, with_grad=True)
    step = Step(w, inp, dev)
    NT = sum((L + 63) // 64 for L in w.seq_lens)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _abi.profile_report()
    with Clocks(dev.index if dev.index is not None else 0) as clk:
        launches0 = _abi.launch_count()
        _abi.profile_enable(True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        e1.synchronize()
        _abi.profile_enable(False)
        launches = _abi.launch_count() - launches0
    ms = e0.elapsed_time(e1) / args.steps
    prof = _abi.profile_report()
    torch.cuda.synchronize()
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
        torch.distributed.barrier()
    value = world * w.T / (ms / 1e3)

    # dominant kernel and its roofline
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        pass
    top = max(prof.items(), key=lambda kv: kv[1][1])
    name, (nl, tot_ms) = top
    avg_ms = tot_ms / nl
    bound, amount, unit = kernel_cost(name, w, NT)
    hbm_peak = peaks.get("hbm_gbs")
    peak_src = "measured" if hbm_peak else "fallback"
    hbm_peak = hbm_peak or 6800.0
    achieved = amount / (avg_ms / 1e3) / 1e9 if amount else None
    roof = {"kernel": name, "bound": bound, "achieved": achieved, "peak": hbm_peak,
            "unit": "GB/s", "frac": achieved / hbm_peak if achieved else None,
            "traffic": (TRAFFIC_64K.get(name) if args.workload == "qwen38_flash_64k"
                        and not args.tokens else None),
            "traffic_unit": "B per launch",
            "peak_source": peak_src, "avg_launch_ms": avg_ms,
            "step_share": tot_ms / sum(v[1] for v in prof.values())}
    path_bytes = w.T * (2 * w.C * 2 + 4 * w.h_v * 2 + 2 * w.h_v * D * 2) \
        + w.T * (2 * w.C * 2 + 2 * w.h_v * D * 2 + 2 * w.h_v * D * 2 + 4 * w.h_v * 2 +
                 w.C * 2)
    kernels = {k: {"launches": v[0], "ms_per_step": v[1] / args.steps} for k, v in prof.items()}

    # end to end: pinned host inputs -> device, step, results -> pinned host
    e2e = None
    if not args.no_e2e and rank == 0 or (not args.no_e2e and world > 1):
        host_in = {k: inp[k].pin_memory() for k in Step.INPUTS}
        host_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in step.outputs()]
        h2d = sum(v.numel() * v.element_size() for v in host_in.values())
        d2h = sum(o.numel() * o.element_size() for o in host_out)
        torch.cuda.synchronize()
        e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2.record(stream)
        for _ in range(args.e2e_steps):
            for k, v in host_in.items():
                step.t[k].copy_(v, non_blocking=True)
            step()
            for h, o in zip(host_out, step.outputs()):
                h.copy_(o, non_blocking=True)
        e3.record(stream)
        e3.synchronize()
        e2e_ms = e2.elapsed_time(e3) / args.e2e_steps
        if world > 1:
            t = torch.tensor([e2e_ms], device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            e2e_ms = float(t.item())
        e2e = {"value": world * w.T / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_tokens)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "tokens": w.T, "seqs": w.N, "h_k": w.h_k,
                       "h_v": w.h_v, "d_k": D, "d_v": D, "chunk": 64, "conv_k": 4,
                       "io": w.io, "state": "fp32",
                       "mma": "tf32 tcgen05 (chunk kernels, reverse state pass), "
                              "tf32 mma.sync (forward state pass)",
                       "qkv": "conv output stored at tf32 precision",
                       "passes": "fwd+bwd (conv, chunk rule, fused gated norm)",
                       "l2": "inputs larger than L2 (x alone is %.2f GB)" % (
                           w.T * w.C * 2 / 1e9),
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": roof,
            "path_roofline": {"bound": "hbm", "algorithmic_bytes_per_step": path_bytes,
                              "achieved_gbs": path_bytes / (ms / 1e3) / 1e9,
                              "frac": path_bytes / (ms / 1e3) / 1e9 / hbm_peak},
            "kernels": kernels,
            "gpu_launches": launches,
            "clocks": clk.summary(),
            "e2e": e2e,
            "cpu_baseline": cpu,
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
    oracle.backward(**args, dy=dy)
    dt = time.perf_counter() - t0
    return {"value": tokens / dt, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"fp64 oracle fwd+bwd of all {w.h_v} v-heads over the first {tokens} "
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

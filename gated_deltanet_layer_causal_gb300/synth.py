"""Seeded synthetic inputs for the GDN core.

This module holds no arithmetic of the method: it only draws random tensors
with the shapes and value distributions of the workloads and rounds them to
the I/O dtype.  Both the CUDA path and the fp64 oracle are fed from here, so
they read bit-identical inputs (the oracle widens the rounded values to fp64).

Distributions (per workload): x ~ N(0, 1) over the flat [q | k | v] conv
channels; conv weight ~ U(-0.5, 0.5); a, b ~ N(0, 1); A_log = ln U(1, 16);
dt_bias = 0; z ~ N(0, 1); norm weight ~ N(0, 0.02); zero initial state;
output gradients ~ N(0, 1).  Random numbers come from numpy's PCG64, which
gives the same stream on x86 and Arm.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seq_lens: tuple          # lengths of the packed sequences
    h_k: int
    h_v: int
    d: int = 128
    conv_k: int = 4
    io: str = "bf16"         # activation dtype: "bf16" or "fp32"
    backward: bool = False
    seed: int = 0
    dt_bias: float = 0.0

    @property
    def T(self) -> int:
        return int(sum(self.seq_lens))

    @property
    def N(self) -> int:
        return len(self.seq_lens)

    @property
    def C(self) -> int:
        return 2 * self.h_k * self.d + self.h_v * self.d

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.io == "bf16" else torch.float32

    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seq_lens)]).astype(np.int32)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def varlen_lengths(n: int, total: int, lo: int, hi: int, seed: int) -> tuple:
    """n lengths drawn log-uniform in [lo, hi], rescaled to sum to ``total``.

    Draw u_i ~ U(ln lo, ln hi), L_i = e^{u_i}; scale by total / sum(L), floor,
    then add one to the first (total - sum) lengths.  After rescaling a length
    may leave [lo, hi] slightly."""
    rng = np.random.default_rng(seed)
    L = np.exp(rng.uniform(math.log(lo), math.log(hi), size=n))
    L = np.floor(L * (total / L.sum())).astype(np.int64)
    L[: total - int(L.sum())] += 1
    assert int(L.sum()) == total
    return tuple(int(v) for v in L)


# The five workloads: a tiny fp32 forward, the Qwen3.5-9B-shaped forward
# (16 k-heads / 32 v-heads), the Qwen3.8-Flash-shaped forward+backward at 64k
# (16 / 48), a 64-sequence varlen batch at 128k and a 128k long-context run
# (with a 256-wide decode batch).
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", (512,), 2, 4, io="fp32", seed=0),
    "qwen35_9b_16k": Workload("qwen35_9b_16k", (16384,), 16, 32, seed=1),
    "qwen38_flash_64k": Workload("qwen38_flash_64k", (65536,), 16, 48, backward=True, seed=2),
    "varlen64_128k": Workload("varlen64_128k", varlen_lengths(64, 131072, 256, 8192, 3), 16, 32,
                              backward=True, seed=3),
    "long_128k": Workload("long_128k", (131072,), 16, 48, backward=True, seed=4),
}
DECODE_BATCH = 256


def _round(a: np.ndarray, dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dtype)


def make_inputs(w: Workload, with_grad: bool | None = None) -> dict:
    """Draw one batch of inputs for workload ``w`` as CPU torch tensors.

    Activations (x, a, b, z, dy) are in the I/O dtype; parameters (conv_w,
    A_log, dt_bias, norm_w) are fp32; cu_seqlens is int32."""
    rng = np.random.default_rng(w.seed)
    T, C, H, d = w.T, w.C, w.h_v, w.d
    dt = w.torch_dtype
    out = {
        "x": _round(rng.standard_normal((T, C), dtype=np.float32), dt),
        "conv_w": _round(rng.uniform(-0.5, 0.5, size=(C, w.conv_k)), torch.float32),
        "a": _round(rng.standard_normal((T, H), dtype=np.float32), dt),
        "b": _round(rng.standard_normal((T, H), dtype=np.float32), dt),
        "A_log": _round(np.log(rng.uniform(1.0, 16.0, size=H)), torch.float32),
        "dt_bias": torch.full((H,), float(w.dt_bias), dtype=torch.float32),
        "z": _round(rng.standard_normal((T, H, d), dtype=np.float32), dt),
        "norm_w": _round(rng.normal(0.0, 0.02, size=d), torch.float32),
        "cu_seqlens": torch.from_numpy(w.cu_seqlens()),
    }
    if with_grad if with_grad is not None else w.backward:
        out["dy"] = _round(rng.standard_normal((T, H, d), dtype=np.float32), dt)
    return out


def make_state(n: int, h_v: int, d: int, seed: int, scale: float = 0.1) -> torch.Tensor:
    """Random fp32 recurrent states [n, h_v, d_v, d_k] ~ N(0, scale^2)."""
    rng = np.random.default_rng(seed)
    return torch.from_numpy(rng.standard_normal((n, h_v, d, d), dtype=np.float32) * scale)


def make_conv_state(n: int, C: int, k: int, seed: int, dtype) -> torch.Tensor:
    """Random conv caches [n, C, k-1] ~ N(0, 1) in the I/O dtype."""
    rng = np.random.default_rng(seed)
    return _round(rng.standard_normal((n, C, k - 1), dtype=np.float32), dtype)


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Widen a (rounded) tensor to a float64 numpy array for the oracle."""
    return t.detach().to("cpu", torch.float64).numpy()

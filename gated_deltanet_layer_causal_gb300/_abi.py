"""ctypes view of libgdn.so's C ABI (include/gdn.h).  Marshalling only.

The library is loaded on first use.  If it is missing, every call raises: there
is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libgdn.so")

# status codes (gdn_status)
GDN_OK = 0
GDN_ERR_INVALID_ARG = 1
GDN_ERR_UNSUPPORTED = 2
GDN_ERR_WORKSPACE = 3
GDN_ERR_CUDA = 4
GDN_ERR_DEVICE_TIMEOUT = 5
GDN_ERR_DEVICE_CHECK = 6
# dtypes (gdn_dtype)
GDN_F32 = 0
GDN_BF16 = 1
# output gates (gdn_gate) and channel layouts (gdn_layout)
GDN_GATE_SILU = 0
GDN_GATE_SIGMOID = 1
GDN_LAYOUT_FLAT = 0
GDN_LAYOUT_GROUP = 1
GATES = {"silu": GDN_GATE_SILU, "sigmoid": GDN_GATE_SIGMOID}
LAYOUTS = {"flat": GDN_LAYOUT_FLAT, "group": GDN_LAYOUT_GROUP}
# workspace kinds
GDN_WS_FWD = 0
GDN_WS_BWD = 1
GDN_WS_CONV_BWD = 2
GDN_WS_NORM_BWD = 3
# rows (tokens * v-heads) gdn_gated_rmsnorm_bwd_noalloc accepts
GDN_NOALLOC_NORM_BWD_MAX_ROWS = 524288


# GDN_ABI_VERSION of include/gdn.h that GdnDims and SIGNATURES mirror
ABI_VERSION = 300


class GdnDims(ctypes.Structure):
    """Mirror of gdn_dims."""
    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("total_tokens", ctypes.c_int64),
        ("h_k", ctypes.c_int32),
        ("h_v", ctypes.c_int32),
        ("d_k", ctypes.c_int32),
        ("d_v", ctypes.c_int32),
        ("conv_k", ctypes.c_int32),
        ("chunk", ctypes.c_int32),
        ("io_dtype", ctypes.c_int32),
        ("l2_eps", ctypes.c_float),
        ("norm_eps", ctypes.c_float),
        ("qkv_tf32", ctypes.c_int32),
        ("gate", ctypes.c_int32),
        ("layout", ctypes.c_int32),
    ]


_P = ctypes.c_void_p
_S = ctypes.c_size_t
_DP = ctypes.POINTER(GdnDims)

# name -> argtypes (every entry point returns gdn_status as int)
SIGNATURES = {
    "gdn_workspace_size": [_DP, _P, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)],
    "gdn_conv1d_silu": [_DP, _P, _P, _P, _P, _P, _P, _P, _P],
    "gdn_conv1d_silu_bwd": [_DP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _S, _P],
    "gdn_chunk_fwd": [_DP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _S, _P],
    "gdn_chunk_bwd": [_DP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _S, _P, _P, _P, _P, _P,
                      _P, _P, _P, _P, _P, _P, _S, _P],
    "gdn_gated_rmsnorm": [_DP, _P, _P, _P, _P, _P, _P],
    "gdn_gated_rmsnorm_bwd": [_DP, _P, _P, _P, _P, _P, _P, _P, _P, _S, _P],
    "gdn_gated_rmsnorm_bwd_noalloc": [_DP, _P, _P, _P, _P, _P, _P, _P, _P],
    "gdn_recurrent_step": [_DP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "gdn_read_status": [_P, ctypes.POINTER(ctypes.c_int32), _P],
    "gdn_selftest_bounded_wait": [_P, _S, ctypes.c_int32, ctypes.c_int32, _P],
    "gdn_profile_enable": [ctypes.c_int32],
    "gdn_profile_report": [ctypes.c_char_p, _S],
}

_lib = None


def load():
    """Load libgdn.so (built by ``build.py``); raise if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"libgdn.so not found at {LIB_PATH}: build it with "
            "`python -m gated_deltanet_layer_causal_gb300.build` (there is no fallback path)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, args in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.gdn_status_string.argtypes = [ctypes.c_int]
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_launch_count.argtypes = []
    lib.gdn_launch_count.restype = ctypes.c_int64
    lib.gdn_abi_version.argtypes = []
    lib.gdn_abi_version.restype = ctypes.c_int32
    if lib.gdn_abi_version() != ABI_VERSION:
        raise RuntimeError(f"libgdn.so at {LIB_PATH} has ABI {lib.gdn_abi_version()}, this "
                           f"binding expects {ABI_VERSION}: rebuild it")
    _lib = lib
    return lib


class GdnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        name = load().gdn_status_string(status).decode()
        super().__init__(f"{fn} failed: {name} ({status})")
        self.status = status


def call(name: str, *args) -> None:
    """Call entry point ``name`` and raise GdnError on a non-OK status."""
    st = getattr(load(), name)(*args)
    if st != GDN_OK:
        raise GdnError(name, st)


def dims(num_seqs, total_tokens, h_k, h_v, io_bf16, l2_eps=1e-6, norm_eps=1e-6, d=128,
         conv_k=4, chunk=64, qkv_tf32=False, gate="silu", layout="flat") -> GdnDims:
    """gate: "silu" | "sigmoid" (output gate of the gated norm); layout: "flat" |
    "group" (q/k/v channel order of x, conv_w and the conv states)."""
    return GdnDims(int(num_seqs), int(total_tokens), int(h_k), int(h_v), d, d, conv_k, chunk,
                   GDN_BF16 if io_bf16 else GDN_F32, float(l2_eps), float(norm_eps),
                   1 if qkv_tf32 else 0, GATES[gate], LAYOUTS[layout])


def launch_count() -> int:
    """Kernel launches made by libgdn.so in this process."""
    return int(load().gdn_launch_count())


def profile_enable(on: bool) -> None:
    call("gdn_profile_enable", 1 if on else 0)


def profile_report() -> dict:
    """{kernel name: (timed launches, total ms)} since the last report."""
    buf = ctypes.create_string_buffer(1 << 16)
    call("gdn_profile_report", buf, len(buf))
    out = {}
    for line in buf.value.decode().splitlines():
        name, n, ms = line.split()
        out[name] = (int(n), float(ms))
    return out

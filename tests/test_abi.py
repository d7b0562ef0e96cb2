"""The C-ABI library builds, loads and exports every symbol include/gdn.h
declares; host-side validation rejects bad input before any launch.  No GPU:
only entry points that fail validation (and so never touch CUDA) are called."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

from gated_deltanet_layer_causal_gb300 import _abi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _abi.load()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_core_entry_points():
    names = _declared()
    for n in ("gdn_conv1d_silu", "gdn_chunk_fwd", "gdn_chunk_bwd", "gdn_gated_rmsnorm",
              "gdn_recurrent_step"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert lib.gdn_abi_version() == _abi.ABI_VERSION


def test_status_strings(lib):
    for code in range(7):
        s = lib.gdn_status_string(code).decode()
        assert s.startswith("GDN_")


def _ws(lib, d, cu, kind):
    n = ctypes.c_size_t(0)
    cu_t = torch.tensor(cu, dtype=torch.int32)
    st = lib.gdn_workspace_size(ctypes.byref(d), ctypes.c_void_p(cu_t.data_ptr()), kind,
                                ctypes.byref(n))
    return st, n.value


def test_workspace_sizes(lib):
    d = _abi.dims(2, 130, 2, 4, True)
    st, fwd = _ws(lib, d, [0, 65, 130], _abi.GDN_WS_FWD)
    assert st == 0
    # 4 chunks (2 per sequence): the per-chunk states alone are 4 * 4 * 128 * 128 * 4 bytes
    assert fwd >= 4 * 4 * 128 * 128 * 4 + 3 * 130 * 4 * 128 * 4
    st, bwd = _ws(lib, d, [0, 65, 130], _abi.GDN_WS_BWD)
    assert st == 0 and bwd > fwd / 2
    st, _ = _ws(lib, d, [0, 65, 130], _abi.GDN_WS_CONV_BWD)
    assert st == 0


def test_dims_struct_layout_matches_the_header(tmp_path):
    """ctypes' GdnDims has gdn_dims' size and field offsets (gcc on the header)."""
    fields = [f for f, _ in _abi.GdnDims._fields_]
    src = tmp_path / "layout.c"
    src.write_text(
        "#include <stddef.h>\n#include <stdio.h>\n#include \"gdn.h\"\n"
        "int main(void) {\n  printf(\"%zu\", sizeof(gdn_dims));\n"
        + "".join(f'  printf(" %zu", offsetof(gdn_dims, {f}));\n' for f in fields)
        + "  printf(\" %d\\n\", GDN_ABI_VERSION);\n  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)],
                   check=True)
    out = [int(v) for v in subprocess.run([str(exe)], check=True, capture_output=True,
                                          text=True).stdout.split()]
    assert out[0] == ctypes.sizeof(_abi.GdnDims)
    assert out[1:-1] == [getattr(_abi.GdnDims, f).offset for f in fields]
    assert out[-1] == _abi.ABI_VERSION


@pytest.mark.parametrize("cu,why", [([0, 70, 60], "decreasing"), ([1, 65, 130], "cu[0] != 0"),
                                    ([0, 65, 129], "cu[N] != T")])
def test_bad_cu_seqlens_rejected(lib, cu, why):
    d = _abi.dims(2, 130, 2, 4, True)
    st, _ = _ws(lib, d, cu, _abi.GDN_WS_FWD)
    assert st == _abi.GDN_ERR_INVALID_ARG, why


@pytest.mark.parametrize("field,value,code", [
    ("d_k", 64, _abi.GDN_ERR_UNSUPPORTED), ("conv_k", 3, _abi.GDN_ERR_UNSUPPORTED),
    ("chunk", 32, _abi.GDN_ERR_UNSUPPORTED), ("h_v", 5, _abi.GDN_ERR_INVALID_ARG),
    ("io_dtype", 7, _abi.GDN_ERR_UNSUPPORTED), ("h_k", 0, _abi.GDN_ERR_INVALID_ARG),
    ("qkv_tf32", 2, _abi.GDN_ERR_INVALID_ARG)])
def test_bad_dims_rejected(lib, field, value, code):
    d = _abi.dims(1, 64, 2, 4, True)
    setattr(d, field, value)
    st, _ = _ws(lib, d, [0, 64], _abi.GDN_WS_FWD)
    assert st == code


def test_null_and_misaligned_pointers_rejected_before_launch(lib):
    d = _abi.dims(1, 64, 2, 4, True)
    cu = torch.tensor([0, 64], dtype=torch.int32)
    P = ctypes.c_void_p
    st = lib.gdn_conv1d_silu(ctypes.byref(d), P(16), P(cu.data_ptr()), None, P(16), None, P(16),
                             None, None)
    assert st == _abi.GDN_ERR_INVALID_ARG
    st = lib.gdn_conv1d_silu(ctypes.byref(d), P(16), P(cu.data_ptr()), P(8), P(16), None, P(16),
                             None, None)
    assert st == _abi.GDN_ERR_INVALID_ARG
    # missing workspace
    st = lib.gdn_chunk_fwd(ctypes.byref(d), P(16), P(cu.data_ptr()), P(16), P(16), P(16), P(16),
                           P(16), None, None, None, P(16), None, None, None, 0, None)
    assert st == _abi.GDN_ERR_WORKSPACE
    # decode step wants total_tokens == num_seqs
    d2 = _abi.dims(4, 5, 2, 4, True)
    st = lib.gdn_recurrent_step(ctypes.byref(d2), *([P(16)] * 10), None, P(16), None)
    assert st == _abi.GDN_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_abi, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_abi, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        _abi.load()


def test_binding_rejects_a_library_of_another_abi(lib, monkeypatch):
    monkeypatch.setattr(_abi, "ABI_VERSION", _abi.ABI_VERSION + 1)
    monkeypatch.setattr(_abi, "_lib", None)
    with pytest.raises(RuntimeError, match="rebuild"):
        _abi.load()

"""The device-side failure path: a bounded mbarrier wait that gives up sets
GDN_ERR_DEVICE_TIMEOUT in the workspace status word and returns, leaving the
context usable (gdn_selftest_bounded_wait runs that path on purpose with
nothing in flight).  Argument checks run without a GPU."""
import ctypes

import pytest
import torch

import oracle
from gated_deltanet_layer_causal_gb300 import _abi, core, synth
from gdn_testutil import check_against, full_args, gpu_run


def _wait(ws, limit, arrive):
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    _abi.call("gdn_selftest_bounded_wait", ctypes.c_void_p(ws.data_ptr()), ws.numel(), limit,
              arrive, s)


@pytest.mark.gpu
def test_bounded_wait_gives_up_and_reports_timeout():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    _wait(ws, 1000, 0)   # nothing completes the barrier: the wait runs out
    assert core.read_status(ws) == _abi.GDN_ERR_DEVICE_TIMEOUT
    assert core.read_status(ws) == 0   # the read cleared it
    _wait(ws, 1000, 1)   # the barrier completes: no timeout
    assert core.read_status(ws) == 0
    # the context is still usable: a small forward + backward matches the oracle
    w = synth.Workload("after", (130,), 1, 2, io="bf16", backward=True, seed=37, dt_bias=-4.0)
    inp = synth.make_inputs(w)
    out = gpu_run(inp, w, backward=True)
    assert out["status_fwd"] == 0
    ref = oracle.backward(**full_args(inp, w), dy=synth.to_f64(inp["dy"]))
    check_against(out, ref, True, tag="after a timeout")


def test_selftest_argument_checks():
    lib = _abi.load()
    P = ctypes.c_void_p
    assert lib.gdn_selftest_bounded_wait(None, 64, 10, 0, None) == _abi.GDN_ERR_INVALID_ARG
    assert lib.gdn_selftest_bounded_wait(P(16), 2, 10, 0, None) == _abi.GDN_ERR_INVALID_ARG
    assert lib.gdn_selftest_bounded_wait(P(8), 64, 10, 0, None) == _abi.GDN_ERR_INVALID_ARG
    assert lib.gdn_selftest_bounded_wait(P(16), 64, 0, 0, None) == _abi.GDN_ERR_INVALID_ARG
    assert lib.gdn_selftest_bounded_wait(P(16), 64, (1 << 24) + 1, 0, None) == \
        _abi.GDN_ERR_INVALID_ARG
    assert lib.gdn_selftest_bounded_wait(P(16), 64, 10, 2, None) == _abi.GDN_ERR_INVALID_ARG

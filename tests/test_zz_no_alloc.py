"""The allocation-free conv2d entry point, fc_conv2d_epi_noalloc.

It serves callers that cannot allocate device memory (host callbacks,
allocator hooks, allocation-free real-time paths, plug-ins whose host owns the
memory pool): instead of a caller-provided workspace it uses a fixed 1 MiB
device array inside the library.  These tests call it through the C ABI and
check it against fc_conv2d_epi (which takes a workspace) at the suite's
tolerance, atol = rtol = 1e-4, on two calls in a row with different inputs --
the second call runs on whatever the first left in the shared array.  The
file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

from convolution_epilogue_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-4


def _fc():
    from convolution_epilogue_gb300 import _build
    _build.build()
    import convolution_epilogue_gb300 as fc
    return fc


def _close(got, ref, what):
    got = got.double().cpu().numpy()
    ref = ref.double().cpu().numpy()
    err = np.abs(got - ref)
    ok = err <= ATOL + RTOL * np.abs(ref)
    assert ok.all(), f"{what}: {(~ok).sum()} outputs differ (max abs err {err.max():.3g})"


def _case(seed, shape, cout, ops_kind):
    st = synth.seeded(seed)
    N, C, H, W = shape
    bound = 1.0 / np.sqrt(9 * C)
    x = torch.from_numpy(st.normal(shape)).cuda()
    w = torch.from_numpy(st.uniform((cout, C, 3, 3), bound)).cuda()
    b = torch.from_numpy(st.uniform((cout,), bound)).cuda()
    if ops_kind == "rh":
        ops = (("relu",), ("hardswish",))
    else:
        s = torch.from_numpy(st.normal((cout,))).cuda()
        ops = (("leaky_relu", 0.2), ("add_channel", s), ("clamp", -1.0, 1.0), ("gelu_erf",))
    return x, w, b, ops


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    fc = _fc()
    cases = [
        _case(901, (4, 8, 32, 32), 64, "rh"),     # the small conv2d workload's shape
        _case(902, (2, 12, 21, 150), 70, "gelu"),  # different shape, C_out > 64, wide rows
    ]
    for i, (x, w, b, ops) in enumerate(cases):
        N, C, H, W = x.shape
        CO = w.shape[0]
        y = torch.full((N, CO, H - 2, W - 2), float("nan"), device="cuda")
        fc.fc_conv2d_epi_noalloc(x, w, y, b, ops)
        ref = fc.fc_conv2d_epi(x, w, b, ops)
        torch.cuda.synchronize()
        assert fc.get_last_device_error() == 0
        _close(y, ref, f"call {i + 1}")


def test_noalloc_refuses_shapes_beyond_its_array():
    fc = _fc()
    L = fc.lib()
    # 256 -> 256 channels need well over 1 MiB of packed weights
    x = torch.zeros((1, 256, 8, 8), device="cuda")
    w = torch.zeros((256, 256, 3, 3), device="cuda")
    y = torch.zeros((1, 256, 6, 6), device="cuda")
    assert fc.workspace_bytes(0, (1, 256, 8, 8, 256, 3, 0)) > (1 << 20)
    e, _keep = fc.make_epilogue(None, ())
    st = L.fc_conv2d_epi_noalloc(ctypes.c_void_p(x.data_ptr()), 1, 256, 8, 8,
                                 ctypes.c_void_p(w.data_ptr()), 256, 3, 3, 1, 0, 1,
                                 ctypes.byref(e), ctypes.c_void_p(y.data_ptr()), None)
    assert st == 4  # FC_ERR_WORKSPACE
    assert L.fc_status_string(st).decode().startswith("FC_ERR_WORKSPACE")

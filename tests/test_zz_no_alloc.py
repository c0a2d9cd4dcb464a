"""The allocation-free conv2d entry point, fc_conv2d_epi_noalloc.

It serves callers that cannot allocate device memory (host callbacks,
allocator hooks, allocation-free real-time paths, plug-ins whose host owns the
memory pool): instead of a caller-provided workspace it uses a fixed 1 MiB
device array inside the library.  These tests call it through the C ABI, on
two calls in a row with different inputs -- the second call runs on whatever
the first left in the shared array -- for the CUDA-core variant and both
tensor-core variants (whose packed weights then live in that array), and
check each call against the CPU oracle and against fc_conv2d_epi (which takes
a workspace) at the suite's tolerance, atol = rtol = 1e-4.  A second test
checks that, once every kernel involved has been loaded, the calls leave the
device's free memory unchanged.  The file is named so that pytest collects it
last.
"""
import ctypes

import numpy as np
import pytest

import oracle
from convolution_epilogue_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-4
VARIANTS = ["ffma", "tc_tf32x3", "tc_f16x3"]


def _fc():
    from convolution_epilogue_gb300 import _build
    _build.build()
    import convolution_epilogue_gb300 as fc
    return fc


def _close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    ok = err <= ATOL + RTOL * np.abs(ref)
    assert ok.all(), f"{what}: {(~ok).sum()} outputs differ (max abs err {err.max():.3g})"


def _case(seed, shape, cout, ops_kind, pad):
    """Host inputs, their device copies and the oracle's result."""
    st = synth.seeded(seed)
    N, C, H, W = shape
    bound = 1.0 / np.sqrt(9 * C)
    x = st.normal(shape)
    w = st.uniform((cout, C, 3, 3), bound)
    b = st.uniform((cout,), bound)
    if ops_kind == "rh":
        ops_h = ops_d = (("relu",), ("hardswish",))
    else:
        s = st.normal((cout,))
        ops_h = (("leaky_relu", 0.2), ("add_channel", s), ("clamp", -1.0, 1.0), ("gelu_erf",))
        ops_d = (("leaky_relu", 0.2), ("add_channel", torch.from_numpy(s).cuda()),
                 ("clamp", -1.0, 1.0), ("gelu_erf",))
    ref = oracle.conv_epi(x, w, b, ops_h, pad=pad)
    d = dict(x=torch.from_numpy(x).cuda(), w=torch.from_numpy(w).cuda(),
             b=torch.from_numpy(b).cuda(), ops=ops_d, pad=pad, ref=ref)
    d["y"] = torch.full(ref.shape, float("nan"), dtype=torch.float32, device="cuda")
    return d


def _cases():
    return [
        _case(901, (4, 8, 32, 32), 64, "rh", 0),      # the small conv2d workload's shape
        _case(902, (2, 12, 21, 150), 70, "gelu", 1),  # C_in 12, C_out > 64, 128-column strips
    ]


def test_noalloc_matches_oracle_and_workspace_entry_on_two_calls_in_a_row():
    fc = _fc()
    fc.profile_enable(False)
    cases = _cases()
    try:
        for v in VARIANTS:
            fc.set_variant(v)
            for i, c in enumerate(cases):
                c["y"].fill_(float("nan"))
                fc.fc_conv2d_epi_noalloc(c["x"], c["w"], c["y"], c["b"], c["ops"], pad=c["pad"])
                assert fc.last_variant() == v
                ref_ws = fc.fc_conv2d_epi(c["x"], c["w"], c["b"], c["ops"], pad=c["pad"])
                torch.cuda.synchronize()
                assert fc.get_last_device_error() == 0
                got = c["y"].cpu().numpy()
                _close(got, c["ref"], f"[{v}] call {i + 1} vs the oracle")
                _close(got, ref_ws.cpu().numpy().astype(np.float64),
                       f"[{v}] call {i + 1} vs fc_conv2d_epi")
    finally:
        fc.set_variant("auto")


def test_noalloc_calls_allocate_nothing():
    """After one round of calls has looked up the array's address and
    loaded every kernel involved, further calls on preallocated tensors
    leave the device's free memory where it was."""
    fc = _fc()
    fc.profile_enable(False)
    cases = _cases()
    try:
        for v in VARIANTS:  # warm-up round: address look-up and kernel loading
            fc.set_variant(v)
            for c in cases:
                fc.fc_conv2d_epi_noalloc(c["x"], c["w"], c["y"], c["b"], c["ops"], pad=c["pad"])
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        for v in VARIANTS:
            fc.set_variant(v)
            for c in cases:
                c["y"].fill_(float("nan"))
                fc.fc_conv2d_epi_noalloc(c["x"], c["w"], c["y"], c["b"], c["ops"], pad=c["pad"])
            torch.cuda.synchronize()
            free1, _ = torch.cuda.mem_get_info()
            assert free1 == free0, f"[{v}] free device memory moved by {free0 - free1} bytes"
            for i, c in enumerate(cases):
                _close(c["y"].cpu().numpy(), c["ref"], f"[{v}] call {i + 1}")
        assert fc.get_last_device_error() == 0
    finally:
        fc.set_variant("auto")


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

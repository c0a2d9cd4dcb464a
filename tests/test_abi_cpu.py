"""C-ABI checks that need no GPU: the library builds, loads, exports every
symbol include/fusedconv.h declares, and rejects bad arguments on the host
before it touches the device."""
import ctypes
import os
import re

import pytest

import convolution_epilogue_gb300 as fc
from convolution_epilogue_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include",
                      "fusedconv.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return fc.lib()


def _declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"FC_API\s+[\w\s\*]+?\b(fc_\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("fc_conv2d_epi", "fc_conv3d_epi", "fc_convT2d_pool_mean"):
        assert n in names
    assert sorted(fc.EXPORTS) == names


def test_every_declared_symbol_is_exported(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_status_strings(L):
    for code, name in fc.STATUS_NAMES.items():
        assert L.fc_status_string(code).decode().startswith(name)
    assert L.fc_version() >= 100


def test_workspace_sizes(L):
    w0 = fc.workspace_bytes(0, (128, 8, 128, 128, 64, 3, 0))
    w1 = fc.workspace_bytes(1, (128, 8, 16, 64, 64, 64, 3, 0))
    w2 = fc.workspace_bytes(2, (128, 64, 256, 256, 64, 3, 1))
    assert w0 >= 8 * 9 * 64 * 4 and w0 % 256 == 0
    assert w1 >= 8 * 27 * 64 * 4 and w1 % 256 == 0
    # w2 holds the packed weights and one fp32 partial per (n, tile, c_out)
    assert w2 >= 64 * 9 * 64 * 4 + 128 * 64 * 4
    assert fc.workspace_bytes(7, (1, 1, 1, 1, 1, 3, 0)) == 0


def _epi(ops=()):
    e, keep = fc.make_epilogue(None, ops)
    return e, keep


def _conv2d(L, N=1, C=8, H=8, W=8, CO=64, k=3, stride=1, pad=0, x=16, w=16,
            y=16, ops=(), ws=256, ws_bytes=1 << 20, dilation=1):
    e, _ = _epi(ops)
    return L.fc_conv2d_epi(ctypes.c_void_p(x), N, C, H, W, ctypes.c_void_p(w), CO,
                           k, k, stride, pad, dilation, ctypes.byref(e), ctypes.c_void_p(y),
                           ctypes.c_void_p(ws), ws_bytes, None)


def test_host_validation_rejects_before_launch(L):
    INVALID, UNSUP, ALIGN = 1, 2, 3
    assert _conv2d(L, N=-1) == INVALID
    assert _conv2d(L, C=0) == INVALID
    assert _conv2d(L, stride=0) == INVALID
    assert _conv2d(L, stride=5) == UNSUP  # strides 1 .. 4 are supported
    assert _conv2d(L, k=8) == UNSUP      # kernel sizes 1 .. 7
    assert _conv2d(L, k=9, H=20, W=20) == UNSUP
    assert _conv2d(L, pad=65) == UNSUP   # padding up to 64
    assert _conv2d(L, dilation=0) == INVALID
    assert _conv2d(L, dilation=5) == UNSUP  # dilations 1 .. 4
    assert _conv2d(L, stride=4, k=7, dilation=4, pad=3, H=30, W=30, N=0) == 0  # valid
    assert _conv2d(L, H=2) == INVALID  # Ho = 0
    assert _conv2d(L, H=4, dilation=2) == INVALID  # window of 5 rows over 4
    assert _conv2d(L, H=4, W=4, dilation=2, pad=1, N=0) == 0  # 6 padded rows: valid
    assert _conv2d(L, x=0) == INVALID  # NULL x
    assert _conv2d(L, x=18) == ALIGN
    assert _conv2d(L, ops=(("maxpool2x2",),)) == UNSUP
    assert _conv2d(L, ops=(("clamp", 1.0, -1.0),)) == INVALID
    assert _conv2d(L, N=0) == 0  # empty batch: nothing to launch


def test_pool_entry_requires_exact_chain(L):
    e, _ = _epi((("maxpool2x2",), ("hardtanh", -1, 1), ("tanh",)))
    st = L.fc_convT2d_pool_mean(ctypes.c_void_p(16), 1, 4, 8, 8, ctypes.c_void_p(16),
                                4, 3, 1, 1, 0, ctypes.byref(e), ctypes.c_void_p(16),
                                ctypes.c_void_p(256), 1 << 20, None)
    assert st == 2
    e, _ = _epi(fc.pool_mean_ops())
    st = L.fc_convT2d_pool_mean(ctypes.c_void_p(16), 1, 4, 8, 8, ctypes.c_void_p(16),
                                4, 3, 5, 1, 0, ctypes.byref(e), ctypes.c_void_p(16),
                                ctypes.c_void_p(256), 1 << 20, None)
    assert st == 2  # stride 5 is not supported (1 .. 4 are)
    st = L.fc_convT2d_pool_mean(ctypes.c_void_p(16), 1, 4, 8, 8, ctypes.c_void_p(16),
                                4, 3, 1, 1, 1, ctypes.byref(e), ctypes.c_void_p(16),
                                ctypes.c_void_p(256), 1 << 20, None)
    assert st == 1  # output padding must be below the stride
    st = L.fc_convT2d_pool_mean(ctypes.c_void_p(16), 1, 4, 8, 8, ctypes.c_void_p(16),
                                4, 8, 1, 1, 0, ctypes.byref(e), ctypes.c_void_p(16),
                                ctypes.c_void_p(256), 1 << 20, None)
    assert st == 2  # kernel sizes 1 .. 7


def test_no_cpu_fallback_without_gpu(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # a fully valid call cannot run anywhere but the GPU
    assert _conv2d(L) == 5  # FC_ERR_CUDA


def test_set_variant(L):
    assert L.fc_set_variant(9) == 1
    for v in range(4):
        assert L.fc_set_variant(v) == 0
    assert L.fc_set_variant(0) == 0


def test_pool_mean_tail_host_validation(L):
    """The standalone tail rejects bad extents, windows and clamps on the
    host, before any CUDA call (no GPU here)."""
    import ctypes
    P = ctypes.c_void_p

    def call(N=2, C=3, H=8, W=8, k=2, s=2, lo=-1.0, hi=1.0, x=256, y=512):
        return L.fc_pool_mean_tail(P(x), N, C, H, W, k, s, ctypes.c_float(lo),
                                   ctypes.c_float(hi), P(y), None)
    L.fc_pool_mean_tail.restype = ctypes.c_int
    L.fc_pool_mean_tail.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                    P, P]
    INVALID = 1
    assert call(N=-1) == INVALID
    assert call(C=0) == INVALID
    assert call(k=0) == INVALID
    assert call(s=0) == INVALID
    assert call(k=9) == INVALID          # window wider than the plane
    assert call(lo=1.0, hi=-1.0) == INVALID
    assert call(x=0) == INVALID          # NULL with N > 0
    assert call(N=0) == 0                # nothing to do


def test_general_pool_chain_validation(L):
    """The pooled entry's general max pool: window and stride integers in
    1..4, stride-1 transposed conv only; the op is refused by the elementwise
    entries.  All rejected on the host before any device work."""
    UNSUP = 2
    assert _conv2d(L, ops=(("maxpool", 3.0, 2.0),)) == UNSUP

    def pool_call(pool, stride=1, out_pad=0):
        e, _ = _epi(fc.pool_mean_ops(pool=pool))
        return L.fc_convT2d_pool_mean(ctypes.c_void_p(16), 1, 4, 8, 8, ctypes.c_void_p(16),
                                      4, 3, stride, 1, out_pad, ctypes.byref(e),
                                      ctypes.c_void_p(16), ctypes.c_void_p(256), 1 << 20, None)
    assert pool_call((5, 2)) == UNSUP      # window above 4
    assert pool_call((3, 0)) == UNSUP      # stride below 1
    assert pool_call((2.5, 2)) == UNSUP    # not an integer
    # workspace entry 3 (general pool) covers its per-tile partials, at any
    # supported stride / output padding
    assert fc.workspace_bytes(3, (2, 8, 20, 20, 64, 3, 1, 1, 0, 3, 2)) > 0
    assert fc.workspace_bytes(3, (2, 8, 20, 20, 64, 3, 1, 2, 1, 3, 2)) > 0
    assert fc.workspace_bytes(3, (2, 8, 20, 20, 64, 3, 1, 2, 2, 3, 2)) == 0  # out_pad >= stride


def test_binding_refuses_wrong_output_shapes_before_any_launch():
    """A caller-provided y (or bias / per-channel tensor) whose shape is not
    the one the call writes is refused by the binding with ValueError before
    it checks devices or calls the library: the kernels write every element
    of the call's output shape, so a smaller tensor would be overrun."""
    import torch
    x = torch.zeros((2, 8, 10, 12))
    w = torch.zeros((64, 8, 3, 3))
    bad = torch.zeros((2, 64, 10, 12))  # pad-1 extents, called with pad 0
    with pytest.raises(ValueError):
        fc.fc_conv2d_epi(x, w, None, (), pad=0, y=bad)
    with pytest.raises(ValueError):
        fc.fc_conv2d_epi_noalloc(x, w, bad, None, (), pad=0)
    with pytest.raises(ValueError):
        fc.fc_conv2d_epi(x, w, torch.zeros(32), (), pad=1)  # bias of 32 for C_out 64
    with pytest.raises(ValueError):
        fc.fc_conv2d_epi(x, w, None, (("add_channel", torch.zeros(63)),), pad=1)
    with pytest.raises(ValueError):
        fc.fc_conv2d_epi(x, w, None, (), stride=2, y=torch.zeros((2, 64, 5, 5)))
    x3 = torch.zeros((1, 8, 5, 6, 7))
    w3 = torch.zeros((16, 8, 3, 3, 3))
    with pytest.raises(ValueError):
        fc.fc_conv3d_epi(x3, w3, None, (), y=torch.zeros((1, 16, 3, 4, 6)))
    with pytest.raises(ValueError):
        fc.fc_conv2d_epi_nhwc(torch.zeros((1, 10, 12, 8)), w, None, (),
                              y=torch.zeros((1, 64, 8, 10)))  # channels-first y
    with pytest.raises(ValueError):
        fc.fc_conv3d_epi_ndhwc(torch.zeros((1, 5, 6, 7, 8)), w3, None, (),
                               y=torch.zeros((1, 3, 4, 5, 15)))
    wt = torch.zeros((8, 64, 3, 3))
    with pytest.raises(ValueError):
        fc.fc_convT2d_pool_mean(x, wt, None, y=torch.zeros((2, 63, 1, 1)))
    with pytest.raises(ValueError):
        fc.fc_pool_mean_tail(torch.zeros((2, 4, 8, 8)), y=torch.zeros((2, 4)))
    with pytest.raises(ValueError):
        fc.fc_conv2d_epi(torch.zeros((2, 8, 10)), w, None, ())  # rank 3 x
    # the right shapes get past the shape checks to the device checks
    with pytest.raises(TypeError):
        fc.fc_conv2d_epi(x, w, None, (), pad=1, y=bad)

"""libfusedconv Python binding: argument marshalling over the C ABI only.

Every computation runs in the CUDA kernels of ``_build/libfusedconv.so``
(declared in ``include/fusedconv.h``); PyTorch only supplies device memory
and streams.  There is no CPU fallback: if the library is missing or the
device is unusable, these functions raise.

Elementwise ops are tuples::

    ("relu",) ("hardswish",) ("leaky_relu", slope) ("add_channel", t[C_out])
    ("clamp", lo, hi) ("gelu_erf",) ("hardtanh", lo, hi) ("tanh",)
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libfusedconv.so")

FC_OK = 0
STATUS_NAMES = {0: "FC_OK", 1: "FC_ERR_INVALID_ARG", 2: "FC_ERR_UNSUPPORTED",
                3: "FC_ERR_ALIGNMENT", 4: "FC_ERR_WORKSPACE", 5: "FC_ERR_CUDA",
                6: "FC_ERR_TIMEOUT", 7: "FC_ERR_RANGE"}
EPI = {"relu": 1, "hardswish": 2, "leaky_relu": 3, "add_channel": 4, "clamp": 5,
       "gelu_erf": 6, "maxpool2x2": 7, "hardtanh": 8, "mean_hw": 9, "tanh": 10,
       "maxpool": 11}
VARIANTS = {"auto": 0, "ffma": 1, "tc_tf32x3": 2, "tc_f16x3": 3}
VARIANT_NAMES = {v: k for k, v in VARIANTS.items()}
MAX_OPS = 8

# every symbol include/fusedconv.h declares
EXPORTS = ("fc_conv2d_epi", "fc_conv2d_epi_noalloc", "fc_conv3d_epi", "fc_convT2d_pool_mean",
           "fc_conv2d_epi_nhwc", "fc_conv3d_epi_ndhwc",
           "fc_workspace_bytes", "fc_set_variant", "fc_set_staging", "fc_select_variant",
           "fc_last_variant", "fc_last_staging",
           "fc_last_launch_count", "fc_status_string",
           "fc_get_last_device_error", "fc_version", "fc_profile_enable",
           "fc_profile_read", "fc_profile_reset", "fc_wait_report",
           "fc_selftest_wait_timeout", "fc_pool_mean_tail")


class FcError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


class _Op(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("a", ctypes.c_float),
                ("b", ctypes.c_float), ("chan", ctypes.c_void_p)]


class _Epilogue(ctypes.Structure):
    _fields_ = [("bias", ctypes.c_void_p), ("n_ops", ctypes.c_int),
                ("ops", _Op * MAX_OPS)]


_lib = None
_lock = threading.Lock()


def lib():
    """The loaded libfusedconv (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libfusedconv is not built ({LIB_PATH} missing); run "
                    "convolution_epilogue_gb300._build.build()")
            L = ctypes.CDLL(LIB_PATH)
            P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            L.fc_conv2d_epi.restype = I
            L.fc_conv2d_epi.argtypes = [P, I, I, I, I, P, I, I, I, I, I, I, P, P, P, S, P]
            L.fc_conv2d_epi_nhwc.restype = I
            L.fc_conv2d_epi_nhwc.argtypes = [P, I, I, I, I, P, I, I, I, I, I, I, P, P, P, S, P]
            L.fc_conv3d_epi_ndhwc.restype = I
            L.fc_conv3d_epi_ndhwc.argtypes = [P, I, I, I, I, I, P, I, I, I, I, I, I, I, P,
                                              P, P, S, P]
            L.fc_conv2d_epi_noalloc.restype = I
            L.fc_conv2d_epi_noalloc.argtypes = [P, I, I, I, I, P, I, I, I, I, I, I, P, P, P]
            L.fc_conv3d_epi.restype = I
            L.fc_conv3d_epi.argtypes = [P, I, I, I, I, I, P, I, I, I, I, I, I, I, P,
                                        P, P, S, P]
            L.fc_convT2d_pool_mean.restype = I
            L.fc_convT2d_pool_mean.argtypes = [P, I, I, I, I, P, I, I, I, I, I, P, P,
                                               P, S, P]
            L.fc_workspace_bytes.restype = S
            L.fc_workspace_bytes.argtypes = [I, ctypes.POINTER(I)]
            L.fc_set_variant.restype = I
            L.fc_set_variant.argtypes = [I]
            L.fc_set_staging.restype = I
            L.fc_set_staging.argtypes = [I]
            L.fc_select_variant.restype = I
            L.fc_select_variant.argtypes = [I, ctypes.POINTER(I)]
            L.fc_last_variant.restype = I
            L.fc_last_staging.restype = I
            L.fc_last_launch_count.restype = I
            L.fc_status_string.restype = ctypes.c_char_p
            L.fc_status_string.argtypes = [I]
            L.fc_get_last_device_error.restype = I
            L.fc_get_last_device_error.argtypes = [P]
            L.fc_version.restype = I
            L.fc_profile_enable.restype = I
            L.fc_profile_enable.argtypes = [I]
            L.fc_profile_read.restype = I
            L.fc_profile_read.argtypes = [I, ctypes.POINTER(ctypes.c_double),
                                          ctypes.POINTER(I)]
            L.fc_profile_reset.restype = None
            L.fc_wait_report.restype = I
            L.fc_wait_report.argtypes = [P, ctypes.POINTER(ctypes.c_uint), I]
            L.fc_selftest_wait_timeout.restype = I
            L.fc_selftest_wait_timeout.argtypes = [ctypes.c_uint, P]
            F = ctypes.c_float
            L.fc_pool_mean_tail.restype = I
            L.fc_pool_mean_tail.argtypes = [P, I, I, I, I, I, I, F, F, P, P]
            _lib = L
    return _lib


def _check(status, what):
    if status != FC_OK:
        msg = lib().fc_status_string(status).decode()
        raise FcError(status, f"{what} ({msg})")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _require_cuda_f32(name, t):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32:
        raise TypeError(f"{name} must be a CUDA float32 tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _dims(name, t, ndim):
    """Shape of a tensor argument, checked for its rank (any device: shapes
    are checked before anything touches the GPU)."""
    shape = tuple(getattr(t, "shape", ()))
    if len(shape) != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {shape}")
    return shape


def _check_out(name, t, shape):
    """A caller-provided output must have exactly the shape the call
    writes: the kernels write every element of that shape, so a smaller
    tensor would be written past its end."""
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}; this call writes {tuple(shape)}")


def _check_vec(name, t, n):
    if t is not None and tuple(t.shape) != (n,) and int(t.numel()) != n:
        raise ValueError(f"{name} must hold {n} values (one per output channel), "
                         f"got shape {tuple(t.shape)}")


def _check_ops(ops, cout):
    for op in ops:
        if op[0] not in EPI:
            raise ValueError(f"unknown epilogue op {op[0]!r}")
        if op[0] == "add_channel":
            _check_vec("add_channel tensor", op[1], cout)


def _ws_bytes(ws):
    return int(ws.numel()) * int(ws.element_size())


def _stream_handle(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_epilogue(bias, ops):
    """Build the C epilogue descriptor; returns (struct, keepalive list)."""
    if bias is not None:
        _require_cuda_f32("bias", bias)
    e = _Epilogue()
    keep = []
    e.bias = None if bias is None else bias.data_ptr()
    if bias is not None:
        keep.append(bias)
    if len(ops) > MAX_OPS:
        raise ValueError("at most 8 epilogue ops")
    e.n_ops = len(ops)
    for i, op in enumerate(ops):
        name = op[0]
        e.ops[i].kind = EPI[name]
        if name == "leaky_relu":
            e.ops[i].a = float(op[1])
        elif name in ("clamp", "hardtanh", "maxpool"):
            e.ops[i].a, e.ops[i].b = float(op[1]), float(op[2])
        elif name == "add_channel":
            t = op[1]
            _require_cuda_f32("add_channel tensor", t)
            e.ops[i].chan = t.data_ptr()
            keep.append(t)
    return e, keep


def workspace_bytes(entry: int, dims) -> int:
    arr = (ctypes.c_int * len(dims))(*[int(d) for d in dims])
    return int(lib().fc_workspace_bytes(int(entry), arr))


def _workspace(nbytes, device):
    import torch
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def set_variant(name: str = "auto"):
    _check(lib().fc_set_variant(VARIANTS[name]), "fc_set_variant")


def select_variant(entry: int, dims) -> str:
    """The variant a call would run for a problem (fc_select_variant);
    "none" for an invalid or unsupported one.  Needs no device."""
    arr = (ctypes.c_int * len(dims))(*[int(d) for d in dims])
    return VARIANT_NAMES.get(int(lib().fc_select_variant(int(entry), arr)), "none")


STAGING = {"auto": -1, "loads": 0, "tma": 1}


def set_staging(mode: str = "auto"):
    """Input staging of the tensor-core variants: "auto" (chosen per shape
    from the measured table), "tma" (tensor copies where the plan allows
    them) or "loads" (producer register loads)."""
    _check(lib().fc_set_staging(STAGING[mode]), "fc_set_staging")


def last_staging() -> str:
    return "tma" if lib().fc_last_staging() == 1 else "loads"


def last_variant() -> str:
    return VARIANT_NAMES.get(lib().fc_last_variant(), "none")


def last_launch_count() -> int:
    return int(lib().fc_last_launch_count())


def selftest_wait_timeout(limit_us: int, stream=None):
    """Launch the bounded-wait self-test (see fc_selftest_wait_timeout)."""
    _check(lib().fc_selftest_wait_timeout(int(limit_us), _stream_handle(stream)),
           "fc_selftest_wait_timeout")


def get_last_device_error(stream=None) -> int:
    return int(lib().fc_get_last_device_error(_stream_handle(stream)))


def wait_report(stream=None):
    """Records of timed-out kernel waits since the last call (diagnostics
    for FC_ERR_TIMEOUT): a list of dicts, cleared on read."""
    buf = (ctypes.c_uint * (1 + 32 * 8))()
    n = lib().fc_wait_report(_stream_handle(stream), buf, len(buf))
    if n < 0:
        raise FcError(5, "fc_wait_report")
    recs = []
    for i in range(min(n, 32)):
        r = buf[1 + 8 * i:1 + 8 * i + 8]
        recs.append({"block": r[0], "thread": r[1], "barrier": r[2], "parity": r[3],
                     "tag": hex(r[4]), "word": hex(r[5] | (r[6] << 32))})
    return n, recs


def profile_enable(on: bool = True):
    _check(lib().fc_profile_enable(1 if on else 0), "fc_profile_enable")


def profile_reset():
    lib().fc_profile_reset()


def profile_read(entry: int):
    """(total_ms, launches) of the main kernels of one entry since reset."""
    ms = ctypes.c_double()
    n = ctypes.c_int()
    _check(lib().fc_profile_read(int(entry), ctypes.byref(ms), ctypes.byref(n)),
           "fc_profile_read")
    return ms.value, n.value


def _extent(n_in, k, stride, pad, dilation):
    return (n_in + 2 * pad - dilation * (k - 1) - 1) // stride + 1


def fc_conv2d_epi(x, w, bias=None, ops=(), pad=0, y=None, ws=None, stream=None, stride=1,
                  dilation=1):
    """Conv2d(k=3, stride 1 or 2, pad, dilation 1 or 2) + bias + elementwise
    ops -> y [N,CO,Ho,Wo]."""
    import torch
    N, C, H, W = _dims("x", x, 4)
    CO, C2, KH, KW = _dims("w", w, 4)
    if C2 != C:
        raise ValueError("weight C_in mismatch")
    Ho, Wo = _extent(H, KH, stride, pad, dilation), _extent(W, KW, stride, pad, dilation)
    _check_out("y", y, (N, CO, Ho, Wo))
    _check_vec("bias", bias, CO)
    _check_ops(ops, CO)
    _require_cuda_f32("x", x)
    _require_cuda_f32("w", w)
    if y is None:
        y = torch.empty((N, CO, Ho, Wo), dtype=torch.float32, device=x.device)
    _require_cuda_f32("y", y)
    if ws is None:
        ws = _workspace(workspace_bytes(0, (N, C, H, W, CO, KH, pad)), x.device)
    e, keep = make_epilogue(bias, ops)
    st = lib().fc_conv2d_epi(_ptr(x), N, C, H, W, _ptr(w), CO, KH, KW, int(stride), pad,
                             int(dilation), ctypes.byref(e), _ptr(y), _ptr(ws), _ws_bytes(ws),
                             _stream_handle(stream))
    _check(st, "fc_conv2d_epi")
    del keep
    return y


def fc_conv2d_epi_noalloc(x, w, y, bias=None, ops=(), pad=0, stream=None):
    """fc_conv2d_epi without a workspace argument, for callers that cannot
    allocate device memory: the library uses its own fixed 1 MiB device
    array (shared by all calls on a device; overlapping calls race).  The
    caller passes every tensor, including the output y, whose shape must be
    the call's output shape; nothing is allocated here."""
    N, C, H, W = _dims("x", x, 4)
    CO, C2, KH, KW = _dims("w", w, 4)
    if C2 != C:
        raise ValueError("weight C_in mismatch")
    _check_out("y", y, (N, CO, _extent(H, KH, 1, pad, 1), _extent(W, KW, 1, pad, 1)))
    _check_vec("bias", bias, CO)
    _check_ops(ops, CO)
    _require_cuda_f32("x", x)
    _require_cuda_f32("w", w)
    _require_cuda_f32("y", y)
    e, keep = make_epilogue(bias, ops)
    st = lib().fc_conv2d_epi_noalloc(_ptr(x), N, C, H, W, _ptr(w), CO, KH, KW, 1, pad, 1,
                                     ctypes.byref(e), _ptr(y), _stream_handle(stream))
    _check(st, "fc_conv2d_epi_noalloc")
    del keep
    return y


def fc_conv3d_epi(x, w, bias=None, ops=(), pad=0, y=None, ws=None, stream=None, stride=1,
                  dilation=1):
    """Conv3d(k=3, stride 1 or 2, pad, dilation 1 or 2) + bias + elementwise ops."""
    import torch
    N, C, D, H, W = _dims("x", x, 5)
    CO, C2, KD, KH, KW = _dims("w", w, 5)
    if C2 != C:
        raise ValueError("weight C_in mismatch")
    Do, Ho, Wo = (_extent(D, KD, stride, pad, dilation), _extent(H, KH, stride, pad, dilation),
                  _extent(W, KW, stride, pad, dilation))
    _check_out("y", y, (N, CO, Do, Ho, Wo))
    _check_vec("bias", bias, CO)
    _check_ops(ops, CO)
    _require_cuda_f32("x", x)
    _require_cuda_f32("w", w)
    if y is None:
        y = torch.empty((N, CO, Do, Ho, Wo), dtype=torch.float32, device=x.device)
    _require_cuda_f32("y", y)
    if ws is None:
        ws = _workspace(workspace_bytes(1, (N, C, D, H, W, CO, KD, pad)), x.device)
    e, keep = make_epilogue(bias, ops)
    st = lib().fc_conv3d_epi(_ptr(x), N, C, D, H, W, _ptr(w), CO, KD, KH, KW, int(stride),
                             pad, int(dilation), ctypes.byref(e), _ptr(y), _ptr(ws),
                             _ws_bytes(ws), _stream_handle(stream))
    _check(st, "fc_conv3d_epi")
    del keep
    return y


def fc_conv2d_epi_nhwc(x, w, bias=None, ops=(), pad=0, y=None, ws=None, stream=None, stride=1,
                       dilation=1):
    """Channels-last conv2d: x [N,H,W,C_in], w [C_out,C_in,3,3] -> y [N,Ho,Wo,C_out]."""
    import torch
    N, H, W, C = _dims("x", x, 4)
    CO, C2, KH, KW = _dims("w", w, 4)
    if C2 != C:
        raise ValueError("weight C_in mismatch")
    Ho, Wo = _extent(H, KH, stride, pad, dilation), _extent(W, KW, stride, pad, dilation)
    _check_out("y", y, (N, Ho, Wo, CO))
    _check_vec("bias", bias, CO)
    _check_ops(ops, CO)
    _require_cuda_f32("x", x)
    _require_cuda_f32("w", w)
    if y is None:
        y = torch.empty((N, Ho, Wo, CO), dtype=torch.float32, device=x.device)
    _require_cuda_f32("y", y)
    if ws is None:
        ws = _workspace(workspace_bytes(0, (N, C, H, W, CO, KH, pad)), x.device)
    e, keep = make_epilogue(bias, ops)
    st = lib().fc_conv2d_epi_nhwc(_ptr(x), N, C, H, W, _ptr(w), CO, KH, KW, int(stride), pad,
                                  int(dilation), ctypes.byref(e), _ptr(y), _ptr(ws),
                                  _ws_bytes(ws), _stream_handle(stream))
    _check(st, "fc_conv2d_epi_nhwc")
    del keep
    return y


def fc_conv3d_epi_ndhwc(x, w, bias=None, ops=(), pad=0, y=None, ws=None, stream=None, stride=1,
                        dilation=1):
    """Channels-last conv3d: x [N,D,H,W,C_in], w [C_out,C_in,3,3,3] -> y [N,Do,Ho,Wo,C_out]."""
    import torch
    N, D, H, W, C = _dims("x", x, 5)
    CO, C2, KD, KH, KW = _dims("w", w, 5)
    if C2 != C:
        raise ValueError("weight C_in mismatch")
    Do, Ho, Wo = (_extent(D, KD, stride, pad, dilation), _extent(H, KH, stride, pad, dilation),
                  _extent(W, KW, stride, pad, dilation))
    _check_out("y", y, (N, Do, Ho, Wo, CO))
    _check_vec("bias", bias, CO)
    _check_ops(ops, CO)
    _require_cuda_f32("x", x)
    _require_cuda_f32("w", w)
    if y is None:
        y = torch.empty((N, Do, Ho, Wo, CO), dtype=torch.float32, device=x.device)
    _require_cuda_f32("y", y)
    if ws is None:
        ws = _workspace(workspace_bytes(1, (N, C, D, H, W, CO, KD, pad)), x.device)
    e, keep = make_epilogue(bias, ops)
    st = lib().fc_conv3d_epi_ndhwc(_ptr(x), N, C, D, H, W, _ptr(w), CO, KD, KH, KW, int(stride),
                                   pad, int(dilation), ctypes.byref(e), _ptr(y), _ptr(ws),
                                   _ws_bytes(ws), _stream_handle(stream))
    _check(st, "fc_conv3d_epi_ndhwc")
    del keep
    return y


def pool_mean_ops(lo=-1.0, hi=1.0, pool=(2, 2)):
    """The pooled entry's chain; pool = (window, stride) of the max pool."""
    mp = ("maxpool2x2",) if tuple(pool) == (2, 2) else ("maxpool", float(pool[0]), float(pool[1]))
    return (mp, ("hardtanh", lo, hi), ("mean_hw",), ("tanh",))


def fc_convT2d_pool_mean(x, w, bias=None, hardtanh=(-1.0, 1.0), pad=1, y=None,
                         ws=None, stream=None, stride=1, out_pad=0, pool=(2, 2)):
    """ConvTranspose2d(k=3, stride 1 or 2, p=1, out_pad) + bias -> maxpool
    (window, stride) = pool -> hardtanh -> mean(H,W) -> tanh.
    w: [C_in, C_out, 3, 3]; returns y [N, C_out, 1, 1]."""
    import torch
    N, C, H, W = _dims("x", x, 4)
    C2, CO, K, _ = _dims("w", w, 4)
    if C2 != C:
        raise ValueError("weight C_in mismatch")
    _check_out("y", y, (N, CO, 1, 1))
    _check_vec("bias", bias, CO)
    _require_cuda_f32("x", x)
    _require_cuda_f32("w", w)
    if y is None:
        y = torch.empty((N, CO, 1, 1), dtype=torch.float32, device=x.device)
    _require_cuda_f32("y", y)
    if ws is None:
        if tuple(pool) == (2, 2):
            nb = workspace_bytes(2, (N, C, H, W, CO, K, pad))
        else:
            nb = workspace_bytes(3, (N, C, H, W, CO, K, pad, stride, out_pad, pool[0], pool[1]))
        ws = _workspace(nb, x.device)
    e, keep = make_epilogue(bias, pool_mean_ops(*hardtanh, pool=pool))
    st = lib().fc_convT2d_pool_mean(_ptr(x), N, C, H, W, _ptr(w), CO, K, int(stride), pad,
                                    int(out_pad),
                                    ctypes.byref(e), _ptr(y), _ptr(ws), _ws_bytes(ws),
                                    _stream_handle(stream))
    _check(st, "fc_convT2d_pool_mean")
    del keep
    return y


def fc_pool_mean_tail(x, k=2, s=2, hardtanh=(-1.0, 1.0), y=None, stream=None):
    """MaxPool(k, s) -> hardtanh -> mean(H, W) -> tanh on a conv output
    x [N, C, H, W]; returns y [N, C, 1, 1]."""
    import torch
    N, C, H, W = _dims("x", x, 4)
    _check_out("y", y, (N, C, 1, 1))
    _require_cuda_f32("x", x)
    if y is None:
        y = torch.empty((N, C, 1, 1), dtype=torch.float32, device=x.device)
    _require_cuda_f32("y", y)
    _check(lib().fc_pool_mean_tail(_ptr(x), N, C, H, W, int(k), int(s), float(hardtanh[0]),
                                   float(hardtanh[1]), _ptr(y), _stream_handle(stream)),
           "fc_pool_mean_tail")
    return y

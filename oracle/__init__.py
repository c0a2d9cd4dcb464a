"""CPU oracle for the fused convolution + epilogue chains.

TEST INFRASTRUCTURE ONLY.  The product path (the ``convolution_epilogue_gb300``
package and its CUDA library) never imports, links or calls anything in this
directory; only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg do.

The arithmetic lives in ``fc_oracle.c`` (plain C, fp64 sums over fp32 inputs);
this module compiles it with gcc and marshals numpy arrays through ctypes.
Each entry states the definition it follows:

* ``conv_epi``            cross-correlation + bias, then an elementwise chain
                          (Kimi-K2.6 l2_p57 trace, "simplest kernel" paragraph;
                          Kimi-K2.6 l2_p90 trace, conv3d FLOP paragraph).
* ``convT2d``             transposed conv in scatter form (Kimi-K2.6 l2_p10
                          trace, ConvTranspose2d formula paragraph).
* ``convT_pool_mean``     convT -> MaxPool2d -> hardtanh -> mean(H,W) -> tanh
                          (Kimi-K2.6 l2_p10 trace, tail-kernel paragraphs).

Elementwise ops are given as tuples::

    ("relu",) ("hardswish",) ("leaky_relu", slope) ("add_channel", s[CO])
    ("clamp", lo, hi) ("gelu_erf",) ("hardtanh", lo, hi) ("tanh",)

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, delta kernels, brute force against an independent loop, and
the values the pages print).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fc_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

OPS = {
    "relu": 1,
    "hardswish": 2,
    "leaky_relu": 3,
    "add_channel": 4,
    "clamp": 5,
    "gelu_erf": 6,
    "hardtanh": 7,
    "tanh": 8,
}


def build(force: bool = False) -> str:
    """Compile fc_oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            L = ctypes.c_long
            D = ctypes.c_double
            lib.or_apply_op.restype = D
            lib.or_apply_op.argtypes = [I, D, D, P, I, D]
            lib.or_conv_epi.restype = None
            lib.or_conv_epi.argtypes = [P, I, I, I, I, I, P, I, I, I, I, I, I,
                                        I, P, I, P, P, P, P, P]
            lib.or_conv_epi_points.restype = None
            lib.or_conv_epi_points.argtypes = [P, I, I, I, I, I, P, I, I, I, I,
                                               I, I, I, P, I, P, P, P, P, P, L,
                                               P]
            lib.or_convT2d.restype = None
            lib.or_convT2d.argtypes = [P, I, I, I, I, P, I, I, I, I, I, P, P]
            lib.or_maxpool2d.restype = None
            lib.or_maxpool2d.argtypes = [P, L, I, I, I, I, P]
            lib.or_mean_hw.restype = None
            lib.or_mean_hw.argtypes = [P, L, L, P]
            lib.or_convT_pool_mean_points.restype = None
            lib.or_convT_pool_mean_points.argtypes = [P, I, I, I, I, P, I, I,
                                                      I, I, I, P, I, I, D, D,
                                                      P, L, P]
            lib.or_convT_pool_mean.restype = None
            lib.or_convT_pool_mean.argtypes = [P, I, I, I, I, P, I, I, I, I,
                                               I, P, I, I, D, D, P]
            _lib = lib
    return _lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _chain(ops, CO):
    """Marshal an op list into (n, kinds, a, b, chan) arrays kept alive by
    the caller."""
    n = len(ops)
    kinds = np.zeros(max(n, 1), dtype=np.int32)
    a = np.zeros(max(n, 1), dtype=np.float64)
    b = np.zeros(max(n, 1), dtype=np.float64)
    chan = np.zeros((max(n, 1), CO), dtype=np.float32)
    for i, op in enumerate(ops):
        name = op[0]
        kinds[i] = OPS[name]
        if name == "leaky_relu":
            a[i] = float(op[1])
        elif name in ("clamp", "hardtanh"):
            a[i], b[i] = float(op[1]), float(op[2])
        elif name == "add_channel":
            chan[i, :] = np.asarray(op[1], dtype=np.float32).reshape(-1)[:CO]
    return n, kinds, a, b, chan


def apply_op(name, v, a=0.0, b=0.0, chan=None, co=0):
    """One elementwise op on one scalar, in double (for pin tests)."""
    lib = _load()
    c = None
    if chan is not None:
        c = _f32(chan)
    return lib.or_apply_op(OPS[name], float(a), float(b), _ptr(c), int(co),
                           float(v))


def conv_out_extent(n_in, k, stride=1, pad=0, dilation=1):
    """Output extent of a cross-correlation: (n + 2p - d(k-1) - 1) // s + 1."""
    return (n_in + 2 * pad - dilation * (k - 1) - 1) // stride + 1


def convT_out_extent(n_in, k, stride=1, pad=0, out_pad=0):
    """Output extent of a transposed conv: (n-1)s - 2p + k + op."""
    return (n_in - 1) * stride - 2 * pad + k + out_pad


def conv_epi(x, w, bias, ops=(), stride=1, pad=0, dilation=1):
    """Conv2d (x [N,C,H,W], w [CO,C,kh,kw]) or Conv3d (x [N,C,D,H,W],
    w [CO,C,kd,kh,kw]) + bias, then the elementwise chain.  Output o reads
    input o*stride + k*dilation - pad on every axis.  Returns float64."""
    lib = _load()
    x = _f32(x)
    w = _f32(w)
    bias = None if bias is None else _f32(bias)
    if x.ndim == 4:
        N, C, H, W = x.shape
        D = 1
        CO, _, KH, KW = w.shape
        KD = 1
    else:
        N, C, D, H, W = x.shape
        CO, _, KD, KH, KW = w.shape
    pad_d = 0 if x.ndim == 4 else pad
    Do = conv_out_extent(D, KD, stride, pad_d, dilation)
    Ho = conv_out_extent(H, KH, stride, pad, dilation)
    Wo = conv_out_extent(W, KW, stride, pad, dilation)
    y = np.empty((N, CO, Do, Ho, Wo), dtype=np.float64)
    n, kinds, a, b, chan = _chain(ops, CO)
    lib.or_conv_epi(_ptr(x), N, C, D, H, W, _ptr(w), CO, KD, KH, KW, stride,
                    pad, dilation, _ptr(bias), n, _ptr(kinds), _ptr(a), _ptr(b),
                    _ptr(chan), _ptr(y))
    return y.reshape((N, CO, Ho, Wo)) if x.ndim == 4 else y


def conv_epi_points(x, w, bias, ops, flat_idx, stride=1, pad=0, dilation=1):
    """conv_epi evaluated at the given flat output indices only."""
    lib = _load()
    x = _f32(x)
    w = _f32(w)
    bias = None if bias is None else _f32(bias)
    if x.ndim == 4:
        N, C, H, W = x.shape
        D, KD = 1, 1
        CO, _, KH, KW = w.shape
    else:
        N, C, D, H, W = x.shape
        CO, _, KD, KH, KW = w.shape
    idx = np.ascontiguousarray(flat_idx, dtype=np.int64)
    out = np.empty(idx.shape[0], dtype=np.float64)
    n, kinds, a, b, chan = _chain(ops, CO)
    lib.or_conv_epi_points(_ptr(x), N, C, D, H, W, _ptr(w), CO, KD, KH, KW,
                           stride, pad, dilation, _ptr(bias), n, _ptr(kinds), _ptr(a),
                           _ptr(b), _ptr(chan), _ptr(idx), idx.shape[0],
                           _ptr(out))
    return out


def convT2d(x, w, bias, stride=1, pad=0, out_pad=0):
    """Scatter-form ConvTranspose2d + bias.  w: [CI, CO, K, K]."""
    lib = _load()
    x = _f32(x)
    w = _f32(w)
    bias = None if bias is None else _f32(bias)
    N, CI, H, W = x.shape
    _, CO, K, _ = w.shape
    Ho = convT_out_extent(H, K, stride, pad, out_pad)
    Wo = convT_out_extent(W, K, stride, pad, out_pad)
    y = np.empty((N, CO, Ho, Wo), dtype=np.float64)
    lib.or_convT2d(_ptr(x), N, CI, H, W, _ptr(w), CO, K, stride, pad, out_pad,
                   _ptr(bias), _ptr(y))
    return y


def maxpool2d(y, k=2, s=2):
    """MaxPool2d(k, s) over the last two dims of a float64 array (floor)."""
    lib = _load()
    y = np.ascontiguousarray(y, dtype=np.float64)
    *lead, H, W = y.shape
    NC = int(np.prod(lead)) if lead else 1
    Hp, Wp = (H - k) // s + 1, (W - k) // s + 1
    out = np.empty((*lead, Hp, Wp), dtype=np.float64)
    lib.or_maxpool2d(_ptr(y), NC, H, W, k, s, _ptr(out))
    return out


def mean_hw(y):
    """Mean over the last two dims, keepdim."""
    lib = _load()
    y = np.ascontiguousarray(y, dtype=np.float64)
    *lead, H, W = y.shape
    NC = int(np.prod(lead)) if lead else 1
    out = np.empty((*lead, 1, 1), dtype=np.float64)
    lib.or_mean_hw(_ptr(y), NC, H * W, _ptr(out))
    return out


def convT_pool_mean(x, w, bias, stride=1, pad=1, out_pad=0, pool=(2, 2),
                    hardtanh=(-1.0, 1.0)):
    """ConvTranspose2d + bias -> MaxPool2d -> hardtanh -> mean -> tanh.
    Returns [N, CO, 1, 1] float64."""
    lib = _load()
    x = _f32(x)
    w = _f32(w)
    bias = None if bias is None else _f32(bias)
    N, CI, H, W = x.shape
    _, CO, K, _ = w.shape
    out = np.empty((N, CO, 1, 1), dtype=np.float64)
    lib.or_convT_pool_mean(_ptr(x), N, CI, H, W, _ptr(w), CO, K, stride, pad,
                           out_pad, _ptr(bias), pool[0], pool[1],
                           float(hardtanh[0]), float(hardtanh[1]), _ptr(out))
    return out


def convT_pool_mean_points(x, w, bias, nc_pairs, stride=1, pad=1, out_pad=0,
                           pool=(2, 2), hardtanh=(-1.0, 1.0)):
    """convT_pool_mean for selected (n, co) pairs only."""
    lib = _load()
    x = _f32(x)
    w = _f32(w)
    bias = None if bias is None else _f32(bias)
    N, CI, H, W = x.shape
    _, CO, K, _ = w.shape
    nc = np.ascontiguousarray(nc_pairs, dtype=np.int32).reshape(-1, 2)
    out = np.empty(nc.shape[0], dtype=np.float64)
    lib.or_convT_pool_mean_points(_ptr(x), N, CI, H, W, _ptr(w), CO, K,
                                  stride, pad, out_pad, _ptr(bias), pool[0],
                                  pool[1], float(hardtanh[0]),
                                  float(hardtanh[1]), _ptr(nc), nc.shape[0],
                                  _ptr(out))
    return out

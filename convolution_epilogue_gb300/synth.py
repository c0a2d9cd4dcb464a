"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke
check.

This module holds no convolution or epilogue arithmetic: only a
counter-based random generator and the input shapes of the five workloads.
The same host bytes feed both the CPU oracle and the CUDA library.

Generator (stated so that anyone can regenerate the bytes):

* splitmix64 in counter form: draw ``i`` of stream ``seed`` is
  ``mix(seed * 2**32 + 0x9E3779B97F4A7C15 * (i + 1))`` where ``mix`` is the
  splitmix64 finaliser (xor-shift 30, multiply 0xBF58476D1CE4E5B9,
  xor-shift 27, multiply 0x94D049BB133111EB, xor-shift 31), all mod 2**64.
* uniform double in (0, 1): ``((z >> 11) + 0.5) * 2**-53``.
* standard normal: Box-Muller on draws (2j, 2j+1):
  ``sqrt(-2 ln u1) * cos(2 pi u2)`` for element 2j and ``* sin`` for 2j+1,
  computed in double and rounded to fp32.
* U(-a, a): ``a * (2u - 1)`` in double, rounded to fp32.
* Tensors of one workload are drawn in the order x, W, b, s from one
  stream (seed = workload number 1..5), each starting where the previous
  one stopped.

Distributions (the workloads' stated ones): x ~ N(0, 1); W and b ~
U(-1/sqrt(fan_in), 1/sqrt(fan_in)) with fan_in = C_in * k^d (576 for the
64 -> 64 3x3 transposed conv); s ~ N(0, 1).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z):
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def raw_u64(seed: int, start: int, count: int) -> np.ndarray:
    """Draws start .. start+count-1 of stream `seed` as uint64."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        base = np.uint64((seed << 32) & 0xFFFFFFFFFFFFFFFF)
        return _mix(base + _GOLDEN * i)


def _uniform01(seed, start, count):
    z = raw_u64(seed, start, count)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def _normal_chunk(seed, start_draw, first_elem, count):
    """Normals first_elem .. first_elem+count-1 of a tensor whose draws
    start at start_draw."""
    j0 = first_elem // 2
    j1 = (first_elem + count + 1) // 2
    u = _uniform01(seed, start_draw + 2 * j0, 2 * (j1 - j0))
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * math.pi * u2
    z = np.empty(2 * (j1 - j0), dtype=np.float64)
    z[0::2] = r * np.cos(t)
    z[1::2] = r * np.sin(t)
    off = first_elem - 2 * j0
    return z[off:off + count].astype(np.float32)


class Stream:
    """Sequential tensor draws from one seeded stream."""

    def __init__(self, seed: int):
        self.seed = int(seed)
        self.pos = 0

    def normal(self, shape, threads: int | None = None) -> np.ndarray:
        n = int(np.prod(shape))
        out = np.empty(n, dtype=np.float32)
        start = self.pos
        chunks = [(c, min(_CHUNK, n - c)) for c in range(0, n, _CHUNK)]

        def work(ck):
            c, m = ck
            out[c:c + m] = _normal_chunk(self.seed, start, c, m)

        nthr = threads or min(16, os.cpu_count() or 1)
        if len(chunks) > 1 and nthr > 1:
            with ThreadPoolExecutor(nthr) as ex:
                list(ex.map(work, chunks))
        else:
            for ck in chunks:
                work(ck)
        self.pos += 2 * ((n + 1) // 2)
        return out.reshape(shape)

    def uniform(self, shape, bound: float) -> np.ndarray:
        n = int(np.prod(shape))
        u = _uniform01(self.seed, self.pos, n)
        self.pos += n
        return (bound * (2.0 * u - 1.0)).astype(np.float32).reshape(shape)


# The five workloads.  kind: conv2d / conv3d / convT_pool_mean.
WORKLOADS = {
    1: dict(name="conv2d_relu_hardswish_small", kind="conv2d",
            x=(4, 8, 32, 32), cout=64, k=3, fan_in=72),
    2: dict(name="convT2d_pool_mean_small", kind="convT_pool_mean",
            x=(2, 64, 32, 32), cout=64, k=3, fan_in=576),
    3: dict(name="conv2d_relu_hardswish_128x8x128x128", kind="conv2d",
            x=(128, 8, 128, 128), cout=64, k=3, fan_in=72),
    4: dict(name="conv3d_leaky_add_clamp_gelu_128x8x16x64x64", kind="conv3d",
            x=(128, 8, 16, 64, 64), cout=64, k=3, fan_in=216),
    5: dict(name="convT2d_pool_mean_128x64x256x256", kind="convT_pool_mean",
            x=(128, 64, 256, 256), cout=64, k=3, fan_in=576),
}


def make_inputs(wid: int, x_shape=None, first_images=None):
    """Seeded inputs of workload `wid` (optionally with another x shape of
    the same kind, for the small edge-case sweeps).  Returns a dict with
    x, w, b and (conv3d only) s, all fp32 numpy arrays.  With
    `first_images=n` only the first n images of x are drawn (the same bytes
    as the full draw) and W, b, s are the full workload's."""
    spec = WORKLOADS[wid]
    xs = tuple(x_shape) if x_shape is not None else spec["x"]
    st = Stream(wid)
    k = spec["k"]
    cin = xs[1]
    cout = spec["cout"]
    if first_images is None:
        out = {"x": st.normal(xs)}
    else:
        n = int(np.prod(xs))
        part = (int(first_images),) + tuple(xs[1:])
        out = {"x": st.normal(part)}
        st.pos = 2 * ((n + 1) // 2)
    if spec["kind"] == "conv2d":
        wshape = (cout, cin, k, k)
        fan_in = cin * k * k
    elif spec["kind"] == "conv3d":
        wshape = (cout, cin, k, k, k)
        fan_in = cin * k * k * k
    else:
        wshape = (cin, cout, k, k)
        fan_in = cout * k * k
    bound = 1.0 / math.sqrt(fan_in)
    out["w"] = st.uniform(wshape, bound)
    out["b"] = st.uniform((cout,), bound)
    if spec["kind"] == "conv3d":
        out["s"] = st.normal((cout, 1, 1, 1))
    return out


def seeded(seed: int):
    """A fresh stream for ad-hoc test tensors."""
    return Stream(seed)

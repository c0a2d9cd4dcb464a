"""Coefficients of the short GELU polynomial used by the fused conv3d chain.

For |v| <= 1 (the chain clamps to [-1, 1] before GELU) write
    GELU(v) = v/2 + v/2 erf(v / sqrt 2) = v/2 + s R(s),   s = v^2,
where R(s) = (GELU(v) - v/2) / s is an even, entire function of v.  This
script fits R on s in [0, 1] by a degree-4 polynomial p(s) that minimises
the GELU error max |s (R(s) - p(s))|: a weighted least-squares fit refined
by Lawson's iteration (C. L. Lawson, 1961: reweighting each sample by its
error drives the least-squares fit to the minimax one).  R is sampled from
Python's math.erf in double precision.

Run `python gen_gelu_poly.py` to print the coefficients and the errors:
the fit's own error is about 4e-9; evaluated in fp32 by Horner's rule the
result is within 1e-7 of GELU on [-1, 1], the fp32 rounding level of the
result.  The printed constants are the ones in fc_epi.cuh (kGeluR0 .. 4).
"""
from math import erf, pi, sqrt

import numpy as np

DEG = 4


def r_exact(s: np.ndarray) -> np.ndarray:
    out = np.empty_like(s)
    for i, ss in enumerate(s):
        if ss < 1e-12:
            out[i] = 1.0 / sqrt(2.0 * pi)  # limit of R at s = 0
        else:
            v = sqrt(ss)
            out[i] = (0.5 * v * erf(v / sqrt(2.0))) / ss
    return out


def fit(deg: int = DEG, samples: int = 20001, iters: int = 60):
    s = np.linspace(0.0, 1.0, samples)
    r = r_exact(s)
    V = np.vander(s, deg + 1, increasing=True)
    w = np.ones_like(s)
    for _ in range(iters):
        W = np.sqrt(w) * np.maximum(s, 1e-6)
        c, *_ = np.linalg.lstsq(V * W[:, None], r * W, rcond=None)
        e = np.abs(s * (V @ c - r))
        w = w * (e + 1e-30)
        w /= w.sum()
    return c, float(e.max())


def fp32_error(c) -> float:
    c32 = np.asarray(c, dtype=np.float32)
    v = np.linspace(-1.0, 1.0, 200001).astype(np.float32)
    s = (v * v).astype(np.float32)
    p = np.full_like(s, c32[-1])
    for k in range(len(c32) - 2, -1, -1):
        p = (p * s + c32[k]).astype(np.float32)
    g = (s * p + np.float32(0.5) * v).astype(np.float32)
    ref = np.array([0.5 * x * (1.0 + erf(x / sqrt(2.0))) for x in v.astype(np.float64)])
    return float(np.abs(g - ref).max())


if __name__ == "__main__":
    c, e = fit()
    print(f"// degree {DEG}, fit error {e:.3g}, fp32 Horner error {fp32_error(c):.3g}")
    print("constexpr float kGeluR[%d] = {" % (DEG + 1))
    for k, ck in enumerate(c):
        print(f"    {np.float32(ck)!r}f,  // s^{k}".replace("np.float32(", "").replace(")f", "f"))
    print("};")

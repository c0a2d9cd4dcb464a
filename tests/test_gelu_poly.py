"""The fused conv3d chain's GELU polynomial: the constants compiled into the
kernels are the ones the committed generator computes, and the polynomial
stays within 2e-7 of GELU on [-1, 1] in fp32 (CPU only)."""
import importlib.util
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "convolution_epilogue_gb300", "csrc")


def _gen():
    spec = importlib.util.spec_from_file_location("gen_gelu_poly", os.path.join(CSRC, "gen_gelu_poly.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_kernel_constants_match_generator():
    gen = _gen()
    c, fit_err = gen.fit()
    assert fit_err < 1e-8
    src = open(os.path.join(CSRC, "fc_epi.cuh")).read()
    got = [float(re.search(rf"kGeluR{k} = ([-+0-9.e]+)f", src).group(1)) for k in range(5)]
    np.testing.assert_array_equal(np.float32(got), np.float32(c))
    assert gen.fp32_error(np.float32(got)) < 2e-7

"""Pins for the CPU oracle: checks it against things other than itself.

* values the pages print for worked examples (tests/golden/page_values.txt),
* closed forms (all-ones inputs, delta kernels, constant planes),
* brute force against independent pure-Python loops on tiny inputs,
* the transposed conv's scatter definition against a separately derived
  gather form with flipped taps and swapped channels (and the un-flipped
  variant that one page derives must DISAGREE).
"""
import math
import os

import numpy as np
import pytest

import oracle
from convolution_epilogue_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_values.txt")


def _golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            body, _cite = line.split("|", 1)
            key, val, tol = body.split()
            vals[key] = (float(val), float(tol))
    return vals


G = _golden()


def _rng(seed):
    return synth.seeded(1000 + seed)


# --------------------------------------------------------------- page values
@pytest.mark.parametrize("x", [0, 3, 6])
def test_hardswish_page_points(x):
    v, tol = G[f"hardswish@{x}"]
    assert abs(oracle.apply_op("hardswish", x) - v) <= tol


def test_gelu_exact_matches_page_not_tanh_approx():
    v, tol = G["gelu_erf@1"]
    g = oracle.apply_op("gelu_erf", 1.0)
    assert abs(g - v) <= tol
    # closed form: GELU(1) = Phi(1) = 0.5 (1 + erf(1/sqrt 2))
    assert abs(g - 0.8413447460685429) < 1e-15
    vt, _ = G["gelu_tanh_approx@1"]
    # the oracle must not reproduce the value the page prints for the
    # rejected tanh approximation
    assert abs(g - vt) > 1e-3
    # The page's own arithmetic for that value is off (it takes tanh(0.8336)
    # as 0.6869; it is 0.6823).  The true tanh approximation still misses
    # the exact form by more than the 1e-4 tolerance at x = 1, so the
    # page's conclusion (use erf) stands.
    tanh_form = 0.5 * (1 + math.tanh(math.sqrt(2 / math.pi) * (1 + 0.044715)))
    assert abs(tanh_form - 0.8411919906082768) < 1e-15
    assert abs(g - tanh_form) > 1e-4


def test_output_extents_match_pages():
    assert oracle.conv_out_extent(128, 3) == G["conv2d_out_extent@128,k3,p0"][0]
    assert oracle.conv_out_extent(16, 3) == G["conv3d_out_extent@16,k3,p0"][0]
    assert oracle.conv_out_extent(64, 3) == G["conv3d_out_extent@64,k3,p0"][0]
    assert (oracle.convT_out_extent(256, 3, 1, 1, 0)
            == G["convT_out_extent@256,k3,s1,p1,op0"][0])
    assert ((256 - 2) // 2 + 1) ** 2 == G["pool_windows@256x256,k2,s2"][0]


def test_counts_match_pages():
    # output elements and MACs of the full-size workloads, from the shapes
    assert 128 * 64 * 14 * 62 * 62 == G["conv3d_output_elements@cfg4"][0]
    assert 128 * 64 * 14 * 62 * 62 * 8 * 27 == G["conv3d_macs@cfg4"][0]
    assert 128 * 64 * 256 * 256 * 64 * 9 == G["convT_macs@cfg5"][0]
    assert 128 * 64 * 126 * 126 == G["conv2d_output_elements@cfg3"][0]


# ------------------------------------------------------------- activations
def test_activation_known_points():
    A = oracle.apply_op
    assert A("relu", -1.0) == 0.0 and A("relu", 2.5) == 2.5
    assert A("hardswish", -3.0) == 0.0
    assert abs(A("hardswish", 1.0) - 2.0 / 3.0) < 1e-15
    assert A("hardswish", -4.0) == 0.0  # clamp lower bound active
    assert abs(A("hardswish", -1.0) - (-1.0 / 3.0)) < 1e-15
    assert abs(A("leaky_relu", -1.0, 0.2) + 0.2) < 1e-15
    assert A("leaky_relu", 3.0, 0.2) == 3.0
    assert A("gelu_erf", 0.0) == 0.0
    assert abs(A("gelu_erf", -1.0) + 0.15865525393145707) < 1e-15
    assert abs(A("tanh", 1.0) - 0.7615941559557649) < 1e-15
    assert A("hardtanh", 2.0, -1.0, 1.0) == 1.0
    assert A("hardtanh", -2.0, -1.0, 1.0) == -1.0
    assert A("clamp", 0.25, -1.0, 1.0) == 0.25
    s = np.arange(4, dtype=np.float32)
    assert A("add_channel", 1.0, chan=s, co=3) == 4.0


def test_relu_then_hardswish_identity():
    # after ReLU, hardswish(x) = x * min(x + 3, 6) / 6 (l2_p57 simplification)
    for x in np.linspace(0.0, 9.0, 37):
        lhs = oracle.apply_op("hardswish", oracle.apply_op("relu", x))
        assert abs(lhs - x * min(x + 3.0, 6.0) / 6.0) < 1e-14
    # ... and skipping the ReLU is wrong for x < 0
    assert oracle.apply_op("hardswish", -1.0) != 0.0


# ----------------------------------------------------------------- conv
def _brute_conv2d(x, w, b, pad=0):
    """Independent loop: output position outermost, then kw, kh, ci."""
    N, C, H, W = x.shape
    CO, _, K, _ = w.shape
    Ho, Wo = H + 2 * pad - K + 1, W + 2 * pad - K + 1
    y = np.zeros((N, CO, Ho, Wo))
    for n in range(N):
        for oh in range(Ho):
            for ow in range(Wo):
                for co in range(CO):
                    s = float(b[co])
                    for kw in range(K):
                        for kh in range(K):
                            ih, iw = oh + kh - pad, ow + kw - pad
                            if 0 <= ih < H and 0 <= iw < W:
                                for ci in range(C):
                                    s += float(x[n, ci, ih, iw]) * float(w[co, ci, kh, kw])
                    y[n, co, oh, ow] = s
    return y


def _brute_conv3d(x, w, b):
    N, C, D, H, W = x.shape
    CO, _, K, _, _ = w.shape
    y = np.zeros((N, CO, D - K + 1, H - K + 1, W - K + 1))
    for idx in np.ndindex(*y.shape):
        n, co, od, oh, ow = idx
        patch = x[n, :, od:od + K, oh:oh + K, ow:ow + K].astype(np.float64)
        y[idx] = float(b[co]) + float((patch * w[co].astype(np.float64)).sum())
    return y


def test_conv2d_brute_force_tiny():
    st = _rng(1)
    x = st.normal((2, 3, 6, 7))
    w = st.uniform((4, 3, 3, 3), 0.5)
    b = st.uniform((4,), 0.5)
    for pad in (0, 1):
        got = oracle.conv_epi(x, w, b, (), pad=pad)
        ref = _brute_conv2d(x, w, b, pad)
        assert got.shape == ref.shape
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_conv3d_brute_force_tiny():
    st = _rng(2)
    x = st.normal((2, 3, 4, 5, 6))
    w = st.uniform((5, 3, 3, 3, 3), 0.5)
    b = st.uniform((5,), 0.5)
    got = oracle.conv_epi(x, w, b, ())
    np.testing.assert_allclose(got, _brute_conv3d(x, w, b), rtol=0, atol=1e-12)


def _brute_conv2d_strided(x, w, b, stride, pad):
    """Independent loop for a strided conv: out (oh, ow) reads input rows
    oh*stride + kh - pad and columns ow*stride + kw - pad."""
    N, C, H, W = x.shape
    CO, _, K, _ = w.shape
    Ho, Wo = (H + 2 * pad - K) // stride + 1, (W + 2 * pad - K) // stride + 1
    y = np.zeros((N, CO, Ho, Wo))
    for n, co, oh, ow in np.ndindex(N, CO, Ho, Wo):
        s = float(b[co])
        for ci in range(C):
            for kh in range(K):
                for kw in range(K):
                    ih, iw = oh * stride + kh - pad, ow * stride + kw - pad
                    if 0 <= ih < H and 0 <= iw < W:
                        s += float(x[n, ci, ih, iw]) * float(w[co, ci, kh, kw])
        y[n, co, oh, ow] = s
    return y


def test_conv2d_stride2_brute_force_and_extent():
    st = _rng(11)
    x = st.normal((2, 3, 9, 8))
    w = st.uniform((4, 3, 3, 3), 0.5)
    b = st.uniform((4,), 0.5)
    for pad in (0, 1, 2):
        got = oracle.conv_epi(x, w, b, (), stride=2, pad=pad)
        ref = _brute_conv2d_strided(x, w, b, 2, pad)
        assert got.shape == ref.shape == (2, 4, (9 + 2 * pad - 3) // 2 + 1, (8 + 2 * pad - 3) // 2 + 1)
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_conv_stride2_delta_kernel_subsamples():
    # centre tap, stride 2, pad 0: y[i, j] = x[2i + 1, 2j + 1] + b
    st = _rng(12)
    x = st.normal((1, 3, 9, 11))
    w = np.zeros((3, 3, 3, 3), np.float32)
    for c in range(3):
        w[c, c, 1, 1] = 1.0
    b = st.uniform((3,), 1.0)
    y = oracle.conv_epi(x, w, b, (), stride=2)
    ref = x[:, :, 1:-1:2, 1:-1:2].astype(np.float64) + b[None, :, None, None]
    np.testing.assert_array_equal(y, ref)
    # 3-D: tap (kd, kh, kw) = (2, 0, 1) picks x[2od + 2, 2oh, 2ow + 1]
    x3 = st.normal((1, 2, 7, 7, 8))
    w3 = np.zeros((1, 2, 3, 3, 3), np.float32)
    w3[0, 1, 2, 0, 1] = 1.0
    y3 = oracle.conv_epi(x3, w3, None, (), stride=2)
    np.testing.assert_array_equal(y3[0, 0], x3[0, 1, 2:7:2, 0:5:2, 1:7:2])


def _brute_conv2d_dilated(x, w, b, stride, pad, dil):
    """Independent loop for a dilated, strided conv: out (oh, ow) reads input
    row oh*stride + kh*dil - pad and column ow*stride + kw*dil - pad; the
    extent counts the outputs whose window start oh*stride - pad keeps the
    last tap (k-1)*dil inside the padded input."""
    N, C, H, W = x.shape
    CO, _, K, _ = w.shape
    span = (K - 1) * dil + 1
    Ho = len([o for o in range(H + 2 * pad) if o * stride + span <= H + 2 * pad])
    Wo = len([o for o in range(W + 2 * pad) if o * stride + span <= W + 2 * pad])
    y = np.zeros((N, CO, Ho, Wo))
    for n, co, oh, ow in np.ndindex(N, CO, Ho, Wo):
        s = float(b[co])
        for ci in range(C):
            for kh in range(K):
                for kw in range(K):
                    ih, iw = oh * stride + kh * dil - pad, ow * stride + kw * dil - pad
                    if 0 <= ih < H and 0 <= iw < W:
                        s += float(x[n, ci, ih, iw]) * float(w[co, ci, kh, kw])
        y[n, co, oh, ow] = s
    return y


def test_conv2d_dilation2_brute_force_and_extent():
    st = _rng(13)
    x = st.normal((2, 3, 11, 9))
    w = st.uniform((4, 3, 3, 3), 0.5)
    b = st.uniform((4,), 0.5)
    for stride in (1, 2):
        for pad in (0, 1, 2, 3, 4):
            got = oracle.conv_epi(x, w, b, (), stride=stride, pad=pad, dilation=2)
            ref = _brute_conv2d_dilated(x, w, b, stride, pad, 2)
            assert got.shape == ref.shape
            assert got.shape[2:] == (oracle.conv_out_extent(11, 3, stride, pad, 2),
                                     oracle.conv_out_extent(9, 3, stride, pad, 2))
            np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    # the extent of a 3-tap window at dilation 2 (span 5) over 10 inputs, pad 0
    assert oracle.conv_out_extent(10, 3, 1, 0, 2) == 6
    assert oracle.conv_out_extent(10, 3, 2, 2, 2) == 5  # "same"-padded, stride 2


def test_conv_dilation2_equals_zero_inserted_kernel():
    """A 3-tap kernel at dilation 2 is the 5-tap kernel with zeros between
    its taps at dilation 1 (2-D and 3-D; same terms in the same order)."""
    st = _rng(14)
    x = st.normal((2, 3, 10, 12))
    w = st.uniform((4, 3, 3, 3), 0.5)
    b = st.uniform((4,), 0.5)
    w5 = np.zeros((4, 3, 5, 5), np.float32)
    w5[:, :, ::2, ::2] = w
    for stride, pad in ((1, 2), (2, 1), (1, 0)):
        np.testing.assert_array_equal(
            oracle.conv_epi(x, w, b, (), stride=stride, pad=pad, dilation=2),
            oracle.conv_epi(x, w5, b, (), stride=stride, pad=pad))
    x3 = st.normal((1, 2, 7, 8, 9))
    w3 = st.uniform((3, 2, 3, 3, 3), 0.5)
    w35 = np.zeros((3, 2, 5, 5, 5), np.float32)
    w35[:, :, ::2, ::2, ::2] = w3
    np.testing.assert_array_equal(
        oracle.conv_epi(x3, w3, None, (), stride=1, pad=2, dilation=2),
        oracle.conv_epi(x3, w35, None, (), stride=1, pad=2))


def test_conv_dilation2_delta_kernel_shifts():
    # tap (kh, kw) = (2, 0) at dilation 2, pad 2: y[i, j] = x[i + 2, j - 2]
    st = _rng(15)
    x = st.normal((1, 1, 8, 9))
    w = np.zeros((1, 1, 3, 3), np.float32)
    w[0, 0, 2, 0] = 1.0
    y = oracle.conv_epi(x, w, None, (), pad=2, dilation=2)
    ref = np.zeros((8, 9))
    ref[:6, 2:] = x[0, 0, 2:, :7]
    np.testing.assert_array_equal(y[0, 0], ref)
    # 3-D, stride 2: tap (kd, kh, kw) = (1, 2, 1) at dilation 2, pad 0 picks
    # x[2od + 2, 2oh + 4, 2ow + 2]
    x3 = st.normal((1, 1, 9, 10, 11))
    w3 = np.zeros((1, 1, 3, 3, 3), np.float32)
    w3[0, 0, 1, 2, 1] = 1.0
    y3 = oracle.conv_epi(x3, w3, None, (), stride=2, dilation=2)
    np.testing.assert_array_equal(y3[0, 0], x3[0, 0, 2:7:2, 4:10:2, 2:9:2])


@pytest.mark.parametrize("k,stride,pad,dil", [
    (1, 1, 0, 1), (1, 3, 1, 1), (5, 1, 2, 1), (5, 3, 4, 2), (7, 1, 3, 1), (7, 4, 6, 3),
    (4, 2, 1, 1), (2, 1, 0, 4), (3, 3, 2, 3), (6, 4, 5, 1)])
def test_conv2d_general_layer_brute_force(k, stride, pad, dil):
    """Kernel sizes 1..7 (odd and even), strides and dilations 1..4 and
    paddings, against the independent loop: out (oh, ow) reads input
    oh*stride + kh*dil - pad, extent (n + 2p - d(k-1) - 1)//s + 1."""
    st = _rng(40 + k + 10 * stride + 100 * dil)
    x = st.normal((2, 3, 13, 16))
    w = st.uniform((4, 3, k, k), 0.4)
    b = st.uniform((4,), 0.4)
    got = oracle.conv_epi(x, w, b, (), stride=stride, pad=pad, dilation=dil)
    ref = _brute_conv2d_dilated(x, w, b, stride, pad, dil)
    assert got.shape == ref.shape
    assert got.shape[2:] == (oracle.conv_out_extent(13, k, stride, pad, dil),
                             oracle.conv_out_extent(16, k, stride, pad, dil))
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_conv_general_kernel_delta_and_pointwise():
    """Closed forms at other kernel sizes: a 1x1 kernel is a matrix product
    over channels at every pixel; a 7x7 delta tap at (kh, kw) with pad 3
    shifts the input by (kh - 3, kw - 3); a 5x5x5 3-D delta at stride 2
    subsamples."""
    st = _rng(50)
    x = st.normal((2, 5, 6, 7))
    w = st.uniform((3, 5, 1, 1), 0.5)
    y = oracle.conv_epi(x, w, None, ())
    ref = np.einsum("oc,nchw->nohw", w[:, :, 0, 0].astype(np.float64), x.astype(np.float64))
    np.testing.assert_allclose(y, ref, atol=1e-12)
    w7 = np.zeros((1, 1, 7, 7), np.float32)
    w7[0, 0, 1, 5] = 1.0
    x1 = st.normal((1, 1, 9, 10))
    y7 = oracle.conv_epi(x1, w7, None, (), pad=3)
    ref7 = np.zeros((9, 10))
    ref7[2:, :8] = x1[0, 0, :7, 2:]
    np.testing.assert_array_equal(y7[0, 0], ref7)
    x3 = st.normal((1, 1, 11, 12, 13))
    w5 = np.zeros((1, 1, 5, 5, 5), np.float32)
    w5[0, 0, 4, 0, 2] = 1.0
    y3 = oracle.conv_epi(x3, w5, None, (), stride=2)
    np.testing.assert_array_equal(y3[0, 0], x3[0, 0, 4:11:2, 0:8:2, 2:11:2])


def test_conv_all_ones_closed_form():
    b = np.array([0.5, -1.0], dtype=np.float32)
    y2 = oracle.conv_epi(np.ones((1, 8, 5, 5), np.float32),
                         np.ones((2, 8, 3, 3), np.float32), b)
    assert np.all(y2[0, 0] == 72.5) and np.all(y2[0, 1] == 71.0)
    y3 = oracle.conv_epi(np.ones((1, 8, 4, 4, 4), np.float32),
                         np.ones((2, 8, 3, 3, 3), np.float32), b)
    assert np.all(y3[0, 0] == 216.5) and np.all(y3[0, 1] == 215.0)


def test_conv_delta_kernel_is_centred_crop():
    st = _rng(3)
    x = st.normal((2, 4, 7, 9))
    w = np.zeros((4, 4, 3, 3), np.float32)
    for c in range(4):
        w[c, c, 1, 1] = 1.0
    b = st.uniform((4,), 1.0)
    y = oracle.conv_epi(x, w, b)
    ref = x[:, :, 1:-1, 1:-1].astype(np.float64) + b[None, :, None, None]
    np.testing.assert_array_equal(y, ref)
    # off-centre tap (kh=0, kw=2) picks x[oh, ow+2]
    w2 = np.zeros_like(w)
    w2[1, 2, 0, 2] = 1.0
    y2 = oracle.conv_epi(x, w2, None)
    np.testing.assert_array_equal(y2[:, 1], x[:, 2, 0:5, 2:9])
    # 3-D delta
    x3 = st.normal((1, 2, 5, 5, 5))
    w3 = np.zeros((2, 2, 3, 3, 3), np.float32)
    w3[0, 1, 2, 0, 1] = 1.0
    y3 = oracle.conv_epi(x3, w3, None)
    np.testing.assert_array_equal(y3[0, 0], x3[0, 1, 2:5, 0:3, 1:4])


def test_conv_linear_in_weights():
    st = _rng(4)
    x = st.normal((1, 3, 6, 6))
    w1 = st.uniform((2, 3, 3, 3), 1.0)
    w2 = st.uniform((2, 3, 3, 3), 1.0)
    y1 = oracle.conv_epi(x, w1, None)
    y2 = oracle.conv_epi(x, w2, None)
    y12 = oracle.conv_epi(x, (w1.astype(np.float64) + w2).astype(np.float32), None)
    # w1 + w2 is rounded to fp32, so compare with the rounding bound
    np.testing.assert_allclose(y12, y1 + y2, atol=1e-5)


def test_conv_points_match_full():
    st = _rng(5)
    x = st.normal((2, 3, 5, 6, 7))
    w = st.uniform((4, 3, 3, 3, 3), 0.5)
    b = st.uniform((4,), 0.5)
    s = st.normal((4,))
    ops = (("leaky_relu", 0.2), ("add_channel", s), ("clamp", -1, 1), ("gelu_erf",))
    full = oracle.conv_epi(x, w, b, ops)
    idx = np.array([0, 7, 100, full.size - 1, 333])
    pts = oracle.conv_epi_points(x, w, b, ops, idx)
    np.testing.assert_array_equal(pts, full.reshape(-1)[idx])


def test_epilogue_chains_elementwise():
    st = _rng(6)
    x = st.normal((2, 3, 6, 6))
    w = st.uniform((4, 3, 3, 3), 1.0)
    b = st.uniform((4,), 1.0)
    raw = oracle.conv_epi(x, w, b)
    y = oracle.conv_epi(x, w, b, (("relu",), ("hardswish",)))
    r = np.maximum(raw, 0.0)
    np.testing.assert_allclose(y, r * np.clip((r + 3.0) / 6.0, 0.0, 1.0),
                               atol=1e-15)
    s = st.normal((4,))
    y2 = oracle.conv_epi(x, w, b, (("leaky_relu", 0.2), ("add_channel", s),
                                   ("clamp", -1.0, 1.0), ("gelu_erf",)))
    t = np.where(raw > 0, raw, 0.2 * raw) + s.astype(np.float64)[None, :, None, None]
    t = np.clip(t, -1.0, 1.0)
    erf = np.vectorize(math.erf)
    np.testing.assert_allclose(y2, 0.5 * t * (1.0 + erf(t / math.sqrt(2.0))),
                               atol=1e-15)


# ------------------------------------------------------------ transposed conv
def _gather_flip(x, w, b, pad):
    """ConvT (stride 1) written as a plain conv: swap W's channel axes, flip
    both taps, pad with k-1-p.  Derived independently of the scatter form."""
    K = w.shape[2]
    wc = np.ascontiguousarray(np.transpose(w, (1, 0, 2, 3))[:, :, ::-1, ::-1])
    return _brute_conv2d(x, wc, b, pad=K - 1 - pad)


def _gather_noflip(x, w, b, pad):
    """The variant with swapped channels but NO flip (one trace derives this)."""
    wc = np.ascontiguousarray(np.transpose(w, (1, 0, 2, 3)))
    return _brute_conv2d(x, wc, b, pad=pad)


@pytest.mark.parametrize("pad", [0, 1, 2])
def test_convT_scatter_equals_flipped_gather(pad):
    st = _rng(7 + pad)
    x = st.normal((2, 3, 5, 6))
    w = st.uniform((3, 4, 3, 3), 0.5)
    b = st.uniform((4,), 0.5)
    y = oracle.convT2d(x, w, b, 1, pad, 0)
    assert y.shape == (2, 4, 5 + 2 - 2 * pad, 6 + 2 - 2 * pad)
    np.testing.assert_allclose(y, _gather_flip(x, w, b, pad), rtol=0, atol=1e-12)


def test_convT_noflip_reading_disagrees():
    st = _rng(11)
    x = st.normal((1, 3, 5, 5))
    w = st.uniform((3, 4, 3, 3), 0.5)
    b = st.uniform((4,), 0.5)
    y = oracle.convT2d(x, w, b, 1, 1, 0)
    assert np.max(np.abs(y - _gather_noflip(x, w, b, 1))) > 1e-2


def test_convT_delta_tap_shifts_input():
    st = _rng(12)
    x = st.normal((1, 2, 6, 6))
    for kh, kw in [(0, 0), (0, 2), (2, 1), (1, 1)]:
        w = np.zeros((2, 2, 3, 3), np.float32)
        w[1, 0, kh, kw] = 1.0
        y = oracle.convT2d(x, w, None, 1, 1, 0)
        ref = np.zeros((6, 6))
        for i in range(6):
            for j in range(6):
                oi, oj = i + kh - 1, j + kw - 1
                if 0 <= oi < 6 and 0 <= oj < 6:
                    ref[oi, oj] = x[0, 1, i, j]
        np.testing.assert_array_equal(y[0, 0], ref)
        assert np.all(y[0, 1] == 0.0)


def test_convT_all_ones_pad1():
    CI = 64
    y = oracle.convT2d(np.ones((1, CI, 8, 8), np.float32),
                       np.ones((CI, 2, 3, 3), np.float32),
                       np.array([0.25, 0.0], np.float32), 1, 1, 0)
    p = y[0, 0]
    assert np.all(p[1:-1, 1:-1] == 9 * CI + 0.25)
    assert np.all(p[0, 1:-1] == 6 * CI + 0.25) and np.all(p[1:-1, -1] == 6 * CI + 0.25)
    for c in (p[0, 0], p[0, -1], p[-1, 0], p[-1, -1]):
        assert c == 4 * CI + 0.25


def test_convT_stride2_brute_force():
    st = _rng(13)
    x = st.normal((1, 2, 3, 4))
    w = st.uniform((2, 3, 3, 3), 1.0)
    y = oracle.convT2d(x, w, None, 2, 1, 1)
    Ho = (3 - 1) * 2 - 2 + 3 + 1
    Wo = (4 - 1) * 2 - 2 + 3 + 1
    ref = np.zeros((3, Ho, Wo))
    for ci in range(2):
        for i in range(3):
            for j in range(4):
                for co in range(3):
                    for kh in range(3):
                        for kw in range(3):
                            oi, oj = 2 * i + kh - 1, 2 * j + kw - 1
                            if 0 <= oi < Ho and 0 <= oj < Wo:
                                ref[co, oi, oj] += float(x[0, ci, i, j]) * float(w[ci, co, kh, kw])
    np.testing.assert_allclose(y[0], ref, atol=1e-12)


# ------------------------------------------------------ pool / mean / tanh
def test_maxpool_brute_force_and_checkerboard():
    st = _rng(14)
    a = st.normal((2, 3, 4, 5)).astype(np.float64)
    p = oracle.maxpool2d(a, 2, 2)
    assert p.shape == (2, 3, 2, 2)  # floor extent drops the 5th column
    for idx in np.ndindex(*p.shape):
        n, c, i, j = idx
        assert p[idx] == a[n, c, 2 * i:2 * i + 2, 2 * j:2 * j + 2].max()
    cb = np.indices((4, 4)).sum(axis=0) % 2 * 2.0 - 1.0  # +-1 checkerboard
    assert np.all(oracle.maxpool2d(cb[None, None], 2, 2) == 1.0)


def test_mean_permutation_invariant():
    st = _rng(15)
    a = st.normal((1, 1, 8, 8)).astype(np.float64)
    m = oracle.mean_hw(a)[0, 0, 0, 0]
    perm = a.reshape(-1)[np.argsort(st.uniform((64,), 1.0))].reshape(1, 1, 8, 8)
    assert abs(oracle.mean_hw(perm)[0, 0, 0, 0] - m) < 1e-15
    assert abs(m - a.sum() / 64.0) < 1e-15


def test_convT_pool_mean_constant_plane():
    # zero input => conv output is the bias everywhere
    b = np.array([0.3, -2.0, 5.0], np.float32)
    out = oracle.convT_pool_mean(np.zeros((1, 4, 6, 6), np.float32),
                                 np.ones((4, 3, 3, 3), np.float32), b)
    exp = np.tanh(np.clip(b.astype(np.float64), -1, 1))
    np.testing.assert_allclose(out[0, :, 0, 0], exp, atol=1e-15)


def test_convT_pool_mean_composition():
    st = _rng(16)
    x = st.normal((2, 4, 6, 8))
    w = st.uniform((4, 3, 3, 3), 0.3)
    b = st.uniform((3,), 0.3)
    y = oracle.convT2d(x, w, b, 1, 1, 0)
    # independent tail: numpy max over reshaped windows, clip, mean, tanh
    N, C, H, W = y.shape
    pooled = y.reshape(N, C, H // 2, 2, W // 2, 2).max(axis=(3, 5))
    ref = np.tanh(np.clip(pooled, -1, 1).mean(axis=(2, 3)))
    out = oracle.convT_pool_mean(x, w, b)
    np.testing.assert_allclose(out[:, :, 0, 0], ref, atol=1e-14)
    pts = oracle.convT_pool_mean_points(x, w, b, [(1, 2), (0, 0)])
    np.testing.assert_allclose(pts, [ref[1, 2], ref[0, 0]], atol=1e-14)


def test_convT_pool_mean_odd_extent_floor():
    st = _rng(17)
    x = st.normal((1, 2, 5, 7))
    w = st.uniform((2, 2, 3, 3), 0.3)
    b = st.uniform((2,), 0.3)
    y = oracle.convT2d(x, w, b, 1, 1, 0)  # 5 x 7 output
    pooled = y[:, :, :4, :6].reshape(1, 2, 2, 2, 3, 2).max(axis=(3, 5))
    ref = np.tanh(np.clip(pooled, -1, 1).mean(axis=(2, 3)))
    np.testing.assert_allclose(oracle.convT_pool_mean(x, w, b)[:, :, 0, 0], ref,
                               atol=1e-14)


def _brute_convT(x, w, b, s, p, op):
    """Scatter loop for a transposed conv: x[ci, i, j] adds x * w[ci, co, kh, kw]
    to output (i*s + kh - p, j*s + kw - p)."""
    N, C, H, W = x.shape
    CO, K = w.shape[1], w.shape[2]
    Ho, Wo = (H - 1) * s - 2 * p + K + op, (W - 1) * s - 2 * p + K + op
    y = np.zeros((N, CO, Ho, Wo)) + b.astype(np.float64)[None, :, None, None]
    for n, ci, i, j in np.ndindex(N, C, H, W):
        for co, kh, kw in np.ndindex(CO, K, K):
            oi, oj = i * s + kh - p, j * s + kw - p
            if 0 <= oi < Ho and 0 <= oj < Wo:
                y[n, co, oi, oj] += float(x[n, ci, i, j]) * float(w[ci, co, kh, kw])
    return y


@pytest.mark.parametrize("op", [0, 1])
def test_convT_stride2_pool_mean_composition(op):
    """Stride-2 transposed conv (pad 1, output padding 0 or 1) -> 2x2 max
    pool (floor extent) -> hardtanh -> mean -> tanh, against an independent
    scatter loop and a numpy tail."""
    st = _rng(18 + op)
    x = st.normal((2, 3, 5, 6))
    w = st.uniform((3, 4, 3, 3), 0.4)
    b = st.uniform((4,), 0.3)
    y = _brute_convT(x, w, b, 2, 1, op)
    assert y.shape[2:] == ((5 - 1) * 2 + 1 + op, (6 - 1) * 2 + 1 + op)
    Hp, Wp = y.shape[2] // 2, y.shape[3] // 2
    pooled = y[:, :, :2 * Hp, :2 * Wp].reshape(2, 4, Hp, 2, Wp, 2).max(axis=(3, 5))
    ref = np.tanh(np.clip(pooled, -1, 1).mean(axis=(2, 3)))
    out = oracle.convT_pool_mean(x, w, b, stride=2, pad=1, out_pad=op)
    np.testing.assert_allclose(out[:, :, 0, 0], ref, atol=1e-13)
    np.testing.assert_allclose(oracle.convT2d(x, w, b, 2, 1, op), y, atol=1e-12)


@pytest.mark.parametrize("k,s,p,op", [(3, 3, 1, 2), (3, 4, 0, 3), (3, 2, 0, 1), (3, 2, 2, 0),
                                      (5, 2, 2, 1), (1, 3, 0, 0), (7, 1, 3, 0), (4, 2, 1, 0),
                                      (5, 1, 0, 0)])
def test_convT_general_layer_scatter_and_pool_mean(k, s, p, op):
    """The transposed conv at other kernel sizes, strides 1..4, paddings and
    output paddings below the stride, against the independent scatter loop
    (extent (H-1)s - 2p + k + op); then the 2x2 pool chain against a numpy
    tail on that loop's output."""
    st = _rng(60 + k + 10 * s + 100 * p + 1000 * op)
    x = st.normal((2, 3, 5, 6))
    w = st.uniform((3, 4, k, k), 0.4)
    b = st.uniform((4,), 0.3)
    y = _brute_convT(x, w, b, s, p, op)
    assert y.shape[2:] == (oracle.convT_out_extent(5, k, s, p, op),
                           oracle.convT_out_extent(6, k, s, p, op))
    np.testing.assert_allclose(oracle.convT2d(x, w, b, s, p, op), y, atol=1e-12)
    Hp, Wp = y.shape[2] // 2, y.shape[3] // 2
    pooled = y[:, :, :2 * Hp, :2 * Wp].reshape(2, 4, Hp, 2, Wp, 2).max(axis=(3, 5))
    ref = np.tanh(np.clip(pooled, -1, 1).mean(axis=(2, 3)))
    out = oracle.convT_pool_mean(x, w, b, stride=s, pad=p, out_pad=op)
    np.testing.assert_allclose(out[:, :, 0, 0], ref, atol=1e-13)


@pytest.mark.parametrize("pool", [(3, 2), (2, 1), (3, 3), (4, 2)])
def test_convT_pool_mean_general_window(pool):
    """Stride-1 transposed conv -> max pool of window k, stride s (floor
    extent, overlapping when k > s) -> hardtanh -> mean -> tanh, against an
    independent scatter loop and explicit window loops."""
    k, s = pool
    st = _rng(20 + k + s)
    x = st.normal((2, 3, 9, 10))
    w = st.uniform((3, 2, 3, 3), 0.4)
    b = st.uniform((2,), 0.3)
    y = _brute_convT(x, w, b, 1, 1, 0)
    Hp, Wp = (y.shape[2] - k) // s + 1, (y.shape[3] - k) // s + 1
    pooled = np.empty(y.shape[:2] + (Hp, Wp))
    for i in range(Hp):
        for j in range(Wp):
            pooled[:, :, i, j] = y[:, :, i * s:i * s + k, j * s:j * s + k].max(axis=(2, 3))
    ref = np.tanh(np.clip(pooled, -0.5, 0.8).mean(axis=(2, 3)))
    out = oracle.convT_pool_mean(x, w, b, pool=pool, hardtanh=(-0.5, 0.8))
    np.testing.assert_allclose(out[:, :, 0, 0], ref, atol=1e-13)


# ------------------------------------------------------------ the generator
def test_synth_generator_is_deterministic_and_distributed():
    a = synth.make_inputs(1)
    b = synth.make_inputs(1)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])
    x = a["x"].astype(np.float64)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1.0) < 0.02
    bound = 1.0 / math.sqrt(72)
    assert np.abs(a["w"]).max() <= bound and np.abs(a["w"]).max() > 0.9 * bound
    # chunked generation equals one-shot generation
    st1 = synth.Stream(9)
    big = st1.normal((3 * (1 << 22) + 5,), threads=4)
    st2 = synth.Stream(9)
    one = st2.normal((3 * (1 << 22) + 5,), threads=1)
    np.testing.assert_array_equal(big, one)

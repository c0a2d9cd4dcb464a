"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle,
element by element, at atol = rtol = 1e-4 (the tolerance the traces' harness
uses for fp32: Kimi-K2.6__l2_p10 trace, evaluator paragraph; Kimi-K2.6__l2_p90
trace, problem statement).

* small workloads 1 and 2: every output, every variant;
* ragged shapes (several tiles plus a ragged tail, C_out not a multiple of
  64, odd extents, padding) for every variant and chain;
* full-size workloads 3-5, in the launch configuration the benchmark times,
  on every output (the oracle runs once per workload on all host cores);
* widened forms at full size on sampled outputs the oracle computes one by
  one.
"""
import numpy as np
import pytest

import oracle
from convolution_epilogue_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-4
VARIANTS = ["ffma", "tc_tf32x3", "tc_f16x3"]


def fc():
    import convolution_epilogue_gb300 as m
    return m


def _check(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} outside atol=rtol=1e-4; worst at {i}: "
            f"gpu={got[i]!r} oracle={ref[i]!r} (max abs err {err.max():.3g})")


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _ops_torch(ops):
    out = []
    for op in ops:
        if op[0] == "add_channel":
            out.append(("add_channel", _dev(np.asarray(op[1], np.float32).reshape(-1))))
        else:
            out.append(op)
    return tuple(out)


def _run_conv(variant, x, w, b, ops, pad=0):
    m = fc()
    m.set_variant(variant)
    try:
        xt, wt, bt = _dev(x), _dev(w), _dev(b) if b is not None else None
        f = m.fc_conv2d_epi if x.ndim == 4 else m.fc_conv3d_epi
        y = f(xt, wt, bt, _ops_torch(ops), pad=pad)
        assert m.last_variant() == variant
        assert m.get_last_device_error() == 0
        return y.cpu().numpy()
    finally:
        m.set_variant("auto")


def _run_pool(variant, x, w, b, ht=(-1.0, 1.0)):
    m = fc()
    m.set_variant(variant)
    try:
        y = m.fc_convT2d_pool_mean(_dev(x), _dev(w), _dev(b) if b is not None else None,
                                   hardtanh=ht)
        assert m.last_variant() == variant
        assert m.get_last_device_error() == 0
        return y.cpu().numpy()
    finally:
        m.set_variant("auto")


def _supported(variant):
    return True


CHAIN_RH = (("relu",), ("hardswish",))


def chain_gelu(s):
    return (("leaky_relu", 0.2), ("add_channel", s), ("clamp", -1.0, 1.0), ("gelu_erf",))


# ------------------------------------------------------------ workloads 1, 2
@pytest.mark.parametrize("variant", VARIANTS)
def test_workload1_full(variant):
    inp = synth.make_inputs(1)
    ref = oracle.conv_epi(inp["x"], inp["w"], inp["b"], CHAIN_RH)
    got = _run_conv(variant, inp["x"], inp["w"], inp["b"], CHAIN_RH)
    _check(got, ref, f"workload 1 [{variant}]")


@pytest.mark.parametrize("variant", VARIANTS)
def test_workload2_full(variant):
    inp = synth.make_inputs(2)
    ref = oracle.convT_pool_mean(inp["x"], inp["w"], inp["b"])
    got = _run_pool(variant, inp["x"], inp["w"], inp["b"])
    _check(got, ref, f"workload 2 [{variant}]")


# --------------------------------------------------------------- ragged shapes
RAGGED_2D = [
    # (N, C, H, W, CO, pad, chain)
    (2, 3, 9, 37, 10, 0, "rh"),
    (1, 8, 33, 130, 64, 0, "rh"),       # W > 128: two column tiles
    (3, 12, 17, 20, 70, 1, "gelu"),     # C_in not a multiple of 8, CO > 64
    (1, 16, 5, 260, 64, 2, "generic"),  # wide rows, pad 2
    (2, 8, 3, 3, 64, 0, "none"),        # 1x1 output
]


def _chain(name, CO, st):
    if name == "rh":
        return CHAIN_RH
    if name == "gelu":
        return chain_gelu(st.normal((CO,)))
    if name == "generic":
        return (("tanh",), ("leaky_relu", 0.1), ("clamp", -0.5, 0.75), ("hardswish",))
    return ()


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", RAGGED_2D)
def test_conv2d_ragged(variant, shape):
    N, C, H, W, CO, pad, chain = shape
    st = synth.seeded(hash(shape) % 1000 + 50)
    x = st.normal((N, C, H, W))
    w = st.uniform((CO, C, 3, 3), 1.0 / np.sqrt(9 * C))
    b = st.uniform((CO,), 1.0 / np.sqrt(9 * C))
    ops = _chain(chain, CO, st)
    ref = oracle.conv_epi(x, w, b, ops, pad=pad)
    got = _run_conv(variant, x, w, b, ops, pad=pad)
    _check(got, ref, f"conv2d {shape} [{variant}]")


RAGGED_3D = [
    (1, 5, 5, 7, 9, 70, 0),
    (2, 8, 4, 12, 66, 64, 0),   # W > 64: ragged column tile
    (1, 8, 3, 6, 6, 16, 1),
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", RAGGED_3D)
def test_conv3d_ragged(variant, shape):
    N, C, D, H, W, CO, pad = shape
    st = synth.seeded(hash(shape) % 1000 + 60)
    x = st.normal((N, C, D, H, W))
    w = st.uniform((CO, C, 3, 3, 3), 1.0 / np.sqrt(27 * C))
    b = st.uniform((CO,), 1.0 / np.sqrt(27 * C))
    ops = chain_gelu(st.normal((CO,)))
    ref = oracle.conv_epi(x, w, b, ops, pad=pad)
    got = _run_conv(variant, x, w, b, ops, pad=pad)
    _check(got, ref, f"conv3d {shape} [{variant}]")


RAGGED_T = [
    (2, 5, 7, 10, 3),      # odd H: floor drops the last row
    (1, 64, 18, 140, 64),  # W > 128
    (2, 16, 2, 2, 64),     # one window
    (1, 9, 33, 31, 65),
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", RAGGED_T)
def test_convT_pool_mean_ragged(variant, shape):
    N, C, H, W, CO = shape
    st = synth.seeded(hash(shape) % 1000 + 70)
    x = st.normal((N, C, H, W))
    w = st.uniform((C, CO, 3, 3), 1.0 / np.sqrt(9 * CO))
    b = st.uniform((CO,), 1.0 / np.sqrt(9 * CO))
    ref = oracle.convT_pool_mean(x, w, b)
    got = _run_pool(variant, x, w, b)
    _check(got, ref, f"convT pool mean {shape} [{variant}]")


def test_convT_pool_mean_hardtanh_params():
    st = synth.seeded(80)
    x = st.normal((1, 8, 10, 12))
    w = st.uniform((8, 8, 3, 3), 0.2)
    b = st.uniform((8,), 0.2)
    ref = oracle.convT_pool_mean(x, w, b, hardtanh=(-0.25, 0.5))
    for v in VARIANTS:
        _check(_run_pool(v, x, w, b, ht=(-0.25, 0.5)), ref, f"hardtanh params [{v}]")


def test_pool_mean_deterministic():
    inp = synth.make_inputs(2)
    for v in VARIANTS:
        a = _run_pool(v, inp["x"], inp["w"], inp["b"])
        for _ in range(3):
            np.testing.assert_array_equal(_run_pool(v, inp["x"], inp["w"], inp["b"]), a)


def test_empty_batch_is_a_noop():
    m = fc()
    x = torch.empty((0, 8, 8, 8), device="cuda")
    w = torch.zeros((64, 8, 3, 3), device="cuda")
    y = m.fc_conv2d_epi(x, w, None, CHAIN_RH)
    assert y.shape == (0, 64, 6, 6)


# -------------------------------------------------------- full-size, sampled
_FULL = {}


def _full_inputs(wid):
    if wid not in _FULL:
        _FULL[wid] = synth.make_inputs(wid)
    return _FULL[wid]


def _sample_idx(shape, n, seed):
    rng = np.random.default_rng(seed)
    size = int(np.prod(shape))
    idx = rng.integers(0, size, n)
    # plus the corners of the first and last planes and a row edge
    extra = [0, size - 1, shape[-1] - 1, size - shape[-1]]
    return np.concatenate([idx, np.array(extra)])


_REF = {}


def _full_ref(wid):
    """The oracle's result for every output of a full-size workload,
    computed once per session (float64)."""
    if wid not in _REF:
        inp = _full_inputs(wid)
        if wid == 3:
            _REF[wid] = oracle.conv_epi(inp["x"], inp["w"], inp["b"], CHAIN_RH)
        elif wid == 4:
            _REF[wid] = oracle.conv_epi(inp["x"], inp["w"], inp["b"],
                                        chain_gelu(inp["s"].reshape(-1)))
        else:
            _REF[wid] = oracle.convT_pool_mean(inp["x"], inp["w"], inp["b"])
    return _REF[wid]


def _check_whole(got, ref, what, chunk=1 << 24):
    """Element-by-element allclose over every output, in chunks (the
    full-size outputs hold up to 441 M values).  Returns the largest
    tolerance use max |g - o| / (atol + rtol |o|)."""
    g = np.asarray(got).reshape(-1)
    r = np.asarray(ref).reshape(-1)
    assert g.size == r.size, f"{what}: {g.size} outputs vs {r.size} in the oracle"
    worst = 0.0
    for c in range(0, g.size, chunk):
        gc = g[c:c + chunk].astype(np.float64)
        rc = r[c:c + chunk]
        use = np.abs(gc - rc) / (ATOL + RTOL * np.abs(rc))
        m = float(np.nanmax(use)) if use.size else 0.0
        if not np.all(use <= 1.0):  # NaN fails too
            i = int(np.argmax(np.where(np.isnan(use), np.inf, use)))
            raise AssertionError(
                f"{what}: {(~(use <= 1.0)).sum()} outputs in chunk at {c} outside "
                f"atol=rtol=1e-4; worst flat index {c + i}: gpu={gc[i]!r} oracle={rc[i]!r}")
        worst = max(worst, m)
    return worst


@pytest.mark.parametrize("variant", ["auto"] + VARIANTS)
def test_workload3_full_size_every_output(variant):
    """conv2d [128,8,128,128] + ReLU + HardSwish: all 130 M outputs against
    the oracle, in the launch configuration the benchmark times."""
    inp = _full_inputs(3)
    ref = _full_ref(3)
    m = fc()
    m.set_variant(variant)
    try:
        y = m.fc_conv2d_epi(_dev(inp["x"]), _dev(inp["w"]), _dev(inp["b"]), CHAIN_RH)
        assert m.get_last_device_error() == 0
        assert tuple(y.shape) == (128, 64, 126, 126)
        got = y.cpu().numpy()
        del y
    finally:
        m.set_variant("auto")
    use = _check_whole(got, ref, f"workload 3 every output [{variant}]")
    print(f"workload 3 [{variant}] max tolerance use {use:.4f}")


@pytest.mark.parametrize("variant", ["auto"] + VARIANTS)
def test_workload4_full_size_every_output(variant):
    """conv3d [128,8,16,64,64] + LeakyReLU + add + clamp + GELU: all 441 M
    outputs against the oracle."""
    inp = _full_inputs(4)
    ref = _full_ref(4)
    m = fc()
    m.set_variant(variant)
    s = inp["s"].reshape(-1)
    try:
        y = m.fc_conv3d_epi(_dev(inp["x"]), _dev(inp["w"]), _dev(inp["b"]),
                            _ops_torch(chain_gelu(s)))
        assert m.get_last_device_error() == 0
        assert tuple(y.shape) == (128, 64, 14, 62, 62)
        got = y.cpu().numpy()
        del y
    finally:
        m.set_variant("auto")
    use = _check_whole(got, ref, f"workload 4 every output [{variant}]")
    print(f"workload 4 [{variant}] max tolerance use {use:.4f}")


@pytest.mark.parametrize("variant", ["auto"] + VARIANTS)
def test_workload5_full_size_every_output(variant):
    """Transposed conv [128,64,256,256] -> pool -> hardtanh -> mean -> tanh:
    all 8192 (n, c) outputs against the oracle."""
    inp = _full_inputs(5)
    ref = _full_ref(5)
    m = fc()
    m.set_variant(variant)
    try:
        y = m.fc_convT2d_pool_mean(_dev(inp["x"]), _dev(inp["w"]), _dev(inp["b"]))
        assert m.get_last_device_error() == 0
        got = y.cpu().numpy()
    finally:
        m.set_variant("auto")
    use = _check_whole(got, ref, f"workload 5 every output [{variant}]")
    print(f"workload 5 [{variant}] max tolerance use {use:.4f}")
    # every output is inside tanh's range for clamped means
    assert np.all(np.abs(got) <= np.tanh(1.0) + 1e-6)


def test_workload5_deterministic_over_ten_calls():
    """The pooled mean is reduced in a fixed order (per-tile partials, then
    an index-order sum): ten calls on the full-size workload give bitwise
    the same 8192 outputs, on every variant."""
    inp = _full_inputs(5)
    m = fc()
    x, w, b = _dev(inp["x"]), _dev(inp["w"]), _dev(inp["b"])
    for v in ["auto"] + VARIANTS:
        m.set_variant(v)
        try:
            first = m.fc_convT2d_pool_mean(x, w, b).cpu().numpy()
            for _ in range(9):
                again = m.fc_convT2d_pool_mean(x, w, b).cpu().numpy()
                np.testing.assert_array_equal(again, first, err_msg=f"[{v}]")
            assert m.get_last_device_error() == 0
        finally:
            m.set_variant("auto")


def test_f16_split_range_boundary():
    """tc_f16x3 splits each x into an fp16 hi part and a scaled fp16 lo part.
    While the hi part stays finite (|x| < 65520; 65510 rounds to fp16's
    largest finite value, 65504) the result meets the tolerance; once it
    overflows (|x| >= 65520) the call reports FC_ERR_RANGE (7) in the device
    status word rather than a wrong result."""
    st = synth.seeded(777)
    x = st.normal((1, 8, 12, 12))
    w = st.uniform((64, 8, 3, 3), 1.0 / np.sqrt(72.0))
    b = st.uniform((64,), 1.0 / np.sqrt(72.0))
    x[0, 3, 5, 5] = 65510.0
    ref = oracle.conv_epi(x, w, b, ())
    _check(_run_conv("tc_f16x3", x, w, b, ()), ref, "x = 65510")
    x[0, 3, 5, 5] = -70000.0
    m = fc()
    m.set_variant("tc_f16x3")
    try:
        m.fc_conv2d_epi(_dev(x), _dev(w), _dev(b), ())
        assert m.last_variant() == "tc_f16x3"
        assert m.get_last_device_error() == 7
        assert m.get_last_device_error() == 0  # reading clears the word
    finally:
        m.set_variant("auto")


@pytest.mark.parametrize("scale_exp", [8, 16, 24])
def test_small_magnitudes_relative_accuracy(scale_exp):
    """x and w scaled by 2^-e, compared with rtol = 1e-4 and atol = 0 on the
    outputs that are not near zero (so the relative error decides, which
    the suite's atol hides at the workloads' scales).  tf32x3 keeps fp32's
    exponent range: it passes at every scale.  f16x3's parts are fp16: it
    passes while the data's largest magnitude is at least 2^-12 (x ~ N(0,1)
    2^-8 has max ~2^-6, w ~ 2^-11) and reports FC_ERR_RANGE below that
    (2^-16, 2^-24) instead of a less accurate result."""
    st = synth.seeded(3000 + scale_exp)
    x = (st.normal((2, 8, 20, 36)) * np.float32(2.0 ** -scale_exp)).astype(np.float32)
    w = (st.uniform((64, 8, 3, 3), 1.0 / np.sqrt(72.0)) * np.float32(2.0 ** -scale_exp)).astype(
        np.float32)
    ref = oracle.conv_epi(x, w, None, (), pad=1)
    sel = np.abs(ref) >= 0.05 * np.abs(ref).max()
    m = fc()
    for variant in ("tc_tf32x3", "tc_f16x3"):
        m.set_variant(variant)
        try:
            y = m.fc_conv2d_epi(_dev(x), _dev(w), None, (), pad=1).cpu().numpy()
            assert m.last_variant() == variant
            status = m.get_last_device_error()
        finally:
            m.set_variant("auto")
        if variant == "tc_f16x3" and scale_exp >= 16:
            assert status == 7, f"f16x3 at 2^-{scale_exp}: status {status}, FC_ERR_RANGE expected"
            continue
        assert status == 0
        rel = np.abs(y[sel] - ref[sel]) / np.abs(ref[sel])
        assert rel.max() <= 1e-4, f"{variant} at 2^-{scale_exp}: max relative error {rel.max():.3g}"


@pytest.mark.parametrize("k,s,shape,ht", [
    (2, 2, (2, 5, 36, 40), (-1.0, 1.0)),    # the configs' pooling, even extents
    (2, 2, (1, 3, 37, 41), (-1.0, 1.0)),    # odd extents: last row / column dropped
    (3, 2, (2, 4, 19, 23), (-0.5, 0.75)),   # overlapping windows, other clamp
    (2, 3, (1, 6, 20, 17), (-2.0, 2.0)),    # gaps between windows
    (1, 1, (1, 2, 7, 9), (-1.0, 1.0)),      # no pooling at all
])
def test_pool_mean_tail_against_oracle(k, s, shape, ht):
    """The standalone tail: maxpool(k, s) -> hardtanh -> mean -> tanh, vs
    the oracle's max-pool and mean composed with clamp and tanh in double."""
    st = synth.seeded(600 + 10 * k + s)
    x = st.normal(shape)
    m = fc()
    y = m.fc_pool_mean_tail(_dev(x), k=k, s=s, hardtanh=ht)
    assert m.get_last_device_error() == 0
    pooled = np.clip(oracle.maxpool2d(x.astype(np.float64), k, s), ht[0], ht[1])
    ref = np.tanh(oracle.mean_hw(pooled))
    _check(y.cpu().numpy(), ref, f"tail k={k} s={s} {shape}")


def test_unfused_conv_then_tail_matches_fused_entry():
    """The pooled entry's result equals the unfused pipeline the pages
    describe (the transposed conv as a conv with swapped, flipped weights
    and padding k - 1 - p, materialised, then the standalone tail), and
    both match the oracle."""
    inp = synth.make_inputs(2)
    x, w, b = inp["x"], inp["w"], inp["b"]
    m = fc()
    fused = m.fc_convT2d_pool_mean(_dev(x), _dev(w), _dev(b)).cpu().numpy()
    w_conv = np.ascontiguousarray(np.flip(w.transpose(1, 0, 2, 3), axis=(2, 3)))
    conv = m.fc_conv2d_epi(_dev(x), _dev(w_conv), _dev(b), (), pad=1)
    unfused = m.fc_pool_mean_tail(conv).cpu().numpy()
    assert m.get_last_device_error() == 0
    ref = oracle.convT_pool_mean(x, w, b)
    _check(fused, ref, "fused")
    _check(unfused, ref, "unfused")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape,pad,ops", [
    ((2, 8, 33, 37), 0, (("relu",), ("hardswish",))),
    ((1, 5, 20, 71), 1, (("leaky_relu", 0.2), ("clamp", -1.0, 1.0), ("gelu_erf",))),
    ((2, 16, 9, 12), 2, ()),
    ((1, 8, 11, 300), 1, (("relu",),)),       # 128-column strips plus a tail
    ((2, 64, 20, 150), 1, (("hardswish",),)),  # several channel chunks
])
def test_conv2d_stride2(variant, shape, pad, ops):
    """Stride 2 vs the oracle for every variant: odd and even extents, pads
    0-2, row-packed tiles and column strips, ragged tails.  The tensor-core
    variants stage the input in even/odd row x column sub-planes."""
    st = synth.seeded(700 + pad + shape[1])
    N, C, H, W = shape
    x = st.normal(shape)
    w = st.uniform((70, C, 3, 3), 1.0 / np.sqrt(9.0 * C))
    b = st.uniform((70,), 0.1)
    got = _run_conv_strided(variant, x, w, b, ops, pad, 2)
    _check(got, oracle.conv_epi(x, w, b, ops, stride=2, pad=pad), f"{variant} stride2 {shape} pad {pad}")


def _run_conv_strided(variant, x, w, b, ops, pad, stride, dilation=1):
    m = fc()
    m.set_variant(variant)
    try:
        f = m.fc_conv2d_epi if x.ndim == 4 else m.fc_conv3d_epi
        y = f(_dev(x), _dev(w), _dev(b), _ops_torch(ops), pad=pad, stride=stride,
              dilation=dilation)
        assert m.last_variant() == variant
        assert m.get_last_device_error() == 0
        return y.cpu().numpy()
    finally:
        m.set_variant("auto")


@pytest.mark.parametrize("variant", VARIANTS)
def test_conv3d_stride2(variant):
    st = synth.seeded(710)
    x = st.normal((2, 8, 9, 12, 35))
    w = st.uniform((64, 8, 3, 3, 3), 1.0 / np.sqrt(216.0))
    b = st.uniform((64,), 0.1)
    s = st.normal((64,))
    ops = (("leaky_relu", 0.2), ("add_channel", s), ("clamp", -1.0, 1.0), ("gelu_erf",))
    got = _run_conv_strided(variant, x, w, b, ops, 1, 2)
    _check(got, oracle.conv_epi(x, w, b, ops, stride=2, pad=1), f"{variant} conv3d stride 2")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape,stride,pad,ops", [
    ((2, 8, 33, 37), 1, 0, (("relu",), ("hardswish",))),
    ((1, 5, 20, 71), 1, 3, (("leaky_relu", 0.2), ("clamp", -1.0, 1.0), ("gelu_erf",))),
    ((1, 8, 11, 300), 1, 4, (("relu",),)),        # 128-column strips plus a tail
    ((2, 64, 20, 150), 1, 2, (("hardswish",),)),  # several channel chunks
    ((2, 8, 33, 37), 2, 2, (("relu",), ("hardswish",))),
    ((1, 8, 15, 300), 2, 1, ()),
    ((2, 16, 9, 12), 2, 4, (("tanh",),)),
])
def test_conv2d_dilation2(variant, shape, stride, pad, ops):
    """Dilation 2 (strides 1 and 2, pads 0-4) vs the oracle for every
    variant: row-packed tiles, column strips, ragged tails."""
    st = synth.seeded(720 + pad + shape[1] + 10 * stride)
    N, C, H, W = shape
    x = st.normal(shape)
    w = st.uniform((70, C, 3, 3), 1.0 / np.sqrt(9.0 * C))
    b = st.uniform((70,), 0.1)
    got = _run_conv_strided(variant, x, w, b, ops, pad, stride, dilation=2)
    ref = oracle.conv_epi(x, w, b, ops, stride=stride, pad=pad, dilation=2)
    _check(got, ref, f"{variant} dilation 2 stride {stride} {shape} pad {pad}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape,stride,pad", [
    ((2, 8, 9, 12, 35), 1, 2),
    ((2, 8, 11, 12, 20), 2, 2),
])
def test_conv3d_dilation2(variant, shape, stride, pad):
    st = synth.seeded(730 + stride)
    x = st.normal(shape)
    w = st.uniform((64, shape[1], 3, 3, 3), 1.0 / np.sqrt(27.0 * shape[1]))
    b = st.uniform((64,), 0.1)
    s = st.normal((64,))
    ops = (("leaky_relu", 0.2), ("add_channel", s), ("clamp", -1.0, 1.0), ("gelu_erf",))
    got = _run_conv_strided(variant, x, w, b, ops, pad, stride, dilation=2)
    ref = oracle.conv_epi(x, w, b, ops, stride=stride, pad=pad, dilation=2)
    _check(got, ref, f"{variant} conv3d dilation 2 stride {stride}")


@pytest.mark.parametrize("variant", ["auto"] + VARIANTS)
@pytest.mark.parametrize("stride,pad,dilation", [(2, 0, 1), (1, 2, 2)])
def test_widened_conv2d_full_size_sampled(variant, stride, pad, dilation):
    """The widened layer parameters on the full conv2d workload input
    [128,8,128,128], in the launch configuration the benchmark times, on
    sampled outputs."""
    inp = _full_inputs(3)
    m = fc()
    m.set_variant(variant)
    try:
        y = m.fc_conv2d_epi(_dev(inp["x"]), _dev(inp["w"]), _dev(inp["b"]), CHAIN_RH,
                            stride=stride, pad=pad, dilation=dilation)
        assert m.get_last_device_error() == 0
        shape = tuple(y.shape)
        e = oracle.conv_out_extent(128, 3, stride, pad, dilation)
        assert shape == (128, 64, e, e)
        idx = _sample_idx(shape, 4000, 30 + stride)
        got = y.reshape(-1)[torch.from_numpy(idx).cuda()].cpu().numpy()
    finally:
        m.set_variant("auto")
    ref = oracle.conv_epi_points(inp["x"], inp["w"], inp["b"], CHAIN_RH, idx, stride=stride,
                                 pad=pad, dilation=dilation)
    _check(got, ref, f"widened s{stride} p{pad} d{dilation} sampled [{variant}]")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", [(2, 8, 21, 40), (1, 8, 6, 7, 30)])
def test_generic_chain_every_op(variant, shape):
    """An op sequence outside the fixed chains, using every elementwise op
    (per-channel add included), with 70 output channels so the last channel
    group is partial."""
    st = synth.seeded(740 + len(shape))
    x = st.normal(shape)
    C, taps = shape[1], 9 if len(shape) == 4 else 27
    w = st.uniform((70, C) + (3,) * (len(shape) - 2), 1.0 / np.sqrt(taps * C))
    b = st.uniform((70,), 0.1)
    s = st.normal((70,))
    ops = (("relu",), ("add_channel", s), ("leaky_relu", 0.3), ("hardtanh", -0.8, 0.9),
           ("gelu_erf",), ("tanh",), ("hardswish",), ("clamp", -0.2, 0.6))
    got = _run_conv_strided(variant, x, w, b, ops, 1, 1)
    _check(got, oracle.conv_epi(x, w, b, ops, pad=1), f"{variant} generic chain {shape}")


# ------------------------------------------- stride-2 transposed conv + pool
def _run_pool_s2(variant, x, w, b, op, ht=(-1.0, 1.0)):
    m = fc()
    m.set_variant(variant)
    try:
        y = m.fc_convT2d_pool_mean(_dev(x), _dev(w), _dev(b) if b is not None else None,
                                   hardtanh=ht, stride=2, out_pad=op)
        if variant != "auto":
            assert m.last_variant() == variant
        assert m.get_last_device_error() == 0
        return y.cpu().numpy()
    finally:
        m.set_variant("auto")


@pytest.mark.parametrize("variant", ["auto", "tc_tf32x3", "tc_f16x3"])
@pytest.mark.parametrize("shape,op", [
    ((2, 64, 16, 20, 64), 1),   # several pooled rows per tile
    ((1, 8, 9, 33, 64), 0),     # C_in 8: paired taps; odd extents (floor pool)
    ((2, 16, 12, 140, 70), 1),  # 128-column strips, C_out > 64
    ((1, 3, 5, 7, 64), 0),      # C_in not a multiple of 8, tiny image
    ((1, 8, 6, 127, 64), 1),    # one pooled row of 127 per tile
])
def test_convT_stride2_pool_mean(variant, shape, op):
    """Stride-2 transposed conv (pad 1, output padding 0 or 1) + 2x2 max pool
    + hardtanh + mean + tanh, computed per output parity class, against the
    oracle's scatter-form transposed conv."""
    N, C, H, W, CO = shape
    st = synth.seeded(760 + C + op)
    x = st.normal((N, C, H, W))
    w = st.uniform((C, CO, 3, 3), 1.0 / np.sqrt(9.0 * C))
    b = st.uniform((CO,), 0.1)
    ht = (-0.5, 0.7)
    got = _run_pool_s2(variant, x, w, b, op, ht)
    ref = oracle.convT_pool_mean(x, w, b, stride=2, pad=1, out_pad=op, hardtanh=ht)
    _check(got, ref, f"{variant} convT stride 2 {shape} op {op}")


@pytest.mark.parametrize("shape,op", [((2, 16, 12, 20, 64), 1), ((1, 8, 9, 33, 70), 0)])
def test_convT_stride2_pool_mean_cuda_cores(shape, op):
    """The CUDA-core variant computes the stride-2 transposed conv with the
    general kernel (zero-inserted input staged in shared memory)."""
    N, C, H, W, CO = shape
    st = synth.seeded(765 + C + op)
    x = st.normal((N, C, H, W))
    w = st.uniform((C, CO, 3, 3), 1.0 / np.sqrt(9.0 * C))
    b = st.uniform((CO,), 0.1)
    got = _run_pool_s2("ffma", x, w, b, op, (-0.5, 0.7))
    ref = oracle.convT_pool_mean(x, w, b, stride=2, pad=1, out_pad=op, hardtanh=(-0.5, 0.7))
    _check(got, ref, f"ffma convT stride 2 {shape} op {op}")


# ------------------------------------------------------ the general layer
GENERAL_2D = [
    # (shape N C H W, C_out, k, stride, pad, dilation, chain)
    ((2, 5, 17, 23), 70, 1, 1, 0, 1, "rh"),
    ((1, 8, 20, 37), 64, 5, 1, 2, 1, "gelu"),
    ((2, 3, 19, 31), 10, 7, 2, 3, 1, "generic"),
    ((1, 16, 23, 29), 64, 5, 3, 4, 2, "rh"),
    ((1, 4, 30, 35), 64, 3, 4, 1, 3, "none"),
    ((2, 6, 14, 18), 33, 4, 2, 1, 1, "rh"),      # even kernel size
    ((1, 8, 9, 130), 64, 3, 3, 2, 4, "gelu"),    # stride 3, dilation 4, wide rows
    ((1, 64, 12, 16), 64, 7, 1, 3, 1, "none"),  # 7x7 over 64 channels (smaller chunks)
]


@pytest.mark.parametrize("variant", ["auto", "ffma"])
@pytest.mark.parametrize("case", GENERAL_2D)
def test_conv2d_general_layer(variant, case):
    """Kernel sizes 1-7, strides 3-4, dilations 3-4 and other paddings: the
    general CUDA-core kernel, against the oracle."""
    shape, CO, k, stride, pad, dil, chain = case
    st = synth.seeded(850 + k + 7 * stride + 31 * dil)
    N, C, H, W = shape
    x = st.normal(shape)
    w = st.uniform((CO, C, k, k), 1.0 / np.sqrt(k * k * C))
    b = st.uniform((CO,), 0.1)
    ops = _chain(chain, CO, st)
    m = fc()
    m.set_variant(variant)
    try:
        y = m.fc_conv2d_epi(_dev(x), _dev(w), _dev(b), _ops_torch(ops), pad=pad, stride=stride,
                            dilation=dil)
        assert m.last_variant() == "ffma"
        assert m.get_last_device_error() == 0
        got = y.cpu().numpy()
    finally:
        m.set_variant("auto")
    _check(got, oracle.conv_epi(x, w, b, ops, stride=stride, pad=pad, dilation=dil),
           f"{variant} general conv2d {case}")


@pytest.mark.parametrize("case", [
    ((1, 5, 6, 9, 11), 64, 1, 1, 0, 1),
    ((1, 8, 9, 12, 14), 70, 5, 1, 2, 1),
    ((2, 4, 11, 13, 12), 16, 3, 3, 1, 2),
    ((1, 3, 8, 9, 10), 20, 5, 2, 3, 1),
])
def test_conv3d_general_layer(case):
    shape, CO, k, stride, pad, dil = case
    st = synth.seeded(870 + k + stride)
    C = shape[1]
    x = st.normal(shape)
    w = st.uniform((CO, C, k, k, k), 1.0 / np.sqrt(k ** 3 * C))
    b = st.uniform((CO,), 0.1)
    ops = chain_gelu(st.normal((CO,)))
    got = _run_conv_strided("ffma", x, w, b, ops, pad, stride, dilation=dil)
    _check(got, oracle.conv_epi(x, w, b, ops, stride=stride, pad=pad, dilation=dil),
           f"general conv3d {case}")


@pytest.mark.parametrize("variant", ["auto", "ffma"])
@pytest.mark.parametrize("case", [
    # (N C H W, C_out, k, stride, pad, out_pad, pool)
    ((2, 8, 9, 11), 64, 3, 3, 1, 2, (2, 2)),
    ((1, 16, 7, 8), 70, 3, 4, 0, 3, (3, 2)),
    ((2, 5, 10, 9), 64, 3, 2, 0, 1, (2, 2)),
    ((1, 8, 12, 13), 64, 3, 2, 2, 0, (3, 3)),
    ((2, 4, 8, 10), 33, 5, 2, 2, 1, (2, 2)),
    ((1, 12, 11, 9), 64, 7, 1, 3, 0, (4, 2)),
    ((1, 8, 6, 7), 64, 1, 3, 0, 2, (2, 1)),
    ((2, 64, 9, 10), 64, 3, 1, 0, 0, (2, 2)),  # stride 1, pad 0: equivalent conv with pad 2
    ((1, 8, 10, 12), 64, 4, 2, 1, 0, (2, 2)),  # even kernel size
])
def test_convT_general_layer_pool_mean(variant, case):
    """Transposed conv at kernel sizes 1-7, strides 1-4, paddings and output
    paddings, with 2x2 and general pools, against the oracle's scatter form."""
    shape, CO, k, stride, pad, op, pool = case
    st = synth.seeded(890 + k + 5 * stride + 13 * pad + 29 * op)
    N, C, H, W = shape
    x = st.normal(shape)
    w = st.uniform((C, CO, k, k), 1.0 / np.sqrt(k * k * C))
    b = st.uniform((CO,), 0.1)
    ht = (-0.6, 0.8)
    m = fc()
    m.set_variant(variant)
    try:
        y = m.fc_convT2d_pool_mean(_dev(x), _dev(w), _dev(b), hardtanh=ht, pad=pad,
                                   stride=stride, out_pad=op, pool=pool)
        assert m.get_last_device_error() == 0
        got = y.cpu().numpy()
    finally:
        m.set_variant("auto")
    ref = oracle.convT_pool_mean(x, w, b, stride=stride, pad=pad, out_pad=op, pool=pool,
                                 hardtanh=ht)
    _check(got, ref, f"{variant} general convT pool mean {case}")


@pytest.mark.parametrize("variant", ["auto", "tc_tf32x3", "tc_f16x3"])
@pytest.mark.parametrize("case", [
    # (N C H W, C_out, k, stride, pad, dilation, chain, tf32 plan fits)
    ((2, 8, 20, 36), 64, 1, 1, 0, 1, "rh", True),
    ((1, 64, 9, 40), 70, 1, 1, 0, 1, "none", True),
    ((2, 8, 21, 37), 64, 5, 1, 2, 1, "gelu", True),
    ((1, 16, 19, 140), 64, 5, 2, 1, 1, "rh", True),
    ((1, 8, 25, 60), 64, 5, 1, 4, 2, "generic", True),
    ((1, 8, 23, 44), 64, 7, 1, 3, 1, "rh", False),
    ((1, 8, 30, 70), 64, 7, 2, 6, 2, "none", False),
])
def test_conv2d_kernel_sizes_tensor_cores(variant, case):
    """Square odd kernels 1, 5, 7 on the tensor-core kernel (a longer tap
    table of shifted descriptor starts), strides / dilations 1-2."""
    shape, CO, k, stride, pad, dil, chain, tf32_fits = case
    if variant == "tc_tf32x3" and not tf32_fits:
        pytest.skip("the tf32 split's K steps do not fit shared memory at this size")
    st = synth.seeded(900 + k + 7 * stride + 31 * dil)
    N, C, H, W = shape
    x = st.normal(shape)
    w = st.uniform((CO, C, k, k), 1.0 / np.sqrt(k * k * C))
    b = st.uniform((CO,), 0.1)
    ops = _chain(chain, CO, st)
    m = fc()
    m.set_variant(variant)
    try:
        y = m.fc_conv2d_epi(_dev(x), _dev(w), _dev(b), _ops_torch(ops), pad=pad, stride=stride,
                            dilation=dil)
        if variant != "auto":
            assert m.last_variant() == variant
        assert m.get_last_device_error() == 0
        got = y.cpu().numpy()
    finally:
        m.set_variant("auto")
    _check(got, oracle.conv_epi(x, w, b, ops, stride=stride, pad=pad, dilation=dil),
           f"{variant} kernel {k} conv2d {case}")


@pytest.mark.parametrize("variant", ["tc_tf32x3", "tc_f16x3"])
def test_conv3d_pointwise_tensor_cores(variant):
    st = synth.seeded(905)
    x = st.normal((1, 8, 6, 9, 20))
    w = st.uniform((64, 8, 1, 1, 1), 0.3)
    b = st.uniform((64,), 0.1)
    ops = chain_gelu(st.normal((64,)))
    got = _run_conv_strided(variant, x, w, b, ops, 0, 1)
    _check(got, oracle.conv_epi(x, w, b, ops), f"{variant} conv3d 1x1x1")


@pytest.mark.parametrize("variant", ["auto", "tc_f16x3", "ffma"])
def test_convT_kernel5_stride1_pool_mean(variant):
    """A 5 x 5 transposed conv (stride 1, pad 2) as the equivalent conv with
    flipped weights on the tensor cores, or the general CUDA-core kernel."""
    st = synth.seeded(906)
    x = st.normal((2, 16, 18, 20))
    w = st.uniform((16, 64, 5, 5), 1.0 / np.sqrt(400.0))
    b = st.uniform((64,), 0.1)
    m = fc()
    m.set_variant(variant)
    try:
        y = m.fc_convT2d_pool_mean(_dev(x), _dev(w), _dev(b), pad=2)
        if variant != "auto":
            assert m.last_variant() == variant
        assert m.get_last_device_error() == 0
        got = y.cpu().numpy()
    finally:
        m.set_variant("auto")
    _check(got, oracle.convT_pool_mean(x, w, b, pad=2), f"{variant} convT k5")


def test_general_layer_refused_by_tensor_cores():
    """Parameters outside the fixed-size kernels run on the general CUDA-core
    kernel only: the tensor-core variants refuse them, AUTO takes FFMA."""
    m = fc()
    x = _dev(np.zeros((1, 8, 12, 12), np.float32))
    w4 = _dev(np.zeros((64, 8, 4, 4), np.float32))  # even kernel size
    for v in ("tc_tf32x3", "tc_f16x3"):
        m.set_variant(v)
        try:
            with pytest.raises(m.FcError):
                m.fc_conv2d_epi(x, w4, None, (), pad=2)
            with pytest.raises(m.FcError):
                m.fc_conv2d_epi(x, _dev(np.zeros((64, 8, 3, 3), np.float32)), None, (),
                                stride=3)
            with pytest.raises(m.FcError):
                m.fc_convT2d_pool_mean(x, _dev(np.zeros((8, 64, 3, 3), np.float32)), None,
                                       stride=3, out_pad=0)
        finally:
            m.set_variant("auto")
    m.fc_conv2d_epi(x, w4, None, (), pad=2)
    assert m.last_variant() == "ffma"


def test_pooled_batch_1024_beyond_2_31_elements():
    """x [1024,64,256,256] has 2^32 elements (16 GiB): the pooled workload's
    128 images eight times over.  Offsets are 64-bit, so the call is
    accepted and every block of 128 images gives bitwise the batch-128
    result, which the whole-output test checks against the oracle."""
    inp = _full_inputs(5)
    m = fc()
    x1 = _dev(inp["x"])
    w, b = _dev(inp["w"]), _dev(inp["b"])
    y1 = m.fc_convT2d_pool_mean(x1, w, b).cpu().numpy()
    x8 = x1.repeat(8, 1, 1, 1)
    del x1
    assert x8.numel() == 1 << 32
    y8 = m.fc_convT2d_pool_mean(x8, w, b).cpu().numpy()
    assert m.get_last_device_error() == 0
    del x8
    torch.cuda.empty_cache()
    for r in range(8):
        np.testing.assert_array_equal(y8[128 * r:128 * (r + 1)], y1)
    _check(y8[:128], _full_ref(5), "batch 1024 vs the oracle")


def test_pooled_cta_pairs_ragged_strips():
    """x [32,64,256,200]: 8192 pooled units, so the fp16 split runs on CTA
    pairs, with a ragged second column strip (72 of 128 columns).  Sampled
    (n, c) outputs against the oracle, and the first 16 images bitwise
    against a 16-image call (4096 units: single CTAs)."""
    inp = _full_inputs(5)
    x = np.ascontiguousarray(inp["x"][:32, :, :, :200])
    w, b = inp["w"], inp["b"]
    m = fc()
    m.set_variant("tc_f16x3")
    try:
        y32 = m.fc_convT2d_pool_mean(_dev(x), _dev(w), _dev(b)).cpu().numpy().reshape(32, 64)
        assert m.get_last_device_error() == 0
        y16 = m.fc_convT2d_pool_mean(_dev(x[:16]), _dev(w), _dev(b)).cpu().numpy().reshape(16, 64)
        assert m.get_last_device_error() == 0
    finally:
        m.set_variant("auto")
    np.testing.assert_array_equal(y32[:16], y16)
    rng = np.random.default_rng(11)
    pairs = [(0, 0), (31, 63), (17, 5)] + [(int(rng.integers(32)), int(rng.integers(64)))
                                           for _ in range(13)]
    ref = oracle.convT_pool_mean_points(x, w, b, pairs)
    got = np.array([y32[n, c] for n, c in pairs])
    _check(got, ref, "CTA pairs, ragged strips")


@pytest.mark.parametrize("variant", ["auto", "tc_tf32x3", "tc_f16x3"])
def test_convT_stride2_full_size_sampled(variant):
    """x [128,64,128,128] -> transposed conv 256 x 256 (stride 2, output
    padding 1) -> pooled 128 x 128 -> mean: sampled (n, c) outputs."""
    inp = _full_inputs(5)
    x = inp["x"][:, :, ::2, ::2].copy()  # 128 x 64 x 128 x 128 from the same draw
    m = fc()
    m.set_variant(variant)
    try:
        y = m.fc_convT2d_pool_mean(_dev(x), _dev(inp["w"]), _dev(inp["b"]), stride=2, out_pad=1)
        assert m.get_last_device_error() == 0
        ynp = y.cpu().numpy().reshape(128, 64)
    finally:
        m.set_variant("auto")
    rng = np.random.default_rng(7)
    pairs = [(0, 0), (127, 63)] + [(int(rng.integers(128)), int(rng.integers(64)))
                                   for _ in range(14)]
    ref = oracle.convT_pool_mean_points(x, inp["w"], inp["b"], pairs, stride=2, pad=1, out_pad=1)
    got = np.array([ynp[n, c] for n, c in pairs])
    _check(got, ref, f"convT stride 2 sampled [{variant}]")


# ------------------------------------------- general max-pool windows (fused)
@pytest.mark.parametrize("variant", ["auto", "ffma", "tc_tf32x3", "tc_f16x3"])
@pytest.mark.parametrize("shape,pool", [
    ((2, 16, 17, 21, 64), (3, 2)),   # overlapping windows, odd extents
    ((1, 8, 12, 40, 70), (2, 1)),    # stride 1: every conv output in 4 windows
    ((2, 64, 13, 14, 64), (3, 3)),   # non-overlapping 3x3
    ((1, 5, 9, 35, 64), (4, 2)),     # 4x4 windows, C_in not a multiple of 8
    ((1, 8, 6, 7, 64), (1, 1)),      # window 1: plain mean of the clamped conv
    ((1, 8, 20, 40, 70), (4, 4)),    # non-overlapping 4x4, TMA-eligible width
    ((1, 64, 9, 300, 64), (3, 3)),   # 128-column strips of 42 windows
    ((2, 8, 9, 260, 64), (3, 2)),    # strips of 63 overlapping windows
])
def test_convT_general_pool_mean(variant, shape, pool):
    """Transposed conv (stride 1, pad 1) + max pool of any window / stride
    (floor extent) + hardtanh + mean + tanh in one pass, against the oracle:
    the CUDA-core kernel (each thread its window) and the tensor-core kernel
    (one tile per window row, the windows taken in shared memory)."""
    N, C, H, W, CO = shape
    st = synth.seeded(780 + pool[0] * 4 + pool[1])
    x = st.normal((N, C, H, W))
    w = st.uniform((C, CO, 3, 3), 1.0 / np.sqrt(9.0 * C))
    b = st.uniform((CO,), 0.1)
    ht = (-0.6, 0.9)
    m = fc()
    m.set_variant(variant)
    try:
        y = m.fc_convT2d_pool_mean(_dev(x), _dev(w), _dev(b), hardtanh=ht, pool=pool)
        if variant != "auto":
            assert m.last_variant() == variant
        assert m.get_last_device_error() == 0
        got = y.cpu().numpy()
    finally:
        m.set_variant("auto")
    ref = oracle.convT_pool_mean(x, w, b, pool=pool, hardtanh=ht)
    _check(got, ref, f"{variant} general pool {pool} {shape}")


@pytest.mark.parametrize("variant", ["tc_tf32x3", "tc_f16x3"])
def test_general_pool_deterministic_tensor_cores(variant):
    st = synth.seeded(788)
    x = st.normal((2, 16, 17, 21))
    w = st.uniform((16, 64, 3, 3), 0.08)
    b = st.uniform((64,), 0.1)
    m = fc()
    m.set_variant(variant)
    try:
        a = m.fc_convT2d_pool_mean(_dev(x), _dev(w), _dev(b), pool=(3, 2)).cpu().numpy()
        for _ in range(3):
            np.testing.assert_array_equal(
                m.fc_convT2d_pool_mean(_dev(x), _dev(w), _dev(b), pool=(3, 2)).cpu().numpy(), a)
    finally:
        m.set_variant("auto")


# ------------------------------------------------ channels-last (N(D)HWC)
@pytest.mark.parametrize("variant", ["auto", "tc_tf32x3", "tc_f16x3"])
@pytest.mark.parametrize("shape,pad,dil,chain", [
    ((2, 8, 33, 37, 64), 0, 1, "rh"),
    ((1, 12, 17, 20, 70), 1, 1, "gelu"),      # C_in, C_out not multiples of 4 / 64
    ((1, 16, 9, 150, 64), 2, 2, "generic"),   # strips, dilation 2
    ((2, 64, 10, 30, 64), 1, 1, "none"),      # several channel chunks
])
def test_conv2d_channels_last(variant, shape, pad, dil, chain):
    N, C, H, W, CO = shape
    st = synth.seeded(790 + C + pad)
    x = st.normal((N, C, H, W))
    w = st.uniform((CO, C, 3, 3), 1.0 / np.sqrt(9.0 * C))
    b = st.uniform((CO,), 0.1)
    ops = _chain(chain, CO, st)
    m = fc()
    m.set_variant(variant)
    try:
        xl = torch.from_numpy(np.ascontiguousarray(x.transpose(0, 2, 3, 1))).cuda()
        y = m.fc_conv2d_epi_nhwc(xl, _dev(w), _dev(b), _ops_torch(ops), pad=pad, dilation=dil)
        if variant != "auto":
            assert m.last_variant() == variant
        assert m.get_last_device_error() == 0
        got = y.cpu().numpy().transpose(0, 3, 1, 2)
    finally:
        m.set_variant("auto")
    _check(got, oracle.conv_epi(x, w, b, ops, pad=pad, dilation=dil),
           f"{variant} channels-last conv2d {shape}")


@pytest.mark.parametrize("variant", ["auto", "tc_f16x3"])
def test_conv3d_channels_last(variant):
    st = synth.seeded(795)
    x = st.normal((2, 8, 6, 10, 30))
    w = st.uniform((64, 8, 3, 3, 3), 1.0 / np.sqrt(216.0))
    b = st.uniform((64,), 0.1)
    s = st.normal((64,))
    ops = chain_gelu(s)
    m = fc()
    m.set_variant(variant)
    try:
        xl = torch.from_numpy(np.ascontiguousarray(x.transpose(0, 2, 3, 4, 1))).cuda()
        y = m.fc_conv3d_epi_ndhwc(xl, _dev(w), _dev(b), _ops_torch(ops), pad=1)
        assert m.get_last_device_error() == 0
        got = y.cpu().numpy().transpose(0, 4, 1, 2, 3)
    finally:
        m.set_variant("auto")
    _check(got, oracle.conv_epi(x, w, b, ops, pad=1), f"{variant} channels-last conv3d")


def test_channels_last_refused_by_cuda_core_and_stride2():
    m = fc()
    x = torch.zeros((1, 8, 8, 8), device="cuda")
    w = _dev(np.zeros((64, 8, 3, 3), np.float32))
    m.set_variant("ffma")
    try:
        with pytest.raises(m.FcError):
            m.fc_conv2d_epi_nhwc(x, w, None, ())
    finally:
        m.set_variant("auto")
    with pytest.raises(m.FcError):
        m.fc_conv2d_epi_nhwc(x, w, None, (), stride=2)


# ------------------------------------------------------------ size limits
@pytest.mark.parametrize("variant", VARIANTS)
def test_very_wide_rows_sampled(variant):
    """Rows of 2048 outputs: 16 tensor-core column strips plus a ragged one."""
    st = synth.seeded(800)
    x = st.normal((1, 8, 5, 2050))
    w = st.uniform((64, 8, 3, 3), 1.0 / np.sqrt(72.0))
    b = st.uniform((64,), 0.1)
    m = fc()
    m.set_variant(variant)
    try:
        y = m.fc_conv2d_epi(_dev(x), _dev(w), _dev(b), CHAIN_RH, pad=1)
        assert m.get_last_device_error() == 0
        shape = tuple(y.shape)
        idx = _sample_idx(shape, 3000, 800)
        got = y.reshape(-1)[torch.from_numpy(idx).cuda()].cpu().numpy()
    finally:
        m.set_variant("auto")
    ref = oracle.conv_epi_points(x, w, b, CHAIN_RH, idx, pad=1)
    _check(got, ref, f"{variant} wide rows")


@pytest.mark.parametrize("variant", VARIANTS)
def test_largest_channel_block(variant):
    """C_in 256 (16 fp16 chunks) and C_out 512, the most output channels the
    tensor-core kernel stages: the weights no longer fit shared memory and
    stream through the weight ring."""
    st = synth.seeded(801)
    x = st.normal((1, 256, 6, 40))
    w = st.uniform((512, 256, 3, 3), 1.0 / np.sqrt(2304.0))
    b = st.uniform((512,), 0.1)
    got = _run_conv(variant, x, w, b, (("relu",),), pad=1)
    _check(got, oracle.conv_epi(x, w, b, (("relu",),), pad=1), f"{variant} C 256 -> 512")


def test_output_channels_beyond_the_tensor_core_block():
    """C_out 520 > 512: the tensor-core variants refuse (FC_ERR_UNSUPPORTED),
    AUTO runs the CUDA-core kernel."""
    st = synth.seeded(802)
    x = st.normal((1, 8, 7, 9))
    w = st.uniform((520, 8, 3, 3), 1.0 / np.sqrt(72.0))
    b = st.uniform((520,), 0.1)
    m = fc()
    for v in ("tc_tf32x3", "tc_f16x3"):
        m.set_variant(v)
        try:
            with pytest.raises(m.FcError):
                m.fc_conv2d_epi(_dev(x), _dev(w), _dev(b), ())
        finally:
            m.set_variant("auto")
    y = m.fc_conv2d_epi(_dev(x), _dev(w), _dev(b), ())
    assert m.last_variant() == "ffma"
    _check(y.cpu().numpy(), oracle.conv_epi(x, w, b, ()), "C_out 520 auto")

"""Failure detection on the GPU without a fault, and guard bands.

* The conv kernels' waits on mbarriers are bounded: on expiry a wait records
  where it gave up, sets FC_ERR_TIMEOUT in the device status word and raises
  the block's abort flag, which ends the block's other waits.  The self-test
  entry point runs that routine on barriers that nothing completes, with a
  20 ms limit; the status, both wait records and the prompt end of the
  second wait (its own limit is 4 s) are checked, and a conv call afterwards
  shows the context is still usable.
* Guard bands: sentinel bytes before and after y, and after the workspace
  the library asked for, are unchanged after each entry point runs.
"""
import time

import numpy as np
import pytest

import oracle
from convolution_epilogue_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _fc():
    from convolution_epilogue_gb300 import _build
    _build.build()
    import convolution_epilogue_gb300 as fc
    return fc


def test_bounded_wait_gives_up_reports_and_leaves_context_usable():
    fc = _fc()
    fc.get_last_device_error()
    fc.wait_report()  # start from a clean status area
    t0 = time.perf_counter()
    fc.selftest_wait_timeout(20000)  # 20 ms
    status = fc.get_last_device_error()  # synchronises
    dt = time.perf_counter() - t0
    assert status == 6, f"expected FC_ERR_TIMEOUT, got {status}"
    n, recs = fc.wait_report()
    tags = sorted(r["tag"] for r in recs)
    assert n == 2 and tags == ["0x71000001", "0x79000002"], recs
    assert all(r["block"] == 0 for r in recs)
    assert dt < 2.0, f"the abort flag did not end the second wait ({dt:.2f} s)"
    assert fc.get_last_device_error() == 0 and fc.wait_report()[0] == 0
    # the context still runs kernels correctly
    inp = synth.make_inputs(1)
    d = {k: torch.from_numpy(v).cuda() for k, v in inp.items()}
    y = fc.fc_conv2d_epi(d["x"], d["w"], d["b"], (("relu",), ("hardswish",)))
    assert fc.get_last_device_error() == 0
    ref = oracle.conv_epi(inp["x"], inp["w"], inp["b"], (("relu",), ("hardswish",)))
    err = np.abs(y.double().cpu().numpy() - ref)
    assert (err <= 1e-4 + 1e-4 * np.abs(ref)).all()


def test_selftest_rejects_bad_limits():
    fc = _fc()
    L = fc.lib()
    assert L.fc_selftest_wait_timeout(0, None) == 1
    assert L.fc_selftest_wait_timeout(1000001, None) == 1


G = 1024  # guard elements (4 KiB) on each side


def _guarded(shape):
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * G,), 12345.0, device="cuda")
    return buf, buf[G:G + n].view(*shape)


def _guarded_ws(nbytes):
    buf = torch.full((nbytes + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
    return buf, buf[:nbytes]


def _check_guards(buf, what):
    b = buf.cpu().numpy()
    assert (b[:G] == 12345.0).all() and (b[-G:] == 12345.0).all(), f"{what}: write outside y"


def _check_ws_guard(buf, nbytes, what):
    assert (buf[nbytes:].cpu().numpy() == 0xA5).all(), f"{what}: write past the workspace"


@pytest.mark.parametrize("variant", ["ffma", "tc_tf32x3", "tc_f16x3"])
def test_no_writes_outside_y_or_workspace(variant):
    fc = _fc()
    st = synth.seeded(4242)
    fc.set_variant(variant)
    try:
        # conv2d, ragged: 3 tiles of rows plus a tail, 70 channels
        x = torch.from_numpy(st.normal((2, 8, 19, 40))).cuda()
        w = torch.from_numpy(st.uniform((70, 8, 3, 3), 0.1)).cuda()
        b = torch.from_numpy(st.uniform((70,), 0.1)).cuda()
        buf, y = _guarded((2, 70, 17, 38))
        need = fc.workspace_bytes(0, (2, 8, 19, 40, 70, 3, 0))
        wbuf, ws = _guarded_ws(need)
        fc.fc_conv2d_epi(x, w, b, (("relu",),), y=y, ws=ws)
        assert fc.get_last_device_error() == 0
        _check_guards(buf, "conv2d")
        _check_ws_guard(wbuf, need, "conv2d")
        # conv3d
        x = torch.from_numpy(st.normal((1, 8, 5, 9, 70))).cuda()
        w = torch.from_numpy(st.uniform((64, 8, 3, 3, 3), 0.1)).cuda()
        buf, y = _guarded((1, 64, 3, 7, 68))
        need = fc.workspace_bytes(1, (1, 8, 5, 9, 70, 64, 3, 0))
        wbuf, ws = _guarded_ws(need)
        fc.fc_conv3d_epi(x, w, None, (), y=y, ws=ws)
        assert fc.get_last_device_error() == 0
        _check_guards(buf, "conv3d")
        _check_ws_guard(wbuf, need, "conv3d")
        # pooled transposed conv
        x = torch.from_numpy(st.normal((2, 16, 10, 36))).cuda()
        w = torch.from_numpy(st.uniform((16, 64, 3, 3), 0.1)).cuda()
        buf, y = _guarded((2, 64, 1, 1))
        need = fc.workspace_bytes(2, (2, 16, 10, 36, 64, 3, 1))
        wbuf, ws = _guarded_ws(need)
        fc.fc_convT2d_pool_mean(x, w, None, y=y, ws=ws)
        assert fc.get_last_device_error() == 0
        _check_guards(buf, "convT pool")
        _check_ws_guard(wbuf, need, "convT pool")
    finally:
        fc.set_variant("auto")

"""The benchmark's host-side arithmetic, checked without a GPU.

The reported throughput and roofline fractions rest on a few host
functions of bench.py: the MAC count and the algorithmic bytes of each
workload, the peak of the pipe a variant uses, the roofline time, the DRAM
traffic figure taken from an ncu capture, and the parsing of the clock
samples.  They are checked here against the values the pages print
(tests/golden/page_values.txt), against output extents that PyTorch's own
shape inference gives on meta tensors (no data, no compute), and against
closed forms on made-up peaks.
"""
import os
import shutil
import sys

import pytest
import torch
import torch.nn.functional as F

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from convolution_epilogue_gb300 import synth  # noqa: E402

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


def _meta_output_shape(wid):
    """Output shape of a workload's convolution from PyTorch's shape
    inference on meta tensors (stride 1; the transposed conv has pad 1)."""
    spec = synth.WORKLOADS[wid]
    C, CO, k = spec["x"][1], spec["cout"], spec["k"]
    x = torch.empty(spec["x"], device="meta")
    if spec["kind"] == "conv2d":
        return tuple(F.conv2d(x, torch.empty(CO, C, k, k, device="meta")).shape)
    if spec["kind"] == "conv3d":
        return tuple(F.conv3d(x, torch.empty(CO, C, k, k, k, device="meta")).shape)
    w = torch.empty(C, CO, k, k, device="meta")  # transposed conv: (C_in, C_out, k, k)
    return tuple(F.conv_transpose2d(x, w, stride=1, padding=1).shape)


def _numel(shape):
    n = 1
    for s in shape:
        n *= s
    return n


def _taps(wid):
    spec = synth.WORKLOADS[wid]
    return spec["k"] ** (3 if spec["kind"] == "conv3d" else 2)


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_macs_are_outputs_times_cin_times_taps(wid):
    """Every output sums C_in x taps products (the transposed conv, written
    as a gather with flipped taps, too): MACs = conv outputs x C_in x taps,
    with the conv outputs counted before any pooling."""
    out = _meta_output_shape(wid)
    C = synth.WORKLOADS[wid]["x"][1]
    assert bench.macs_of(wid) == _numel(out) * C * _taps(wid)


def test_macs_match_the_pages():
    assert bench.macs_of(4) == G["conv3d_macs@cfg4"][0]
    assert bench.macs_of(5) == G["convT_macs@cfg5"][0]
    # conv2d: the page's output count times C_in x taps (8 x 9)
    assert bench.macs_of(3) == G["conv2d_output_elements@cfg3"][0] * 8 * 9


def test_algorithmic_bytes_match_the_pages_traffic_paragraph():
    """The conv2d trace itemises the fused kernel's traffic: input, weights,
    output, each once."""
    x_bytes = 4 * _numel(synth.WORKLOADS[3]["x"])
    w_bytes = 4 * 64 * 8 * 9
    v, tol = G["conv2d_input_bytes@cfg3"]
    assert abs(x_bytes - v) <= tol
    v, tol = G["conv2d_weight_bytes@cfg3"]
    assert abs(w_bytes - v) <= tol
    v, tol = G["conv2d_fused_traffic@cfg3"]
    assert abs(bench.algorithmic_bytes(3) - v) <= tol


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_algorithmic_bytes_are_inputs_and_outputs_once(wid):
    spec = synth.WORKLOADS[wid]
    C, CO = spec["x"][1], spec["cout"]
    out = _meta_output_shape(wid)
    nw = CO * C * _taps(wid)
    extra = CO * (2 if spec["kind"] == "conv3d" else 1)  # bias (+ the per-channel addend)
    ny = _numel(out) if spec["kind"] != "convT_pool_mean" else out[0] * CO  # one mean per (n, c)
    assert bench.algorithmic_bytes(wid) == 4 * (_numel(spec["x"]) + nw + extra + ny)


PEAKS = dict(hbm_gbs=6000.0, bf16=1800.0, bf16_sus=1500.0, sm_max_mhz=2000.0, source="test")


def test_pipe_peaks_closed_forms():
    pk, kind, _ = bench.pipe_peak_tflops("tc_f16x3", PEAKS)
    assert kind == "tensor" and pk == pytest.approx(600.0)
    pk, _, _ = bench.pipe_peak_tflops("tc_f16x3", PEAKS, basis="sustained")
    assert pk == pytest.approx(500.0)
    pk, kind, _ = bench.pipe_peak_tflops("tc_tf32x3", PEAKS)
    assert kind == "tensor" and pk == pytest.approx(1800.0 * 1.1 / 2.25 / 3.0)
    pk, kind, _ = bench.pipe_peak_tflops("ffma", PEAKS)
    # 152 SMs x 128 FMA lanes x 2 FLOP x 2.0 GHz
    assert kind == "alu" and pk == pytest.approx(152 * 128 * 2 * 2.0e9 / 1e12)


def test_roofline_takes_the_slower_bound():
    # 600 GFLOP at 600 TF/s = 1 ms; 3 GB at 6000 GB/s = 0.5 ms -> tensor-bound
    ms, bound = bench.roofline_ms(600e9, 3e9, "tc_f16x3", PEAKS)
    assert bound == "tensor" and ms == pytest.approx(1.0)
    # 12 GB at 6000 GB/s = 2 ms -> HBM-bound
    ms, bound = bench.roofline_ms(600e9, 12e9, "tc_f16x3", PEAKS)
    assert bound == "hbm" and ms == pytest.approx(2.0)
    # the nominal 8 TB/s basis replaces only the bandwidth
    ms, bound = bench.roofline_ms(600e9, 12e9, "tc_f16x3", PEAKS, hbm_gbs=bench.NOMINAL_HBM_GBS)
    assert bound == "hbm" and ms == pytest.approx(1.5)


def test_ncu_traffic_is_null_once_the_kernel_sources_change(tmp_path, monkeypatch):
    for key, entry in bench.NCU_TRAFFIC.items():
        monkeypatch.setattr(bench, "kernel_src_digest", lambda e=entry: e["src"])
        assert bench.ncu_traffic(*key) == entry["bytes"]
        monkeypatch.setattr(bench, "kernel_src_digest", lambda: "0" * 16)
        assert bench.ncu_traffic(*key) is None
    monkeypatch.undo()
    assert bench.ncu_traffic(5, "no-such-variant") is None
    # the digest covers every kernel source: one changed byte changes it
    csrc = tmp_path / "convolution_epilogue_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES:
        shutil.copy(os.path.join(ROOT, "convolution_epilogue_gb300", "csrc", f), csrc / f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d0 = bench.kernel_src_digest()
    assert len(d0) == 16
    for f in bench.KERNEL_SOURCES:
        p = csrc / f
        data = p.read_bytes()
        p.write_bytes(data + b" ")
        assert bench.kernel_src_digest() != d0, f
        p.write_bytes(data)
    assert bench.kernel_src_digest() == d0


def test_stored_traffic_is_close_to_the_algorithmic_bytes():
    """A capture whose DRAM bytes sit far above the algorithmic bytes would
    mean re-reads; far below, that the capture missed most of the launch."""
    for (wid, _variant), entry in bench.NCU_TRAFFIC.items():
        r = entry["bytes"] / bench.algorithmic_bytes(wid)
        assert 0.85 < r < 1.10, (wid, r)


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_sampler_parses_medians_and_reasons(tmp_path):
    rows = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1350.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, [N/A], 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage",
    ]
    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(rows) + "\n")
    s = bench.ClockSampler(0)
    s.proc, s.path, s.out = _FakeProc(), str(path), open(os.devnull, "w")
    got = s.stop()
    assert got["sm_mhz"] == 2070.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["sw_power_cap"] and got["samples"] == 3
    assert not path.exists()

    rows = ["0, 1400, 2070, 800.0, 0x8, Active, Not Active, Active, Not Active"] * 3
    path.write_text("\n".join(rows) + "\n")
    s = bench.ClockSampler(0)
    s.proc, s.path, s.out = _FakeProc(), str(path), open(os.devnull, "w")
    got = s.stop()
    assert got["sm_mhz"] == 1400.0
    assert got["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_sampler_without_nvidia_smi():
    s = bench.ClockSampler(0)
    got = s.stop()
    assert got["sm_mhz"] is None and got["reasons"] == ["nvidia-smi unavailable"]


def test_cpu_sample_counts_the_macs_it_runs():
    """One image of conv2d and of conv3d (whole planes) and 16 pooled
    (n, c_out) outputs, each a full 256 x 256 conv plane of 64 x 9 MACs."""
    _run, macs, desc = bench.cpu_sample(1)
    per3 = _numel(_meta_output_shape(3)[1:]) * 8 * 9
    per4 = _numel(_meta_output_shape(4)[1:]) * 8 * 27
    per5 = 256 * 256 * 64 * 9
    assert macs == per3 + per4 + 16 * per5
    assert "1 image(s)" in desc and "16 (n, c_out)" in desc


def _run_bench(args, env_extra=None):
    import subprocess
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT,
                          env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` times the CPU oracle on a bounded sample and
    prints one JSON line with the contract's keys (no GPU needed)."""
    import json
    r = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "0", "--ref-scale", "1"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["warmup"] >= 3 and d["steps"] == 1 and d["value"] > 0
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    _run, macs, desc = bench.cpu_sample(1)
    assert d["value"] == pytest.approx(2.0 * macs / (d["ms_per_step"] * 1e-3) / 1e9, rel=1e-9)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["sample"] == desc == d["config"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "0", "--ref-scale", "1"],
                   {"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_profile_pool_parsing():
    assert bench.parse_pool("3,2") == (3, 2) and bench.parse_pool("2,2") == (2, 2)
    for bad in ("3", "0,2", "5,1", "3,2,1", "a,b", ""):
        with pytest.raises(ValueError):
            bench.parse_pool(bad)
    r = _run_bench(["--profile-workload", "5", "--profile-pool", "9,9"])
    assert r.returncode != 0 and "--profile-pool" in r.stderr


def test_install_variant_table_reproduces_the_committed_header(tmp_path):
    """Installing the committed measurements into copies of the library's
    table files gives the committed files back, byte for byte; a changed
    measurement reaches the header's row."""
    import json
    csrc = os.path.join(ROOT, "convolution_epilogue_gb300", "csrc")
    for f in ("fc_variant_table.h", "fc_variant_table.json"):
        shutil.copy(os.path.join(csrc, f), tmp_path / f)
    src = tmp_path / "measured.json"
    shutil.copy(os.path.join(csrc, "fc_variant_table.json"), src)
    n = bench.install_variant_table(str(src), str(tmp_path))
    for f in ("fc_variant_table.h", "fc_variant_table.json"):
        with open(os.path.join(csrc, f), "rb") as a:
            assert (tmp_path / f).read_bytes() == a.read(), f
    tab = json.loads(src.read_text())
    assert n == len(tab["rows"])
    tab["rows"][0]["ms"][0] = 9.87654
    tab["gpu"] = "TEST GPU"
    src.write_text(json.dumps(tab))
    bench.install_variant_table(str(src), str(tmp_path))
    h = (tmp_path / "fc_variant_table.h").read_text()
    assert "{9.87654f," in h and "// Measured on TEST GPU (fc_variant_table.json" in h

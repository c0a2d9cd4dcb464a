"""The automatic choice against the measured table it compiles in (no GPU).

`python bench.py --variant-table T.json` times every (variant, input
staging) pair on a grid of shapes on a GB300 and writes the measurements;
`python bench.py --install-variant-table T.json` copies them into
convolution_epilogue_gb300/csrc/fc_variant_table.json and the C rows the
library compiles in (fc_variant_table.h).  These tests check that the
compiled rows are those measurements, and that for every measured shape the
library's selection (fc_select_variant, which runs no kernel) is the
variant of the fastest measured pair.
"""
import json
import os

import pytest

import convolution_epilogue_gb300 as fc
from convolution_epilogue_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "convolution_epilogue_gb300", "csrc")
TABLE_JSON = os.path.join(CSRC, "fc_variant_table.json")
TABLE_H = os.path.join(CSRC, "fc_variant_table.h")
COL_VARIANT = ["ffma", "tc_tf32x3", "tc_tf32x3", "tc_f16x3", "tc_f16x3"]


@pytest.fixture(scope="module")
def table():
    if not os.path.exists(TABLE_JSON):
        pytest.skip("no measured table committed")
    _build.build()
    with open(TABLE_JSON) as f:
        return json.load(f)


def _query(row):
    e, d = row["entry"], row["dims"]
    if e == 0:
        return (4 if d[9] else 0), d[:9]
    if e == 1:
        return (5 if d[10] else 1), d[:10]
    return 2, d


def test_compiled_rows_are_the_measurements(table):
    import bench
    text = open(TABLE_H).read()
    assert bench.variant_table_header(table) in text
    assert len(table["rows"]) == len(bench.TABLE_SHAPES)


def test_selection_is_the_fastest_measured_variant(table):
    fc.set_variant("auto")
    fc.set_staging("auto")
    for row in table["rows"]:
        ms = row["ms"]
        cands = [i for i, m in enumerate(ms) if m >= 0]
        assert cands, row
        best = min(cands, key=lambda i: ms[i])
        entry, dims = _query(row)
        got = fc.select_variant(entry, dims)
        assert got == COL_VARIANT[best], (row["dims"], got, ms)


def test_override_and_unsupported_queries(table):
    # an override is reported as such when the problem supports it
    fc.set_variant("ffma")
    try:
        assert fc.select_variant(0, (128, 8, 128, 128, 64, 3, 1, 0, 1)) == "ffma"
        assert fc.select_variant(4, (1, 8, 32, 32, 64, 3, 1, 0, 1)) == "none"  # no channels-last FFMA
    finally:
        fc.set_variant("auto")
    # parameters only the general CUDA-core kernel computes
    assert fc.select_variant(0, (1, 8, 20, 20, 64, 4, 1, 1, 1)) == "ffma"
    assert fc.select_variant(2, (1, 8, 10, 10, 64, 3, 3, 1, 2, 2, 2)) == "ffma"
    # invalid problems
    assert fc.select_variant(0, (1, 8, 2, 2, 64, 3, 1, 0, 1)) == "none"
    assert fc.select_variant(9, (1,) * 11) == "none"

"""The benchmark's byte accounting, on the CPU.

Every GB/s figure is algorithmic bytes over time: inputs read once, outputs written once, gamma
once per launch. These tests pin the counts for the five workloads to the per-element costs of the
method (16-bit input and residual read, residual_output written, E4M3 codes 1 B, packed E2M1
0.5 B, one scale byte per 16 or 32 elements, one fp32 scale per FP8 row, the fp32 global scale
read once). They then check the widened-row variants against the same definitions."""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def _expected(mode, rows, hidden, e, residual, scale_bytes=4):
    n = rows * hidden
    b = n * e + hidden * e                           # input, gamma
    if residual:
        b += 2 * n * e                               # residual in, residual_output out
    if mode == "fp8":
        return b + n + rows * scale_bytes
    if mode == "nvfp4":
        return b + n // 2 + n // 16 + 4
    return b + n // 2 + n // 32


@pytest.mark.parametrize("name,rows,hidden,value", [
    ("fp8_small", None, None, 794_880),
    ("fp8_residual", None, None, 234_921_984),
    ("fp8_gemma", None, None, 939_606_016),
    ("nvfp4", None, None, 601_896_964),
    ("mxfp4_residual", 1, 2048, 17_472),
    ("mxfp4_residual", 65536, 16384, 7_012_909_056),
])
def test_workload_bytes(name, rows, hidden, value):
    w = W.config(name, rows=rows, hidden=hidden)
    assert w.algorithmic_bytes() == value
    assert value == _expected(w.mode, w.rows, w.hidden, 2, w.residual)


def test_bench_step_bytes_are_the_three_launches():
    total = sum(bench.mode_bytes(m, 8192, 4096) for m in bench.MODES)
    assert total == sum(_expected(m, 8192, 4096, 2, True) for m in bench.MODES)
    assert bench.mode_bytes("fp8", 8192, 4096) == 234_921_984


@pytest.mark.parametrize("case", bench.next_row_cases(), ids=lambda c: "%s-%s-%dx%d" % (
    c[1], c[2].mode, c[2].rows, c[2].hidden))
def test_next_row_bytes(case):
    _, name, w, opts = case
    assert bench.variant_bytes(w, {}) == w.algorithmic_bytes()
    e = torch.tensor([], dtype=opts.get("dtype", w.torch_dtype)).element_size()
    got = bench.variant_bytes(w, opts)
    if opts.get("prepass"):
        n = w.rows * w.hidden
        assert got == n * e * (2 if w.residual else 1) + w.hidden * e + 4
    elif "scale_dtype" in opts:
        assert got == _expected(w.mode, w.rows, w.hidden, e, w.residual, scale_bytes=2)
    else:
        assert got == _expected(w.mode, w.rows, w.hidden, e, w.residual)
    if opts.get("swizzled"):
        # whole 128 x 4 tiles: the swizzled layout writes exactly the row-major scale bytes
        import rmsnorm_precision_activation_gb300 as rq
        block = 16 if w.mode == "nvfp4" else 32
        assert rq.swizzled_scale_numel(w.rows, w.hidden, block) == w.rows * w.hidden // block

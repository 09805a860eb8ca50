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


def test_bench_step_is_the_three_large_workloads():
    # the step times each mode on its large workload at the stated shape
    st = bench.STEP_WORKLOADS
    assert (st["fp8"].name, st["fp8"].rows, st["fp8"].hidden, st["fp8"].dtype) == \
        ("fp8_gemma", 16384, 8192, "fp16")
    assert st["fp8"].residual and st["fp8"].weight_offset == 1.0 and st["fp8"].scale_ub == 10.0
    assert (st["nvfp4"].name, st["nvfp4"].rows, st["nvfp4"].hidden, st["nvfp4"].residual) == \
        ("nvfp4", 32768, 7168, False)
    assert (st["mxfp4"].name, st["mxfp4"].rows, st["mxfp4"].hidden, st["mxfp4"].residual) == \
        ("mxfp4_residual", 65536, 16384, True)
    total = sum(w.algorithmic_bytes() for w in st.values())
    assert total == 939_606_016 + 601_896_964 + 7_012_909_056
    assert total == sum(_expected(w.mode, w.rows, w.hidden, 2, w.residual) for w in st.values())


def test_both_arms_report_the_same_config():
    # the reference arm's line carries the config of the step it stands beside
    a = bench.step_config(bench.STEP_WORKLOADS, 1)
    b = bench.step_config(bench.parse_step_workloads(""), 1)
    assert a == b
    assert "fp8_gemma 16384x8192 fp16 +residual offset 1 ub 10" in a["workload"]
    assert "mxfp4_residual 65536x16384 bf16 +residual" in a["workload"]
    # about 5 GB of distinct inputs per step: no L2 flush needed
    assert "no flush" in a["l2"] and int(a["l2"].split()[4]) > 4000


def test_step_override_and_oracle_sample_sizes():
    ws = bench.parse_step_workloads("fp8=fp8_residual,mxfp4=mxfp4_residual:4096:2048")
    assert list(ws) == ["fp8", "mxfp4"] and ws["mxfp4"].rows == 4096
    with pytest.raises(SystemExit):
        bench.parse_step_workloads("fp8=nvfp4")
    s = bench.sample_workloads(bench.STEP_WORKLOADS, 1.0 / 8)
    assert [w.rows for w in s.values()] == [2048, 4096, 8192]
    assert all(w.hidden == bench.STEP_WORKLOADS[m].hidden for m, w in s.items())
    tiny = bench.sample_workloads(bench.STEP_WORKLOADS, 1e-9)
    assert all(w.rows == 1 for w in tiny.values())


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


@pytest.mark.parametrize("name,rows,hidden", [("fp8_gemma", 16384, 8192), ("nvfp4", 32768, 7168),
                                              ("mxfp4_residual", 65536, 16384),
                                              ("mxfp4_residual", 1, 2048), ("fp8_small", 64, 4096)])
@pytest.mark.parametrize("chunk_bytes", [1 << 20, 64 << 20, bench.E2E_CHUNK_BYTES])
def test_e2e_chunks_cover_every_row_once(name, rows, hidden, chunk_bytes):
    w = W.config(name, rows=rows, hidden=hidden)
    ch = bench.e2e_chunks(w, chunk_bytes)
    assert ch[0][0] == 0 and ch[-1][1] == rows
    assert all(a[1] == b[0] for a, b in zip(ch, ch[1:]))        # contiguous, in order
    assert all(r1 > r0 for r0, r1 in ch)
    per_row = hidden * w.torch_dtype.itemsize * (2 if w.residual else 1)
    # every piece starts on a multiple of 16 rows (16-byte aligned row scales); the fewest
    # pieces of at most chunk_bytes on average, each within 16 rows of an even split
    assert all(r0 % 16 == 0 for r0, _ in ch)
    n = min(rows, -(-rows * per_row // chunk_bytes))
    assert len(ch) <= n
    sizes = [r1 - r0 for r0, r1 in ch]
    assert all(k * per_row <= chunk_bytes + 16 * per_row for k in sizes)
    if rows >= 16 * n:
        assert len(ch) == n and max(sizes) - min(sizes) <= 16

"""GPU parity of the FP8 path (rmsnorm_quant_fp8 through the C ABI) against the oracle.

Workloads fp8_small, fp8_residual and fp8_gemma at their full sizes in the launch configuration
the benchmark uses (all rows of fp8_small; sampled rows of the larger ones), both kernel schedules,
plus small shapes that span several CTAs and ragged row lengths."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_common import check_fp8, inputs, sample_rows, schedule

pytestmark = pytest.mark.gpu

SCHEDS = [0, 1, 2]   # automatic, bulk-copy pipeline, register-staged


@pytest.mark.parametrize("sched", SCHEDS)
def test_fp8_small_all_rows(sched):
    w = W.config("fp8_small")
    with schedule(sched):
        rep, _ = check_fp8(w, inputs(w, seed=0))
    assert rep["elements"] == 64 * 4096


@pytest.mark.parametrize("sched", SCHEDS)
@pytest.mark.parametrize("name", ["fp8_residual", "fp8_gemma"])
def test_fp8_full_size_sampled(name, sched):
    w = W.config(name)
    d = inputs(w, seed=0)
    with schedule(sched):
        rep, _ = check_fp8(w, d, idx=sample_rows(w.rows, 96, seed=1))
    # the FP8 kernels form the definition's fp32 values exactly: not even a tolerated code differs
    assert rep["bad"] == 0 and rep["tolerated"] == 0


def test_fp8_gemma_spike_clamps():
    w = W.config("fp8_gemma_spike")
    d = inputs(w, seed=0)
    x = d["input"].float()
    spiky = torch.nonzero((x.abs() > 50).any(-1)).flatten().cpu().numpy()
    assert len(spiky) > 50
    rep, ora = check_fp8(w, d, idx=sample_rows(w.rows, 32, seed=2, extra=spiky[:64]))
    assert rep["clamped_rows"] > 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("rows,hidden", [(1, 64), (3, 8), (157, 520), (300, 4104), (33, 12288)])
@pytest.mark.parametrize("sched", [1, 2])
def test_fp8_shapes(dtype, residual, rows, hidden, sched):
    w = W.Workload("custom", "fp8", rows, hidden, "bf16", residual, scale_ub=1200.0)
    d = inputs(w, seed=rows + hidden, dtype=dtype)
    with schedule(sched):
        check_fp8(w, d)


@pytest.mark.parametrize("hidden", [16384, 32768])
def test_fp8_widest_rows(hidden):
    w = W.Workload("custom", "fp8", 40, hidden, "bf16", True, scale_ub=1200.0)
    check_fp8(w, inputs(w, seed=5))


@pytest.mark.parametrize("sdt", [torch.bfloat16, torch.float16])
def test_fp8_low_precision_scale(sdt):
    w = W.config("fp8_residual", rows=512)
    check_fp8(w, inputs(w, seed=3), scale_dtype=sdt)


def test_fp8_offset_and_tiny_ub():
    w = W.Workload("custom", "fp8", 200, 2048, "fp16", True, weight_offset=1.0, scale_ub=0.5)
    rep, ora = check_fp8(w, inputs(w, seed=4))
    assert rep["clamped_rows"] == 200


@pytest.mark.parametrize("sched", [0, 1, 2, 3])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("rows,hidden", [(37, 64), (301, 520), (1000, 2048), (700, 4104),
                                         (455, 8192), (97, 12288), (60, 16384)])
def test_fp8_weight_offset_shapes(rows, hidden, dtype, sched):
    """The FP8 kernels with a weight offset: the CTA-per-row ring keeps w = gamma + offset in a
    shared-memory table beside one or two ring slots (16-bit input), the other schedules and fp32
    input take w from L1 or registers. Every plan must give the definition's codes exactly."""
    if sched == 3 and hidden * torch.tensor([], dtype=dtype).element_size() > 4096:
        pytest.skip("row per warp holds rows of up to 256 vectors")
    w = W.Workload("custom", "fp8", rows, hidden, "fp16", True, weight_offset=0.75, scale_ub=6.0)
    d = inputs(w, seed=rows * 7 + hidden, dtype=dtype)
    with schedule(sched):
        rep, _ = check_fp8(w, d)
    assert rep["bad"] == 0 and rep["tolerated"] == 0


class _stages:
    def __init__(self, n):
        self.n = n

    def __enter__(self):
        from gpu_common import rq
        rq().rmsq_set_tuning(self.n, 0, 0)

    def __exit__(self, *exc):
        from gpu_common import rq
        rq().rmsq_set_tuning(0, 0, 0)


@pytest.mark.parametrize("dtype,offset,hidden,residual", [
    (torch.float32, 0.0, 8192, True),       # one CTA per row
    (torch.float32, 0.5, 2048 + 64, False),
    (torch.float32, 0.0, 65536, True),      # cluster
    (torch.float16, 1.0, 8192, True),       # one CTA per row, w table
    (torch.bfloat16, 1.0, 65536, True),     # cluster (one slot is its plan)
    (torch.float16, 1.0, 131072, True),
    (torch.float16, 1.0, 65536, False),
])
def test_fp8_one_slot_ring(dtype, offset, hidden, residual):
    # the kernels that hold s in registers refill their slot right after the sum-of-squares
    # barrier, so a ring of one slot is valid for them: every code and scale as the oracle's
    w = W.Workload("custom", "fp8", 37, hidden, "bf16", residual, weight_offset=offset,
                   scale_ub=10.0)
    d = inputs(w, seed=hidden // 64 + int(residual), dtype=dtype)
    with _stages(1):
        rep, _ = check_fp8(w, d)
    assert rep["bad"] == 0

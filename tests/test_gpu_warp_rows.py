"""GPU parity of the row-per-warp schedule (schedule 3) against the oracle.

Every warp owns whole rows with its own bulk-copy ring and reduces with shuffles only, so these
cases cover rows up to 256 vectors of 16 bytes (hidden <= 2048 for 16-bit input, 1024 for
fp32), row counts that leave some warps of the last CTAs without a row, all three modes, three
input dtypes, weight offsets, low-precision FP8 scales, swizzled FP4 scales, guard bytes after
every output, and the fall-back to the CTA schedule for rows a warp cannot hold."""
import pytest
import torch

import workloads as W
from gpu_common import (check_fp8, check_mxfp4, check_nvfp4, guarded, guards_intact, inputs,
                        oracle_global_scale, rq, sample_rows, schedule)

pytestmark = pytest.mark.gpu

WARP = 3
SHAPES = [(1, 64), (3, 256), (157, 520), (1000, 1024), (2049, 2048), (33, 2016)]


def _skip_wide_fp32(dtype, hidden):
    if dtype == torch.float32 and hidden > 1024:
        pytest.skip("fp32 rows wider than 1024 elements take the CTA schedule")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("rows,hidden", SHAPES)
def test_warp_rows_fp8(dtype, residual, rows, hidden):
    _skip_wide_fp32(dtype, hidden)
    w = W.Workload("custom", "fp8", rows, hidden, "bf16", residual, scale_ub=1200.0)
    with schedule(WARP):
        check_fp8(w, inputs(w, seed=rows + 3 * hidden, dtype=dtype))


@pytest.mark.parametrize("hidden", [512, 2048])
def test_warp_rows_fp8_offset_and_clamp(hidden):
    # weight_offset != 0: the FMA-split product path with two warp reductions
    w = W.Workload("custom", "fp8", 700, hidden, "fp16", True, weight_offset=1.0, scale_ub=0.5)
    with schedule(WARP):
        rep, _ = check_fp8(w, inputs(w, seed=hidden))
    assert rep["clamped_rows"] == 700


@pytest.mark.parametrize("sdt", [torch.bfloat16, torch.float16])
def test_warp_rows_fp8_low_precision_scale(sdt):
    w = W.config("fp8_residual", rows=300, hidden=2048)
    with schedule(WARP):
        check_fp8(w, inputs(w, seed=8), scale_dtype=sdt)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("rows,hidden", [(1, 64), (257, 1040), (1500, 2048)])
def test_warp_rows_nvfp4(dtype, residual, rows, hidden):
    _skip_wide_fp32(dtype, hidden)
    w = W.Workload("custom", "nvfp4", rows, hidden, "bf16", residual)
    with schedule(WARP):
        check_nvfp4(w, inputs(w, seed=rows + hidden, dtype=dtype), 3.0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("rows,hidden", [(1, 64), (129, 1024), (4096, 2048)])
def test_warp_rows_mxfp4(dtype, rows, hidden):
    _skip_wide_fp32(dtype, hidden)
    w = W.Workload("custom", "mxfp4", rows, hidden, "bf16", True)
    with schedule(WARP):
        check_mxfp4(w, inputs(w, seed=rows + 5 * hidden, dtype=dtype))


def test_warp_rows_mxfp4_full_size_sampled():
    w = W.config("mxfp4_residual", rows=65536, hidden=2048)
    with schedule(WARP):
        rep, _ = check_mxfp4(w, inputs(w, seed=9), idx=sample_rows(w.rows, 96, seed=4))
    assert rep["bad"] == 0


@pytest.mark.parametrize("rows", [1, 100, 300])
def test_warp_rows_swizzled(rows):
    w = W.Workload("custom", "mxfp4", rows, 2048, "bf16", True)
    wn = W.Workload("custom", "nvfp4", rows, 1024, "bf16", False)
    with schedule(WARP):
        check_mxfp4(w, inputs(w, seed=rows), swizzled=True)
        check_nvfp4(wn, inputs(wn, seed=rows + 1), 2.0, swizzled=True)


@pytest.mark.parametrize("warps", [1, 2, 4, 8, 16])
def test_warp_rows_cta_sizes(warps):
    w = W.Workload("custom", "fp8", 999, 2048, "bf16", True, scale_ub=1200.0)
    wm = W.Workload("custom", "mxfp4", 999, 2048, "bf16", True)
    d, dm = inputs(w, seed=warps), inputs(wm, seed=warps + 100)
    rq().rmsq_set_row_warps(warps)
    try:
        with schedule(WARP):
            check_fp8(w, d)
            check_mxfp4(wm, dm)
    finally:
        rq().rmsq_set_row_warps(0)


@pytest.mark.parametrize("sched", [0, WARP])
@pytest.mark.parametrize("residual", [False, True])
def test_warp_rows_global_scale_prepass(sched, residual):
    # the NVFP4 global-amax pre-pass (one atomic max per warp) on short rows
    w = W.Workload("custom", "nvfp4", 3001, 1024, "bf16", residual)
    d = inputs(w, seed=31 + residual)
    gs = float(oracle_global_scale(w, d))
    with schedule(sched):
        dev = rq().rmsnorm_nvfp4_global_scale(d["input"], d["gamma"], residual=d["residual"],
                                              epsilon=w.eps)
    torch.cuda.synchronize()
    got = float(dev.cpu()[0])
    assert abs(got - gs) <= 2e-6 * gs, (got, gs)


@pytest.mark.parametrize("mode", ["fp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("rows,hidden,residual", [(5000, 256, True), (4000, 512, True),
                                                   (3000, 1024, True), (3000, 2048, False),
                                                   (2000, 2048, True)])
def test_short_rows_automatic_plan(mode, rows, hidden, residual):
    # whatever schedule the planner picks for short rows
    w = W.Workload("custom", mode, rows, hidden, "bf16", residual, scale_ub=1200.0)
    d = inputs(w, seed=rows + hidden)
    if mode == "fp8":
        check_fp8(w, d)
    elif mode == "nvfp4":
        check_nvfp4(w, d, 1.5)
    else:
        check_mxfp4(w, d)


def test_warp_rows_fall_back_for_wide_rows():
    # 4096 bf16 elements are 512 vectors: more than a warp holds, so the CTA schedule runs
    w = W.config("fp8_residual", rows=500)
    with schedule(WARP):
        check_fp8(w, inputs(w, seed=10))


@pytest.mark.parametrize("mode", ["fp8", "nvfp4", "mxfp4"])
def test_warp_rows_guard_bytes(mode):
    rows, H = 97, 2016
    w = W.Workload("custom", mode, rows, H, "bf16", True)
    d = W.generate(w, seed=22, device="cuda")
    ro, ro_raw = guarded(rows * H, torch.bfloat16)
    ro = ro.view(rows, H)
    with schedule(WARP):
        if mode == "fp8":
            q, q_raw = guarded(rows * H, torch.uint8)
            s, s_raw = guarded(rows, torch.float32)
            rq().rmsnorm_quant_fp8(d["input"], d["gamma"], residual=d["residual"], residual_output=ro,
                                   output=q.view(rows, H).view(torch.float8_e4m3fn), scale_output=s)
            raws = (ro_raw, q_raw, s_raw)
        else:
            blk = 16 if mode == "nvfp4" else 32
            q, q_raw = guarded(rows * H // 2, torch.uint8)
            b, b_raw = guarded(rows * H // blk, torch.uint8)
            bs = b.view(rows, H // blk)
            if mode == "nvfp4":
                rq().rmsnorm_quant_nvfp4(d["input"], d["gamma"], residual=d["residual"],
                                         residual_output=ro, output=q.view(rows, H // 2),
                                         block_scale=bs.view(torch.float8_e4m3fn))
            else:
                rq().rmsnorm_quant_mxfp4(d["input"], d["gamma"], residual=d["residual"],
                                         residual_output=ro, output=q.view(rows, H // 2),
                                         block_scale=bs)
            raws = (ro_raw, q_raw, b_raw)
    torch.cuda.synchronize()
    assert guards_intact(raws)
    assert torch.equal(ro, (d["input"].float() + d["residual"].float()).to(torch.bfloat16))

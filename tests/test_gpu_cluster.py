"""GPU parity of the cluster schedule (schedule 4) against the oracle.

Rows wider than one CTA's ring holds are split over a thread-block cluster: CTA k of C takes the
k-th 1/C of every row, and the slices' sums (and maxima) meet in distributed shared memory. The
cases cover:
- the automatic plans for rows of 32768, 65536 and 131072 elements (clusters of 4, 8 and 16 for
  rows with a residual);
- the schedule forced with every cluster size on narrow rows, for all kernel variants: FP8 with
  and without weight offset, blocked NVFP4, MXFP4, fp16 and fp32 inputs, swizzled scales;
- row counts that leave clusters idle;
- the global-scale pre-pass and guard bytes after the outputs."""
import pytest
import torch

import workloads as W
from gpu_common import (check_fp8, check_mxfp4, check_nvfp4, guarded, guards_intact, inputs,
                        oracle_global_scale, rq, schedule)

pytestmark = pytest.mark.gpu

CLUSTER = 4


class cluster_size:
    def __init__(self, c):
        self.c = c

    def __enter__(self):
        rq().rmsq_set_cluster_size(self.c)

    def __exit__(self, *exc):
        rq().rmsq_set_cluster_size(0)


def _check(mode, w, d, gs=1.75, **kw):
    if mode == "fp8":
        return check_fp8(w, d, **kw)
    if mode == "nvfp4":
        return check_nvfp4(w, d, gs, **kw)
    return check_mxfp4(w, d, **kw)


@pytest.mark.parametrize("mode", ["fp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("hidden", [32768, 65536, 131072])
def test_wide_rows_automatic(mode, residual, hidden):
    w = W.Workload("custom", mode, 37, hidden, "bf16", residual, scale_ub=1200.0)
    _check(mode, w, inputs(w, seed=hidden // 256 + residual))


@pytest.mark.parametrize("mode", ["fp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("dtype", [torch.float16, torch.float32])
def test_wide_rows_other_dtypes(mode, dtype):
    hidden = 65536 if dtype == torch.float32 else 131072
    w = W.Workload("custom", mode, 19, hidden, "bf16", True, scale_ub=1200.0)
    _check(mode, w, inputs(w, seed=5, dtype=dtype))


@pytest.mark.parametrize("c", [2, 4, 8, 16])
@pytest.mark.parametrize("mode", ["fp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("rows,hidden", [(1, 4096), (3, 8192), (300, 8192)])
def test_forced_cluster_sizes(c, mode, rows, hidden):
    w = W.Workload("custom", mode, rows, hidden, "bf16", True, scale_ub=1200.0)
    d = inputs(w, seed=c * 100 + rows)
    with schedule(CLUSTER), cluster_size(c):
        _check(mode, w, d)


@pytest.mark.parametrize("c", [2, 8])
def test_forced_cluster_fp8_offset_and_scale_dtype(c):
    w = W.Workload("custom", "fp8", 200, 8192, "fp16", True, weight_offset=1.0, scale_ub=0.5)
    d = inputs(w, seed=c)
    with schedule(CLUSTER), cluster_size(c):
        rep, _ = check_fp8(w, d)
        assert rep["clamped_rows"] == 200
        wb = W.config("fp8_residual", rows=150)
        check_fp8(wb, inputs(wb, seed=c + 1), scale_dtype=torch.bfloat16)


@pytest.mark.parametrize("c", [2, 4])
@pytest.mark.parametrize("dtype", [torch.float16, torch.float32])
def test_forced_cluster_dtypes(c, dtype):
    for mode in ("fp8", "nvfp4", "mxfp4"):
        w = W.Workload("custom", mode, 64, 4096, "bf16", True, scale_ub=1200.0)
        with schedule(CLUSTER), cluster_size(c):
            _check(mode, w, inputs(w, seed=c, dtype=dtype))


@pytest.mark.parametrize("c", [2, 8])
def test_forced_cluster_swizzled_scales(c):
    w = W.Workload("custom", "mxfp4", 300, 8192, "bf16", True)
    wn = W.Workload("custom", "nvfp4", 130, 4096, "bf16", False)
    with schedule(CLUSTER), cluster_size(c):
        check_mxfp4(w, inputs(w, seed=c), swizzled=True)
        check_nvfp4(wn, inputs(wn, seed=c + 1), 2.0, swizzled=True)


def test_wide_rows_swizzled_and_prepass():
    w = W.Workload("custom", "nvfp4", 150, 65536, "bf16", True)
    d = inputs(w, seed=9)
    check_nvfp4(w, d, 1.25, swizzled=True)
    gs = float(oracle_global_scale(w, d))
    dev = rq().rmsnorm_nvfp4_global_scale(d["input"], d["gamma"], residual=d["residual"],
                                          epsilon=w.eps)
    torch.cuda.synchronize()
    got = float(dev.cpu()[0])
    assert abs(got - gs) <= 2e-6 * gs, (got, gs)


@pytest.mark.parametrize("mode", ["fp8", "mxfp4"])
def test_wide_rows_guard_bytes(mode):
    rows, H = 5, 65536 + 256
    w = W.Workload("custom", mode, rows, H, "bf16", True)
    d = W.generate(w, seed=23, device="cuda")
    ro, ro_raw = guarded(rows * H, torch.bfloat16)
    ro = ro.view(rows, H)
    if mode == "fp8":
        q, q_raw = guarded(rows * H, torch.uint8)
        s, s_raw = guarded(rows, torch.float32)
        rq().rmsnorm_quant_fp8(d["input"], d["gamma"], residual=d["residual"], residual_output=ro,
                               output=q.view(rows, H).view(torch.float8_e4m3fn), scale_output=s)
        raws = (ro_raw, q_raw, s_raw)
    else:
        q, q_raw = guarded(rows * H // 2, torch.uint8)
        b, b_raw = guarded(rows * H // 32, torch.uint8)
        rq().rmsnorm_quant_mxfp4(d["input"], d["gamma"], residual=d["residual"], residual_output=ro,
                                 output=q.view(rows, H // 2), block_scale=b.view(rows, H // 32))
        raws = (ro_raw, q_raw, b_raw)
    torch.cuda.synchronize()
    assert guards_intact(raws)
    assert torch.equal(ro, (d["input"].float() + d["residual"].float()).to(torch.bfloat16))
    assert rq().rmsq_device_status() == 0


def _launch(mode, d):
    x, r, g = d["input"], d["residual"], d["gamma"]
    if mode == "fp8":
        return rq().rmsnorm_quant_fp8(x, g, residual=r, scale_ub=1200.0)
    if mode == "nvfp4":
        gs = torch.full((1,), 2.0, dtype=torch.float32, device=x.device)
        return rq().rmsnorm_quant_nvfp4(x, g, global_scale=gs, residual=r)
    return rq().rmsnorm_quant_mxfp4(x, g, residual=r)


def _bits(outs):
    return [o.view(torch.uint8) if o.dtype == torch.float8_e4m3fn else o for o in outs]


@pytest.mark.parametrize("mode", ["fp8", "nvfp4", "mxfp4"])
def test_cluster_ring_depth_leaves_every_bit(mode):
    # deeper rings only change when slices arrive, never the arithmetic
    w = W.Workload("custom", mode, 200, 65536, "bf16", True, scale_ub=1200.0)
    d = inputs(w, seed=61)
    ref = _bits(_launch(mode, d))
    for stages in (3, 4):
        rq().rmsq_set_tuning(stages, 0, 0)
        try:
            got = _bits(_launch(mode, d))
        finally:
            rq().rmsq_set_tuning(0, 0, 0)
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(got, ref)), stages
    _check(mode, w, d)
    assert rq().rmsq_device_status() == 0


class vectors_per_thread:
    def __init__(self, v):
        self.v = v

    def __enter__(self):
        rq().rmsq_set_tuning(0, 0, self.v)

    def __exit__(self, *exc):
        rq().rmsq_set_tuning(0, 0, 0)


@pytest.mark.parametrize("vpt", [4, 8])
@pytest.mark.parametrize("case", ["fp8_bf16_res", "fp8_bf16", "fp8_fp16_offset", "nvfp4_bf16_res",
                                  "mxfp4_bf16_res", "fp8_fp32_res"])
def test_cluster_both_vector_widths(case, vpt):
    # The planner gives 16-bit FP8 and NVFP4 slices 8 vectors per thread and the rest 4 (8 on
    # slices wider than 1024 vectors); both widths of every kernel stay checked, on wide rows
    # (automatic cluster) and on narrow rows with every forced cluster size.
    mode = case.split("_")[0]
    dtype = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[case.split("_")[1]]
    res = case.endswith("res") or case.endswith("offset")
    off = 1.0 if case.endswith("offset") else 0.0
    wide = 65536 if dtype == torch.float32 else 131072
    ww = W.Workload("custom", mode, 23, wide, "bf16", res, weight_offset=off, scale_ub=10.0)
    with vectors_per_thread(vpt):
        _check(mode, ww, inputs(ww, seed=vpt + len(case), dtype=dtype))
        for c in (2, 4, 8, 16):
            w = W.Workload("custom", mode, 97, 8192, "bf16", res, weight_offset=off, scale_ub=10.0)
            with schedule(CLUSTER), cluster_size(c):
                _check(mode, w, inputs(w, seed=c * 7 + vpt, dtype=dtype))
    assert rq().rmsq_device_status() == 0

"""The launch planner, on the CPU (rmsq_plan with GB300's shared-memory limits).

The planner picks schedule, vectors per thread, CTA size, ring depth and cluster size for each
call. These tests pin:
- the plans of the gated workloads, against the kernel templates the committed ncu summaries
  were taken on (profiles/ncu_traffic.json), so a planner change that leaves those summaries
  describing another kernel fails here;
- the documented rules: row per warp for short rows, one CTA per row, clusters for wide rows,
  the cluster sizes and vectors per thread;
- invariants over every accepted width: the plan fits the shared memory, covers the row, keeps
  FP4 scale blocks whole within a cluster slice, and stays within 512 threads;
- the argument checks, which are the entry points' own."""
import ctypes
import json
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

BF16, FP16, F32 = torch.bfloat16, torch.float16, torch.float32
PIPE, REG, WARP, CLUSTER = 1, 2, 3, 4
MODE_ID = {"fp8": 0, "nvfp4": 1, "mxfp4": 2, "global_scale": 3}
DT_ID = {BF16: 0, FP16: 1, F32: 2}


@pytest.fixture(scope="module")
def rq():
    from rmsnorm_precision_activation_gb300 import build
    build.build()
    import rmsnorm_precision_activation_gb300 as m
    return m


def plan(rq, mode, dtype, hidden, residual=False, offset=0.0, smem=None):
    kw = {} if smem is None else {"smem": smem}
    return rq.rmsq_plan(mode, dtype, hidden, residual=residual, weight_offset=offset, **kw)


def template_of(p, mode, dtype, residual):
    """The rmsq_row_kernel<DT, RES, MODE, VPT, SCHED, W16> instantiation a plan launches."""
    return (DT_ID[dtype], int(residual), MODE_ID[mode], p["vectors_per_thread"], p["schedule"],
            p["w16"])


def test_bench_step_plans_are_the_profiled_kernels(rq):
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        rec = json.load(f)["kernels"]
    cases = {"fp8": ("fp8", FP16, 8192, True, 1.0),          # fp8_gemma 16384 x 8192
             "nvfp4": ("nvfp4", BF16, 7168, False, 0.0),     # nvfp4 32768 x 7168
             "mxfp4": ("mxfp4", BF16, 16384, True, 0.0)}     # mxfp4_residual 65536 x 16384
    for key, (mode, dt, h, res, off) in cases.items():
        p = plan(rq, mode, dt, h, res, off)
        args = tuple(int(v) for v in re.findall(r"\d+", rec[key]["template"].split("<")[1]))
        assert template_of(p, mode, dt, res) == args, (key, p, rec[key]["template"])


def test_profiled_full_captures_are_the_planned_kernels(rq):
    # each --set full summary names the instantiation it captured; the planner still picks it
    cases = {"fp8_gemma_16384x8192_ncu_full.md": ("fp8", FP16, 8192, True, 1.0),
             "nvfp4_32768x7168_ncu_full.md": ("nvfp4", BF16, 7168, False, 0.0),
             "mxfp4_residual_65536x2048_ncu_full.md": ("mxfp4", BF16, 2048, True, 0.0),
             "cluster_fp8_4096x65536_ncu_full.md": ("fp8", BF16, 65536, True, 0.0),
             "cluster_fp8_offset_4096x65536_ncu_full.md": ("fp8", FP16, 65536, True, 1.0),
             "cluster_fp8_fp32_2048x65536_ncu_full.md": ("fp8", F32, 65536, True, 0.0),
             "cluster_fp8_2048x131072_ncu_full.md": ("fp8", BF16, 131072, True, 0.0)}
    for fn, (mode, dt, h, res, off) in cases.items():
        text = open(os.path.join(ROOT, "profiles", fn)).read()
        m = re.search(r"`void rmsq_row_kernel<([\d, ]+)>\(Params\)`", text)
        assert m, fn
        args = tuple(int(v) for v in m.group(1).split(","))
        assert template_of(plan(rq, mode, dt, h, res, off), mode, dt, res) == args, fn


def test_gated_plans(rq):
    p = plan(rq, "fp8", FP16, 8192, True, 1.0)
    # the offset FP8 kernel: 4 vectors per thread, w table beside one ring slot
    assert (p["schedule"], p["vectors_per_thread"], p["threads"], p["stages"], p["w16"]) == \
        (PIPE, 4, 256, 1, 0)
    assert p["smem_bytes"] >= 32 * 1024 + 8192 * 2 * 2          # w table (32 B/vector) + x, r
    p = plan(rq, "nvfp4", BF16, 7168)
    assert (p["schedule"], p["vectors_per_thread"], p["threads"], p["stages"]) == (PIPE, 8, 128, 2)
    # MXFP4 with a residual: one vector per thread up to 256 vectors, two up to 1024, then as
    # many as make 512 threads; a third ring slot from 2048 vectors
    for h, vpt, threads, stages in [(2048, 1, 256, 2), (5120, 2, 320, 2), (8192, 2, 512, 2),
                                    (16384, 4, 512, 3)]:
        p = plan(rq, "mxfp4", BF16, h, True)
        assert (p["schedule"], p["vectors_per_thread"], p["threads"], p["stages"]) == \
            (PIPE, vpt, threads, stages), (h, p)


def test_short_rows_take_a_warp_each(rq):
    for h in (64, 512, 1024, 2048):                      # up to 256 vectors without a residual
        assert plan(rq, "fp8", BF16, h)["schedule"] == WARP, h
    assert plan(rq, "fp8", BF16, 4096)["schedule"] == PIPE
    assert plan(rq, "mxfp4", BF16, 512, True)["schedule"] == WARP   # up to 64 with one
    assert plan(rq, "mxfp4", BF16, 1024, True)["schedule"] == PIPE


@pytest.mark.parametrize("mode", ["fp8", "nvfp4", "mxfp4", "global_scale"])
def test_wide_rows_take_a_cluster(mode, rq):
    # beyond 4096 vectors (one CTA covers 512 threads x 8 vectors), or a ring that does not fit
    assert plan(rq, mode, BF16, 32768)["schedule"] == PIPE
    assert plan(rq, mode, BF16, 32768 + 256)["schedule"] == CLUSTER
    assert plan(rq, mode, F32, 16384)["schedule"] == PIPE
    assert plan(rq, mode, F32, 16384 + 256)["schedule"] == CLUSTER
    assert plan(rq, mode, BF16, 32768, True)["schedule"] == CLUSTER    # 2 x 128 KB slots


@pytest.mark.parametrize("mode,dtype,hidden,res,off,cluster,vpt", [
    ("fp8", BF16, 65536, True, 0.0, 8, 8),
    ("fp8", BF16, 131072, True, 0.0, 16, 8),       # no longer moved to 8 CTAs of 512 threads
    ("fp8", BF16, 32768, True, 0.0, 4, 4),         # W16 with a residual on a cluster of 4 keeps 4
    ("fp8", BF16, 65536, False, 0.0, 4, 8),
    ("fp8", BF16, 131072, False, 0.0, 8, 8),
    ("fp8", FP16, 65536, True, 1.0, 4, 8),         # the offset kernel: one slot of up to 64 KB
    ("fp8", FP16, 131072, True, 1.0, 8, 8),
    ("fp8", FP16, 32768, True, 1.0, 2, 8),
    ("fp8", FP16, 65536, False, 1.0, 2, 8),
    ("fp8", BF16, 65536, True, 1.0, 4, 8),
    ("fp8", F32, 65536, True, 0.0, 8, 8),          # fp32 FP8: two exchanges, one slot
    ("fp8", F32, 32768, False, 0.0, 2, 8),
    ("nvfp4", BF16, 65536, True, 0.0, 8, 8),
    ("nvfp4", BF16, 131072, True, 0.0, 16, 8),
    ("nvfp4", F32, 65536, True, 0.0, 16, 8),
    ("mxfp4", F32, 65536, True, 0.0, 16, 4),       # MXFP4 keeps 4 whatever the input
    ("mxfp4", BF16, 65536, True, 0.0, 8, 4),       # MXFP4 keeps 4
    ("mxfp4", BF16, 131072, True, 0.0, 16, 4),
    ("mxfp4", BF16, 131072, False, 0.0, 8, 8),     # 8 where 4 would take 512 threads
])
def test_cluster_sizes_and_vectors(mode, dtype, hidden, res, off, cluster, vpt, rq):
    p = plan(rq, mode, dtype, hidden, res, off)
    assert p["schedule"] == CLUSTER
    assert (p["cluster"], p["vectors_per_thread"]) == (cluster, vpt), p
    nvc = hidden // (8 if dtype != F32 else 4) // cluster
    assert p["threads"] == ((nvc + vpt - 1) // vpt + 31) // 32 * 32
    # pipelined kernels (one exchange per row) keep three slots; the FP8 kernels with two
    # exchanges (an offset, or fp32 input) refill their one slot right after the first
    one_exchange = mode != "fp8" or (dtype != F32 and off == 0.0)
    assert p["stages"] == (3 if one_exchange else 1)


def _widths(mode, dtype):
    step = {"fp8": 8 if dtype != F32 else 4, "nvfp4": 16, "mxfp4": 32, "global_scale": 16}[mode]
    one_cta = 32768 if dtype != F32 else 16384
    top = 131072 if dtype != F32 else 65536
    narrow = list(range(step, 4096 + 1, step))
    mid = list(range(4096 + step, one_cta + 1, step * 16))
    wide = list(range(one_cta + 256, top + 1, 256 * 7)) + [top]
    return narrow + mid + wide


@pytest.mark.parametrize("mode", ["fp8", "nvfp4", "mxfp4", "global_scale"])
@pytest.mark.parametrize("dtype", [BF16, FP16, F32])
def test_every_width_gets_a_plan_that_fits(mode, dtype, rq):
    optin, per_sm, reserved = rq.GB300_SMEM
    epv = 8 if dtype != F32 else 4
    block = {"fp8": 1, "nvfp4": 16, "mxfp4": 32, "global_scale": 16}[mode]
    for res in (False, True):
        for off in ((0.0, 1.0) if mode == "fp8" else (0.0,)):
            for h in _widths(mode, dtype):
                p = plan(rq, mode, dtype, h, res, off)
                nv = h // epv
                where = (mode, dtype, res, off, h, p)
                assert p["smem_bytes"] <= optin, where
                assert 32 <= p["threads"] <= 512 and p["threads"] % 32 == 0, where
                assert p["vectors_per_thread"] in (1, 2, 4, 8), where
                if p["schedule"] == WARP:
                    assert 32 * p["vectors_per_thread"] >= nv, where
                    assert p["stages"] >= 2, where
                    continue
                c = p["cluster"]
                assert nv % c == 0, where
                nvc = nv // c
                assert p["threads"] * p["vectors_per_thread"] >= nvc, where
                assert (p["threads"] - 32) * p["vectors_per_thread"] < nvc, where   # no idle warp
                if c > 1:
                    assert p["schedule"] == CLUSTER and c in (2, 4, 8, 16), where
                    assert (nvc * epv) % block == 0, where
                if p["schedule"] in (PIPE, CLUSTER):
                    assert p["stages"] >= 1, where
                    # the ring's slots alone (x, and the residual unless it has its own slot)
                    assert p["stages"] * nvc * 16 <= p["smem_bytes"], where
                assert p["w16"] == int(dtype != F32 and off == 0.0), where


def test_smaller_devices_still_get_plans_that_fit(rq):
    # the planner only assumes the limits it is given
    for smem in [(101376, 102400, 1024), (166912, 167936, 1024)]:
        for mode in ("fp8", "nvfp4", "mxfp4"):
            for h in (2048, 8192, 16384, 32768, 65536, 131072):
                for res in (False, True):
                    try:
                        p = plan(rq, mode, BF16, h, res, smem=smem)
                    except rq.RmsqError as e:
                        assert e.status == 2          # no plan: RMSQ_ERR_SHAPE, never a bad one
                        continue
                    assert p["smem_bytes"] <= smem[0], (smem, mode, h, res, p)


def test_tuning_settings_are_reflected(rq):
    base = plan(rq, "mxfp4", BF16, 8192, True)
    rq.rmsq_set_schedule(CLUSTER)
    rq.rmsq_set_cluster_size(2)
    try:
        p = plan(rq, "mxfp4", BF16, 8192, True)
        assert (p["schedule"], p["cluster"]) == (CLUSTER, 2)
    finally:
        rq.rmsq_set_schedule(0)
        rq.rmsq_set_cluster_size(0)
    rq.rmsq_set_tuning(3, 0, 2)
    try:
        p = plan(rq, "mxfp4", BF16, 8192, True)
        assert (p["stages"], p["vectors_per_thread"]) == (3, 2)
    finally:
        rq.rmsq_set_tuning(0, 0, 0)
    # one slot: honoured where s is held in registers (FP8 with an offset or fp32 input), two or
    # three slots at least elsewhere
    rq.rmsq_set_tuning(1, 0, 0)
    try:
        assert plan(rq, "fp8", F32, 8192, True)["stages"] == 1
        assert plan(rq, "fp8", F32, 65536, True)["stages"] == 1
        assert plan(rq, "fp8", FP16, 8192, True, 1.0)["stages"] == 1
        assert plan(rq, "fp8", BF16, 8192, True)["stages"] == 2
        assert plan(rq, "mxfp4", BF16, 512, True)["stages"] == 2        # row per warp
        assert plan(rq, "nvfp4", BF16, 65536, True)["stages"] == 3      # split residual ring
        assert plan(rq, "nvfp4", BF16, 65536)["stages"] == 2
    finally:
        rq.rmsq_set_tuning(0, 0, 0)
    assert plan(rq, "mxfp4", BF16, 8192, True) == base


def test_argument_checks(rq):
    def status(*args):
        info = rq.PlanInfo()
        return rq.lib().rmsq_plan(*args, *rq.GB300_SMEM, ctypes.byref(info))

    assert status(0, 0, 0, 0.0, 4096) == 0
    assert status(4, 0, 0, 0.0, 4096) == 6                 # unknown mode
    assert status(0, 3, 0, 0.0, 4096) == 4                 # unknown dtype
    assert status(1, 0, 0, 0.0, 4104) == 2                 # NVFP4: not a multiple of 16
    assert status(2, 0, 0, 0.0, 4112) == 2                 # MXFP4: not a multiple of 32
    assert status(0, 0, 0, 0.0, 32768 + 8) == 2            # cluster rows: multiples of 256
    assert status(0, 0, 0, 0.0, 131072 + 256) == 2         # beyond the widest row
    assert status(0, 2, 0, 0.0, 65536 + 256) == 2          # fp32: half of it
    assert status(0, 0, 0, float("nan"), 4096) == 6
    info = rq.PlanInfo()
    assert rq.lib().rmsq_plan(0, 0, 0, 0.0, 4096, 1024, 512, 0, ctypes.byref(info)) == 6
    assert rq.lib().rmsq_plan(0, 0, 0, 0.0, 4096, *rq.GB300_SMEM, None) == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="a device is present")
def test_device_limits_need_a_device(rq):
    # smem=None asks for the current device's limits: without a GPU that is RMSQ_ERR_DEVICE
    with pytest.raises(rq.RmsqError) as e:
        rq.rmsq_plan("fp8", BF16, 4096, smem=None)
    assert e.value.status == 7

"""GPU parity of the NVFP4 and MXFP4 paths and the global-scale pre-pass against the oracle.

nvfp4 at its full size (32768 x 7168, sampled rows) with gs = 448 * 6 / amax(y) from the oracle;
the MXFP4 + residual sweep over rows {1, 16, 128, 4096, 65536} x hidden {2048, 5120, 8192, 16384};
row-major and swizzled 128x4 scale layouts; bf16, fp16 and fp32 inputs."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_common import (check_mxfp4, check_nvfp4, host_bits, inputs, oracle_global_scale, rq,
                        sample_rows, schedule)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nvfp4_full():
    w = W.config("nvfp4")
    d = inputs(w, seed=0)
    return w, d, oracle_global_scale(w, d)


@pytest.mark.parametrize("sched", [0, 1, 2])
def test_nvfp4_full_size_sampled(nvfp4_full, sched):
    w, d, gs = nvfp4_full
    with schedule(sched):
        rep, _ = check_nvfp4(w, d, float(gs), idx=sample_rows(w.rows, 64, seed=3))
    assert rep["bad"] == 0


def test_nvfp4_global_scale_prepass(nvfp4_full):
    w, d, gs = nvfp4_full
    dev = rq().rmsnorm_nvfp4_global_scale(d["input"], d["gamma"], epsilon=w.eps)
    torch.cuda.synchronize()
    got = float(dev.cpu()[0])
    assert abs(got - float(gs)) <= 2e-6 * float(gs), (got, float(gs))


@pytest.mark.parametrize("gs", [1.0, 0.03, 250.0])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("residual", [False, True])
def test_nvfp4_small(gs, dtype, residual):
    w = W.Workload("custom", "nvfp4", 257, 1040, "bf16", residual)
    check_nvfp4(w, inputs(w, seed=11, dtype=dtype), gs)


@pytest.mark.parametrize("rows", W.MXFP4_ROWS)
@pytest.mark.parametrize("hidden", W.MXFP4_HIDDEN)
def test_mxfp4_sweep(rows, hidden):
    w = W.config("mxfp4_residual", rows=rows, hidden=hidden)
    d = inputs(w, seed=rows * 7 + hidden)
    check_mxfp4(w, d, idx=sample_rows(rows, 64, seed=rows))


@pytest.mark.parametrize("sched", [1, 2])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_mxfp4_dtypes(sched, dtype):
    w = W.Workload("custom", "mxfp4", 300, 3072, "bf16", True)
    with schedule(sched):
        check_mxfp4(w, inputs(w, seed=12, dtype=dtype))


@pytest.mark.parametrize("rows,hidden", [(300, 2048), (128, 64), (1, 32 * 6)])
def test_fp4_swizzled_layout(rows, hidden):
    w = W.Workload("custom", "mxfp4", rows, hidden, "bf16", True)
    d = inputs(w, seed=13)
    check_mxfp4(w, d, swizzled=True)
    wn = W.Workload("custom", "nvfp4", rows, hidden, "bf16", False)
    check_nvfp4(wn, inputs(wn, seed=14), 2.0, swizzled=True)


def test_swizzled_padding_untouched():
    rows, H = 130, 96                      # 2 row tiles (126 padded rows), 6 -> 8 scales per row
    x = torch.randn(rows, H, device="cuda").to(torch.bfloat16)
    g = torch.ones(H, device="cuda", dtype=torch.bfloat16)
    n = rq().swizzled_scale_numel(rows, H, 16)
    bs = torch.full((n,), 0xA5, dtype=torch.uint8, device="cuda")
    rq().rmsnorm_quant_nvfp4(x, g, block_scale=bs.view(torch.float8_e4m3fn), swizzled=True)
    torch.cuda.synchronize()
    flat = bs.cpu().numpy()
    used = {oracle.scale_offset(r, s, H // 16, True) for r in range(rows) for s in range(H // 16)}
    pad = np.array(sorted(set(range(n)) - used))
    assert len(pad) > 0 and np.all(flat[pad] == 0xA5)


def test_global_scale_prepass_reuses_its_scratch_slots():
    """The pre-pass is one launch whose last CTA turns the launch's running max into gs and
    leaves its two scratch words at 0. Launches take their slot from a pool of 4096 in turn, so
    4200 launches (alternating two inputs whose global scales differ, with and without a
    residual, and one with no rows) reuse slots; every gs must still be that input's."""
    wa = W.Workload("custom", "nvfp4", 48, 2048, "bf16", True)
    wb = W.Workload("custom", "nvfp4", 300, 1024, "bf16", False)
    da, db = inputs(wa, seed=61), inputs(wb, seed=62)
    db["input"] = db["input"] * 3
    ga, gb = float(oracle_global_scale(wa, da)), float(oracle_global_scale(wb, db))
    n = 4200
    out = torch.empty(n + 1, dtype=torch.float32, device="cuda")
    for i in range(n):
        w, d = (wa, da) if i % 2 == 0 else (wb, db)
        rq().rmsnorm_nvfp4_global_scale(d["input"], d["gamma"], residual=d["residual"],
                                        epsilon=w.eps, out=out[i:i + 1])
    empty = torch.empty(0, 2048, dtype=torch.bfloat16, device="cuda")
    rq().rmsnorm_nvfp4_global_scale(empty, da["gamma"], epsilon=wa.eps, out=out[n:n + 1])
    got = out.cpu().numpy()
    assert np.all(np.abs(got[0:n:2] - ga) <= 2e-6 * ga)
    assert np.all(np.abs(got[1:n:2] - gb) <= 2e-6 * gb)
    assert got[n] == 1.0
    assert rq().rmsq_device_status() == 0

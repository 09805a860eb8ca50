"""Seeded random cases through all three entry points, every output checked against the oracle.

Each case draws a mode, an input dtype, a residual or none, a weight offset, a scale layout (FP4)
or scale dtype (FP8), and a ragged shape, so the planner's choices (row per warp, CTA per row with
one, two or three ring slots, the FP8 w table, clusters for the widest rows) are crossed with the
options. Rows are few enough that the oracle checks every element."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_common import check_fp8, check_mxfp4, check_nvfp4, inputs, oracle_global_scale

pytestmark = pytest.mark.gpu

_DT = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def _case(i):
    rng = np.random.default_rng(1000 + i)
    mode = ["fp8", "nvfp4", "mxfp4"][i % 3]
    dtype = ["bf16", "fp16", "fp32"][rng.integers(3)]
    residual = bool(rng.integers(2))
    offset = float(rng.choice([0.0, 0.0, 1.0, -0.5]))
    step = {"fp8": 8 if dtype != "fp32" else 4, "nvfp4": 16, "mxfp4": 32}[mode]
    cap = 65536 if dtype != "fp32" else 32768
    # a width from 1 to 64 blocks of step (short rows) or up to the cluster range (wide rows)
    u = rng.random()
    if u < 0.15:
        hidden = step * int(rng.integers(1, 9))                       # a few blocks
    elif u < 0.75:
        hidden = step * int(rng.integers(1, 1024 // step + 2)) * int(rng.choice([1, 4, 16]))
    else:
        hidden = 256 * int(rng.integers(1, cap // 256 + 1))
    hidden = min(max(hidden, step), cap)
    one_cta = 32768 if dtype != "fp32" else 16384
    if hidden > one_cta:                    # rows split over a cluster: a multiple of 256
        hidden = hidden // 256 * 256
    rows = int(rng.integers(1, max(2, min(3000, 6_000_000 // hidden))))
    opt = bool(rng.integers(2))
    return mode, dtype, residual, offset, rows, hidden, opt


CASES = [_case(i) for i in range(96)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%s-%s-res%d-off%g-%dx%d-%d" % c)
def test_random_case_matches_oracle(case):
    mode, dtype, residual, offset, rows, hidden, opt = case
    w = W.Workload("custom", mode, rows, hidden, "bf16", residual, weight_offset=offset,
                   scale_ub=float(np.random.default_rng(rows).choice([1.0, 10.0, 1200.0])))
    d = inputs(w, seed=rows + hidden, dtype=_DT[dtype])
    if mode == "fp8":
        sd = torch.bfloat16 if opt else torch.float32
        rep, _ = check_fp8(w, d, scale_dtype=sd)
        assert rep["bad"] == 0
    elif mode == "nvfp4":
        check_nvfp4(w, d, float(oracle_global_scale(w, d)), swizzled=opt)
    else:
        check_mxfp4(w, d, swizzled=opt)

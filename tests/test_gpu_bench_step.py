"""The launches bench.py times, checked against the oracle.

bench.py's step runs the FP8, NVFP4 and MXFP4 kernels on three resident [8192 x 4096] bf16
batches with a residual. It uses the fp8_residual workload's distributions, FP8 with
scale_ub 1200, and NVFP4 with the global scale from the device pre-pass. This test builds that
same Step, runs its launches back to back on one stream as the timed loop does (twice, so the
second pass reuses the buffers and counters), and checks sampled rows of every output against
the oracle. The device global scale is compared with the oracle's amax, then used as the
oracle's input for the NVFP4 codes."""
import numpy as np
import pytest
import torch

import oracle
import parity as P
from gpu_common import ODT, host_bits, rq, sample_rows

pytestmark = pytest.mark.gpu


def test_bench_step_launches_match_oracle():
    import bench
    dev = torch.device("cuda", 0)
    step = bench.Step(rq(), 8192, 4096, dev)
    for _ in range(2):
        for m in bench.MODES:
            step.launch(m)
    torch.cuda.synchronize()
    w = step.w
    idx = sample_rows(8192, 48, seed=17)
    t_idx = torch.as_tensor(idx, device=dev)

    def rows(t):
        return None if t is None else t[t_idx]

    # FP8
    d = step.batches["fp8"]
    q, sc, ro = step.out["fp8"]
    ora = oracle.quant_fp8(host_bits(rows(d["input"])), host_bits(rows(d["residual"])),
                           host_bits(d["gamma"]), dtype=ODT[torch.bfloat16], eps=w.eps,
                           weight_offset=w.weight_offset, scale_ub=w.scale_ub, want_pre=True)
    P.compare_fp8(rows(q.view(torch.uint8)).cpu().numpy(), rows(sc).cpu().numpy(),
                  host_bits(rows(ro)), ora).check()

    # NVFP4 with the device global scale
    d = step.batches["nvfp4"]
    gs = float(step.gs.cpu()[0])
    y = oracle.rmsnorm(host_bits(d["input"]), host_bits(d["residual"]), host_bits(d["gamma"]),
                       dtype=ODT[torch.bfloat16], eps=w.eps)["y"]
    gs_ora = float(oracle.nvfp4_global_scale(np.abs(y).max()))
    assert abs(gs - gs_ora) <= 2e-6 * gs_ora, (gs, gs_ora)
    q, bs, ro = step.out["nvfp4"]
    ora = oracle.quant_nvfp4(host_bits(rows(d["input"])), host_bits(rows(d["residual"])),
                             host_bits(d["gamma"]), gs, dtype=ODT[torch.bfloat16], eps=w.eps,
                             want_y=True, want_pre=True)
    P.compare_nvfp4(rows(q).cpu().numpy(), rows(bs.view(torch.uint8)).cpu().numpy(),
                    host_bits(rows(ro)), ora, gs).check()

    # MXFP4
    d = step.batches["mxfp4"]
    q, bs, ro = step.out["mxfp4"]
    ora = oracle.quant_mxfp4(host_bits(rows(d["input"])), host_bits(rows(d["residual"])),
                             host_bits(d["gamma"]), dtype=ODT[torch.bfloat16], eps=w.eps,
                             want_y=True, want_pre=True)
    P.compare_mxfp4(rows(q).cpu().numpy(), rows(bs).cpu().numpy(), host_bits(rows(ro)), ora).check()
    assert rq().rmsq_device_status() == 0

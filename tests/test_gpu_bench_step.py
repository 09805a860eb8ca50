"""The launches bench.py times, checked against the oracle.

bench.py's step runs the FP8, NVFP4 and MXFP4 kernels, each on its large workload at the stated
shape: fp8_gemma (16384 x 8192 fp16 + residual, weight_offset 1, scale_ub 10), nvfp4
(32768 x 7168 bf16, global scale from the device pre-pass) and mxfp4_residual at
65536 x 16384. This test builds that same Step, runs its launches back to back on one stream as
the timed loop does (twice, so the second pass reuses the buffers and row counters), and checks
sampled rows of every output against the oracle. The device global scale is compared with the
oracle's, computed over the whole nvfp4 tensor, then used as the oracle's input for the NVFP4
codes."""
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
    step = bench.Step(rq(), dev)
    assert step.modes == ("fp8", "nvfp4", "mxfp4")
    for _ in range(2):
        for m in step.modes:
            step.launch(m)
    torch.cuda.synchronize()

    def rows_of(t, idx):
        return None if t is None else t[torch.as_tensor(idx, device=dev)]

    def bits(t, idx):
        return None if t is None else host_bits(rows_of(t, idx))

    # FP8 on fp8_gemma, with the rows whose input was scaled x200 among the samples
    w, d = step.workloads["fp8"], step.batches["fp8"]
    big = torch.nonzero(d["input"].float().abs().amax(-1) > 50).flatten().cpu().numpy()
    assert len(big) > 50
    idx = sample_rows(w.rows, 48, seed=17, extra=big[:16])
    q, sc, ro = step.out["fp8"]
    ora = oracle.quant_fp8(bits(d["input"], idx), bits(d["residual"], idx), host_bits(d["gamma"]),
                           dtype=ODT[d["input"].dtype], eps=w.eps,
                           weight_offset=w.weight_offset, scale_ub=w.scale_ub, want_pre=True)
    rep = P.compare_fp8(rows_of(q.view(torch.uint8), idx).cpu().numpy(),
                        rows_of(sc, idx).cpu().numpy(), bits(ro, idx), ora).check()
    assert rep["bad"] == 0

    # NVFP4 with the device global scale
    w, d = step.workloads["nvfp4"], step.batches["nvfp4"]
    gs = float(step.gs.cpu()[0])
    y = oracle.rmsnorm(host_bits(d["input"]), None, host_bits(d["gamma"]),
                       dtype=ODT[d["input"].dtype], eps=w.eps)["y"]
    gs_ora = float(oracle.nvfp4_global_scale(np.abs(y).max()))
    del y
    assert abs(gs - gs_ora) <= 2e-6 * gs_ora, (gs, gs_ora)
    idx = sample_rows(w.rows, 48, seed=18)
    q, bs, ro = step.out["nvfp4"]
    assert ro is None
    ora = oracle.quant_nvfp4(bits(d["input"], idx), None, host_bits(d["gamma"]), gs,
                             dtype=ODT[d["input"].dtype], eps=w.eps, want_y=True, want_pre=True)
    P.compare_nvfp4(rows_of(q, idx).cpu().numpy(), rows_of(bs.view(torch.uint8), idx).cpu().numpy(),
                    None, ora, gs).check()

    # MXFP4 at 65536 x 16384
    w, d = step.workloads["mxfp4"], step.batches["mxfp4"]
    idx = sample_rows(w.rows, 32, seed=19)
    q, bs, ro = step.out["mxfp4"]
    ora = oracle.quant_mxfp4(bits(d["input"], idx), bits(d["residual"], idx), host_bits(d["gamma"]),
                             dtype=ODT[d["input"].dtype], eps=w.eps, want_y=True, want_pre=True)
    P.compare_mxfp4(rows_of(q, idx).cpu().numpy(), rows_of(bs, idx).cpu().numpy(),
                    bits(ro, idx), ora).check()
    del step
    torch.cuda.empty_cache()
    assert rq().rmsq_device_status() == 0


def test_row_chunks_equal_the_whole_batch():
    # bench.py's end-to-end leg queues each batch as row chunks (one entry-point call per chunk,
    # between the copies in and out); the outputs must be those of one call on the whole batch
    import bench
    import workloads as W
    dev = torch.device("cuda", 0)
    wl = {"fp8": W.config("fp8_gemma", rows=3001), "nvfp4": W.config("nvfp4", rows=2999),
          "mxfp4": W.config("mxfp4_residual", rows=3003, hidden=16384)}
    step = bench.Step(rq(), dev, workloads=wl, seed=5)
    for m in step.modes:
        step.launch(m)
    torch.cuda.synchronize()
    whole = {m: [None if t is None else t.view(torch.uint8).clone() for t in step.out[m]]
             for m in step.modes}
    for m in step.modes:
        for t in step.out[m]:
            if t is not None:
                t.view(torch.uint8).fill_(0xA5)
        chunks = bench.e2e_chunks(step.workloads[m], 8 << 20)
        assert len(chunks) > 2, m
        for r0, r1 in chunks:
            step.launch(m, rows=(r0, r1))
    torch.cuda.synchronize()
    for m in step.modes:
        for a, b in zip(step.out[m], whole[m]):
            if a is not None:
                assert torch.equal(a.view(torch.uint8), b), m
    assert rq().rmsq_device_status() == 0

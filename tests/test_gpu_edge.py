"""GPU edge cases: empty calls, guard bytes after every output, degenerate rows (all zero,
constant, one spike), argument errors reported without a launch, the bounded-wait timeout
report, and the device conversion instructions against the oracle's encoders over a sweep of
fp32 bit patterns."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_common import check_fp8, check_mxfp4, check_nvfp4, guarded, guards_intact, host_bits, rq

pytestmark = pytest.mark.gpu

def test_empty_call_launches_nothing():
    x = torch.empty(0, 4096, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(4096, dtype=torch.bfloat16, device="cuda")
    before = rq().rmsq_launch_count()
    q, s, _ = rq().rmsnorm_quant_fp8(x, g)
    q4, b4, _ = rq().rmsnorm_quant_mxfp4(x, g)
    assert rq().rmsq_launch_count() == before
    assert q.shape == (0, 4096) and s.shape == (0,) and q4.shape == (0, 2048)


@pytest.mark.parametrize("mode", ["fp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("sched", [1, 2])
def test_guard_bytes_untouched(mode, sched):
    rows, H = 97, 2080
    w = W.Workload("custom", mode, rows, H, "bf16", True)
    d = W.generate(w, seed=21, device="cuda")
    ro, ro_raw = guarded(rows * H, torch.bfloat16)
    ro = ro.view(rows, H)
    prev = rq().rmsq_set_schedule(sched)
    try:
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
            fn = rq().rmsnorm_quant_nvfp4 if mode == "nvfp4" else rq().rmsnorm_quant_mxfp4
            bs = b.view(rows, H // blk)
            fn(d["input"], d["gamma"], residual=d["residual"], residual_output=ro,
               output=q.view(rows, H // 2), block_scale=bs.view(torch.float8_e4m3fn) if mode == "nvfp4" else bs)
            raws = (ro_raw, q_raw, b_raw)
    finally:
        rq().rmsq_set_schedule(prev)
    torch.cuda.synchronize()
    assert guards_intact(raws)
    assert torch.equal(ro, (d["input"].float() + d["residual"].float()).to(torch.bfloat16))


def _rows_tensor(rows):
    return torch.tensor(np.array(rows, np.float32)).to(torch.bfloat16).cuda()


def test_degenerate_rows():
    H = 4096
    zero = np.zeros(H)
    const = np.full(H, -3.0)
    spike = np.zeros(H)
    spike[77] = 1000.0
    tiny = np.full(H, 1e-30)
    x = _rows_tensor([zero, const, spike, tiny])
    d = dict(input=x, residual=None, gamma=torch.ones(H, dtype=torch.bfloat16, device="cuda"))
    w = W.Workload("custom", "fp8", 4, H, "bf16", False, scale_ub=10.0)
    rep, ora = check_fp8(w, d)
    assert ora["scale"][0] == 0 and ora["scale"][2] == np.float32(10.0 / 448.0)
    wn = W.Workload("custom", "nvfp4", 4, H, "bf16", False)
    check_nvfp4(wn, d, 1.0)
    wm = W.Workload("custom", "mxfp4", 4, H, "bf16", False)
    check_mxfp4(wm, d)


def test_argument_errors_do_not_launch():
    H = 256
    x = torch.randn(8, H, device="cuda").to(torch.bfloat16)
    g = torch.ones(H, dtype=torch.bfloat16, device="cuda")
    lib = rq().lib()
    q = torch.empty(8, H, dtype=torch.uint8, device="cuda")
    s = torch.empty(8, dtype=torch.float32, device="cuda")
    p = lambda t, off=0: t.data_ptr() + off
    before = rq().rmsq_launch_count()
    st = rq().lib().rmsnorm_quant_fp8
    assert st(p(x, 2), None, None, p(g), 8, H, 0, 1e-6, 0.0, 10.0, p(q), p(s), 2, None) == 3
    assert st(p(x), p(x), None, p(g), 8, H, 0, 1e-6, 0.0, 10.0, p(q), p(s), 2, None) == 1
    assert st(p(x), None, None, p(g), 8, H + 4, 0, 1e-6, 0.0, 10.0, p(q), p(s), 2, None) == 2
    assert st(p(x), None, None, p(g), 8, H, 7, 1e-6, 0.0, 10.0, p(q), p(s), 2, None) == 4
    assert st(p(x), None, None, p(g), 8, H, 0, -1.0, 0.0, 10.0, p(q), p(s), 2, None) == 6
    assert st(p(x), None, None, p(g), 8, H, 0, 1e-6, 0.0, 0.0, p(q), p(s), 2, None) == 6
    assert st(p(x), None, None, p(g), -1, H, 0, 1e-6, 0.0, 10.0, p(q), p(s), 2, None) == 2
    assert lib.rmsnorm_quant_mxfp4(p(x), None, None, p(g), 8, 48, 0, 1e-6, 0.0, p(q), p(s), 0, None) == 2
    assert lib.rmsnorm_quant_nvfp4(p(x), None, None, p(g), 8, H, 0, 1e-6, 0.0, None, p(q), p(s), 0, None) == 1
    assert lib.rmsnorm_quant_nvfp4(p(x), None, None, p(g), 8, H, 0, 1e-6, 0.0, p(s), p(q), p(s), 5, None) == 4
    assert rq().rmsq_launch_count() == before


def test_bounded_wait_reports_timeout_and_context_survives():
    assert rq().rmsq_device_status() == 0
    rq().rmsq_selftest_wait_timeout(2_000_000)        # 2 ms; nothing completes the barrier
    assert rq().rmsq_device_status() == 8               # RMSQ_ERR_TIMEOUT, flag now cleared
    assert rq().rmsq_device_status() == 0
    w = W.config("fp8_small")
    check_fp8(w, W.generate(w, device="cuda"))          # the context is still usable


def _sweep_values():
    """All fp32 bit patterns whose magnitude lies in [2^-12, 2^10), both signs (the range where
    E4M3 and E2M1 rounding decides something), plus a strided sample of every other pattern."""
    e_lo, e_hi = 127 - 12, 127 + 10
    mags = np.arange(e_lo << 23, e_hi << 23, dtype=np.uint32)
    other = np.arange(0, 1 << 31, 4099, dtype=np.uint32)
    bits = np.concatenate([mags, other, mags | np.uint32(1 << 31), other | np.uint32(1 << 31)])
    vals = bits.view(np.float32)
    return vals[np.isfinite(vals)]


@pytest.mark.parametrize("fmt", [0, 1])
def test_device_conversions_match_oracle_encoders(fmt):
    vals = _sweep_values()
    chunk = 1 << 26
    mism = 0
    for i in range(0, vals.size, chunk):
        v = vals[i:i + chunk]
        dev = rq().rmsq_debug_convert(fmt, torch.from_numpy(v).cuda()).cpu().numpy()
        ref = oracle.e4m3_encode(v) if fmt == 0 else oracle.e2m1_encode(v)
        mask = 0x7F if fmt == 0 else 0x7
        both_zero = ((dev & mask) == 0) & ((ref & mask) == 0)
        mism += int(((dev != ref) & ~both_zero).sum())
    assert mism == 0

"""Pins of the oracle's row math against closed forms, torch CPU library routines and brute force.

What each test would catch:
  residual add      wrong rounding of the pre-norm sum         -> torch (a.float()+b.float()).to(dt)
  rmsnorm           dropped eps, wrong mean, offset misapplied -> torch.nn.functional.rms_norm (f64)
  constant row      rstd / scale / saturation closed form
  zero row          eps keeps rstd finite, scale 0, codes 0
  spike row         scale_ub clamp on amax, satfinite at 448
  fp8 quant         y / scale rounding                          -> torch float8_e4m3fn cast
  nvfp4 / mxfp4     block scale, element factor, nibble order   -> brute-force search per block
  invariants        |dequant - y| <= half a quantisation step (unclamped elements)
  fp32 input        the fp32 sum rounded elsewhere, or y off    -> torch fp32 add, rms_norm (f64)
  global scale      gs inverted or off by a factor             -> largest block scale is 448
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads as W


def _bits(t):
    return W.bits(t)


def _rand(rows, H, dtype=torch.bfloat16, seed=0, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(rows, H, generator=g) * std).to(dtype)


ODT = {torch.bfloat16: oracle.BF16, torch.float16: oracle.FP16}


# ------------------------------------------------------------------------------------------
# residual add and RMSNorm
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
def test_residual_add_matches_torch(dt):
    x = _rand(8, 512, dt, 1, 3.0)
    r = _rand(8, 512, dt, 2, 0.01)
    g = torch.ones(512, dtype=dt)
    out = oracle.quant_fp8(_bits(x), _bits(r), _bits(g), dtype=ODT[dt])
    ref = (x.float() + r.float()).to(dt)
    assert np.array_equal(out["residual_output"], _bits(ref))


@pytest.mark.parametrize("dt,offset", [(torch.bfloat16, 0.0), (torch.float16, 1.0), (torch.bfloat16, 0.5)])
@pytest.mark.parametrize("residual", [False, True])
def test_rmsnorm_matches_torch_rms_norm(dt, offset, residual):
    rows, H = 16, 1024
    x = _rand(rows, H, dt, 3, 2.0)
    r = _rand(rows, H, dt, 4) if residual else None
    g = (torch.randn(H, generator=torch.Generator().manual_seed(5)) * 0.1 + (0.0 if offset else 1.0)).to(dt)
    out = oracle.rmsnorm(_bits(x), None if r is None else _bits(r), _bits(g), dtype=ODT[dt],
                         eps=1e-6, weight_offset=offset)
    s = (x.float() + r.float()).to(dt) if residual else x
    w = (g.float() + offset).double()
    ref = F.rms_norm(s.double(), (H,), weight=w, eps=float(np.float32(1e-6))).numpy()
    y = out["y"].astype(np.float64)
    # y = RN32(s * RN32(rstd) * w): two fp32 roundings away from the exact value
    assert np.all(np.abs(y - ref) <= 2.5 * 2.0 ** -24 * np.abs(ref) + 1e-30)
    rstd_ref = 1.0 / np.sqrt((s.double() ** 2).mean(-1).numpy() + float(np.float32(1e-6)))
    assert np.all(np.abs(out["rstd"] - rstd_ref) <= 2.0 ** -24 * rstd_ref)


def test_constant_row_closed_form():
    H = 256
    for c in (0.75, -3.0, 100.0):
        x = torch.full((1, H), c, dtype=torch.bfloat16)
        g = torch.ones(H, dtype=torch.bfloat16)
        out = oracle.quant_fp8(_bits(x), None, _bits(g), eps=1e-6, scale_ub=1200.0, want_y=True)
        cb = float(x[0, 0])
        rstd = np.float32(1.0 / math.sqrt(cb * cb + float(np.float32(1e-6))))
        y = np.float32(cb * float(rstd))
        assert np.all(out["y"] == y)
        assert out["scale"][0] == np.float32(abs(float(y)) / 448.0)
        want = 0x7E if c > 0 else 0xFE
        assert np.all(out["q"] == want)


def test_zero_row():
    H = 512
    x = torch.zeros((2, H), dtype=torch.bfloat16)
    g = torch.ones(H, dtype=torch.bfloat16)
    out = oracle.quant_fp8(_bits(x), None, _bits(g), want_y=True)
    assert np.all(out["y"] == 0) and np.all(out["scale"] == 0) and np.all(out["q"] == 0)
    nv = oracle.quant_nvfp4(_bits(x), None, _bits(g), 1.0)
    assert np.all(nv["q"] == 0) and np.all(nv["block_scale"] == 0)
    mx = oracle.quant_mxfp4(_bits(x), None, _bits(g))
    assert np.all(mx["q"] == 0) and np.all(mx["block_scale"] == 0)
    rs = oracle.rmsnorm(_bits(x), None, _bits(g))["rstd"]
    assert np.all(rs == np.float32(1.0 / math.sqrt(float(np.float32(1e-6)))))


def test_spike_row_clamps_scale_ub():
    H = 4096
    x = torch.zeros((1, H), dtype=torch.bfloat16)
    x[0, 123] = 1000.0
    g = torch.ones(H, dtype=torch.bfloat16)
    out = oracle.quant_fp8(_bits(x), None, _bits(g), scale_ub=10.0, want_y=True)
    y_spike = float(out["y"][0, 123])
    assert abs(y_spike - math.sqrt(H)) < 1e-3          # y = 1000 / sqrt(1e6 / H) = sqrt(H) = 64
    assert out["scale"][0] == np.float32(10.0 / 448.0)  # amax 64 > ub 10
    assert out["q"][0, 123] == 0x7E                     # 64 / (10/448) = 2867 saturates to 448
    assert np.count_nonzero(out["q"]) == 1


# ------------------------------------------------------------------------------------------
# FP8 against torch's cast, and the half-step invariant
# ------------------------------------------------------------------------------------------

def _e4m3_midpoints():
    v = oracle.e4m3_values()
    v = np.unique(np.abs(v[~np.isnan(v)]))
    return (v[1:] + v[:-1]) / 2


def _near(v, mids, rel=1e-6):
    a = np.abs(v)
    idx = np.clip(np.searchsorted(mids, a), 1, len(mids) - 1)
    d = np.minimum(np.abs(a - mids[idx - 1]), np.abs(a - mids[idx]))
    return d <= rel * a


def test_fp8_quant_matches_torch_cast():
    w = W.config("fp8_residual", rows=64)
    d = W.generate(w, seed=7)
    out = oracle.quant_fp8(_bits(d["input"]), _bits(d["residual"]), _bits(d["gamma"]),
                           scale_ub=w.scale_ub, want_y=True, want_pre=True)
    y = torch.from_numpy(out["y"]).double()
    amax = y.abs().amax(-1, keepdim=True).clamp(max=w.scale_ub)
    scale = (amax / 448.0).float()
    assert np.array_equal(scale.numpy()[:, 0], out["scale"])
    ref = (y / scale.double()).float().clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    diff = (ref != out["q"]) & ((ref & 0x7F) | (out["q"] & 0x7F) != 0)
    assert np.all(_near(out["pre"][diff], _e4m3_midpoints()))


def test_fp8_half_step_invariant():
    w = W.config("fp8_gemma_spike", rows=300, hidden=1024)
    d = W.generate(w, seed=8)
    out = oracle.quant_fp8(_bits(d["input"]), _bits(d["residual"]), _bits(d["gamma"]),
                           dtype=oracle.FP16, weight_offset=1.0, scale_ub=10.0, want_y=True,
                           want_pre=True)
    v = out["pre"]
    dq = oracle.e4m3_values()[out["q"]]
    ok = np.abs(v) <= 448.0
    step = np.exp2(np.maximum(np.floor(np.log2(np.maximum(np.abs(v), 1e-300))), -6) - 3)
    assert np.all(np.abs(dq - v)[ok] <= step[ok] / 2)
    assert np.all(dq[~ok] == np.sign(v[~ok]) * 448.0)
    assert (~ok).any()              # the spike rows do clamp


# ------------------------------------------------------------------------------------------
# NVFP4 / MXFP4 against brute force
# ------------------------------------------------------------------------------------------

E2M1_MAGS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _nearest_code(v, mags, max_code):
    """Brute-force nearest magnitude code with ties to the even code, saturating at max."""
    a = min(abs(v), mags[max_code])
    best = min(range(max_code + 1), key=lambda c: (abs(a - mags[c]), c % 2))
    return best


def _brute_nvfp4_block(y, gs):
    e4 = torch.arange(0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    a = max(abs(float(v)) for v in y)
    t = min(gs * a / 6.0, 448.0)
    s = _nearest_code(t, e4, 0x7E)
    ds = e4[s]
    codes = []
    for v in y:
        if ds == 0:
            codes.append(0)
            continue
        x = float(v) * gs / ds
        c = _nearest_code(x, E2M1_MAGS, 7)
        codes.append(c | (8 if x < 0 else 0))
    return s, codes


def _pack(codes):
    return [codes[2 * k] | (codes[2 * k + 1] << 4) for k in range(len(codes) // 2)]


def _strip_zero_sign(b):
    b = np.asarray(b, np.uint8)
    lo, hi = b & 0xF, b >> 4
    lo = np.where((lo & 7) == 0, 0, lo)
    hi = np.where((hi & 7) == 0, 0, hi)
    return lo | (hi << 4)


@pytest.mark.parametrize("gs", [1.0, 37.5, 0.01])
def test_nvfp4_matches_brute_force(gs):
    w = W.config("nvfp4", rows=6, hidden=256)
    d = W.generate(w, seed=9)
    out = oracle.quant_nvfp4(_bits(d["input"]), None, _bits(d["gamma"]), gs, want_y=True)
    for r in range(w.rows):
        for b in range(w.hidden // 16):
            yb = out["y"][r, b * 16:(b + 1) * 16]
            s, codes = _brute_nvfp4_block(yb, gs)
            assert out["block_scale"][r, b] == s
            got = _strip_zero_sign(out["q"][r, b * 8:(b + 1) * 8])
            assert np.array_equal(got, _strip_zero_sign(_pack(codes))), (r, b)


def test_mxfp4_matches_brute_force():
    w = W.config("mxfp4_residual", rows=6, hidden=512)
    d = W.generate(w, seed=10)
    out = oracle.quant_mxfp4(_bits(d["input"]), _bits(d["residual"]), _bits(d["gamma"]), want_y=True)
    for r in range(w.rows):
        for b in range(w.hidden // 32):
            yb = out["y"][r, b * 32:(b + 1) * 32].astype(np.float64)
            a = np.abs(yb).max()
            e = math.ceil(math.log2(a / 6.0))
            if 6.0 * 2.0 ** (e - 1) >= a:   # guard the float log2 at exact powers of two
                e -= 1
            code = e + 127
            assert out["block_scale"][r, b] == code
            codes = []
            for v in yb:
                x = v * 2.0 ** (127 - code)
                c = _nearest_code(x, E2M1_MAGS, 7)
                codes.append(c | (8 if x < 0 else 0))
            got = _strip_zero_sign(out["q"][r, b * 16:(b + 1) * 16])
            assert np.array_equal(got, _strip_zero_sign(_pack(codes))), (r, b)


def test_fp4_nibble_order():
    # element 0 -> 6.0 (code 7, low nibble), element 1 -> 0.5 (code 1, high nibble)
    H = 64
    x = torch.zeros((1, H), dtype=torch.bfloat16)
    x[0, 0], x[0, 1] = 12.0, 1.0
    g = torch.ones(H, dtype=torch.bfloat16)
    mx = oracle.quant_mxfp4(_bits(x), None, _bits(g), want_y=True)
    # y0 = 12 / sqrt(145 / 64) = 7.97: code 128 (factor 1/2), so y0 -> 3.99 -> 4 (code 6) and
    # y1 = y0 / 12 -> 0.33 -> 0.5 (code 1)
    assert mx["block_scale"][0, 0] == 128
    assert mx["q"][0, 0] == 0x16
    nv = oracle.quant_nvfp4(_bits(x), None, _bits(g), 1.0)
    # t = 7.97 / 6 = 1.33 -> E4M3 1.375 (code 0x3B); 7.97 / 1.375 = 5.8 -> 6 (code 7, low nibble);
    # 0.664 / 1.375 = 0.48 -> 0.5 (code 1, high nibble)
    assert nv["block_scale"][0, 0] == 0x3B
    assert nv["q"][0, 0] == 0x17


def test_fp4_half_step_invariant():
    w = W.config("nvfp4", rows=64, hidden=1024)
    d = W.generate(w, seed=11)
    gs = 3.0
    nv = oracle.quant_nvfp4(_bits(d["input"]), None, _bits(d["gamma"]), gs, want_y=True, want_pre=True)
    codes = np.stack([nv["q"] & 0xF, nv["q"] >> 4], -1).reshape(w.rows, w.hidden)
    dq = oracle.e2m1_values()[codes]
    v = nv["pre"]
    step = np.where(np.abs(v) < 2, 0.5, np.where(np.abs(v) < 4, 1.0, 2.0))
    ok = np.abs(v) <= 6.0
    assert np.all(np.abs(dq - v)[ok] <= step[ok] / 2)
    assert np.all(np.abs(dq[~ok]) == 6.0)
    # the block scale never exceeds the block's needs by more than one E4M3 rounding
    e4 = oracle.e4m3_values()
    s = e4[nv["block_scale"]]
    t = nv["t"]
    assert np.all(np.abs(s - t) <= np.maximum(np.exp2(np.floor(np.log2(np.maximum(t, 1e-300))) - 4), 2.0 ** -10))


@pytest.mark.parametrize("sdt,tdt", [(oracle.BF16, torch.bfloat16), (oracle.FP16, torch.float16)])
def test_fp8_rounded_scale_dtype(sdt, tdt):
    w = W.config("fp8_residual", rows=32, hidden=512)
    d = W.generate(w, seed=12)
    args = (_bits(d["input"]), _bits(d["residual"]), _bits(d["gamma"]))
    f32 = oracle.quant_fp8(*args, want_y=True)
    low = oracle.quant_fp8(*args, scale_dtype=sdt, want_y=True, want_pre=True)
    want = torch.from_numpy(f32["scale"]).to(tdt).float().numpy()
    assert np.array_equal(low["scale"], want)
    assert np.allclose(low["pre"], low["y"].astype(np.float64) / want[:, None].astype(np.float64))
    assert np.array_equal(low["q"], oracle.e4m3_encode(low["pre"]))


# ------------------------------------------------------------------------------------------
# fp32 input and the NVFP4 global scale
# ------------------------------------------------------------------------------------------

def test_fp32_input_rows_match_torch():
    # fp32 input: the residual sum is the fp32 sum itself, and y follows rms_norm in f64
    rows, H = 16, 1024
    gen = torch.Generator().manual_seed(11)
    x = torch.randn(rows, H, generator=gen) * 2.0
    r = torch.randn(rows, H, generator=gen)
    g = torch.randn(H, generator=gen) * 0.1 + 1.0
    out = oracle.quant_fp8(x.numpy(), r.numpy(), g.numpy(), dtype=oracle.F32, want_y=True)
    s = x + r
    assert np.array_equal(np.asarray(out["residual_output"]).view(np.uint32), s.numpy().view(np.uint32))
    ref = F.rms_norm(s.double(), (H,), weight=g.double(), eps=float(np.float32(1e-6))).numpy()
    y = out["y"].astype(np.float64)
    assert np.all(np.abs(y - ref) <= 2.5 * 2.0 ** -24 * np.abs(ref) + 1e-30)


def test_global_scale_puts_the_largest_block_on_448():
    # gs maps the tensor's largest |y| onto the largest block scale (448) times the largest E2M1
    # magnitude (6): the block holding it gets the E4M3 code of 448 and no block scale exceeds it
    rows, H = 32, 512
    x = _rand(rows, H, torch.bfloat16, 21, 1.0)
    x[5, 77] = 40.0                                  # one outlier decides the tensor's max
    g = (torch.randn(H, generator=torch.Generator().manual_seed(22)) * 0.1 + 1.0).to(torch.bfloat16)
    y = oracle.rmsnorm(_bits(x), None, _bits(g))["y"]
    r, c = np.unravel_index(np.argmax(np.abs(y)), y.shape)
    gs = oracle.nvfp4_global_scale(np.abs(y).max())
    out = oracle.quant_nvfp4(_bits(x), None, _bits(g), float(gs))
    bs = out["block_scale"].reshape(rows, H // 16)
    assert bs[r, c // 16] == 0x7E                    # 448
    assert bs.max() == 0x7E
    # the element at the max lands on E2M1 6 (code 7), with the sign of y
    q = out["q"].reshape(rows, H // 2)[r, c // 2]
    nib = (q >> (4 * (c % 2))) & 0xF
    assert nib & 0x7 == 0x7 and (nib >> 3) == (1 if y[r, c] < 0 else 0)

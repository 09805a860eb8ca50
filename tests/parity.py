"""Comparison of the CUDA path's outputs with the oracle's, under the parity rules:

  * residual_output bit-exact;
  * FP8 row scales within 1e-6 relative (exactly 0 on all-zero rows);
  * codes exact, except that a code may be one step away from the oracle's when the oracle's
    pre-rounding value lies within 1e-6 relative of a rounding boundary (a midpoint between two
    adjacent representable magnitudes); such elements are at most 1e-4 of all elements;
  * NVFP4 E4M3 block-scale codes and MXFP4 UE8M0 codes follow the same adjacent-code rule on their
    own pre-rounding values (t, and a / 6 against a power of two). A block whose scale code
    legitimately differs is re-checked against the oracle's element rule applied with the GPU's
    scale code;
  * +0 and -0 codes are equal (the sign a zero code carries is not part of the result).
"""
from __future__ import annotations

import numpy as np

import oracle

REL = 1e-6
MAX_FRACTION = 1e-4


def _mids(values):
    v = np.unique(np.abs(values[~np.isnan(values)]))
    return (v[1:] + v[:-1]) / 2


E4M3_MIDS = _mids(oracle.e4m3_values())
E2M1_MIDS = _mids(oracle.e2m1_values())


def near_boundary(v, mids, rel=REL):
    a = np.abs(np.asarray(v, np.float64))
    idx = np.clip(np.searchsorted(mids, a), 1, len(mids) - 1)
    d = np.minimum(np.abs(a - mids[idx - 1]), np.abs(a - mids[idx]))
    return d <= rel * np.maximum(a, 1e-300)


def _mag_sign(codes, bits):
    codes = np.asarray(codes).astype(np.int64)
    mag = codes & ((1 << (bits - 1)) - 1)
    sign = (codes >> (bits - 1)) & 1
    sign = np.where(mag == 0, 0, sign)
    return mag, sign


def code_diff(a, b, bits):
    """0 where equal (+-0 equal), 1 where adjacent magnitudes of one sign, 2 otherwise."""
    ma, sa = _mag_sign(a, bits)
    mb, sb = _mag_sign(b, bits)
    eq = (ma == mb) & (sa == sb)
    adj = (np.abs(ma - mb) == 1) & ((sa == sb) | (ma == 0) | (mb == 0))
    return np.where(eq, 0, np.where(adj, 1, 2))


def unpack_e2m1(packed, hidden):
    p = np.asarray(packed, np.uint8).reshape(-1, hidden // 2)
    return np.stack([p & 0xF, p >> 4], -1).reshape(-1, hidden)


class Report(dict):
    def check(self):
        assert self["bad"] == 0, self
        assert self["tolerated"] <= MAX_FRACTION * max(self["elements"], 1) + 0, self
        return self


def check_codes(gpu, ora, pre, bits, mids, report):
    d = code_diff(gpu, ora, bits)
    tol = (d == 1) & near_boundary(pre, mids)
    report["bad"] += int(((d == 2) | ((d == 1) & ~tol)).sum())
    report["tolerated"] += int(tol.sum())
    report["elements"] += int(d.size)
    if report["bad"] and "first_bad" not in report:
        idx = np.argwhere((d == 2) | ((d == 1) & ~tol))[:5]
        report["first_bad"] = [(tuple(int(j) for j in i), int(np.asarray(gpu)[tuple(i)]),
                                int(np.asarray(ora)[tuple(i)]), float(np.asarray(pre)[tuple(i)]))
                               for i in idx]


def compare_residual(gpu_res, ora_res, report):
    if ora_res is None:
        return
    diff = int((np.asarray(gpu_res) != np.asarray(ora_res)).sum())
    report["residual_mismatch"] = report.get("residual_mismatch", 0) + diff
    report["bad"] += diff


def compare_fp8(gpu_q, gpu_scale, gpu_res, ora, report=None):
    """gpu_q uint8 [rows, H], gpu_scale float32 [rows]; ora from oracle.quant_fp8(want_pre=True)."""
    report = report if report is not None else Report(bad=0, tolerated=0, elements=0)
    compare_residual(gpu_res, ora["residual_output"], report)
    so, sg = ora["scale"].astype(np.float64), np.asarray(gpu_scale, np.float64)
    scale_bad = (np.abs(sg - so) > REL * np.abs(so)) | ((so == 0) != (sg == 0))
    report["scale_bad"] = report.get("scale_bad", 0) + int(scale_bad.sum())
    report["bad"] += int(scale_bad.sum())
    check_codes(gpu_q, ora["q"], ora["pre"], 8, E4M3_MIDS, report)
    return report


def compare_nvfp4(gpu_q, gpu_bs, gpu_res, ora, gs, report=None):
    """Row-major block scales. ora from oracle.quant_nvfp4(want_y=True, want_pre=True)."""
    report = report if report is not None else Report(bad=0, tolerated=0, elements=0)
    compare_residual(gpu_res, ora["residual_output"], report)
    rows, H = ora["y"].shape
    nsf = H // 16
    gbs = np.asarray(gpu_bs, np.uint8).reshape(rows, nsf)
    sd = code_diff(gbs, ora["block_scale"], 8)
    scale_tol = (sd == 1) & near_boundary(ora["t"], E4M3_MIDS)
    report["scale_bad"] = report.get("scale_bad", 0) + int(((sd == 2) | ((sd == 1) & ~scale_tol)).sum())
    report["bad"] += int(((sd == 2) | ((sd == 1) & ~scale_tol)).sum())
    report["scale_tolerated"] = report.get("scale_tolerated", 0) + int(scale_tol.sum())
    gq = unpack_e2m1(gpu_q, H)
    oq = unpack_e2m1(ora["q"], H)
    pre = ora["pre"].copy()
    # blocks whose scale legitimately differs: expected codes from the GPU's scale code
    for r, b in np.argwhere(scale_tol):
        ds = oracle.e4m3_decode(int(gbs[r, b]))
        yb = ora["y"][r, b * 16:(b + 1) * 16].astype(np.float64)
        v = yb * float(gs) / ds if ds != 0 else np.zeros(16)
        oq[r, b * 16:(b + 1) * 16] = oracle.e2m1_encode(v) if ds != 0 else 0
        pre[r, b * 16:(b + 1) * 16] = v
    check_codes(gq, oq, pre, 4, E2M1_MIDS, report)
    return report


def _near_pow2(v, rel=REL):
    v = np.asarray(v, np.float64)
    with np.errstate(divide="ignore"):
        e = np.round(np.log2(np.maximum(v, 1e-300)))
    p = np.exp2(e)
    return np.abs(v - p) <= rel * p


def compare_mxfp4(gpu_q, gpu_bs, gpu_res, ora, report=None):
    """Row-major block scales. ora from oracle.quant_mxfp4(want_y=True, want_pre=True)."""
    report = report if report is not None else Report(bad=0, tolerated=0, elements=0)
    compare_residual(gpu_res, ora["residual_output"], report)
    rows, H = ora["y"].shape
    nsf = H // 32
    gbs = np.asarray(gpu_bs, np.uint8).reshape(rows, nsf).astype(np.int64)
    obs = ora["block_scale"].astype(np.int64)
    sd = np.abs(gbs - obs)
    scale_tol = (sd == 1) & _near_pow2(ora["a"] / 6.0)
    nbad = int(((sd > 1) | ((sd == 1) & ~scale_tol)).sum())
    report["scale_bad"] = report.get("scale_bad", 0) + nbad
    report["bad"] += nbad
    report["scale_tolerated"] = report.get("scale_tolerated", 0) + int(scale_tol.sum())
    gq = unpack_e2m1(gpu_q, H)
    oq = unpack_e2m1(ora["q"], H)
    pre = ora["pre"].copy()
    for r, b in np.argwhere(scale_tol):
        code = int(gbs[r, b])
        yb = ora["y"][r, b * 32:(b + 1) * 32].astype(np.float64)
        v = np.ldexp(yb, 127 - code) if code else np.zeros(32)
        oq[r, b * 32:(b + 1) * 32] = oracle.e2m1_encode(v) if code else 0
        pre[r, b * 32:(b + 1) * 32] = v
    check_codes(gq, oq, pre, 4, E2M1_MIDS, report)
    return report


def unswizzle(flat, rows, nsf):
    """Swizzled 128x4 block scales -> row-major [rows, nsf], via the oracle's index function."""
    flat = np.asarray(flat, np.uint8)
    out = np.zeros((rows, nsf), np.uint8)
    for r in range(rows):
        for s in range(nsf):
            out[r, s] = flat[oracle.scale_offset(r, s, nsf, True)]
    return out

"""Pins of the oracle's number-format code against things other than itself.

E4M3: the decode table and in-range RNE encoding are checked against torch's CPU float8_e4m3fn
casts (a library routine). E2M1: the code table is checked against a golden fixture and the
encoder against brute-force nearest-value search. bf16 / fp16: decode and rounding against torch
CPU casts. UE8M0: against an exact search over integer exponents with rational arithmetic.
"""
import fractions
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line.split())
    return rows


def _torch_e4m3_table():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().double().numpy()


# ------------------------------------------------------------------------------------------
# E4M3
# ------------------------------------------------------------------------------------------

def test_e4m3_decode_matches_torch_all_codes():
    ours = oracle.e4m3_values()
    ref = _torch_e4m3_table()
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_e4m3_constants_match_golden():
    consts = {k: float(v) for k, v in _golden("format_constants.txt")}
    vals = oracle.e4m3_values()
    assert np.nanmax(vals) == consts["e4m3_max"] == 448.0
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_roundtrip_every_finite_code():
    vals = oracle.e4m3_values()
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    back = oracle.e4m3_encode(vals[codes])
    assert np.array_equal(back, codes.astype(np.uint8))


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(1)
    mags = np.exp2(rng.uniform(-14, math.log2(464.0), 400_000))
    v = (mags * rng.choice([-1.0, 1.0], mags.size)).astype(np.float32)
    # add every representable value, every midpoint and its fp32 neighbours
    vals = np.unique(np.abs(oracle.e4m3_values()[~np.isnan(oracle.e4m3_values())]))
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)
    extra = np.concatenate([vals.astype(np.float32), mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9)])
    v = np.concatenate([v, extra, -extra, np.float32([464.0, -464.0])])
    ours = oracle.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    zero = (ours & 0x7F) == 0
    assert np.array_equal(ours[~zero], ref[~zero])
    assert np.array_equal(ref[zero] & 0x7F, np.zeros(zero.sum(), np.uint8))


def test_e4m3_ties_go_to_even_mantissa():
    table = _torch_e4m3_table()
    pos = [(c, table[c]) for c in range(0x7F)]          # 0x00 .. 0x7E, ascending values
    for (c0, v0), (c1, v1) in zip(pos[:-1], pos[1:]):
        mid = (v0 + v1) / 2
        got = int(oracle.e4m3_encode(np.float64([mid]))[0])
        assert got == (c0 if c0 % 2 == 0 else c1), (c0, c1, mid)
        below = int(oracle.e4m3_encode(np.float64([mid * (1 - 1e-9)]))[0])
        above = int(oracle.e4m3_encode(np.float64([mid * (1 + 1e-9)]))[0])
        assert (below, above) == (c0, c1)


@pytest.mark.parametrize("v", [448.0, 449.0, 463.99, 464.0, 465.0, 480.0, 1e6, 3e38, math.inf])
def test_e4m3_satfinite(v):
    assert int(oracle.e4m3_encode(np.float64([v]))[0]) == 0x7E
    assert int(oracle.e4m3_encode(np.float64([-v]))[0]) == 0xFE


def test_e4m3_nan_and_signed_zero():
    assert int(oracle.e4m3_encode(np.float64([math.nan]))[0]) == 0x7F
    assert int(oracle.e4m3_encode(np.float64([-0.0]))[0]) == 0x80
    assert int(oracle.e4m3_encode(np.float64([-1e-9]))[0]) == 0x80   # rounds to -0
    assert int(oracle.e4m3_encode(np.float64([2.0 ** -10]))[0]) == 0x00  # tie 0 / 2^-9: even
    assert int(oracle.e4m3_encode(np.float64([3 * 2.0 ** -11]))[0]) == 0x01


# ------------------------------------------------------------------------------------------
# E2M1
# ------------------------------------------------------------------------------------------

def test_e2m1_table_matches_golden():
    table = {int(c): float(v) for c, v in _golden("e2m1_values.txt")}
    for code in range(16):
        got = oracle.e2m1_decode(code)
        assert got == table[code]
        assert math.copysign(1, got) == math.copysign(1, table[code])
    consts = {k: float(v) for k, v in _golden("format_constants.txt")}
    assert max(table.values()) == consts["e2m1_max"]


def _e2m1_brute(v):
    """Nearest of the 8 magnitudes, ties to the even code, saturating at 6."""
    table = [float(x) for _, x in _golden("e2m1_values.txt")][:8]
    a = min(abs(v), 6.0)
    best = min(range(8), key=lambda c: (abs(a - table[c]), c % 2))
    return best | (8 if math.copysign(1, v) < 0 else 0)


def test_e2m1_encode_brute_force():
    rng = np.random.default_rng(2)
    v = np.concatenate([rng.uniform(-8, 8, 20000), rng.uniform(-0.6, 0.6, 5000)])
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    v = np.concatenate([v, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 9), [6.0, 7.0, 1e9]])
    ours = oracle.e2m1_encode(v)
    for x, c in zip(v, ours):
        want = _e2m1_brute(x)
        if (want & 7) == 0 and (c & 7) == 0:
            continue  # +-0: sign compared separately below
        assert c == want, (x, c, want)
    assert int(oracle.e2m1_encode(np.float64([-0.2]))[0]) == 0x8


def test_e2m1_roundtrip():
    for code in range(16):
        assert int(oracle.e2m1_encode(np.float64([oracle.e2m1_decode(code)]))[0]) == code


# ------------------------------------------------------------------------------------------
# bf16 / fp16
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("dt,tdt", [(oracle.BF16, torch.bfloat16), (oracle.FP16, torch.float16)])
def test_16bit_decode_all_codes(dt, tdt):
    codes = np.arange(65536, dtype=np.uint16)
    ours = oracle.decode_bits(codes, dt)
    ref = torch.from_numpy(codes.view(np.int16)).view(tdt).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


@pytest.mark.parametrize("dt,tdt", [(oracle.BF16, torch.bfloat16), (oracle.FP16, torch.float16)])
def test_16bit_rounding_matches_torch(dt, tdt):
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 32, 1_000_000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    if dt == oracle.FP16:  # keep to the fp16 range plus a margin of overflow
        f = np.concatenate([np.clip(f, -70000, 70000), rng.uniform(-70000, 70000, 100000).astype(np.float32),
                            rng.uniform(-1e-4, 1e-4, 100000).astype(np.float32)])
    ours = oracle.round_to_dtype(f.astype(np.float64), dt)
    ref = torch.from_numpy(f).to(tdt).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# ------------------------------------------------------------------------------------------
# UE8M0
# ------------------------------------------------------------------------------------------

def _ue8m0_exact(a: float) -> int:
    """Smallest integer e with 6 * 2^e >= a, by search in exact rationals, plus the bias 127,
    clamped to [0, 255]; 0 for a <= 0."""
    if a <= 0:
        return 0
    fa = fractions.Fraction(a)
    e = -300
    while fractions.Fraction(6) * fractions.Fraction(2) ** e < fa:
        e += 1
    return max(0, min(255, e + 127))


def test_ue8m0_exact_ceiling_brute_force():
    consts = {k: float(v) for k, v in _golden("format_constants.txt")}
    assert consts["ue8m0_bias"] == 127
    vals = [0.0, -1.0]
    for e in range(-130, 131):
        base = 6.0 * 2.0 ** e
        for d in (0.0, 2.0 ** -23, -(2.0 ** -24), 1e-3, -1e-3, 0.3, -0.3):
            with np.errstate(over="ignore"):
                a = float(np.float32(base * (1 + d)))
            if np.isfinite(a):
                vals.append(a)
    vals += [float(np.float32(x)) for x in (1e-45, 1e-40, 1.17549435e-38, 3.4e38)]
    ours = oracle.ue8m0_code(np.array(vals))
    for a, c in zip(vals, ours):
        assert int(c) == _ue8m0_exact(a), (a, c)
    assert int(oracle.ue8m0_code(np.array([6.0]))[0]) == 127
    assert int(oracle.ue8m0_code(np.array([float(np.float32(6.0000005))]))[0]) == 128


# ------------------------------------------------------------------------------------------
# Swizzled scale layout
# ------------------------------------------------------------------------------------------

def test_swizzle_offsets_match_hand_worked_golden():
    for rows, nsf, r, sf, off in (map(int, x) for x in _golden("swizzle_offsets.txt")):
        assert oracle.scale_offset(r, sf, nsf, True) == off
        assert oracle.scale_offset(r, sf, nsf, False) == r * nsf + sf


def test_swizzle_is_injective_and_fills_whole_tiles():
    for rows, nsf in ((256, 8), (200, 6), (1, 1), (130, 448)):
        offs = [oracle.scale_offset(r, s, nsf, True) for r in range(rows) for s in range(nsf)]
        assert len(set(offs)) == len(offs)
        assert max(offs) < oracle.swizzled_scale_size(rows, nsf)
        if rows % 128 == 0 and nsf % 4 == 0:
            assert sorted(offs) == list(range(oracle.swizzled_scale_size(rows, nsf)))

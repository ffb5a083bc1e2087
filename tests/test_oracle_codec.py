"""Pins of the oracle's FP8 codec against what the pages and mathematics fix.

Independent sources used here (none of them is the oracle's own code):
  * named values printed on the pages (tests/golden/fp8_named_values.txt);
  * the unit roundoff printed on "FP8 Mixed-Precision Serving in Production"
    (tests/golden/unit_roundoff.txt);
  * torch's float8_e4m3fn / float8_e5m2 dtypes (a library decode, and a library
    round-to-nearest-even cast that agrees with a saturating encoder wherever
    it does not overflow);
  * IEEE binary16: E5M2 keeps half precision's 5-bit exponent and bias 15, so
    code c is the top byte of a binary16 value;
  * two independent encoders inside the oracle agreeing on all 2^32 fp32 inputs.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FMT = {"E4M3": E4M3, "E5M2": E5M2}
TORCH_DT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("|")[0].strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_named_values_from_pages():
    rows = _golden("fp8_named_values.txt")
    assert len(rows) >= 12
    for fmt_name, code, value in rows:
        got = oracle.decode(np.array([int(code, 16)]), FMT[fmt_name])[0]
        if value == "nan":
            assert math.isnan(got), (fmt_name, code)
        else:
            assert got == float(value), (fmt_name, code, got, value)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_decode_all_codes_match_torch_float8(fmt):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.decode(codes, fmt)
    ref = torch.from_numpy(codes.copy()).view(TORCH_DT[fmt]).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.all(both_nan | (ours == ref))
    assert np.array_equal(np.signbit(ours[~both_nan]), np.signbit(ref[~both_nan]))


def test_e5m2_is_top_byte_of_binary16():
    codes = np.arange(256, dtype=np.uint16)
    half = (codes << 8).astype(np.uint16).view(np.float16).astype(np.float64)
    ours = oracle.decode(codes.astype(np.uint8), E5M2)
    nan = np.isnan(half)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], half[~nan])


@pytest.mark.parametrize("fmt,n_finite,n_nan", [(E4M3, 254, 2), (E5M2, 248, 6)])
def test_code_space_structure(fmt, n_finite, n_nan):
    v = oracle.decode(np.arange(256, dtype=np.uint8), fmt)
    assert int(np.isnan(v).sum()) == n_nan
    assert int(np.isfinite(v).sum()) == n_finite
    if fmt == E4M3:
        assert not np.isinf(v).any()  # E4M3 has no infinities
    pos = v[:128]
    fin = pos[np.isfinite(pos)]
    assert np.all(np.diff(fin) > 0)  # positive codes are monotone in value
    assert np.array_equal(v[128:][np.isfinite(v[128:])], -fin)  # sign bit is a pure sign
    # homework 1 of "07 - The FP8 Family": max normal, min normal, min subnormal
    assert oracle.fmt_max(fmt) == (448.0 if fmt == E4M3 else 57344.0)
    assert fin[1] == (2.0 ** -9 if fmt == E4M3 else 2.0 ** -16)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encoders_agree_on_every_fp32(fmt):
    bad, first = oracle.encoders_disagree(0, 1 << 32, fmt)
    assert bad == 0, hex(first)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_decode_roundtrip_every_code(fmt):
    codes = np.arange(256, dtype=np.uint8)
    v = oracle.decode(codes, fmt)
    fin = np.isfinite(v)
    back = oracle.encode(v[fin].astype(np.float32), fmt)
    assert np.array_equal(back, codes[fin])


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_matches_torch_cast_on_every_inrange_bf16(fmt):
    bits = np.arange(1 << 16, dtype=np.uint32)
    x = (bits << 16).astype(np.uint32).view(np.float32)
    keep = np.isfinite(x) & (np.abs(x) <= oracle.fmt_max(fmt))
    x = x[keep]
    ours = oracle.encode(x, fmt)
    ref = torch.from_numpy(x.copy()).to(TORCH_DT[fmt]).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_matches_torch_cast_on_random_fp32(fmt):
    rng = np.random.default_rng(1234)
    m = oracle.fmt_max(fmt)
    x = np.concatenate([
        rng.uniform(-m, m, 200000),
        rng.standard_normal(200000) * 2.0 ** rng.integers(-24, 4, 200000),
    ]).astype(np.float32)
    ours = oracle.encode(x, fmt)
    ref = torch.from_numpy(x.copy()).to(TORCH_DT[fmt]).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("fmt,maxc", [(E4M3, 0x7E), (E5M2, 0x7B)])
def test_saturation_instead_of_overflow(fmt, maxc):
    # satfinite: anything beyond the largest finite value, inf included, clamps to it
    m = oracle.fmt_max(fmt)
    for x in [m * 1.0001, m * 1.5, 1e30, 3.0e38, float("inf")]:
        assert oracle.encode_nearest(x, fmt) == maxc
        assert oracle.encode_nearest(-x, fmt) == 0x80 | maxc
    assert oracle.is_nan_code(oracle.encode_nearest(float("nan"), fmt), fmt)


def test_ties_to_even_examples():
    # 2^-10 is half the smallest E4M3 subnormal: ties to the even code, i.e. zero
    assert oracle.encode_nearest(2.0 ** -10, E4M3) == 0x00
    assert oracle.encode_nearest(-(2.0 ** -10), E4M3) == 0x80
    # 3 * 2^-10 lies between codes 1 and 2: ties to the even code 2
    assert oracle.encode_nearest(3 * 2.0 ** -10, E4M3) == 0x02
    # 1 + 1/16 lies between 1 (M=0) and 1.125 (M=1): ties to M=0
    assert oracle.encode_nearest(1.0625, E4M3) == 0x38
    # 1 + 3/16 lies between M=1 and M=2: ties to M=2
    assert oracle.encode_nearest(1.1875, E4M3) == 0x3A
    # 464 is the midpoint of 448 and the missing 480: stays at 448
    assert oracle.encode_nearest(464.0, E4M3) == 0x7E
    # E5M2: 1 + 1/8 between 1 and 1.25 -> 1 ; 1 + 3/8 -> 1.5
    assert oracle.encode_nearest(1.125, E5M2) == 0x3C
    assert oracle.encode_nearest(1.375, E5M2) == 0x3E
    # values just off a midpoint go to the nearer neighbour
    assert oracle.encode_nearest(np.nextafter(np.float32(1.0625), np.float32(2)), E4M3) == 0x39
    # sign of zero is kept
    assert oracle.encode_nearest(-0.0, E4M3) == 0x80
    assert oracle.encode_nearest(-1e-30, E5M2) == 0x80


@pytest.mark.parametrize("fmt_name", ["E4M3", "E5M2"])
def test_unit_roundoff_printed_on_page(fmt_name):
    fmt = FMT[fmt_name]
    u = dict((r[0], float(r[1])) for r in _golden("unit_roundoff.txt"))[fmt_name]
    rng = np.random.default_rng(7)
    mn = 2.0 ** (-6 if fmt == E4M3 else -14)
    m = oracle.fmt_max(fmt)
    x = np.exp(rng.uniform(np.log(mn), np.log(m), 400000)).astype(np.float32)
    # include the exact midpoints just above powers of two, where the bound is attained
    e = np.arange(int(np.log2(mn)), int(np.log2(m)))
    x = np.concatenate([x, (2.0 ** e * (1 + u)).astype(np.float32)])
    xh = oracle.decode(oracle.encode(x, fmt), fmt)
    rel = np.abs(xh - x) / np.abs(xh)
    assert rel.max() == u


def test_encode_is_monotone():
    x = np.sort(np.random.default_rng(3).standard_normal(100000).astype(np.float32) * 100)
    for fmt in (E4M3, E5M2):
        v = oracle.decode(oracle.encode(x, fmt), fmt)
        assert np.all(np.diff(v) >= 0)


def test_bf16_conversions():
    bits = np.arange(1 << 16, dtype=np.uint16)
    f = oracle.bf16_to_f32(bits)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(f.view(np.uint32), t.view(np.uint32))
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(20000) * 10.0 ** rng.uniform(-30, 30, 20000)).astype(np.float32)
    ours = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)

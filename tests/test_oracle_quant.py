"""Pins of the oracle's quantizers, dequantizer and MX scale layout.

What fixes the expected values (not the oracle's own code):
  * closed forms of the scale rule s = amax/V_max, 1/s in fp32: the amax
    element of every group lands on +-V_max (code 0x7E/0xFE for E4M3,
    0x7B/0xFB for E5M2) -- fp32 rounding moves amax*(1/s) by at most 3 ulp
    around V_max, and V_max's neighbours are far;
  * groups built with a known power-of-two amax, so the expected scale, the
    expected MX exponent and the position of the max code are known in
    advance for each group (this pins the scale layouts);
  * s = 1 (static scaling) reduces the quantizer to the plain cast, compared
    with torch's float8 cast;
  * the error bound of round-to-nearest (unit roundoff printed on "FP8
    Mixed-Precision Serving in Production") for quantize -> dequantize;
  * the E4M3 underflow probe of the "FP8 Serving" guide, section 2;
  * the MX tiled layout: a bijection with the positions of the documented
    128x4 tile.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import BLOCK_128x128, E4M3, E5M2, MX32, SF_LINEAR, SF_TILED, TENSOR, TILE_1x128, TOKEN
from fp8_block_scaled_04_gb300 import synth

MAXC = {E4M3: 0x7E, E5M2: 0x7B}
VMAX = {E4M3: 448.0, E5M2: 57344.0}


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def _f32(b):
    return oracle.bf16_to_f32(b)


def _groups(rows, cols, gran):
    """Yield (row slice, col slice, scale index) for each group of a gran (not MX)."""
    if gran == TENSOR:
        yield slice(0, rows), slice(0, cols), 0
    elif gran == TOKEN:
        for r in range(rows):
            yield slice(r, r + 1), slice(0, cols), r
    elif gran == TILE_1x128:
        for kb in range(cols // 128):
            for r in range(rows):
                yield slice(r, r + 1), slice(kb * 128, kb * 128 + 128), kb * rows + r
    elif gran == BLOCK_128x128:
        nkb = cols // 128
        for rb in range((rows + 127) // 128):
            for kb in range(nkb):
                yield slice(rb * 128, min(rows, rb * 128 + 128)), slice(kb * 128, kb * 128 + 128), rb * nkb + kb


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("gran", [TENSOR, TOKEN, TILE_1x128, BLOCK_128x128])
def test_amax_element_hits_vmax(fmt, gran):
    x = synth.bf16_matrix(200, 384, 1.0, 11, 12, 0.02, 40.0)
    q, s = oracle.quantize(x, fmt, gran)
    xf = np.abs(_f32(x))
    for rs, cs, si in _groups(200, 384, gran):
        g = xf[rs, cs]
        amax = g.max()
        hit = q[rs, cs][g == amax] & 0x7F
        assert np.all(hit == MAXC[fmt])
        assert np.float32(amax) / np.float32(VMAX[fmt]) == s[si]
        # no element of the group exceeds V_max after scaling, none saturates but the max
        assert np.all((q[rs, cs][g < amax] & 0x7F) <= MAXC[fmt])


@pytest.mark.parametrize("gran", [TOKEN, TILE_1x128, BLOCK_128x128])
def test_scale_layout_with_known_group_amax(gran):
    rows, cols = 256, 512
    rng = np.random.default_rng(9)
    x = rng.uniform(-0.5, 0.5, (rows, cols)).astype(np.float32)
    expect = {}
    for rs, cs, si in _groups(rows, cols, gran):
        e = (si * 7) % 23 - 11  # distinct-ish power-of-two amax per group
        g = x[rs, cs] * 2.0 ** e
        r_rel = si % (rs.stop - rs.start)
        c_rel = (si * 13) % (cs.stop - cs.start)
        g[r_rel, c_rel] = 2.0 ** e  # the amax element, exactly 2^e
        x[rs, cs] = g
        expect[si] = (e, rs.start + r_rel, cs.start + c_rel)
    xb = _bf16(x)
    q, s = oracle.quantize(xb, E4M3, gran)
    for si, (e, r, c) in expect.items():
        # 2^e / 448 in fp32: 448 = 7 * 2^6, so the scale is 2^(e-6)/7 rounded once
        assert s[si] == np.float32(2.0 ** (e - 6) / 7.0)
        assert q[r, c] == 0x7E


def test_mx_exponent_and_layout_with_known_group_amax():
    rows, cols = 160, 384  # ragged in rows (160 = 128 + 32) and in 128-col blocks
    ng = cols // 32
    rng = np.random.default_rng(10)
    x = rng.uniform(-0.25, 0.25, (rows, cols)).astype(np.float32)
    js = {}
    for r in range(rows):
        for j in range(ng):
            e = (r * 3 + j * 5) % 30 - 15
            x[r, j * 32:(j + 1) * 32] *= 2.0 ** e
            x[r, j * 32 + (r + j) % 32] = 2.0 ** e
            js[(r, j)] = e
    xb = _bf16(x)
    ql, sl = oracle.quantize(xb, E4M3, MX32, SF_LINEAR)
    qt, st = oracle.quantize(xb, E4M3, MX32, SF_TILED)
    assert np.array_equal(ql, qt)
    assert st.size == ((rows + 127) // 128) * ((ng + 3) // 4) * 512
    for (r, j), e in js.items():
        # 2^e / 448 = 2^(e-8) / 1.75 -> ceil(log2) = e - 8; SF byte = 127 + e - 8
        b = 127 + e - 8
        assert sl[r * ng + j] == b
        assert st[((r // 128) * ((ng + 3) // 4) + j // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + j % 4] == b
        # the amax element becomes 2^e * 2^-(e-8) = 256 = code 0x78 (E=15, M=0)
        assert ql[r, j * 32 + (r + j) % 32] == 0x78


def test_mx_amax_lands_in_upper_half_of_range():
    x = synth.bf16_matrix(64, 1024, 1.0, 21, 22, 0.01, 80.0)
    for fmt in (E4M3, E5M2):
        q, sf = oracle.quantize(x, fmt, MX32)
        xf = np.abs(_f32(x)).reshape(64, 32, 32)
        dec = np.abs(oracle.decode(q, fmt)).reshape(64, 32, 32)
        amax_idx = xf.argmax(axis=2)
        top = np.take_along_axis(dec, amax_idx[..., None], axis=2)[..., 0]
        # before rounding amax * 2^-e lies in (V/2, V]; rounding to the format keeps it in [V/2, V]
        assert np.all(top >= VMAX[fmt] / 2) and np.all(top <= VMAX[fmt])
        assert np.any(top > VMAX[fmt] / 2)


def test_mx_exponent_closed_form():
    for j in range(-20, 21):
        assert oracle.mx_exponent(2.0 ** j, E4M3) == j - 8
        assert oracle.mx_exponent(448.0 * 2.0 ** j, E4M3) == j  # exact power-of-two ratio: no ceil step
        assert oracle.mx_exponent(448.0 * 2.0 ** j * 1.0000001, E4M3) == j + 1
    assert oracle.mx_exponent(0.0, E4M3) == -127
    assert oracle.mx_exponent(3.0e38, E4M3) == 120  # 3e38/448 ~ 2^119.3: ceil -> 120, no clamp needed
    assert oracle.mx_exponent(3.0e38, E5M2) == 113
    # bf16's smallest subnormal: ceil(log2(2^-133 / 448)) = -141 lies below UE8M0's range and clamps to -127
    assert oracle.mx_exponent(2.0 ** -133, E4M3) == -127
    assert oracle.mx_exponent(2.0 ** -110, E4M3) == -118  # fp32-normal ratio 2^-118.8 -> -118


def test_mx_tiled_layout_is_documented_bijection():
    rows, ng = 300, 13
    nrb, ncb = (rows + 127) // 128, (ng + 3) // 4
    size = oracle.mx_tiled_bytes(rows, ng)
    assert size == nrb * ncb * 512
    seen = np.zeros(size, dtype=np.int64)
    for r in range(nrb * 128):
        for j in range(ncb * 4):
            seen[oracle.mx_tiled_offset(r, j, rows, ng)] += 1
    assert np.all(seen == 1)
    # positions inside one 128x4 tile: 32 lines of 16 bytes, line = row % 32,
    # 4-byte word = (row / 32) % 4, byte = group % 4
    assert oracle.mx_tiled_offset(0, 0, rows, ng) == 0
    assert oracle.mx_tiled_offset(0, 3, rows, ng) == 3
    assert oracle.mx_tiled_offset(1, 0, rows, ng) == 16
    assert oracle.mx_tiled_offset(31, 0, rows, ng) == 496
    assert oracle.mx_tiled_offset(32, 0, rows, ng) == 4
    assert oracle.mx_tiled_offset(127, 3, rows, ng) == 31 * 16 + 3 * 4 + 3
    assert oracle.mx_tiled_offset(0, 4, rows, ng) == 512
    assert oracle.mx_tiled_offset(128, 0, rows, ng) == ncb * 512


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_static_unit_scale_is_plain_cast(fmt):
    x = synth.bf16_matrix(64, 256, 3.0, 31)
    q, s = oracle.quantize(x, fmt, TENSOR, static_scale=1.0)
    assert s[0] == 1.0
    ref = torch.from_numpy(_f32(x).copy()).to({E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}[fmt])
    assert np.array_equal(q, ref.view(torch.uint8).numpy())


def test_tensor_static_scale_used_verbatim():
    x = synth.bf16_matrix(32, 128, 1.0, 41)
    q, s = oracle.quantize(x, E4M3, TENSOR, static_scale=0.5)
    assert s[0] == 0.5
    ref = oracle.encode(_f32(x) * np.float32(2.0), E4M3)
    assert np.array_equal(q, ref)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("gran", [TENSOR, TOKEN, TILE_1x128, BLOCK_128x128, MX32])
def test_roundtrip_error_within_unit_roundoff(fmt, gran):
    x = synth.bf16_matrix(130, 640, 1.0, 51, 52, 0.01, 60.0)
    q, s = oracle.quantize(x, fmt, gran)
    xh = _f32(oracle.dequantize(q, s, fmt, gran)).astype(np.float64)
    xf = _f32(x).astype(np.float64)
    u = 2.0 ** -4 if fmt == E4M3 else 2.0 ** -3
    # per-element scale from the group max: values below the format's smallest
    # normal (after scaling) are held to the subnormal spacing instead
    if gran == MX32:
        sc = np.repeat(2.0 ** (s.reshape(130, -1).astype(np.float64) - 127), 32, axis=1)
    elif gran == TENSOR:
        sc = np.full(xf.shape, float(s[0]))
    elif gran == TOKEN:
        sc = np.repeat(s.astype(np.float64)[:, None], 640, axis=1)
    elif gran == TILE_1x128:
        sc = np.repeat(s.reshape(5, 130).T.astype(np.float64), 128, axis=1)
    else:
        blk = s.reshape(2, 5).astype(np.float64)
        sc = np.repeat(np.repeat(blk, 128, axis=0)[:130], 128, axis=1)
    sub = (2.0 ** -9 if fmt == E4M3 else 2.0 ** -16) * sc
    err = np.abs(xh - xf)
    bf16_half_ulp = np.abs(xh) * 2.0 ** -8  # the final bf16 rounding (8 significant bits)
    assert np.all(err <= u * np.abs(xf) + sub / 2 + bf16_half_ulp + 1e-45)


def test_quantize_is_monotone_within_group():
    x = synth.bf16_matrix(1, 4096, 1.0, 61)
    order = np.argsort(_f32(x)[0], kind="stable")
    for gran in (TENSOR, TOKEN):
        q, s = oracle.quantize(x, E4M3, gran)
        v = oracle.decode(q[0, order], E4M3)
        assert np.all(np.diff(v) >= 0)


def test_all_zero_group_gives_zero_codes_and_zero_scale():
    x = np.zeros((4, 256), dtype=np.uint16)
    x[1, :] = _bf16(np.linspace(-1, 1, 256))
    for gran in (TOKEN, TILE_1x128):
        q, s = oracle.quantize(x, E4M3, gran)
        assert np.all(q[0] == 0) and np.all(q[2:] == 0)
        assert s.reshape(-1)[0] == 0.0
    q, sf = oracle.quantize(x, E4M3, MX32)
    assert np.all(sf.reshape(4, 8)[0] == 0)  # e = -127 for an all-zero block


def _underflow_rows():
    rows = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", "underflow_probe.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                mag, sc, err, fl = line.split()
                rows[(float(mag), sc)] = (float(err), float(fl))
    return rows


def test_underflow_probe_from_guide():
    rows = _underflow_rows()
    rng = np.random.default_rng(77)
    for mag in (1.0, 3e-4):
        x = (rng.uniform(0.5, 1.5, 100000) * rng.choice([-1, 1], 100000) * mag).astype(np.float32)
        xb = _bf16(x)
        xf = _f32(xb).astype(np.float64)
        # scale off: plain cast
        q0, _ = oracle.quantize(xb.reshape(1, -1)[:, :99968], E4M3, TENSOR, static_scale=1.0)
        # scale on: per-tensor current scaling
        q1, s1 = oracle.quantize(xb.reshape(1, -1)[:, :99968], E4M3, TENSOR)
        xs = xf[:99968]
        for q, s, tag in ((q0, 1.0, "off"), (q1, float(s1[0]), "on")):
            xh = oracle.decode(q[0], E4M3) * s
            rel = np.mean(np.abs(xh - xs) / np.abs(xs)) * 100
            flushed = np.mean(xh == 0) * 100
            exp_err, exp_fl = rows[(mag, tag)]
            assert abs(flushed - exp_fl) < 0.5, (mag, tag, flushed)
            if exp_err >= 99:
                assert rel == pytest.approx(100.0)
            else:
                assert 1.5 <= rel <= 3.0, (mag, tag, rel)  # the page prints ~2.1-2.2%


# ------------------------------------------------------------ per-channel
def test_channel_is_token_of_transpose():
    """Per-channel scaling of X is per-token scaling of X^T (one scale per column)."""
    from oracle import CHANNEL

    x = synth.bf16_matrix(96, 272, 1.0, 71, 72, 0.02, 50.0)
    q, s = oracle.quantize(x, E4M3, CHANNEL)
    qt, st = oracle.quantize(np.ascontiguousarray(x.T), E4M3, TOKEN)
    assert np.array_equal(q, qt.T)
    assert np.array_equal(f32(s), f32(st))


def f32(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


def test_channel_amax_hits_vmax_per_column():
    from oracle import CHANNEL

    x = synth.bf16_matrix(130, 64, 1.0, 73, 74, 0.05, 80.0)
    for fmt in (E4M3, E5M2):
        q, s = oracle.quantize(x, fmt, CHANNEL)
        xf = np.abs(_f32(x))
        for k in range(64):
            col = xf[:, k]
            assert np.all((q[:, k][col == col.max()] & 0x7F) == MAXC[fmt])
            assert np.float32(col.max()) / np.float32(VMAX[fmt]) == s[k]


def test_channel_dequantize_roundtrip():
    from oracle import CHANNEL

    x = synth.bf16_matrix(40, 128, 1.0, 75)
    q, s = oracle.quantize(x, E4M3, CHANNEL)
    xh = _f32(oracle.dequantize(q, s, E4M3, CHANNEL)).astype(np.float64)
    xf = _f32(x).astype(np.float64)
    sc = np.repeat(s.astype(np.float64)[None, :], 40, axis=0)
    assert np.all(np.abs(xh - xf) <= 2.0 ** -4 * np.abs(xf) + 2.0 ** -10 * sc + 2.0 ** -8 * np.abs(xh) + 1e-45)


# ------------------------------------------------------------ delayed scaling
def test_delayed_with_own_amax_equals_current_scaling():
    x = synth.bf16_matrix(64, 512, 1.0, 81, 82, 0.01, 20.0)
    amax = float(np.abs(_f32(x)).max())
    for fmt in (E4M3, E5M2):
        qd, sd, nh = oracle.quantize_delayed(x, fmt, [amax, 0.0, 0.0], slot=1)
        qc, sc = oracle.quantize(x, fmt, TENSOR)
        assert np.array_equal(qd, qc) and sd[0] == sc[0]
        assert nh[1] == np.float32(amax) and nh[0] == np.float32(amax) and nh[2] == 0.0


def test_delayed_margin_is_power_of_two_on_scale():
    x = synth.bf16_matrix(32, 256, 1.0, 83)
    hist = np.array([3.5, 1.25, 7.0, 2.0], np.float32)
    q0, s0, _ = oracle.quantize_delayed(x, E4M3, hist, slot=0, margin=0)
    q2, s2, _ = oracle.quantize_delayed(x, E4M3, hist, slot=0, margin=2)
    assert s0[0] == np.float32(7.0) / np.float32(448.0)
    assert s2[0] == s0[0] * 4
    # the codes are those of static scaling with that scale
    qs, _ = oracle.quantize(x, E4M3, TENSOR, static_scale=float(s2[0]))
    assert np.array_equal(q2, qs)


def test_delayed_history_ring_and_saturation():
    hist = np.zeros(4, np.float32)
    xs = [synth.bf16_matrix(16, 128, sig, 90 + i) for i, sig in enumerate([1.0, 1.0, 8.0, 0.5])]
    for step, x in enumerate(xs):
        q, s, hist2 = oracle.quantize_delayed(x, E4M3, hist, slot=step % 4)
        amax = float(np.abs(_f32(x)).max())
        assert hist2[step % 4] == np.float32(amax)
        if step == 0:
            assert s[0] == 1.0  # empty history: identity scale
        if step == 2:
            # the history only knew the sigma-1 tensors: the sigma-8 outliers saturate at +-448
            dec = np.abs(oracle.decode(q, E4M3))
            assert np.any(dec == 448.0) and np.abs(_f32(x)).max() * (1 / s[0]) > 448.0
        hist = hist2
    assert np.array_equal(hist[:4] > 0, [True, True, True, True])


def test_delayed_nonfinite_history_uses_unit_scale():
    x = synth.bf16_matrix(8, 128, 1.0, 95)
    for bad in (np.inf, np.nan):
        q, s, _ = oracle.quantize_delayed(x, E4M3, [1.0, bad], slot=0)
        assert s[0] == 1.0
        qs, _ = oracle.quantize(x, E4M3, TENSOR, static_scale=1.0)
        assert np.array_equal(q, qs)


# ---------------------------------------------------------------- reading R2: x * fp32(1/s), not x / s
# The pages print the quantize step both as x / s ("07 -- The FP8 Family", Scaling
# is what makes FP8 usable; "FP8 Mixed-Precision Serving", per-tensor scaling
# formula) and as a multiply by the reciprocal ("Low precision: FP8, FP4, and
# microscaling", qdq_e4m3 listing). The two differ in fp32 for some (x, s): the
# product and the quotient can land on opposite sides of an FP8 rounding
# midpoint. The library takes the multiply. These witnesses are found from plain
# fp32 arithmetic (numpy) and encoded with torch's float8 cast (round to nearest
# even), so a divide anywhere in the oracle's encode step fails them.
_R2_AMAX = (6528.0, 816.0, 210.0, 3120.0, 4016.0, 1.3046875, 0.76171875, 334.0, 3760.0, 97.5)


def _r2_witnesses(fmt, amax, limit=6):
    """bf16 x < amax whose multiply and divide forms encode differently, with the multiply's code."""
    vmax = np.float32(VMAX[fmt])
    s = np.float32(np.float32(amax) / vmax)
    s_inv = np.float32(np.float32(1.0) / s)
    bits = (np.arange(1, 0x7F80, dtype=np.uint32) << 16).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[x < np.float32(amax)]
    dt = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}[fmt]

    def cast(v):
        return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(dt).view(torch.uint8).numpy()

    by_mul = cast((x * s_inv).astype(np.float32))
    by_div = cast((x / s).astype(np.float32))
    idx = np.nonzero(by_mul != by_div)[0][:limit]
    return x[idx], by_mul[idx], by_div[idx]


def test_r2_literal_witness_e4m3():
    # amax 816: s = fp32(816/448) = 1.8214285373687744, fp32(1/s) = 0.5490196347236633.
    # x = 0.037353515625 (bf16) times 1/s lies within an fp32 ulp of 0.0205078125, the
    # midpoint between E4M3 0x0a (0.01953125) and 0x0b (0.021484375): the fp32
    # product rounds above it (code 0x0b), the fp32 quotient x / s lands exactly on
    # it and ties to the even code 0x0a.
    s = np.float32(np.float32(816.0) / np.float32(448.0))
    s_inv = np.float32(np.float32(1.0) / s)
    x = np.float32(0.037353515625)
    assert np.float32(x * s_inv) > np.float32(0.0205078125) == np.float32(x / s)
    row = np.zeros((1, 128), dtype=np.float32)
    row[0, 0], row[0, 5] = 816.0, x
    q, sc = oracle.quantize(_bf16(row), E4M3, TOKEN)
    assert sc[0] == s
    assert q[0, 5] == 0x0B and q[0, 0] == 0x7E


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("gran", [TOKEN, TILE_1x128, TENSOR])
def test_r2_multiply_by_reciprocal_not_divide(fmt, gran):
    n_wit = 0
    for amax in _R2_AMAX:
        xs, mul, div = _r2_witnesses(fmt, amax)
        if xs.size == 0:
            continue
        n_wit += xs.size
        # one group (row / 1x128 tile / whole tensor) holding amax and the witnesses
        row = np.zeros((1, 128), dtype=np.float32)
        row[0, 0] = amax
        row[0, 3:3 + xs.size] = xs
        q, _ = oracle.quantize(_bf16(row), fmt, gran)
        assert np.array_equal(q[0, 3:3 + xs.size], mul), (amax, xs, mul, div)
        assert np.all(q[0, 3:3 + xs.size] != div)
    assert n_wit >= 10

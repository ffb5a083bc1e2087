"""Pins of the oracle's NVFP4 path ("Low precision: FP8, FP4, and microscaling",
NVFP4 paragraph: blocks of 16, an E4M3 microscale per block, one fp32 scale per
tensor keeping the microscales inside E4M3's range).

The page prints neither the FP4 element format nor the scale arithmetic; the
readings (E2M1 of the OCP Microscaling spec the page cites, and the scale steps
stated in oracle.c) are pinned here by what follows from them independently of
the oracle's code:
  * two encoders written differently (midpoint comparison, binade rounding)
    agree on every non-negative fp32 input;
  * the format's closed forms: 8 magnitudes, one fraction bit per binade,
    largest 6, smallest 0.5, unit roundoff 2^-2 attained at midpoints, ties
    to the even code, saturation;
  * the tensor-scale reading makes the tensor's amax element land on +-6 with
    microscale 448 (E4M3's largest value), the page's "keeps the microscales
    inside E4M3's range";
  * brute force: every code is the nearest E2M1 value of x / S (argmin over
    the 8 magnitudes, numpy), S the block's combined scale;
  * GEMM: exact small-value sums against an integer matmul (numpy), layouts.
"""
import numpy as np
import pytest

import oracle
from oracle import E4M3, SF_LINEAR, SF_TILED
from fp8_block_scaled_04_gb300 import synth

MAGS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def test_e2m1_code_space_closed_forms():
    v = oracle.e2m1_decode(np.arange(16))
    pos, neg = v[:8], v[8:]
    assert np.all(np.diff(pos) > 0)                       # monotone in the code
    assert np.array_equal(neg, -pos) and np.signbit(neg[0])  # the top bit is a pure sign
    assert pos[7] == 6.0 and pos[1] == 0.5                 # largest, smallest non-zero
    # one fraction bit: two values per binade [2^e, 2^(e+1)) for e = 0, 1, 2, spaced 2^(e-1)
    for e in range(3):
        b = pos[(pos >= 2.0 ** e) & (pos < 2.0 ** (e + 1))]
        assert len(b) == 2 and b[1] - b[0] == 2.0 ** (e - 1)
    assert np.array_equal(pos, MAGS)


def test_e2m1_encoders_agree_on_every_nonnegative_fp32():
    bad, first = oracle.e2m1_encoders_disagree(0, 1 << 31)
    assert bad == 0, hex(first)


def test_e2m1_encoders_agree_on_negative_sample():
    rng = np.random.default_rng(9)
    for u in rng.integers(1 << 31, 1 << 32, 20000, dtype=np.uint64):
        bad, first = oracle.e2m1_encoders_disagree(int(u), 1, 1)
        assert bad == 0, hex(first)


def test_e2m1_round_trip_ties_and_saturation():
    for c in range(16):
        if c == 8:  # -0 encodes back to -0
            assert oracle.e2m1_encode_nearest(-0.0) == 8
            continue
        assert oracle.e2m1_encode_nearest(float(oracle.e2m1_decode(c))) == c
    # exact midpoints go to the code whose mantissa bit is 0
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for x, want in ties.items():
        assert oracle.e2m1_decode(oracle.e2m1_encode_nearest(x)) == want, x
        assert oracle.e2m1_decode(oracle.e2m1_encode_nearest(-x)) == -want, x
    for x in [6.0001, 7.0, 1e6, 3e38, float("inf")]:
        assert oracle.e2m1_encode_nearest(x) == 7
        assert oracle.e2m1_encode_nearest(-x) == 15


def test_e2m1_unit_roundoff():
    # normals [1, 6]: |x_hat - x| / |x_hat| <= 2^-2, attained at the midpoints above 1, 2 and 4
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.uniform(1.0, 6.0, 100000), [1.25, 2.5, 5.0]]).astype(np.float32)
    xh = np.array([oracle.e2m1_decode(oracle.e2m1_encode_nearest(float(v))) for v in x])
    rel = np.abs(xh - x) / np.abs(xh)
    assert rel.max() <= 0.25 and np.isclose(rel.max(), 0.25)


def _combined_scales(sf, ts, rows, cols, layout):
    ng = cols // 16
    S = np.zeros((rows, ng))
    for r in range(rows):
        for g in range(ng):
            off = oracle.mx_tiled_offset(r, g, rows, ng) if layout == SF_TILED else r * ng + g
            S[r, g] = np.float32(oracle.decode(np.array([sf[off]], np.uint8), E4M3)[0]) * np.float32(ts)
    return S.astype(np.float32)


def test_amax_element_lands_on_six_with_microscale_448():
    x = synth.bf16_matrix(64, 256, 1.0, 31, 32, 0.02, 20.0)
    q, sf, ts = oracle.quantize_nvfp4(x, SF_LINEAR)
    xf = oracle.bf16_to_f32(x)
    amax = np.abs(xf).max()
    assert ts == np.float32(amax / np.float32(2688.0))
    r, c = np.unravel_index(np.argmax(np.abs(xf)), xf.shape)
    assert sf[r * 16 + c // 16] == 0x7E                       # E4M3 448
    code = (q[r, c // 2] >> (4 * (c % 2))) & 15
    assert oracle.e2m1_decode(code) == np.sign(xf[r, c]) * 6.0


def test_codes_are_the_nearest_value_of_x_over_S():
    x = synth.bf16_matrix(8, 64, 1.0, 41, 42, 0.05, 40.0)
    q, sf, ts = oracle.quantize_nvfp4(x, SF_LINEAR)
    xf = oracle.bf16_to_f32(x).astype(np.float32)
    S = _combined_scales(sf, ts, 8, 64, SF_LINEAR)
    for r in range(8):
        for k in range(64):
            s_inv = np.float32(1.0) / S[r, k // 16] if S[r, k // 16] != 0 else np.float32(0.0)
            t = np.float32(xf[r, k] * s_inv)
            d = np.abs(MAGS - abs(float(t)))
            best = np.flatnonzero(d == d.min())
            want = best[0] if len(best) == 1 else best[best % 2 == 0][0]  # tie: even code
            code = (q[r, k // 2] >> (4 * (k % 2))) & 15
            assert (code & 7) == want and (code >> 3) == (1 if np.signbit(t) else 0), (r, k)


def test_zero_blocks_and_zero_tensor():
    x = synth.bf16_matrix(4, 64, 1.0, 51)
    x[1, 16:32] = 0
    q, sf, ts = oracle.quantize_nvfp4(x, SF_LINEAR)
    assert sf[1 * 4 + 1] == 0 and np.all(q[1, 8:16] == 0)
    z = np.zeros((3, 32), np.uint16)
    qz, sfz, tsz = oracle.quantize_nvfp4(z, SF_LINEAR)
    assert tsz == 1.0 and not qz.any() and not sfz.any()


def test_static_tensor_scale_and_layouts_agree():
    x = synth.bf16_matrix(130, 128, 1.0, 61, 62, 0.01, 30.0)
    q1, sf1, ts1 = oracle.quantize_nvfp4(x, SF_LINEAR)
    q2, sf2, ts2 = oracle.quantize_nvfp4(x, SF_TILED)
    q3, sf3, ts3 = oracle.quantize_nvfp4(x, SF_LINEAR, static_tensor_scale=ts1)
    assert ts1 == ts2 == ts3 and np.array_equal(q1, q2) and np.array_equal(q1, q3) and np.array_equal(sf1, sf3)
    ng = 8
    for r in range(130):
        for g in range(ng):
            assert sf2[oracle.mx_tiled_offset(r, g, 130, ng)] == sf1[r * ng + g]


def test_dequantize_relative_error_bound():
    x = synth.bf16_matrix(32, 256, 1.0, 71)
    q, sf, ts = oracle.quantize_nvfp4(x, SF_TILED)
    xh = oracle.bf16_to_f32(oracle.dequantize_nvfp4(q, sf, ts, 256, SF_TILED)).astype(np.float64)
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    S = _combined_scales(sf, ts, 32, 256, SF_TILED).astype(np.float64)
    Sx = np.repeat(S, 16, axis=1)
    normal = np.abs(xf) >= Sx * (1 + 2 ** -20)
    # E2M1 unit roundoff 2^-2 on normals, plus the bf16 rounding of the result and the S_inv rounding
    assert np.all(np.abs(xh - xf)[normal] <= np.abs(xf)[normal] * (0.25 * (1 + 2 ** -7) + 2 ** -7))
    # the subnormal range: at most half the spacing 0.5 * S
    assert np.all(np.abs(xh - xf)[~normal] <= 0.25 * Sx[~normal] * (1 + 2 ** -6) + 1e-30)


def _pack(codes):
    c = np.asarray(codes, np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def test_gemm_small_values_exact():
    rng = np.random.default_rng(5)
    M, N, K = 24, 40, 256
    ca = rng.integers(0, 16, (M, K)).astype(np.uint8)
    cb = rng.integers(0, 16, (N, K)).astype(np.uint8)
    sfa = np.full(M * (K // 16), 0x38, np.uint8)  # E4M3 1.0
    sfb = np.full(N * (K // 16), 0x40, np.uint8)  # E4M3 2.0
    ref, bound = oracle.gemm_nvfp4(_pack(ca), sfa, 0.5, _pack(cb), sfb, 4.0, SF_LINEAR)
    va = oracle.e2m1_decode(ca) * 2   # integers (units of 0.5)
    vb = oracle.e2m1_decode(cb) * 2
    exact = (va.astype(np.int64) @ vb.astype(np.int64).T).astype(np.float64) * (0.25 * 1.0 * 2.0 * 0.5 * 4.0)
    assert np.array_equal(ref, exact)
    assert np.array_equal(bound, (np.abs(va).astype(np.int64) @ np.abs(vb).astype(np.int64).T) * 1.0)


def test_gemm_matches_numpy_matmul_of_dequantized_and_layouts():
    M, N, K = 40, 72, 320
    x = synth.bf16_matrix(M, K, 1.0, 81, 82, 0.02, 40.0)
    w = synth.bf16_matrix(N, K, 0.02, 83)
    qa, sfa, ta = oracle.quantize_nvfp4(x, SF_TILED)
    qb, sfb, tb = oracle.quantize_nvfp4(w, SF_TILED)
    ref, bound = oracle.gemm_nvfp4(qa, sfa, ta, qb, sfb, tb, SF_TILED)
    ca = np.stack([qa & 15, qa >> 4], axis=2).reshape(M, K)
    cb = np.stack([qb & 15, qb >> 4], axis=2).reshape(N, K)
    xh = oracle.e2m1_decode(ca) * np.repeat(_combined_scales(sfa, 1.0, M, K, SF_TILED).astype(np.float64), 16, axis=1) * ta
    wh = oracle.e2m1_decode(cb) * np.repeat(_combined_scales(sfb, 1.0, N, K, SF_TILED).astype(np.float64), 16, axis=1) * tb
    assert np.allclose(ref, xh @ wh.T, rtol=0, atol=1e-12 * bound.max())
    qa2, sfa2, _ = oracle.quantize_nvfp4(x, SF_LINEAR)
    qb2, sfb2, _ = oracle.quantize_nvfp4(w, SF_LINEAR)
    ref2, _ = oracle.gemm_nvfp4(qa2, sfa2, ta, qb2, sfb2, tb, SF_LINEAR)
    assert np.array_equal(ref, ref2)
    rows, cols = np.array([0, 17, 39]), np.array([71, 3, 40])
    part, _ = oracle.gemm_nvfp4(qa, sfa, ta, qb, sfb, tb, SF_TILED, rows=rows, cols=cols)
    assert np.array_equal(part, ref[np.ix_(rows, cols)])

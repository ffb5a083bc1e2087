"""Pins of the oracle's scaled GEMM (fp64 sum over dequantized operands).

Independent checks:
  * small-integer FP8 operands with power-of-two scales: the exact result is
    an integer matmul (numpy int64) times the scale product;
  * numpy's float64 matmul of operands dequantized by numpy from the decoded
    codes and per-group scale arrays expanded by hand;
  * one-hot weights reproduce the dequantized activations;
  * uniform block scales give the per-tensor result ("07 - The FP8 Family",
    "Scaling is what makes FP8 usable": the scales factor out of the sum);
  * the bound sum_k |x_hat w_hat| dominates |ref| and equals it for
    same-signed operands.
"""
import numpy as np
import pytest

import oracle
from oracle import BLOCK_128x128, E4M3, E5M2, MX32, SF_TILED, TENSOR, TILE_1x128, TOKEN
from fp8_block_scaled_04_gb300 import synth


def _int_codes(vals, fmt=E4M3):
    return oracle.encode(np.asarray(vals, dtype=np.float32), fmt)


def test_small_integer_operands_exact():
    rng = np.random.default_rng(0)
    M, N, K = 24, 40, 256
    xi = rng.integers(-8, 9, (M, K))
    wi = rng.integers(-8, 9, (N, K))
    a = _int_codes(xi)
    b = _int_codes(wi)
    sa = np.array([0.25], dtype=np.float32)
    sb = np.array([4.0], dtype=np.float32)
    ref, bound = oracle.gemm(a, sa, TENSOR, b, sb, TENSOR)
    exact = (xi @ wi.T).astype(np.float64) * 1.0
    assert np.array_equal(ref, exact)
    assert np.array_equal(bound, (np.abs(xi) @ np.abs(wi).T).astype(np.float64))


def _expand(scales, gran, rows, cols):
    s = np.asarray(scales)
    if gran == TENSOR:
        return np.full((rows, cols), float(s[0]))
    if gran == TOKEN:
        return np.repeat(s.astype(np.float64)[:, None], cols, axis=1)
    if gran == TILE_1x128:
        return np.repeat(s.reshape(cols // 128, rows).T.astype(np.float64), 128, axis=1)
    if gran == BLOCK_128x128:
        blk = s.reshape((rows + 127) // 128, cols // 128).astype(np.float64)
        return np.repeat(np.repeat(blk, 128, axis=0)[:rows], 128, axis=1)
    if gran == MX32:
        return np.repeat(2.0 ** (s.reshape(rows, cols // 32).astype(np.float64) - 127), 32, axis=1)
    raise ValueError(gran)


@pytest.mark.parametrize("ga,gb", [(TILE_1x128, BLOCK_128x128), (TENSOR, TENSOR), (TOKEN, TOKEN),
                                   (TOKEN, TENSOR), (TENSOR, TOKEN), (MX32, MX32)])
@pytest.mark.parametrize("fa,fb", [(E4M3, E4M3), (E5M2, E4M3)])
def test_matches_numpy_matmul_of_dequantized(ga, gb, fa, fb):
    M, N, K = 70, 200, 384
    x = synth.bf16_matrix(M, K, 1.0, 100, 101, 0.02, 50.0)
    w = synth.bf16_matrix(N, K, 0.02, 102)
    a, sa = oracle.quantize(x, fa, ga)
    b, sb = oracle.quantize(w, fb, gb)
    ref, bound = oracle.gemm(a, sa, ga, b, sb, gb, fa, fb)
    xh = oracle.decode(a, fa) * _expand(sa, ga, M, K)
    wh = oracle.decode(b, fb) * _expand(sb, gb, N, K)
    np_ref = xh @ wh.T
    np_bound = np.abs(xh) @ np.abs(wh).T
    assert np.allclose(ref, np_ref, rtol=0, atol=1e-12 * np_bound.max())
    assert np.allclose(bound, np_bound, rtol=1e-12)


def test_row_and_col_selection():
    M, N, K = 50, 90, 256
    x = synth.bf16_matrix(M, K, 1.0, 110)
    w = synth.bf16_matrix(N, K, 0.02, 111)
    a, sa = oracle.quantize(x, E4M3, TILE_1x128)
    b, sb = oracle.quantize(w, E4M3, BLOCK_128x128)
    full, fb = oracle.gemm(a, sa, TILE_1x128, b, sb, BLOCK_128x128)
    rows = np.array([0, 7, 49])
    cols = np.array([3, 89, 0, 64])
    part, pb = oracle.gemm(a, sa, TILE_1x128, b, sb, BLOCK_128x128, rows=rows, cols=cols)
    assert np.array_equal(part, full[np.ix_(rows, cols)])
    assert np.array_equal(pb, fb[np.ix_(rows, cols)])


def test_one_hot_weights_reproduce_dequantized_activations():
    M, K = 33, 256
    N = K
    x = synth.bf16_matrix(M, K, 1.0, 120)
    a, sa = oracle.quantize(x, E4M3, TILE_1x128)
    b = np.zeros((N, K), dtype=np.uint8)
    b[np.arange(N), np.arange(K)] = 0x38  # E4M3 1.0
    sb = np.ones(((N + 127) // 128) * (K // 128), dtype=np.float32)
    ref, _ = oracle.gemm(a, sa, TILE_1x128, b, sb, BLOCK_128x128)
    xh = oracle.bf16_to_f32(oracle.dequantize(a, sa, E4M3, TILE_1x128)).astype(np.float64)
    # ref holds the exact products; dequantize rounds q*s to fp32, then to bf16
    # (8 significant bits: at most 2^-8 + 2^-24 relative)
    assert np.all(np.abs(ref - xh) <= np.abs(ref) * (2.0 ** -8 + 2.0 ** -23))
    assert np.mean(np.abs(ref - xh) == 0) > 0.1


def test_uniform_block_scales_equal_per_tensor():
    M, N, K = 40, 130, 512
    rng = np.random.default_rng(3)
    a = rng.integers(0, 256, (M, K), dtype=np.uint8)
    b = rng.integers(0, 256, (N, K), dtype=np.uint8)
    a[(a & 0x7F) == 0x7F] = 0
    b[(b & 0x7F) == 0x7F] = 0
    s1 = np.float32(0.0123)
    s2 = np.float32(3.5)
    ra, _ = oracle.gemm(a, np.full((K // 128) * M, s1, np.float32), TILE_1x128,
                        b, np.full(((N + 127) // 128) * (K // 128), s2, np.float32), BLOCK_128x128)
    rt, _ = oracle.gemm(a, np.array([s1]), TENSOR, b, np.array([s2]), TENSOR)
    assert np.array_equal(ra, rt)


def test_bound_dominates_and_is_tight_for_same_sign():
    M, N, K = 16, 32, 128
    rng = np.random.default_rng(4)
    a = rng.integers(0x08, 0x70, (M, K), dtype=np.uint8)  # positive normals
    b = rng.integers(0x08, 0x70, (N, K), dtype=np.uint8)
    ref, bound = oracle.gemm(a, np.array([1.5], np.float32), TENSOR, b, np.array([0.5], np.float32), TENSOR)
    assert np.array_equal(ref, bound)
    b2 = b | 0x80
    b2[:, ::2] = b[:, ::2]
    ref2, bound2 = oracle.gemm(a, np.array([1.5], np.float32), TENSOR, b2, np.array([0.5], np.float32), TENSOR)
    assert np.all(np.abs(ref2) <= bound2) and np.array_equal(bound2, bound)


def test_mx_tiled_and_linear_scale_layouts_agree():
    M, N, K = 130, 64, 256
    x = synth.bf16_matrix(M, K, 1.0, 130)
    w = synth.bf16_matrix(N, K, 1.0, 131)
    a, sal = oracle.quantize(x, E4M3, MX32)
    _, sat = oracle.quantize(x, E4M3, MX32, SF_TILED)
    b, sbl = oracle.quantize(w, E4M3, MX32)
    _, sbt = oracle.quantize(w, E4M3, MX32, SF_TILED)
    r1, _ = oracle.gemm(a, sal, MX32, b, sbl, MX32)
    r2, _ = oracle.gemm(a, sat, MX32, b, sbt, MX32, a_sf=SF_TILED, b_sf=SF_TILED)
    assert np.array_equal(r1, r2)


def _half_ulp_bf16(v):
    _, ex = np.frexp(np.abs(v))
    return np.ldexp(1.0, ex - 9)


def test_bf16_of_reference_meets_tolerance_on_random_data():
    # without outliers the output rounding alone fits |out - ref| <= 1e-3 * bound + 1e-6
    x, w = synth.tiny()
    a, sa = oracle.quantize(x, E4M3, TILE_1x128)
    b, sb = oracle.quantize(w, E4M3, BLOCK_128x128)
    ref, bound = oracle.gemm(a, sa, TILE_1x128, b, sb, BLOCK_128x128)
    out = oracle.bf16_to_f32(oracle.f32_to_bf16(ref.astype(np.float32))).astype(np.float64)
    assert np.all(np.abs(out - ref) <= 1e-3 * bound + 1e-6)


def test_bf16_output_rounding_needs_half_ulp_term_with_outliers():
    # With outlier channels one product dominates some sums (|ref| ~ bound), and the
    # rounding of the exact result to bf16 (8 significant bits) exceeds 1e-3 * bound:
    # the GEMM parity rule therefore adds half a bf16 ulp of the output.
    M, N, K = 128, 512, 256
    x = synth.bf16_matrix(M, K, 1.0, 138, 276, 0.01, 50.0)
    w = synth.bf16_matrix(N, K, 0.02, 4126)
    a, sa = oracle.quantize(x, E4M3, TILE_1x128)
    b, sb = oracle.quantize(w, E4M3, BLOCK_128x128)
    ref, bound = oracle.gemm(a, sa, TILE_1x128, b, sb, BLOCK_128x128)
    out = oracle.bf16_to_f32(oracle.f32_to_bf16(ref.astype(np.float32))).astype(np.float64)
    err = np.abs(out - ref)
    assert np.any(err > 1e-3 * bound + 1e-6)
    assert np.all(err <= 1e-3 * bound + 1e-6 + _half_ulp_bf16(ref))
    assert np.all(err <= _half_ulp_bf16(ref))

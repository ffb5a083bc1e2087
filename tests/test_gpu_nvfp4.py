"""GPU parity of the NVFP4 path ("Low precision: FP8, FP4, and microscaling",
NVFP4 paragraph) against the CPU oracle.

Quantizer, dequantizer and the element conversion: bit-exact (codes, E4M3
block scales, tensor scale, bf16 output). GEMM: |gpu - ref| <= 1e-3 * bound +
half a bf16 ulp of ref (the same rule as the FP8 GEMMs), and exact for small
values with power-of-two scales.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_04_gb300 import binding as fb
from fp8_block_scaled_04_gb300 import synth
from gpu_util import out_f64, to_dev_bf16, within_tolerance

pytestmark = pytest.mark.gpu


def test_e2m1_encode_every_fp32():
    """The quantizer's element step against the oracle encoder on all 2^32 fp32 patterns."""
    chunk = 1 << 28
    for start in range(0, 1 << 32, chunk):
        bits = torch.arange(start, start + chunk, dtype=torch.int64, device="cuda").to(torch.int32)
        codes = fb.debug_encode_e2m1_f32(bits.view(torch.float32))
        bad, first = oracle.e2m1_check_codes(start, codes.cpu().numpy())
        assert bad == 0, "first mismatch at fp32 pattern 0x%08x" % first


def _quant_dev(x, layout, static=None):
    q, sf, ts = fb.quantize_nvfp4(to_dev_bf16(x), layout,
                                  None if static is None else torch.tensor([static], dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    return q.cpu().numpy(), sf.cpu().numpy(), float(ts.item())


@pytest.mark.parametrize("layout", [fb.SF_LINEAR, fb.SF_TCGEN05])
@pytest.mark.parametrize("shape", [(1, 16), (7, 48), (130, 272), (257, 1024), (300, 4096), (2048, 7168)])
def test_quantize_bit_exact(shape, layout):
    rows, cols = shape
    x = synth.bf16_matrix(rows, cols, 1.0, 900 + rows, 901 + cols, 0.01, 40.0)
    q, sf, ts = _quant_dev(x, layout)
    qo, sfo, tso = oracle.quantize_nvfp4(x, layout)
    assert np.float32(ts) == np.float32(tso)
    assert np.array_equal(q, qo)
    assert np.array_equal(sf[: sfo.size], sfo)


def test_quantize_static_scale_and_extremes():
    rows, cols = 64, 512
    x = synth.bf16_matrix(rows, cols, 1.0, 911, 912, 0.02, 50.0)
    x[3, :] = 0                        # all-zero blocks
    x[5, 16:32] = 0x0001               # smallest bf16 subnormals
    x[6, 32:48] = 0x7F7F               # largest finite bf16
    x[7, 0:16] = 0x8000                # negative zeros
    for static in [None, 0.01, 3.0e-3]:
        q, sf, ts = _quant_dev(x, fb.SF_TCGEN05, static)
        qo, sfo, tso = oracle.quantize_nvfp4(x, fb.SF_TCGEN05, static)
        assert np.float32(ts) == np.float32(tso)
        assert np.array_equal(q, qo), static
        assert np.array_equal(sf, sfo), static


def test_quantize_tiny_static_tensor_scales_subnormal_blocks():
    """Static tensor scales down to fp32 subnormals with bf16 block maxima around
    6 * 2^-126, where fp32(amax_b / 6) is subnormal: bit-exact against the oracle's
    two divisions. Rows 0-1 hold the blocks whose fast-step code would differ
    (maxima 5 and 20 units of 2^-133 under s_t = fp32 bits 0x000A28A2)."""
    rows, cols = 128, 256
    bits = synth.bf16_matrix(rows, cols, 1.0, 931)
    rng = np.random.default_rng(932)
    small = np.arange(1, 0x0580, dtype=np.uint16)  # bf16 magnitudes up to ~64 * 2^-126, subnormals included
    x = rng.choice(small, size=(rows, cols)).astype(np.uint16) | (rng.integers(0, 2, (rows, cols)) << 15).astype(np.uint16)
    x[0, :16] = 0
    x[0, 3] = 5
    x[1, :16] = 0
    x[1, 7] = 20
    x[64:, :] = bits[64:, :] & 0x807F  # tiny normals / subnormals of mixed signs
    s_wit = float(np.array([0x000A28A2], dtype=np.uint32).view(np.float32)[0])
    for static in [s_wit, 5e-40, 1.335e-38, 2.0e-38, 4.7e-37]:
        for layout in (fb.SF_LINEAR, fb.SF_TCGEN05):
            q, sf, ts = _quant_dev(x, layout, static)
            qo, sfo, tso = oracle.quantize_nvfp4(x, layout, static)
            assert np.float32(ts) == np.float32(tso)
            assert np.array_equal(sf[: sfo.size], sfo), (static, layout)
            assert np.array_equal(q, qo), (static, layout)


def _e4m3_midpoint_blocks():
    """bf16 rows of 16-element blocks whose amax is 3 (v_i + v_i+1) for consecutive
    E4M3 values v_i < v_i+1 (exact in bf16): with s_t = 1 the block scale
    amax / 6 / s_t is exactly their midpoint, a rounding tie."""
    vals = sorted({float(v) for v in oracle.decode(np.arange(0x00, 0x7f, dtype=np.uint8), oracle.E4M3)})
    amax = np.array([3.0 * (a + b) for a, b in zip(vals[:-1], vals[1:])], dtype=np.float32)
    x = np.zeros((len(amax), 16), dtype=np.float32)
    x[:, 5] = amax
    x[:, 9] = -0.5 * amax
    bits = oracle.f32_to_bf16(x)
    assert np.array_equal(oracle.bf16_to_f32(bits), x)  # exactly representable
    return bits.reshape(-1, 64) if len(amax) % 4 == 0 else bits[: len(amax) // 4 * 4].reshape(-1, 64)


@pytest.mark.parametrize("k", list(range(-12, 13)))
def test_quantize_block_scales_near_e4m3_midpoints(k):
    """Static tensor scales 1 +- k units in the last place move every block scale a
    few fp32 units off an E4M3 rounding midpoint: the band where the encoder's
    multiply-by-reciprocal step must hand over to the exact divisions."""
    x = _e4m3_midpoint_blocks()
    s_t = float(np.float32(1.0 + k * 2.0 ** -23) if k >= 0 else np.float32(1.0 + k * 2.0 ** -24))
    q, sf, ts = _quant_dev(x, fb.SF_LINEAR, s_t)
    qo, sfo, tso = oracle.quantize_nvfp4(x, fb.SF_LINEAR, s_t)
    assert np.float32(ts) == np.float32(tso)
    assert np.array_equal(sf, sfo), k
    assert np.array_equal(q, qo), k


@pytest.mark.parametrize("layout", [fb.SF_LINEAR, fb.SF_TCGEN05])
def test_dequantize_bit_exact(layout):
    rows, cols = 130, 1024
    x = synth.bf16_matrix(rows, cols, 1.0, 921, 922, 0.01, 40.0)
    qo, sfo, tso = oracle.quantize_nvfp4(x, layout)
    out = fb.dequantize_nvfp4(torch.from_numpy(qo).cuda(), torch.from_numpy(sfo).cuda(),
                              torch.tensor([tso], dtype=torch.float32, device="cuda"), cols, layout)
    torch.cuda.synchronize()
    ref = oracle.dequantize_nvfp4(qo, sfo, tso, cols, layout)
    assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), ref)


def _gemm_dev(qa, sfa, ta, qb, sfb, tb):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    f = lambda v: torch.tensor([v], dtype=torch.float32, device="cuda")
    out = fb.gemm_nvfp4(torch.from_numpy(qa).cuda(), torch.from_numpy(sfa).cuda(), f(ta),
                        torch.from_numpy(qb).cuda(), torch.from_numpy(sfb).cuda(), f(tb), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (130, 272, 512), (1, 16, 256), (300, 640, 1024),
                                   (257, 512, 2048)])
def test_gemm_parity(M, N, K):
    x = synth.bf16_matrix(M, K, 1.0, 930 + M, 931 + K, 0.01, 40.0)
    w = synth.bf16_matrix(N, K, 1.0, 932 + N, 933 + K, 0.01, 40.0)
    qa, sfa, ta = oracle.quantize_nvfp4(x, oracle.SF_TILED)
    qb, sfb, tb = oracle.quantize_nvfp4(w, oracle.SF_TILED)
    out = _gemm_dev(qa, sfa, ta, qb, sfb, tb)
    ref, bound = oracle.gemm_nvfp4(qa, sfa, ta, qb, sfb, tb, oracle.SF_TILED)
    tol = within_tolerance(out_f64(out), ref, bound)
    assert tol.bad == 0, tol


def test_gemm_small_values_exact():
    """E2M1 codes with power-of-two microscales and tensor scales, K <= 512: fp32 sums are exact."""
    rng = np.random.default_rng(17)
    M, N, K = 130, 272, 512

    def operand(rows):
        c = rng.integers(0, 16, (rows, K)).astype(np.uint8)
        q = (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
        sf = np.zeros(oracle.mx_tiled_bytes(rows, K // 16), np.uint8)
        for r in range(rows):
            for g in range(K // 16):
                sf[oracle.mx_tiled_offset(r, g, rows, K // 16)] = [0x30, 0x38, 0x40][(r + g) % 3]  # 0.5, 1, 2
        return q, sf

    qa, sfa = operand(M)
    qb, sfb = operand(N)
    out = _gemm_dev(qa, sfa, 0.5, qb, sfb, 2.0)
    ref, _ = oracle.gemm_nvfp4(qa, sfa, 0.5, qb, sfb, 2.0, oracle.SF_TILED)
    expect = oracle.bf16_to_f32(oracle.f32_to_bf16(ref.astype(np.float32))).astype(np.float64)
    assert np.array_equal(out_f64(out), expect)


def test_gemm_quantized_by_the_gpu_prefill_shape_sampled():
    """GPU quantizer feeding the GPU GEMM at 4096 x 14336 x 4096, sampled rows against the oracle."""
    M, N, K = 4096, 14336, 4096
    x = synth.bf16_matrix(M, K, 1.0, 940, 941, 0.01, 30.0)
    w = synth.bf16_matrix(N, K, 0.02, 942)
    qa, sfa, ta = fb.quantize_nvfp4(to_dev_bf16(x))
    qb, sfb, tb = fb.quantize_nvfp4(to_dev_bf16(w))
    out = fb.gemm_nvfp4(qa, sfa, ta, qb, sfb, tb)
    torch.cuda.synchronize()
    qa_h, sfa_h, ta_h = qa.cpu().numpy(), sfa.cpu().numpy(), float(ta.item())
    qb_h, sfb_h, tb_h = qb.cpu().numpy(), sfb.cpu().numpy(), float(tb.item())
    rows = np.unique(np.concatenate([np.arange(0, M, 509), [M - 1]]))
    ref, bound = oracle.gemm_nvfp4(qa_h, sfa_h, ta_h, qb_h, sfb_h, tb_h, oracle.SF_TILED, rows=rows)
    tol = within_tolerance(out_f64(out)[rows], ref, bound)
    assert tol.bad == 0, tol

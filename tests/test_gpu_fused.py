"""GEMM with quantization fused into its epilogue ("Low precision: FP8, FP4, and
microscaling", practice 4), against the oracle.

The fused kernel rounds its fp32 result to bf16 (the value the unfused GEMM
stores), then quantizes each 128-column group of the row. So the oracle decides
the fused output exactly: take the unfused GEMM's bf16 output (itself checked
against the oracle's fp64 GEMM within the parity tolerance), quantize it with
the oracle at 1x128, and the fused codes and scales must equal that bit for bit.
A second check dequantizes the fused output and bounds it against the fp64 sum.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_04_gb300 import binding as fb
from fp8_block_scaled_04_gb300 import synth
from gpu_util import bf16_host, f32_bits, half_ulp_bf16, out_f64, to_dev_bf16, within_tolerance

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed):
    x = synth.bf16_matrix(M, K, 1.0, seed, seed + 1, 0.01, 40.0)
    w = synth.bf16_matrix(N, K, 0.02, seed + 2)
    qa, sa = oracle.quantize(x, fb.E4M3, fb.TILE_1x128)
    qb, sb = oracle.quantize(w, fb.E4M3, fb.BLOCK_128x128)
    return qa, sa, qb, sb


def _fused_vs_oracle(qa_d, sa_d, qb_d, sb_d, M, N, out_fmt, ref_rows=None, ref=None, bound=None):
    """Fused codes/scales == oracle 1x128 quantize of the unfused GEMM's bf16 output.

    M > 64 throughout: the unfused GEMM then runs the same fold kernel as the fused
    one (with few rows it swaps operands onto another kernel, whose bf16 output may
    round differently within the tolerance)."""
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qf, sf = fb.gemm_blockscaled_quantized_out(qa_d, sa_d, qb_d, sb_d, out_fmt=out_fmt, status=status)
    out = fb.gemm_blockscaled(qa_d, sa_d, fb.TILE_1x128, qb_d, sb_d, fb.BLOCK_128x128, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    if ref is not None:  # the bf16 output the oracle quantizes is itself within tolerance of the fp64 GEMM
        got = out_f64(out if ref_rows is None else out[torch.from_numpy(ref_rows).cuda()])
        tol = within_tolerance(got, ref, bound)
        assert tol.bad == 0, tol
    oq, os_ = oracle.quantize(bf16_host(out), out_fmt, fb.TILE_1x128)
    q_host = qf.cpu().numpy()
    s_host = sf.cpu().numpy().reshape(N // 128, M)
    assert np.array_equal(q_host, oq), int((q_host != oq).sum())
    assert np.array_equal(f32_bits(s_host), f32_bits(os_.reshape(N // 128, M)))


@pytest.mark.parametrize("M,N,K", [(130, 256, 512), (300, 1024, 1152), (1024, 2048, 1024), (2048, 4096, 512),
                                   (65, 128, 256), (257, 384, 640)])
@pytest.mark.parametrize("out_fmt", [fb.E4M3, fb.E5M2])
def test_fused_equals_oracle_quantize_of_gemm_output(M, N, K, out_fmt):
    qa, sa, qb, sb = _operands(M, N, K, 7 + M)
    ref, bound = oracle.gemm(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128)
    a, sad, b, sbd = (torch.from_numpy(t).cuda() for t in (qa, sa, qb, sb))
    _fused_vs_oracle(a, sad, b, sbd, M, N, out_fmt, ref=ref, bound=bound)


@pytest.mark.parametrize("out_fmt", [fb.E4M3, fb.E5M2])
def test_fused_full_prefill_shape(out_fmt):
    """4096 x 14336 x 4096 (the prefill workload), operands quantized on the GPU and
    checked bit-exact first; every fused code and scale against the oracle."""
    M, N, K = 4096, 14336, 4096
    x = synth.prefill_x(M, K)
    w = synth.prefill_w(N, K)
    qa_d, sa_d = fb.quantize(to_dev_bf16(x), fb.E4M3, fb.TILE_1x128)
    qb_d, sb_d = fb.quantize(to_dev_bf16(w), fb.E4M3, fb.BLOCK_128x128)
    qa, sa = oracle.quantize(x, fb.E4M3, fb.TILE_1x128)
    qb, sb = oracle.quantize(w, fb.E4M3, fb.BLOCK_128x128)
    torch.cuda.synchronize()
    assert np.array_equal(qa_d.cpu().numpy(), qa) and np.array_equal(qb_d.cpu().numpy(), qb)
    rows = np.unique(np.concatenate([np.arange(0, M, 61), [M - 1]]))
    ref, bound = oracle.gemm(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128, rows=rows)
    _fused_vs_oracle(qa_d, sa_d, qb_d, sb_d, M, N, out_fmt, ref_rows=rows, ref=ref, bound=bound)


@pytest.mark.parametrize("M,N,K", [(16, 512, 256), (130, 384, 640), (512, 1536, 1024)])
def test_fused_against_oracle(M, N, K):
    qa, sa, qb, sb = _operands(M, N, K, 31 + N)
    a, sad, b, sbd = (torch.from_numpy(t).cuda() for t in (qa, sa, qb, sb))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qf, sf = fb.gemm_blockscaled_quantized_out(a, sad, b, sbd, status=status)
    deq = fb.dequantize(qf, sf, fb.E4M3, fb.TILE_1x128)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, bound = oracle.gemm(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128)
    got = out_f64(deq)
    s_el = np.repeat(sf.cpu().numpy().reshape(N // 128, M).T.astype(np.float64), 128, axis=1)
    y = np.abs(ref) + 1e-3 * bound + 1e-6 + half_ulp_bf16(ref)  # bound on |bf16 GEMM output|
    allowed = (1e-3 * bound + 1e-6 + half_ulp_bf16(ref)  # the GEMM and its bf16 output
               + 2.0 ** -4 * y + 2.0 ** -10 * s_el  # E4M3 rounding of the scaled value
               + 2.0 ** -8 * (y * (1 + 2.0 ** -4)))  # bf16 rounding of the dequantized value
    assert np.all(np.abs(got - ref) <= allowed)
    # scales follow the 1x128 rule on the output: the largest |value| of each group maps to 448
    dec = np.abs(oracle.decode(qf.cpu().numpy(), fb.E4M3)).reshape(M, N // 128, 128)
    assert np.all(dec.max(axis=2)[s_el[:, ::128] > 0] == 448.0)


def test_fused_refuses_ragged_n():
    a = torch.zeros((16, 128), dtype=torch.uint8, device="cuda")
    b = torch.zeros((144, 128), dtype=torch.uint8, device="cuda")
    s = torch.ones(1024, dtype=torch.float32, device="cuda")
    with pytest.raises(fb.Fp8Error) as e:
        fb.gemm_blockscaled_quantized_out(a, s, b, s, q_scales=s)
    assert e.value.code == fb.ERR_UNSUPPORTED_SHAPE

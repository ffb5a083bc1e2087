"""GEMM with quantization fused into its epilogue ("Low precision: FP8, FP4, and
microscaling", practice 4), against the oracle and against the unfused path.

1. The fused output is the unfused bf16 GEMM output quantized at 1x128: the two
   GPU paths are compared bit for bit (each is checked against the oracle
   elsewhere: the GEMM within tolerance, the quantizer bit-exact).
2. Against the oracle: the dequantized fused output stays within the GEMM
   tolerance plus the rounding the two quantization steps add (unit roundoff of
   the FP8 format, half a subnormal step, the final bf16 rounding).
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_04_gb300 import binding as fb
from fp8_block_scaled_04_gb300 import synth
from gpu_util import bf16_host, half_ulp_bf16, out_f64

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed):
    x = synth.bf16_matrix(M, K, 1.0, seed, seed + 1, 0.01, 40.0)
    w = synth.bf16_matrix(N, K, 0.02, seed + 2)
    qa, sa = oracle.quantize(x, fb.E4M3, fb.TILE_1x128)
    qb, sb = oracle.quantize(w, fb.E4M3, fb.BLOCK_128x128)
    return qa, sa, qb, sb


@pytest.mark.parametrize("M,N,K", [(130, 256, 512), (300, 1024, 1152), (1024, 2048, 1024), (2048, 4096, 512)])
@pytest.mark.parametrize("out_fmt", [fb.E4M3, fb.E5M2])
def test_fused_equals_unfused_gpu_path(M, N, K, out_fmt):
    qa, sa, qb, sb = _operands(M, N, K, 7 + M)
    a, sad, b, sbd = (torch.from_numpy(t).cuda() for t in (qa, sa, qb, sb))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qf, sf = fb.gemm_blockscaled_quantized_out(a, sad, b, sbd, out_fmt=out_fmt, status=status)
    out = fb.gemm_blockscaled(a, sad, fb.TILE_1x128, b, sbd, fb.BLOCK_128x128, status=status)
    qu, su = fb.quantize(out, out_fmt, fb.TILE_1x128)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(qf, qu)
    assert torch.equal(sf.view(torch.int32), su.view(torch.int32))


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

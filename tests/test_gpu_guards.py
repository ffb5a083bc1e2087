"""Guard bands around every output buffer (the stand-in for a memory checker,
which this GPU pool does not offer): each output gets 4 KB of a known byte on
both sides, and after the call the bands must be untouched and the outputs must
still match the oracle. The cases are the ones where a stray store is most
likely: ragged M and N (the GEMMs' TMA stores are clipped by their tensor maps),
row and column tails of the quantizers, the padded 128x4 scale atoms of MX and
NVFP4, the split-K decode kernel's cluster reduction, the fused quantized
epilogue and the dequantizers."""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_04_gb300 import binding as fb
from fp8_block_scaled_04_gb300 import synth
from gpu_util import Guarded, f32_bits, out_f64, to_dev_bf16, within_tolerance, x4_layout

pytestmark = pytest.mark.gpu

QSHAPES = [(1, 128), (7, 384), (130, 640), (257, 1152)]
GRANS = [(fb.TENSOR, fb.SF_LINEAR), (fb.TOKEN, fb.SF_LINEAR), (fb.TILE_1x128, fb.SF_LINEAR),
         (fb.BLOCK_128x128, fb.SF_LINEAR), (fb.MX32, fb.SF_LINEAR), (fb.MX32, fb.SF_TCGEN05),
         (fb.CHANNEL, fb.SF_LINEAR)]


@pytest.mark.parametrize("shape", QSHAPES)
@pytest.mark.parametrize("gran,lay", GRANS)
def test_quantize_and_dequantize_stay_in_bounds(shape, gran, lay):
    rows, cols = shape
    x = synth.bf16_matrix(rows, cols, 1.0, 1200 + rows, 1201 + cols, 0.02, 40.0)
    xd = to_dev_bf16(x)
    nb = fb.scales_bytes(rows, cols, gran, lay)
    q = Guarded((rows, cols), torch.uint8)
    sc = Guarded((nb,), torch.uint8)
    scv = sc.t if gran == fb.MX32 else sc.t.view(torch.float32)
    fb.quantize(xd, fb.E4M3, gran, lay, q=q.t, scales=scv)
    assert q.intact() and sc.intact()
    oq, os_ = oracle.quantize(x, fb.E4M3, gran, lay)
    assert np.array_equal(q.t.cpu().numpy(), oq)
    assert np.array_equal(sc.t.cpu().numpy(), np.ascontiguousarray(os_).view(np.uint8).reshape(-1))
    out = Guarded((rows, cols), torch.bfloat16)
    fb.dequantize(q.t, scv, fb.E4M3, gran, lay, out=out.t)
    assert out.intact()
    ref = oracle.dequantize(oq, os_, fb.E4M3, gran, lay)
    assert np.array_equal(out.t.view(torch.int16).cpu().numpy().view(np.uint16), ref)


@pytest.mark.parametrize("M,N,K", [(1, 16, 128), (17, 48, 256), (130, 272, 640), (257, 400, 384),
                                   (16, 2112, 7168), (32, 7168, 4096), (64, 144, 1024)])
def test_fold_gemm_stays_in_bounds(M, N, K):
    """Fold kernels (wide, narrow, operand-swapped, split-K over clusters)."""
    x = synth.bf16_matrix(M, K, 1.0, 1300 + M, 1301 + K, 0.01, 30.0)
    w = synth.bf16_matrix(N, K, 0.02, 1302 + N)
    qa, sa = oracle.quantize(x, fb.E4M3, fb.TILE_1x128)
    qb, sb = oracle.quantize(w, fb.E4M3, fb.BLOCK_128x128)
    out = Guarded((M, N), torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fb.gemm_blockscaled(torch.from_numpy(qa).cuda(), torch.from_numpy(sa).cuda(), fb.TILE_1x128,
                        torch.from_numpy(qb).cuda(), torch.from_numpy(sb).cuda(), fb.BLOCK_128x128, out=out.t,
                        status=status)
    assert out.intact() and int(status.item()) == 0
    rows = np.unique(np.concatenate([np.arange(0, M, max(1, M // 40)), [M - 1]]))
    ref, bound = oracle.gemm(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128, rows=rows)
    tol = within_tolerance(out_f64(out.t)[rows], ref, bound)
    assert tol.bad == 0, tol


@pytest.mark.parametrize("M,N,K", [(130, 256, 512), (300, 1152, 384)])
def test_fused_and_epilogue_scaled_gemms_stay_in_bounds(M, N, K):
    x = synth.bf16_matrix(M, K, 1.0, 1400 + M, 1401, 0.01, 30.0)
    w = synth.bf16_matrix(N, K, 0.02, 1402 + N)
    qa, sa = oracle.quantize(x, fb.E4M3, fb.TILE_1x128)
    qb, sb = oracle.quantize(w, fb.E4M3, fb.BLOCK_128x128)
    a, sad, b, sbd = (torch.from_numpy(t).cuda() for t in (qa, sa, qb, sb))
    qo = Guarded((M, N), torch.uint8)
    so = Guarded(((N // 128) * M,), torch.float32)
    fb.gemm_blockscaled_quantized_out(a, sad, b, sbd, q_out=qo.t, q_scales=so.t)
    assert qo.intact() and so.intact()
    # per-token activations x per-channel weights (epilogue-scaled tensor-memory kernel)
    ta, tsa = oracle.quantize(x, fb.E4M3, fb.TOKEN)
    tb, tsb = oracle.quantize(w, fb.E4M3, fb.TOKEN)
    out = Guarded((M, N), torch.bfloat16)
    fb.gemm_blockscaled(torch.from_numpy(ta).cuda(), torch.from_numpy(tsa).cuda(), fb.TOKEN,
                        torch.from_numpy(tb).cuda(), torch.from_numpy(tsb).cuda(), fb.TOKEN, out=out.t)
    assert out.intact()
    ref, bound = oracle.gemm(ta, tsa, fb.TOKEN, tb, tsb, fb.TOKEN)
    tol = within_tolerance(out_f64(out.t), ref, bound)
    assert tol.bad == 0, tol


@pytest.mark.parametrize("M,N,K", [(130, 272, 512), (257, 144, 1024)])
def test_mx_and_nvfp4_stay_in_bounds(M, N, K):
    x = synth.bf16_matrix(M, K, 1.0, 1500 + M, 1501, 0.01, 30.0)
    w = synth.bf16_matrix(N, K, 1.0, 1502 + N)
    qa, sfa = oracle.quantize(x, fb.E4M3, fb.MX32, fb.SF_TCGEN05)
    qb, sfb = oracle.quantize(w, fb.E4M3, fb.MX32, fb.SF_TCGEN05)
    ref, bound = oracle.gemm(qa, sfa, fb.MX32, qb, sfb, fb.MX32, a_sf=fb.SF_TCGEN05, b_sf=fb.SF_TCGEN05)
    for kernel in ("single", "pairs"):
        out = Guarded((M, N), torch.bfloat16)
        fb.debug_gemm_mx_kernel(kernel, *(torch.from_numpy(t).cuda() for t in (qa, sfa, qb, sfb)), out=out.t)
        assert out.intact(), kernel
        tol = within_tolerance(out_f64(out.t), ref, bound)
        assert tol.bad == 0, (kernel, tol)
    # the staged-four-times scale layout: quantizer scales and the GEMM's output
    sx4 = Guarded((fb.scales_bytes(M, K, fb.MX32, fb.SF_TCGEN05_X4),), torch.uint8)
    qx4 = Guarded((M, K), torch.uint8)
    fb.quantize(to_dev_bf16(x), fb.E4M3, fb.MX32, fb.SF_TCGEN05_X4, q=qx4.t, scales=sx4.t)
    assert sx4.intact() and qx4.intact()
    assert np.array_equal(sx4.t.cpu().numpy(), x4_layout(sfa))
    sw4 = torch.from_numpy(x4_layout(sfb)).cuda()
    out4 = Guarded((M, N), torch.bfloat16)
    fb.gemm_mx(qx4.t, sx4.t, torch.from_numpy(qb).cuda(), sw4, out=out4.t, sf_layout=fb.SF_TCGEN05_X4)
    assert out4.intact()
    tol = within_tolerance(out_f64(out4.t), ref, bound)
    assert tol.bad == 0, ("x4", tol)
    # NVFP4: codes, padded tiled scale atoms, tensor scale, dequantized output, GEMM output
    xd = to_dev_bf16(x)
    q4 = Guarded((M, K // 2), torch.uint8)
    sf4 = Guarded((fb.nvfp4_scales_bytes(M, K),), torch.uint8)
    ts4 = Guarded((1,), torch.float32)
    fb.quantize_nvfp4(xd, fb.SF_TCGEN05, q=q4.t, sf=sf4.t, tensor_scale=ts4.t)
    assert q4.intact() and sf4.intact() and ts4.intact()
    oq4, osf4, ots4 = oracle.quantize_nvfp4(x, fb.SF_TCGEN05)
    assert np.array_equal(q4.t.cpu().numpy(), oq4)
    assert np.array_equal(sf4.t.cpu().numpy()[: osf4.size], osf4)
    d4 = Guarded((M, K), torch.bfloat16)
    fb.dequantize_nvfp4(q4.t, sf4.t, ts4.t, K, fb.SF_TCGEN05, out=d4.t)
    assert d4.intact()
    qw4, sfw4, tw4 = fb.quantize_nvfp4(to_dev_bf16(w), fb.SF_TCGEN05)
    o4 = Guarded((M, N), torch.bfloat16)
    fb.gemm_nvfp4(q4.t, sf4.t, ts4.t, qw4, sfw4, tw4, out=o4.t)
    assert o4.intact()

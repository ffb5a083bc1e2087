"""Parity at the workloads' full sizes, through the same entry points and launch
configurations the bench times. Quantizer outputs are compared in full
(bit-exact); decode GEMMs in full; prefill and MX GEMMs on sampled rows
(every column), which the oracle computes one by one in fp64."""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_04_gb300 import binding as fb
from fp8_block_scaled_04_gb300 import synth
from gpu_util import f32_bits, out_f64, to_dev_bf16, within_tolerance, x4_layout

pytestmark = pytest.mark.gpu


def _sample_rows(M, per_tile=2, seed=0):
    rng = np.random.default_rng(seed)
    rows = {0, M - 1}
    for t in range(0, M, 128):
        for r in rng.integers(t, min(M, t + 128), per_tile):
            rows.add(int(r))
    return np.array(sorted(rows), dtype=np.int64)


@pytest.fixture(scope="module")
def sweep_x():
    return synth.sweep_x(16384, 8192)


@pytest.mark.parametrize("gran", [fb.TENSOR, fb.TOKEN, fb.TILE_1x128, fb.MX32])
@pytest.mark.parametrize("fmt", [fb.E4M3, fb.E5M2])
def test_quantizer_sweep_full_size(sweep_x, fmt, gran):
    xd = to_dev_bf16(sweep_x)
    q, s = fb.quantize(xd, fmt, gran)
    torch.cuda.synchronize()
    oq, os_ = oracle.quantize(sweep_x, fmt, gran)
    assert np.array_equal(q.cpu().numpy(), oq)
    gs = s.cpu().numpy()
    assert np.array_equal(gs, os_) if gran == fb.MX32 else np.array_equal(f32_bits(gs), f32_bits(os_))


@pytest.fixture(scope="module")
def decode_w():
    w = synth.decode_w(18432, 7168)
    qb, sb = oracle.quantize(w, fb.E4M3, fb.BLOCK_128x128)
    return w, qb, sb


@pytest.mark.parametrize("m", [16, 64])
def test_decode_gemm_full_size(decode_w, m):
    w, qb, sb = decode_w
    x = synth.decode_x(m, 7168)
    # the GPU quantizes both operands itself here (the bench's path), checked bit-exact first
    qa_d, sa_d = fb.quantize(to_dev_bf16(x), fb.E4M3, fb.TILE_1x128)
    qb_d, sb_d = fb.quantize(to_dev_bf16(w), fb.E4M3, fb.BLOCK_128x128)
    qa, sa = oracle.quantize(x, fb.E4M3, fb.TILE_1x128)
    assert np.array_equal(qa_d.cpu().numpy(), qa) and np.array_equal(qb_d.cpu().numpy(), qb)
    assert np.array_equal(f32_bits(sb_d.cpu().numpy()), f32_bits(sb))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fb.gemm_blockscaled(qa_d, sa_d, fb.TILE_1x128, qb_d, sb_d, fb.BLOCK_128x128, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, bound = oracle.gemm(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128)
    tol = within_tolerance(out_f64(out), ref, bound)
    assert tol.bad == 0, tol


def test_prefill_gemm_full_size_sampled_rows():
    M, N, K = 4096, 14336, 4096
    x = synth.prefill_x(M, K)
    w = synth.prefill_w(N, K)
    qa_d, sa_d = fb.quantize(to_dev_bf16(x), fb.E4M3, fb.TILE_1x128)
    qb_d, sb_d = fb.quantize(to_dev_bf16(w), fb.E4M3, fb.BLOCK_128x128)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fb.gemm_blockscaled(qa_d, sa_d, fb.TILE_1x128, qb_d, sb_d, fb.BLOCK_128x128, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    qa, sa = oracle.quantize(x, fb.E4M3, fb.TILE_1x128)
    qb, sb = oracle.quantize(w, fb.E4M3, fb.BLOCK_128x128)
    assert np.array_equal(qa_d.cpu().numpy(), qa) and np.array_equal(qb_d.cpu().numpy(), qb)
    rows = _sample_rows(M)
    ref, bound = oracle.gemm(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128, rows=rows)
    got = out_f64(out[torch.from_numpy(rows).cuda()])
    tol = within_tolerance(got, ref, bound)
    assert tol.bad == 0, tol


def test_mx_gemm_full_size_sampled_rows():
    S = 8192
    x = synth.mx_x(S, S)
    w = synth.mx_w(S, S)
    qa_d, sfa_d = fb.quantize(to_dev_bf16(x), fb.E4M3, fb.MX32, fb.SF_TCGEN05)
    qb_d, sfb_d = fb.quantize(to_dev_bf16(w), fb.E4M3, fb.MX32, fb.SF_TCGEN05)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fb.gemm_mx(qa_d, sfa_d, qb_d, sfb_d, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    qa, sfa = oracle.quantize(x, fb.E4M3, fb.MX32, fb.SF_TCGEN05)
    qb, sfb = oracle.quantize(w, fb.E4M3, fb.MX32, fb.SF_TCGEN05)
    assert np.array_equal(qa_d.cpu().numpy(), qa) and np.array_equal(sfa_d.cpu().numpy(), sfa)
    rows = _sample_rows(S, per_tile=1)
    ref, bound = oracle.gemm(qa, sfa, fb.MX32, qb, sfb, fb.MX32, a_sf=fb.SF_TCGEN05, b_sf=fb.SF_TCGEN05, rows=rows)
    got = out_f64(out[torch.from_numpy(rows).cuda()])
    tol = within_tolerance(got, ref, bound)
    assert tol.bad == 0, tol
    # the path the bench times first: scales quantized straight into the
    # staged-four-times layout, fp8_gemm_mx_x4 (the same output, bit for bit)
    _, sfa4_d = fb.quantize(to_dev_bf16(x), fb.E4M3, fb.MX32, fb.SF_TCGEN05_X4)
    _, sfb4_d = fb.quantize(to_dev_bf16(w), fb.E4M3, fb.MX32, fb.SF_TCGEN05_X4)
    assert np.array_equal(sfa4_d.cpu().numpy(), x4_layout(sfa)) and np.array_equal(sfb4_d.cpu().numpy(), x4_layout(sfb))
    out4 = fb.gemm_mx(qa_d, sfa4_d, qb_d, sfb4_d, status=status, sf_layout=fb.SF_TCGEN05_X4)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out.view(torch.int16), out4.view(torch.int16))
    tol4 = within_tolerance(out_f64(out4[torch.from_numpy(rows).cuda()]), ref, bound)
    assert tol4.bad == 0, tol4

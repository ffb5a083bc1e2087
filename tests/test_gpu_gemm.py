"""GPU parity of the scaled FP8 GEMMs against the CPU oracle.

Tolerance (fixed before any kernel ran): |gpu - ref| <= 1e-3 * sum_k |x_hat w_hat| + 1e-6
element-wise, with ref the fp64 sum over dequantized operands. Small-integer
operands with power-of-two scales must match exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_04_gb300 import binding as fb
from fp8_block_scaled_04_gb300 import synth
from gpu_util import bf16_host, out_f64, to_dev_bf16, within_tolerance, x4_layout

pytestmark = pytest.mark.gpu


def _quant_pair(x, w, ga, gb, fa=fb.E4M3, fw=fb.E4M3, layout=fb.SF_LINEAR):
    """Operands quantized by the oracle (CPU) so the GEMM is tested on its own."""
    qa, sa = oracle.quantize(x, fa, ga, layout)
    qb, sb = oracle.quantize(w, fw, gb, layout)
    return qa, sa, qb, sb


def _run_blockscaled(qa, sa, ga, qb, sb, gb, fa=fb.E4M3, fw=fb.E4M3):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fb.gemm_blockscaled(torch.from_numpy(qa).cuda(), torch.from_numpy(sa).cuda(), ga,
                              torch.from_numpy(qb).cuda(), torch.from_numpy(sb).cuda(), gb, fa, fw, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out


def _run_mx(qa, sfa, qb, sfb, fa=fb.E4M3, fw=fb.E4M3):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fb.gemm_mx(torch.from_numpy(qa).cuda(), torch.from_numpy(sfa).cuda(), torch.from_numpy(qb).cuda(),
                     torch.from_numpy(sfb).cuda(), fa, fw, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out


def test_tiny_config_blockscaled():
    x, w = synth.tiny()
    qa, sa, qb, sb = _quant_pair(x, w, fb.TILE_1x128, fb.BLOCK_128x128)
    out = _run_blockscaled(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128)
    ref, bound = oracle.gemm(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128)
    tol = within_tolerance(out_f64(out), ref, bound)
    assert tol.bad == 0, tol


@pytest.mark.parametrize("M,N,K", [(1, 16, 128), (17, 48, 256), (130, 272, 640), (300, 384, 384),
                                   (257, 512, 1152), (128, 4096, 256), (640, 1280, 512)])
def test_fold_ragged_shapes(M, N, K):
    x = synth.bf16_matrix(M, K, 1.0, 10 + M, 20 + K, 0.01, 50.0)
    w = synth.bf16_matrix(N, K, 0.02, 30 + N)
    qa, sa, qb, sb = _quant_pair(x, w, fb.TILE_1x128, fb.BLOCK_128x128)
    out = _run_blockscaled(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128)
    ref, bound = oracle.gemm(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128)
    tol = within_tolerance(out_f64(out), ref, bound)
    assert tol.bad == 0, tol


@pytest.mark.parametrize("M,N,K", [(2048, 2560, 256), (2000, 2480, 384), (4096, 2432, 640), (130, 272, 512),
                                   (1, 16, 128)])
def test_fold_on_cta_pairs(M, N, K):
    """The CTA-pair kernel (cta_group::2, 256 x 256 tiles) on ragged shapes, small ones included."""
    x = synth.bf16_matrix(M, K, 1.0, 60 + M, 61 + K, 0.01, 50.0)
    w = synth.bf16_matrix(N, K, 0.02, 62 + N)
    qa, sa, qb, sb = _quant_pair(x, w, fb.TILE_1x128, fb.BLOCK_128x128)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fb.debug_gemm_blockscaled_pairs(torch.from_numpy(qa).cuda(), torch.from_numpy(sa).cuda(),
                                          torch.from_numpy(qb).cuda(), torch.from_numpy(sb).cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = np.unique(np.concatenate([np.arange(0, M, 97), np.arange(max(0, M - 130), M), np.arange(min(120, M), min(390, M))]))
    ref, bound = oracle.gemm(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128, rows=rows)
    tol = within_tolerance(out_f64(out)[rows], ref, bound)
    assert tol.bad == 0, tol


@pytest.mark.parametrize("M,N,K", [(16, 7168, 16384), (32, 2048, 4096), (64, 4096, 1024), (16, 1040, 2048),
                                   (5, 768, 896), (48, 3072, 7168)])
def test_decode_split_k(M, N, K):
    """Few 128-row weight blocks: the K range of each block is split over a CTA cluster
    (ragged N edge, odd M, K ranges that do not divide evenly)."""
    x = synth.bf16_matrix(M, K, 1.0, 70 + M, 71 + K, 0.01, 50.0)
    w = synth.bf16_matrix(N, K, 0.02, 72 + N)
    qa, sa, qb, sb = _quant_pair(x, w, fb.TILE_1x128, fb.BLOCK_128x128)
    out = _run_blockscaled(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128)
    cols = np.unique(np.concatenate([np.arange(0, N, 7), np.arange(N - 140, N)]))
    ref, bound = oracle.gemm(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128, cols=cols)
    tol = within_tolerance(out_f64(out)[:, cols], ref, bound)
    assert tol.bad == 0, tol


@pytest.mark.parametrize("M,N,K", [(64, 18432, 8192), (60, 18432, 3584), (61, 18432, 2048), (32, 18448, 7040),
                                   (16, 20480, 3584), (48, 20608, 8192), (3, 18432, 1024),
                                   (16, 17536, 16896)])
def test_decode_every_sm_busy(M, N, K):
    """The decode kernel when the weight blocks fill the GPU (no K split): scales
    brought by tensor copies in chunks of k-blocks (whole chunks, a partial last
    chunk, activation rows past M read as zero, several tiles per CTA, a ragged
    N edge) and by per-lane loads where the copies cannot describe them
    (M % 4 != 0, K/128 % 4 != 0)."""
    x = synth.bf16_matrix(M, K, 1.0, 80 + M, 81 + K, 0.01, 50.0)
    w = synth.bf16_matrix(N, K, 0.02, 82 + N)
    qa, sa, qb, sb = _quant_pair(x, w, fb.TILE_1x128, fb.BLOCK_128x128)
    out = _run_blockscaled(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128)
    cols = np.unique(np.concatenate([np.arange(0, N, 97), np.arange(N - 140, N)]))
    ref, bound = oracle.gemm(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128, cols=cols)
    tol = within_tolerance(out_f64(out)[:, cols], ref, bound)
    assert tol.bad == 0, tol


def test_decode_scale_paths_agree_bit_for_bit():
    """The same decode GEMM with its scale vectors 16-byte aligned (tensor-copy
    path) and shifted by one float (per-lane load path) gives identical bytes:
    both form each product s_w * s_x with the same fp32 multiply."""
    M, N, K = 64, 18432, 3584
    x = synth.bf16_matrix(M, K, 1.0, 90, 91, 0.01, 50.0)
    w = synth.bf16_matrix(N, K, 0.02, 92)
    qa, sa, qb, sb = _quant_pair(x, w, fb.TILE_1x128, fb.BLOCK_128x128)
    a, b = torch.from_numpy(qa).cuda(), torch.from_numpy(qb).cuda()
    outs = []
    for shift in (0, 1):
        sa_d = torch.zeros(sa.size + 4, dtype=torch.float32, device="cuda")[shift:shift + sa.size]
        sb_d = torch.zeros(sb.size + 4, dtype=torch.float32, device="cuda")[shift:shift + sb.size]
        sa_d.copy_(torch.from_numpy(sa))
        sb_d.copy_(torch.from_numpy(sb))
        assert (sa_d.data_ptr() % 16 == 0) == (shift == 0)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        outs.append(fb.gemm_blockscaled(a, sa_d, fb.TILE_1x128, b, sb_d, fb.BLOCK_128x128, status=status))
        torch.cuda.synchronize()
        assert int(status.item()) == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    cols = np.arange(0, N, 61)
    ref, bound = oracle.gemm(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128, cols=cols)
    tol = within_tolerance(out_f64(outs[0])[:, cols], ref, bound)
    assert tol.bad == 0, tol


def test_decode_split_k_small_integers_exact():
    """Split-K partial sums of integer-valued operands with power-of-two scales are exact."""
    rng = np.random.default_rng(11)
    M, N, K = 16, 1024, 512 * 8
    a = oracle.encode(rng.integers(-4, 5, (M, K)).astype(np.float32), fb.E4M3)
    b = oracle.encode(rng.integers(-4, 5, (N, K)).astype(np.float32), fb.E4M3)
    # scales 2^-1..2^1: every partial is a multiple of 2^-2 below 2^18, so fp32 sums are exact
    sa = (2.0 ** rng.integers(-1, 2, (K // 128) * M)).astype(np.float32)
    sb = (2.0 ** rng.integers(-1, 2, ((N + 127) // 128) * (K // 128))).astype(np.float32)
    out = _run_blockscaled(a, sa, fb.TILE_1x128, b, sb, fb.BLOCK_128x128)
    ref, _ = oracle.gemm(a, sa, fb.TILE_1x128, b, sb, fb.BLOCK_128x128)
    expect = oracle.bf16_to_f32(oracle.f32_to_bf16(ref.astype(np.float32))).astype(np.float64)
    assert np.array_equal(out_f64(out), expect)


def test_fold_small_integers_exact():
    """Integer-valued FP8 operands, power-of-two scales, K <= 512: fp32 sums are exact."""
    rng = np.random.default_rng(1)
    M, N, K = 130, 272, 512
    a = oracle.encode(rng.integers(-8, 9, (M, K)).astype(np.float32), fb.E4M3)
    b = oracle.encode(rng.integers(-8, 9, (N, K)).astype(np.float32), fb.E4M3)
    sa = (2.0 ** rng.integers(-3, 4, (K // 128) * M)).astype(np.float32)
    sb = (2.0 ** rng.integers(-3, 4, ((N + 127) // 128) * (K // 128))).astype(np.float32)
    out = _run_blockscaled(a, sa, fb.TILE_1x128, b, sb, fb.BLOCK_128x128)
    ref, _ = oracle.gemm(a, sa, fb.TILE_1x128, b, sb, fb.BLOCK_128x128)
    expect = oracle.bf16_to_f32(oracle.f32_to_bf16(ref.astype(np.float32))).astype(np.float64)
    assert np.array_equal(out_f64(out), expect)


@pytest.mark.parametrize("fa,fw", [(fb.E5M2, fb.E4M3), (fb.E4M3, fb.E5M2), (fb.E5M2, fb.E5M2)])
def test_fold_e5m2_operands(fa, fw):
    x, w = synth.tiny()
    qa, sa, qb, sb = _quant_pair(x, w, fb.TILE_1x128, fb.BLOCK_128x128, fa, fw)
    out = _run_blockscaled(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128, fa, fw)
    ref, bound = oracle.gemm(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128, fa, fw)
    tol = within_tolerance(out_f64(out), ref, bound)
    assert tol.bad == 0, tol


@pytest.mark.parametrize("ga,gb", [(fb.TENSOR, fb.TENSOR), (fb.TOKEN, fb.TOKEN), (fb.TOKEN, fb.TENSOR),
                                   (fb.TENSOR, fb.TOKEN)])
@pytest.mark.parametrize("M,N,K", [(1, 16, 144), (130, 272, 400), (300, 512, 1024)])
def test_epilogue_scaled_modes(ga, gb, M, N, K):
    x = synth.bf16_matrix(M, K, 1.0, 40 + M, 41, 0.01, 30.0)
    w = synth.bf16_matrix(N, K, 0.02, 42 + N)
    qa, sa, qb, sb = _quant_pair(x, w, ga, gb)
    out = _run_blockscaled(qa, sa, ga, qb, sb, gb)
    ref, bound = oracle.gemm(qa, sa, ga, qb, sb, gb)
    tol = within_tolerance(out_f64(out), ref, bound)
    assert tol.bad == 0, tol


def test_uniform_block_scales_match_per_tensor_path():
    x, w = synth.tiny()
    qa, _ = oracle.quantize(x, fb.E4M3, fb.TENSOR)
    qb, _ = oracle.quantize(w, fb.E4M3, fb.TENSOR)
    sa = np.full(4 * 128, 0.5, np.float32)
    sb = np.full(2 * 4, 0.25, np.float32)
    o1 = _run_blockscaled(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128)
    o2 = _run_blockscaled(qa, np.array([0.5], np.float32), fb.TENSOR, qb, np.array([0.25], np.float32), fb.TENSOR)
    ref, bound = oracle.gemm(qa, np.array([0.5], np.float32), fb.TENSOR, qb, np.array([0.25], np.float32), fb.TENSOR)
    tol1 = within_tolerance(out_f64(o1), ref, bound)
    assert tol1.bad == 0, tol1
    tol2 = within_tolerance(out_f64(o2), ref, bound)
    assert tol2.bad == 0, tol2


# ------------------------------------------------------------------ MX
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 256, 512), (130, 272, 416), (1, 16, 32), (300, 640, 1024)])
def test_mx_shapes(M, N, K):
    x = synth.bf16_matrix(M, K, 1.0, 50 + M, 51, 0.005, 50.0)
    w = synth.bf16_matrix(N, K, 1.0, 52 + N, 53, 0.005, 50.0)
    qa, sfa, qb, sfb = _quant_pair(x, w, fb.MX32, fb.MX32, layout=fb.SF_TCGEN05)
    out = _run_mx(qa, sfa, qb, sfb)
    ref, bound = oracle.gemm(qa, sfa, fb.MX32, qb, sfb, fb.MX32, a_sf=fb.SF_TCGEN05, b_sf=fb.SF_TCGEN05)
    tol = within_tolerance(out_f64(out), ref, bound)
    assert tol.bad == 0, tol


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 256, 512), (130, 272, 416), (1, 16, 32), (300, 640, 1024),
                                   (1024, 1536, 4096), (2304, 512, 640)])
def test_mx_x4_layout_same_output_as_tiled(M, N, K):
    """fp8_gemm_mx_x4 on the staged-four-times scales: the same tensor-memory
    scale contents as fp8_gemm_mx, so the same output bit for bit, and within
    the tolerance of the oracle."""
    x = synth.bf16_matrix(M, K, 1.0, 60 + M, 61, 0.005, 50.0)
    w = synth.bf16_matrix(N, K, 1.0, 62 + N, 63, 0.005, 50.0)
    qa, sfa, qb, sfb = _quant_pair(x, w, fb.MX32, fb.MX32, layout=fb.SF_TCGEN05)
    out = _run_mx(qa, sfa, qb, sfb)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out4 = fb.gemm_mx(torch.from_numpy(qa).cuda(), torch.from_numpy(x4_layout(sfa)).cuda(), torch.from_numpy(qb).cuda(),
                      torch.from_numpy(x4_layout(sfb)).cuda(), status=status, sf_layout=fb.SF_TCGEN05_X4)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out.view(torch.int16), out4.view(torch.int16))
    ref, bound = oracle.gemm(qa, sfa, fb.MX32, qb, sfb, fb.MX32, a_sf=fb.SF_TCGEN05, b_sf=fb.SF_TCGEN05)
    tol = within_tolerance(out_f64(out4), ref, bound)
    assert tol.bad == 0, tol


@pytest.mark.parametrize("kernel", ["pairs", "single"])
@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (512, 768, 1024), (300, 640, 1024), (130, 272, 416),
                                   (1, 16, 32), (1024, 1536, 4096), (2304, 512, 640)])
def test_mx_on_each_kernel(kernel, M, N, K):
    """Both MXFP8 kernels, whatever the shape rule picks: CTA pairs (256 x 256
    tiles, each CTA staging its halves of the operands and the scale atoms its
    tensor core reads) and one CTA per 128 x 256 tile; ragged M, N and K, one
    pair tile, several tiles per pair."""
    x = synth.bf16_matrix(M, K, 1.0, 60 + M, 61, 0.005, 50.0)
    w = synth.bf16_matrix(N, K, 1.0, 62 + N, 63, 0.005, 50.0)
    qa, sfa, qb, sfb = _quant_pair(x, w, fb.MX32, fb.MX32, layout=fb.SF_TCGEN05)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fb.debug_gemm_mx_kernel(kernel, *(torch.from_numpy(v).cuda() for v in (qa, sfa, qb, sfb)), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = np.unique(np.concatenate([np.arange(0, M, max(1, M // 64)), [M - 1]]))
    ref, bound = oracle.gemm(qa, sfa, fb.MX32, qb, sfb, fb.MX32, a_sf=fb.SF_TCGEN05, b_sf=fb.SF_TCGEN05, rows=rows)
    tol = within_tolerance(out_f64(out)[rows], ref, bound)
    assert tol.bad == 0, tol


def test_mx_unit_scales_equal_plain_path():
    """SF byte 127 (scale 1) everywhere: the block-scaled MMA must equal the plain one."""
    x, w = synth.tiny()
    qa, _ = oracle.quantize(x, fb.E4M3, fb.TENSOR)
    qb, _ = oracle.quantize(w, fb.E4M3, fb.TENSOR)
    sfa = np.full(oracle.mx_tiled_bytes(128, 512 // 32), 127, np.uint8)
    sfb = np.full(oracle.mx_tiled_bytes(256, 512 // 32), 127, np.uint8)
    o_mx = _run_mx(qa, sfa, qb, sfb)
    one = np.array([1.0], np.float32)
    o_plain = _run_blockscaled(qa, one, fb.TENSOR, qb, one, fb.TENSOR)
    assert torch.equal(o_mx, o_plain)


def test_mx_distinct_scales_per_row_and_group():
    """One-hot scale structure: row r of A and group j carry 2^((r + 3j) % 7 - 3)."""
    M, N, K = 256, 256, 256
    rng = np.random.default_rng(3)
    a = oracle.encode(rng.integers(-4, 5, (M, K)).astype(np.float32), fb.E4M3)
    b = oracle.encode(rng.integers(-4, 5, (N, K)).astype(np.float32), fb.E4M3)
    ng = K // 32
    sfa = np.zeros(oracle.mx_tiled_bytes(M, ng), np.uint8)
    sfb = np.zeros(oracle.mx_tiled_bytes(N, ng), np.uint8)
    for r in range(M):
        for j in range(ng):
            sfa[oracle.mx_tiled_offset(r, j, M, ng)] = 127 + (r + 3 * j) % 7 - 3
    for n in range(N):
        for j in range(ng):
            sfb[oracle.mx_tiled_offset(n, j, N, ng)] = 127 + (2 * n + j) % 5 - 2
    out = _run_mx(a, sfa, b, sfb)
    ref, _ = oracle.gemm(a, sfa, fb.MX32, b, sfb, fb.MX32, a_sf=fb.SF_TCGEN05, b_sf=fb.SF_TCGEN05)
    expect = oracle.bf16_to_f32(oracle.f32_to_bf16(ref.astype(np.float32))).astype(np.float64)
    assert np.array_equal(out_f64(out), expect)


# ------------------------------------------------------------------ status
def test_status_stays_zero_and_launches_counted():
    x, w = synth.tiny()
    qa, sa, qb, sb = _quant_pair(x, w, fb.TILE_1x128, fb.BLOCK_128x128)
    n0 = fb.launch_count()
    _run_blockscaled(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128)
    assert fb.launch_count() == n0 + 1


@pytest.mark.parametrize("M", [16, 64, 256])
def test_dependent_launches_keep_stream_order(M):
    """quantize -> GEMM -> quantize -> GEMM -> GEMM enqueued with no host sync between
    them. The GEMMs are dependent launches that may start before the kernel ahead of
    them has finished; each stage, checked against the oracle on the GPU's own inputs
    to it, must have read its producer's finished output."""
    K1, N1, N2 = 1024, 2048, 1024
    x = synth.bf16_matrix(M, K1, 1.0, 700 + M, 701, 0.01, 30.0)
    w1 = synth.bf16_matrix(N1, K1, 0.02, 702)
    w2 = synth.bf16_matrix(N2, N1, 0.02, 703)
    w3 = synth.bf16_matrix(N2, N1, 0.02, 704)
    dev = lambda a: torch.from_numpy(a).cuda()
    qw = [oracle.quantize(w, fb.E4M3, fb.BLOCK_128x128, fb.SF_LINEAR) for w in (w1, w2, w3)]
    qw_d = [(dev(q), dev(sc)) for q, sc in qw]
    torch.cuda.synchronize()
    xq, xs = fb.quantize(to_dev_bf16(x), fb.E4M3, fb.TILE_1x128)
    o1 = fb.gemm_blockscaled(xq, xs, fb.TILE_1x128, *qw_d[0], fb.BLOCK_128x128)
    hq, hs = fb.quantize(o1, fb.E4M3, fb.TILE_1x128)
    o2 = fb.gemm_blockscaled(hq, hs, fb.TILE_1x128, *qw_d[1], fb.BLOCK_128x128)
    o3 = fb.gemm_blockscaled(hq, hs, fb.TILE_1x128, *qw_d[2], fb.BLOCK_128x128)
    torch.cuda.synchronize()
    xq_o, xs_o = oracle.quantize(x, fb.E4M3, fb.TILE_1x128, fb.SF_LINEAR)
    assert np.array_equal(xq.cpu().numpy(), xq_o) and np.array_equal(xs.cpu().numpy(), xs_o)
    ref, bound = oracle.gemm(xq_o, xs_o, fb.TILE_1x128, *qw[0], fb.BLOCK_128x128)
    tol = within_tolerance(out_f64(o1), ref, bound)
    assert tol.bad == 0, ("o1", tol)
    hq_o, hs_o = oracle.quantize(bf16_host(o1), fb.E4M3, fb.TILE_1x128, fb.SF_LINEAR)
    assert np.array_equal(hq.cpu().numpy(), hq_o) and np.array_equal(hs.cpu().numpy(), hs_o)
    for o, (qb, sb) in ((o2, qw[1]), (o3, qw[2])):
        ref, bound = oracle.gemm(hq_o, hs_o, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128)
        tol = within_tolerance(out_f64(o), ref, bound)
        assert tol.bad == 0, tol


"""GPU parity of the quantizers, the dequantizer and the codec against the CPU oracle.

Quantized codes and scales must match the oracle bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_04_gb300 import binding as fb
from fp8_block_scaled_04_gb300 import synth
from gpu_util import bf16_host, f32_bits, to_dev_bf16, x4_layout

pytestmark = pytest.mark.gpu

FMTS = [fb.E4M3, fb.E5M2]
GRANS = [fb.TENSOR, fb.TOKEN, fb.TILE_1x128, fb.BLOCK_128x128, fb.MX32, fb.CHANNEL]
# ragged rows (not multiples of 128), several 128-wide column blocks, one long row
SHAPES = [(1, 128), (17, 256), (130, 640), (300, 1024), (64, 8192), (3, 20480)]


def _check_quant(x, fmt, gran, layout=fb.SF_LINEAR):
    xd = to_dev_bf16(x)
    q, s = fb.quantize(xd, fmt, gran, layout)
    torch.cuda.synchronize()
    oq, os_ = oracle.quantize(x, fmt, gran, layout)
    gq = q.cpu().numpy()
    assert np.array_equal(gq, oq), "codes differ at %s" % (np.argwhere(gq != oq)[:5].tolist(),)
    gs = s.cpu().numpy()
    if gran == fb.MX32:
        assert np.array_equal(gs, os_)
    else:
        assert np.array_equal(f32_bits(gs), f32_bits(os_))
    return q, s


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("gran", GRANS)
@pytest.mark.parametrize("fmt", FMTS)
def test_quantize_bit_exact(fmt, gran, shape):
    rows, cols = shape
    x = synth.bf16_matrix(rows, cols, 1.0, 1000 + rows, 2000 + cols, 0.01, 60.0)
    _check_quant(x, fmt, gran)


@pytest.mark.parametrize("shape", [(130, 640), (128, 512), (257, 160)])
@pytest.mark.parametrize("fmt", FMTS)
def test_quantize_mx_tiled_layout_bit_exact(fmt, shape):
    rows, cols = shape
    x = synth.bf16_matrix(rows, cols, 1.0, 77, 78, 0.02, 30.0)
    _check_quant(x, fmt, fb.MX32, fb.SF_TCGEN05)


@pytest.mark.parametrize("shape", [(130, 640), (128, 512), (257, 160), (1, 32)])
@pytest.mark.parametrize("fmt", FMTS)
def test_quantize_mx_x4_layout_bit_exact(fmt, shape):
    """MX-32 scales in the staged-four-times layout: codes equal the oracle's and
    the scale bytes equal the oracle's tiled bytes with each 512-byte block
    repeated four times (padding of partial blocks zero in every copy); the
    dequantizer reads them back to the oracle's values."""
    rows, cols = shape
    x = synth.bf16_matrix(rows, cols, 1.0, 79, 80, 0.02, 30.0)
    q, s = fb.quantize(to_dev_bf16(x), fmt, fb.MX32, fb.SF_TCGEN05_X4)
    torch.cuda.synchronize()
    oq, os_ = oracle.quantize(x, fmt, fb.MX32, fb.SF_TCGEN05)
    assert s.numel() == fb.scales_bytes(rows, cols, fb.MX32, fb.SF_TCGEN05_X4) == 4 * os_.size
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy(), x4_layout(os_))
    out = fb.dequantize(q, s, fmt, fb.MX32, fb.SF_TCGEN05_X4)
    ref = oracle.dequantize(oq, os_, fmt, fb.MX32, fb.SF_TCGEN05)
    assert np.array_equal(bf16_host(out), ref)


@pytest.mark.parametrize("layout", [fb.SF_TCGEN05, fb.SF_TCGEN05_X4])
@pytest.mark.parametrize("shape", [(130, 640), (257, 160)])
def test_quantize_mx_tiled_scales_only_4_byte_aligned(layout, shape):
    """A tiled scale array that is 4- but not 16-byte aligned takes the
    byte-store kernel instead of the block kernel: the same bytes."""
    rows, cols = shape
    x = synth.bf16_matrix(rows, cols, 1.0, 81, 82, 0.02, 30.0)
    n = fb.scales_bytes(rows, cols, fb.MX32, layout)
    big = torch.full((n + 16,), 0x5A, dtype=torch.uint8, device="cuda")
    s = big[4:4 + n]
    assert s.data_ptr() % 16 == 4
    q, _ = fb.quantize(to_dev_bf16(x), fb.E4M3, fb.MX32, layout, scales=s)
    torch.cuda.synchronize()
    oq, os_ = oracle.quantize(x, fb.E4M3, fb.MX32, fb.SF_TCGEN05)
    want = os_ if layout == fb.SF_TCGEN05 else x4_layout(os_)
    assert np.array_equal(q.cpu().numpy(), oq)
    got = big.cpu().numpy()
    assert np.array_equal(got[4:4 + n], want)
    assert (got[:4] == 0x5A).all() and (got[4 + n:] == 0x5A).all()


@pytest.mark.parametrize("gran", [fb.TENSOR, fb.TOKEN, fb.TILE_1x128, fb.MX32])
def test_extreme_values(gran):
    rng = np.random.default_rng(5)
    rows, cols = 64, 512
    mag = 2.0 ** rng.integers(-133, 127, (rows, cols)).astype(np.float64)
    x32 = (rng.uniform(1, 2, (rows, cols)) * mag * rng.choice([-1, 1], (rows, cols))).astype(np.float32)
    x32[5, :] = 0.0  # all-zero rows / groups
    x32[6, :] = 2.0 ** -133  # subnormal bf16 only
    x32[7, :128] = 3.0e38  # near the bf16 maximum
    x = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for fmt in FMTS:
        _check_quant(x, fmt, gran)


def test_leading_dimensions():
    x = synth.bf16_matrix(40, 1024, 1.0, 91)
    xd_full = to_dev_bf16(x)
    xd = xd_full[:, 128:640]  # ld_x = 1024 > cols = 512
    q = torch.zeros((40, 768), dtype=torch.uint8, device="cuda")[:, :512]  # ld_q = 768
    for gran in GRANS:
        qq, s = fb.quantize(xd, fb.E4M3, gran, q=q)
        oq, os_ = oracle.quantize(np.ascontiguousarray(x[:, 128:640]), fb.E4M3, gran)
        assert np.array_equal(qq.cpu().numpy(), oq)


@pytest.mark.parametrize("fmt", FMTS)
def test_static_scale(fmt):
    x = synth.bf16_matrix(33, 256, 2.0, 92)
    xd = to_dev_bf16(x)
    st = torch.tensor([0.0078125 if fmt == fb.E4M3 else 0.125], dtype=torch.float32, device="cuda")
    q, s = fb.quantize(xd, fmt, fb.TENSOR, static_scale=st)
    oq, os_ = oracle.quantize(x, fmt, fb.TENSOR, static_scale=float(st.item()))
    assert np.array_equal(q.cpu().numpy(), oq) and float(s.item()) == float(os_[0])


def test_empty_input_is_noop():
    x = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    n0 = fb.launch_count()
    fb.quantize(x, fb.E4M3, fb.TOKEN)
    assert fb.launch_count() == n0


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("gran", GRANS)
def test_dequantize_bit_exact(fmt, gran):
    x = synth.bf16_matrix(130, 640, 1.0, 93, 94, 0.01, 40.0)
    oq, os_ = oracle.quantize(x, fmt, gran)
    qd = torch.from_numpy(oq).cuda()
    sd = torch.from_numpy(os_).cuda()
    out = fb.dequantize(qd, sd, fmt, gran)
    ref = oracle.dequantize(oq, os_, fmt, gran)
    assert np.array_equal(bf16_host(out), ref)


@pytest.mark.parametrize("fmt", FMTS)
def test_dequantize_mx_tiled(fmt):
    x = synth.bf16_matrix(130, 640, 1.0, 95)
    oq, os_ = oracle.quantize(x, fmt, fb.MX32, fb.SF_TCGEN05)
    out = fb.dequantize(torch.from_numpy(oq).cuda(), torch.from_numpy(os_).cuda(), fmt, fb.MX32, fb.SF_TCGEN05)
    assert np.array_equal(bf16_host(out), oracle.dequantize(oq, os_, fmt, fb.MX32, fb.SF_TCGEN05))


@pytest.mark.parametrize("fmt", FMTS)
def test_decode_all_256_codes(fmt):
    codes = np.arange(256, dtype=np.uint8).reshape(16, 16)
    out = fb.dequantize(torch.from_numpy(codes).cuda(), torch.ones(1, device="cuda"), fmt, fb.TENSOR)
    got = out.float().cpu().numpy().astype(np.float64).ravel()
    ref = oracle.decode(codes.ravel(), fmt)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("fmt", FMTS)
def test_encode_every_fp32(fmt):
    """The quantizers' element step against the oracle encoder on all 2^32 fp32 patterns."""
    chunk = 1 << 28
    total_bad = 0
    for start in range(0, 1 << 32, chunk):
        bits = torch.arange(start, start + chunk, dtype=torch.int64, device="cuda").to(torch.int32)
        x = bits.view(torch.float32)
        codes = fb.debug_encode_f32(x, fmt)
        bad, first = oracle.check_codes(start, codes.cpu().numpy(), fmt)
        assert bad == 0, "first mismatch at fp32 pattern 0x%08x" % first
        total_bad += bad
    assert total_bad == 0


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(37, 256), (300, 1024), (2048, 4096)])
def test_delayed_scaling_sequence_bit_exact(fmt, shape):
    """Five steps through a 3-entry amax history with margin 1: codes, scale and
    history match the oracle after every step."""
    rows, cols = shape
    hist_d = torch.zeros(3, dtype=torch.float32, device="cuda")
    hist_o = np.zeros(3, np.float32)
    for step in range(5):
        sigma = [1.0, 2.0, 0.5, 8.0, 1.0][step]
        x = synth.bf16_matrix(rows, cols, sigma, 600 + step, 700 + step, 0.01, 30.0)
        q, s = fb.quantize_delayed(to_dev_bf16(x), fmt, hist_d, slot=step % 3, margin=1)
        torch.cuda.synchronize()
        oq, os_, hist_o = oracle.quantize_delayed(x, fmt, hist_o, slot=step % 3, margin=1)
        assert np.array_equal(q.cpu().numpy(), oq), step
        assert np.array_equal(f32_bits(s.cpu().numpy()), f32_bits(os_)), step
        assert np.array_equal(f32_bits(hist_d.cpu().numpy()), f32_bits(hist_o)), step

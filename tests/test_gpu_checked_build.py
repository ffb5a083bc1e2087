"""The store-checked build (libfp8bs_check.so, -DFP8BS_CHECK): every plain
global store of every kernel family first checks its offset against the extent
the call's shape gives the buffer, skips a store outside it and records the
first one. Run on the small and ragged shapes where a stray store is likeliest,
the checked build must record nothing and produce exactly the product build's
outputs (its checks only skip stores that should not happen)."""
import numpy as np
import pytest
import torch

from fp8_block_scaled_04_gb300 import binding as fb
from fp8_block_scaled_04_gb300 import synth
from gpu_util import to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked():
    L = fb.load(fb.CHECK_LIB_PATH)
    assert L.fp8_debug_checked_build() == 1 and fb.lib().fp8_debug_checked_build() == 0
    L.fp8_debug_oob_read()  # start clean
    return L


def _both(checked, fn):
    """fn() on the product build, then on the checked build; the checked build's
    store record must stay empty. Returns (product outputs, checked outputs)."""
    ref = fn()
    torch.cuda.synchronize()
    saved = fb._lib
    fb._lib = checked
    try:
        got = fn()
        rec = checked.fp8_debug_oob_read()
    finally:
        fb._lib = saved
    assert rec == 0, "out-of-bounds store: line %d, offset %d" % (rec >> 40, rec & ((1 << 40) - 1))
    return ref, got


def _eq(a, b):
    for x, y in zip(a if isinstance(a, tuple) else (a,), b if isinstance(b, tuple) else (b,)):
        assert torch.equal(x.view(torch.uint8) if x.dtype != torch.uint8 else x,
                           y.view(torch.uint8) if y.dtype != torch.uint8 else y)


GRANS = [(fb.TENSOR, fb.SF_LINEAR), (fb.TOKEN, fb.SF_LINEAR), (fb.TILE_1x128, fb.SF_LINEAR),
         (fb.BLOCK_128x128, fb.SF_LINEAR), (fb.MX32, fb.SF_LINEAR), (fb.MX32, fb.SF_TCGEN05),
         (fb.MX32, fb.SF_TCGEN05_X4), (fb.CHANNEL, fb.SF_LINEAR)]


@pytest.mark.parametrize("shape", [(1, 128), (7, 384), (130, 640), (257, 1152), (3, 17408)])
def test_quantizers_record_no_stray_store(checked, shape):
    rows, cols = shape
    x = to_dev_bf16(synth.bf16_matrix(rows, cols, 1.0, 3000 + rows, 3001, 0.02, 40.0))
    for gran, lay in GRANS:
        def run():
            q, s = fb.quantize(x, fb.E4M3, gran, lay)
            d = fb.dequantize(q, s, fb.E4M3, gran, lay)
            return q, s, d
        _eq(*_both(checked, run))
    hist = torch.zeros(4, dtype=torch.float32, device="cuda")

    def delayed():
        h = hist.clone()
        q, s = fb.quantize_delayed(x, fb.E5M2, h, 1)
        return q, s, h
    _eq(*_both(checked, delayed))
    if cols % 16 == 0:
        _eq(*_both(checked, lambda: fb.quantize_nvfp4(x, fb.SF_TCGEN05)))
        _eq(*_both(checked, lambda: fb.quantize_nvfp4(x, fb.SF_LINEAR)))


def _ops(M, N, K, seed):
    x = to_dev_bf16(synth.bf16_matrix(M, K, 1.0, seed, seed + 1, 0.01, 30.0))
    w = to_dev_bf16(synth.bf16_matrix(N, K, 0.02, seed + 2))
    return x, w


@pytest.mark.parametrize("M,N,K", [(1, 16, 128), (130, 272, 640), (2048, 4096, 512), (16, 2112, 7168),
                                   (64, 144, 1024), (300, 384, 256)])
def test_gemms_record_no_stray_store(checked, M, N, K):
    x, w = _ops(M, N, K, 3100 + M)
    qa, sa = fb.quantize(x, fb.E4M3, fb.TILE_1x128)
    qb, sb = fb.quantize(w, fb.E4M3, fb.BLOCK_128x128)
    _eq(*_both(checked, lambda: fb.gemm_blockscaled(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128)))
    _eq(*_both(checked, lambda: fb.debug_gemm_blockscaled_pairs(qa, sa, qb, sb)))
    if N % 128 == 0:
        _eq(*_both(checked, lambda: fb.gemm_blockscaled_quantized_out(qa, sa, qb, sb)))
    ta, tsa = fb.quantize(x, fb.E4M3, fb.TOKEN)
    tb, tsb = fb.quantize(w, fb.E4M3, fb.TOKEN)
    _eq(*_both(checked, lambda: fb.gemm_blockscaled(ta, tsa, fb.TOKEN, tb, tsb, fb.TOKEN)))
    ma, msa = fb.quantize(x, fb.E4M3, fb.MX32, fb.SF_TCGEN05)
    mb, msb = fb.quantize(w, fb.E4M3, fb.MX32, fb.SF_TCGEN05)
    _eq(*_both(checked, lambda: fb.gemm_mx(ma, msa, mb, msb)))
    _, msa4 = fb.quantize(x, fb.E4M3, fb.MX32, fb.SF_TCGEN05_X4)
    _, msb4 = fb.quantize(w, fb.E4M3, fb.MX32, fb.SF_TCGEN05_X4)
    _eq(*_both(checked, lambda: fb.gemm_mx(ma, msa4, mb, msb4, sf_layout=fb.SF_TCGEN05_X4)))
    _eq(*_both(checked, lambda: fb.debug_gemm_mx_kernel("pairs", ma, msa, mb, msb)))
    if K % 256 == 0:
        na, nsa, nta = fb.quantize_nvfp4(x)
        nb, nsb, ntb = fb.quantize_nvfp4(w)
        _eq(*_both(checked, lambda: fb.gemm_nvfp4(na, nsa, nta, nb, nsb, ntb)))
        _eq(*_both(checked, lambda: fb.dequantize_nvfp4(na, nsa, nta, K)))


def test_codec_checks_record_no_stray_store(checked):
    bits = torch.arange(0, 1 << 20, dtype=torch.int64, device="cuda").to(torch.int32) * 4093
    f = bits.view(torch.float32)
    _eq(*_both(checked, lambda: fb.debug_encode_f32(f, fb.E4M3)))
    _eq(*_both(checked, lambda: fb.debug_encode_e2m1_f32(f)))

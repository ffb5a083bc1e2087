"""CPU checks of the C ABI: the library loads, exports every declared entry
point, and refuses bad arguments on the host with the documented codes
(no CUDA call is reached on any of these paths)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from fp8_block_scaled_04_gb300 import binding as fb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from fp8_block_scaled_04_gb300 import build

    build.build()
    return fb.lib()


def test_every_declared_symbol_is_exported(L):
    names = fb.declared_functions()
    assert {"fp8_quantize", "fp8_dequantize", "fp8_gemm_blockscaled", "fp8_gemm_mx"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code, name in enumerate(["FP8_OK", "FP8_ERR_INVALID_ARG", "FP8_ERR_ALIGNMENT", "FP8_ERR_UNSUPPORTED_SHAPE",
                                 "FP8_ERR_WORKSPACE", "FP8_ERR_CUDA", "FP8_ERR_TIMEOUT"]):
        assert fb.status_string(code) == name
    assert fb.status_string(99) == "FP8_ERR_UNKNOWN"


@pytest.mark.parametrize("rows,cols", [(1, 128), (130, 640), (300, 1024), (0, 128)])
@pytest.mark.parametrize("gran", [0, 1, 2, 3, 4, 5])
def test_scales_bytes_match_oracle_layout(L, rows, cols, gran):
    layouts = [fb.SF_LINEAR, fb.SF_TCGEN05] if gran == fb.MX32 else [fb.SF_LINEAR]
    for lay in layouts:
        dt, n = oracle.scales_shape(rows, cols, gran, lay)
        assert fb.scales_bytes(rows, cols, gran, lay) == n * np.dtype(dt).itemsize


def test_scales_bytes_invalid(L):
    assert fb.scales_bytes(4, 100, fb.TILE_1x128) == 0
    assert fb.scales_bytes(4, 48, fb.MX32) == 0
    assert fb.scales_bytes(-1, 128, fb.TOKEN) == 0
    assert fb.workspace_bytes(10, 128, fb.TENSOR) == 256
    assert fb.workspace_bytes(10, 128, fb.TOKEN) == 0


P = ctypes.c_void_p
A16 = P(0x100000)  # fake device addresses: checks fail before any dereference
A16b = P(0x200000)
MIS = P(0x100001)


def _q(L, x=A16, rows=8, cols=128, ldx=128, fmt=0, gran=1, lay=0, st=None, q=A16b, ldq=128, sc=A16, ws=None,
       wsb=0):
    return L.fp8_quantize(x, rows, cols, ldx, fmt, gran, lay, st, q, ldq, sc, ws, wsb, None)


def test_quantize_refusals(L):
    n0 = fb.launch_count()
    assert _q(L, rows=0) == fb.OK  # empty: nothing enqueued
    assert _q(L, fmt=7) == fb.ERR_INVALID_ARG
    assert _q(L, gran=9) == fb.ERR_INVALID_ARG
    assert _q(L, lay=1) == fb.ERR_INVALID_ARG  # tiled SF only for MX32
    assert _q(L, st=A16) == fb.ERR_INVALID_ARG  # static scale only per-tensor
    assert _q(L, x=None) == fb.ERR_INVALID_ARG
    assert _q(L, q=None) == fb.ERR_INVALID_ARG
    assert _q(L, sc=None) == fb.ERR_INVALID_ARG
    assert _q(L, cols=120, ldx=128, ldq=128) == fb.ERR_UNSUPPORTED_SHAPE  # % 16
    assert _q(L, gran=2, cols=144, ldx=144, ldq=144) == fb.ERR_UNSUPPORTED_SHAPE  # % 128
    assert _q(L, gran=4, cols=48, ldx=48, ldq=48) == fb.ERR_UNSUPPORTED_SHAPE  # % 32
    assert _q(L, gran=3, rows=65535 * 128 + 1) == fb.ERR_UNSUPPORTED_SHAPE  # 128x128 row blocks > grid y limit
    assert _q(L, gran=3, rows=65535 * 128, sc=None) == fb.ERR_INVALID_ARG  # the largest accepted row count
    assert _q(L, ldx=64) == fb.ERR_INVALID_ARG  # ld < cols
    assert _q(L, x=MIS) == fb.ERR_ALIGNMENT
    assert _q(L, q=MIS) == fb.ERR_ALIGNMENT
    assert _q(L, ldx=132) == fb.ERR_ALIGNMENT
    assert _q(L, ldq=136) == fb.ERR_ALIGNMENT
    assert _q(L, gran=0) == fb.ERR_WORKSPACE  # dynamic per-tensor needs workspace
    assert _q(L, gran=0, ws=A16, wsb=16) == fb.ERR_WORKSPACE
    assert _q(L, gran=5) == fb.ERR_WORKSPACE  # per-channel needs cols*4 bytes of workspace
    assert _q(L, gran=5, ws=A16, wsb=256) == fb.ERR_WORKSPACE  # 128 cols -> 512 bytes
    assert fb.workspace_bytes(8, 128, fb.CHANNEL) == 512
    d = L.fp8_quantize_delayed
    assert d(A16, 8, 128, 128, 0, A16, 4, 4, 0, A16b, 128, A16, None) == fb.ERR_INVALID_ARG  # slot >= len
    assert d(A16, 8, 128, 128, 0, A16, 4, 0, 200, A16b, 128, A16, None) == fb.ERR_INVALID_ARG  # margin
    assert d(A16, 8, 128, 128, 0, None, 4, 0, 0, A16b, 128, A16, None) == fb.ERR_INVALID_ARG
    assert d(A16, 8, 120, 128, 0, A16, 4, 0, 0, A16b, 128, A16, None) == fb.ERR_UNSUPPORTED_SHAPE
    assert d(A16, 0, 128, 128, 0, A16, 4, 0, 0, A16b, 128, A16, None) == fb.OK
    assert fb.launch_count() == n0


def test_dequantize_refusals(L):
    n0 = fb.launch_count()
    d = L.fp8_dequantize
    assert d(A16, 0, 128, 128, 0, 1, 0, A16, A16b, 128, None) == fb.OK
    assert d(A16, 8, 128, 128, 3, 1, 0, A16, A16b, 128, None) == fb.ERR_INVALID_ARG
    assert d(None, 8, 128, 128, 0, 1, 0, A16, A16b, 128, None) == fb.ERR_INVALID_ARG
    assert d(MIS, 8, 128, 128, 0, 1, 0, A16, A16b, 128, None) == fb.ERR_ALIGNMENT
    assert d(A16, 8, 100, 112, 0, 2, 0, A16, A16b, 128, None) == fb.ERR_UNSUPPORTED_SHAPE
    assert fb.launch_count() == n0


def _g(L, a=A16, sa=A16, ga=2, b=A16b, sb=A16, gb=3, fa=0, fw=0, o=A16, m=16, n=16, k=128, st=None):
    return L.fp8_gemm_blockscaled(a, sa, ga, b, sb, gb, fa, fw, o, m, n, k, st, None)


def test_gemm_refusals(L):
    n0 = fb.launch_count()
    assert _g(L, m=0) == fb.OK
    assert _g(L, ga=3, gb=2) == fb.ERR_INVALID_ARG  # not a valid scale pair
    assert _g(L, ga=2, gb=1) == fb.ERR_INVALID_ARG
    assert _g(L, ga=4, gb=4) == fb.ERR_INVALID_ARG  # MX has its own entry point
    assert _g(L, ga=5, gb=0) == fb.ERR_INVALID_ARG  # per-channel scales do not factor out of K
    qo = L.fp8_gemm_blockscaled_quantized_out
    assert qo(A16, A16, A16b, A16, 0, 0, 0, A16, A16, 16, 144, 128, None, None) == fb.ERR_UNSUPPORTED_SHAPE
    assert qo(A16, A16, A16b, A16, 0, 0, 3, A16, A16, 16, 128, 128, None, None) == fb.ERR_INVALID_ARG
    assert qo(A16, A16, A16b, A16, 0, 0, 0, A16, None, 16, 128, 128, None, None) == fb.ERR_INVALID_ARG
    assert _g(L, fa=5) == fb.ERR_INVALID_ARG
    assert _g(L, n=24) == fb.ERR_UNSUPPORTED_SHAPE  # N % 16
    assert _g(L, k=144) == fb.ERR_UNSUPPORTED_SHAPE  # fold needs K % 128
    assert _g(L, ga=0, gb=0, k=24) == fb.ERR_UNSUPPORTED_SHAPE  # K % 16
    assert _g(L, k=0) == fb.ERR_UNSUPPORTED_SHAPE
    assert _g(L, a=None) == fb.ERR_INVALID_ARG
    assert _g(L, sa=None) == fb.ERR_INVALID_ARG
    assert _g(L, a=MIS) == fb.ERR_ALIGNMENT
    assert _g(L, o=MIS) == fb.ERR_ALIGNMENT
    assert _g(L, st=MIS) == fb.ERR_ALIGNMENT
    assert _g(L, m=1 << 31) == fb.ERR_UNSUPPORTED_SHAPE
    mx = L.fp8_gemm_mx
    assert mx(A16, A16, A16b, A16, 0, 0, A16, 16, 16, 48, None, None) == fb.ERR_UNSUPPORTED_SHAPE  # K % 32
    assert mx(A16, None, A16b, A16, 0, 0, A16, 16, 16, 64, None, None) == fb.ERR_INVALID_ARG
    assert mx(A16, MIS, A16b, A16, 0, 0, A16, 16, 16, 64, None, None) == fb.ERR_ALIGNMENT
    assert L.fp8_debug_wait_probe(None, 1000, None) == fb.ERR_INVALID_ARG
    assert L.fp8_debug_wait_probe(A16, 0, None) == fb.ERR_INVALID_ARG
    assert L.fp8_debug_encode_f32(A16, 12, 0, A16b, None) == fb.ERR_INVALID_ARG
    assert fb.launch_count() == n0


def test_gemm_wait_limit_refusals(L):
    n0 = fb.launch_count()
    g = L.fp8_debug_gemm_blockscaled_wait_limit
    assert g(A16, A16, 2, A16b, A16, 3, 0, 0, A16, 16, 16, 128, None, 1000, None) == fb.ERR_INVALID_ARG  # no status
    assert g(A16, A16, 2, A16b, A16, 3, 0, 0, A16, 16, 16, 128, A16, 0, None) == fb.ERR_INVALID_ARG  # limit 0
    assert g(A16, A16, 2, A16b, A16, 3, 0, 0, A16, 16, 16, 144, A16, 1000, None) == fb.ERR_UNSUPPORTED_SHAPE
    m = L.fp8_debug_gemm_mx_wait_limit
    assert m(A16, A16, A16b, A16, 0, 0, A16, 16, 16, 64, A16, 10 ** 10 + 1, None) == fb.ERR_INVALID_ARG
    assert m(A16, A16, A16b, A16, 0, 0, A16, 16, 16, 48, A16, 1000, None) == fb.ERR_UNSUPPORTED_SHAPE
    assert fb.launch_count() == n0


def test_nvfp4_scales_bytes(L):
    # linear: one byte per 16 elements; tiled: 512-byte atoms of 128 rows x 4 groups, padded
    assert fb.nvfp4_scales_bytes(130, 272, fb.SF_LINEAR) == 130 * 17
    assert fb.nvfp4_scales_bytes(130, 272, fb.SF_TCGEN05) == 2 * 5 * 512
    assert fb.nvfp4_scales_bytes(128, 64, fb.SF_TCGEN05) == 512
    for rows, cols in [(1, 16), (257, 1024), (300, 4096)]:
        assert fb.nvfp4_scales_bytes(rows, cols, fb.SF_TCGEN05) == oracle.mx_tiled_bytes(rows, cols // 16)
    assert fb.nvfp4_scales_bytes(4, 40, fb.SF_LINEAR) == 0   # cols % 16
    assert fb.nvfp4_scales_bytes(-1, 16, fb.SF_LINEAR) == 0
    assert fb.nvfp4_scales_bytes(4, 16, 7) == 0


def _q4(L, x=A16, rows=8, cols=128, ldx=128, lay=1, st=None, q=A16b, ldq=64, sf=A16, ts=A16, ws=A16, wsb=256):
    return L.fp8_quantize_nvfp4(x, rows, cols, ldx, lay, st, q, ldq, sf, ts, ws, wsb, None)


def test_nvfp4_refusals(L):
    n0 = fb.launch_count()
    assert _q4(L, rows=0) == fb.OK
    assert _q4(L, lay=5) == fb.ERR_INVALID_ARG
    assert _q4(L, cols=120, ldx=128) == fb.ERR_UNSUPPORTED_SHAPE  # % 16
    assert _q4(L, x=None) == fb.ERR_INVALID_ARG
    assert _q4(L, sf=None) == fb.ERR_INVALID_ARG
    assert _q4(L, ts=None) == fb.ERR_INVALID_ARG
    assert _q4(L, ldq=32) == fb.ERR_INVALID_ARG  # ld_q < cols / 2
    assert _q4(L, x=MIS) == fb.ERR_ALIGNMENT
    assert _q4(L, ldx=132) == fb.ERR_ALIGNMENT
    assert _q4(L, ldq=68) == fb.ERR_ALIGNMENT
    assert _q4(L, ws=None) == fb.ERR_WORKSPACE  # two-pass needs the amax workspace
    assert _q4(L, wsb=16) == fb.ERR_WORKSPACE
    assert _q4(L, st=MIS, ws=None) == fb.ERR_ALIGNMENT  # static s_t: no workspace, aligned float
    d = L.fp8_dequantize_nvfp4
    assert d(A16, 0, 128, 64, 0, A16, A16, A16b, 128, None) == fb.OK
    assert d(A16, 8, 128, 64, 3, A16, A16, A16b, 128, None) == fb.ERR_INVALID_ARG
    assert d(A16, 8, 100, 64, 0, A16, A16, A16b, 128, None) == fb.ERR_UNSUPPORTED_SHAPE
    assert d(A16, 8, 128, 64, 0, None, A16, A16b, 128, None) == fb.ERR_INVALID_ARG
    assert d(A16, 8, 128, 64, 0, A16, A16, MIS, 128, None) == fb.ERR_ALIGNMENT
    g = L.fp8_gemm_nvfp4
    assert g(A16, A16, A16, A16b, A16, A16, A16, 0, 16, 256, None, None) == fb.OK
    assert g(A16, A16, A16, A16b, A16, A16, A16, 16, 16, 128, None, None) == fb.ERR_UNSUPPORTED_SHAPE  # K % 256
    assert g(A16, A16, A16, A16b, A16, A16, A16, 16, 24, 256, None, None) == fb.ERR_UNSUPPORTED_SHAPE  # N % 16
    assert g(A16, None, A16, A16b, A16, A16, A16, 16, 16, 256, None, None) == fb.ERR_INVALID_ARG
    assert g(A16, A16, None, A16b, A16, A16, A16, 16, 16, 256, None, None) == fb.ERR_INVALID_ARG
    assert g(A16, MIS, A16, A16b, A16, A16, A16, 16, 16, 256, None, None) == fb.ERR_ALIGNMENT
    assert g(A16, A16, A16, A16b, A16, A16, A16, 16, 16, 256, MIS, None) == fb.ERR_ALIGNMENT
    p = L.fp8_debug_gemm_blockscaled_pairs
    assert p(A16, A16, A16b, A16, 0, 0, A16, 16, 16, 144, None, None) == fb.ERR_UNSUPPORTED_SHAPE  # K % 128
    assert p(A16, None, A16b, A16, 0, 0, A16, 16, 16, 128, None, None) == fb.ERR_INVALID_ARG
    assert p(A16, MIS, A16b, A16, 0, 0, A16, 16, 16, 128, None, None) == fb.ERR_ALIGNMENT
    assert p(A16, A16, A16b, A16, 0, 0, A16, 0, 16, 128, None, None) == fb.OK
    e = L.fp8_debug_encode_e2m1_f32
    assert e(A16, 12, A16b, None) == fb.ERR_INVALID_ARG
    assert e(MIS, 16, A16b, None) == fb.ERR_ALIGNMENT
    assert e(A16, 0, A16b, None) == fb.OK
    assert fb.launch_count() == n0


def test_binding_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(fb, "_lib", None)
    monkeypatch.setattr(fb, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libfp8bs.so"))
    with pytest.raises(RuntimeError, match="not built"):
        fb.lib()


def test_oracle_and_cuda_path_share_no_code():
    csrc = os.path.join(ROOT, "fp8_block_scaled_04_gb300", "csrc")
    for f in os.listdir(csrc):
        text = open(os.path.join(csrc, f)).read()
        assert "oracle" not in text.lower(), f
    text = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    assert not re.search(r'#include\s+"', text)  # only system headers
    pkg = os.path.join(ROOT, "fp8_block_scaled_04_gb300")
    for f in os.listdir(pkg):
        if f.endswith(".py"):
            src = open(os.path.join(pkg, f)).read()
            assert not re.search(r"^\s*(from|import)\s+oracle", src, re.M), f

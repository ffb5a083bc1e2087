"""CPU oracle for FP8 quantization and scaled FP8 GEMM (numpy wrapper over liboracle.so).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. It shares no code with the CUDA library and never imports it.

Parity status: every function here is pinned by a CPU test (see
``tests/test_oracle_*.py``) against values printed on the source pages,
closed forms, library routines (torch float8 casts, numpy matmul) or brute
force. The MX shared-exponent rounding rule is a reading (the pages do not
state it); its pins are the closed-form properties of that reading.
"""
import ctypes
import os

import numpy as np

from . import build as _build

E4M3, E5M2 = 0, 1
TENSOR, TOKEN, TILE_1x128, BLOCK_128x128, MX32, CHANNEL = 0, 1, 2, 3, 4, 5
SF_LINEAR, SF_TILED = 0, 1

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        c_i64, c_u64, c_int, vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p
        L.orc_decode.restype = ctypes.c_double
        L.orc_decode.argtypes = [ctypes.c_uint32, c_int]
        L.orc_encode_nearest.restype = ctypes.c_uint8
        L.orc_encode_nearest.argtypes = [ctypes.c_float, c_int]
        L.orc_encode_binade.restype = ctypes.c_uint8
        L.orc_encode_binade.argtypes = [ctypes.c_float, c_int]
        L.orc_encoders_disagree.restype = c_i64
        L.orc_encoders_disagree.argtypes = [c_u64, c_u64, c_int, c_int, ctypes.POINTER(c_u64)]
        L.orc_check_codes.restype = c_i64
        L.orc_check_codes.argtypes = [c_u64, c_u64, c_int, vp, c_int, ctypes.POINTER(c_u64)]
        L.orc_encode_array.restype = None
        L.orc_encode_array.argtypes = [vp, c_i64, c_int, vp]
        L.orc_decode_array.restype = None
        L.orc_decode_array.argtypes = [vp, c_i64, c_int, vp]
        L.orc_is_nan_code.restype = c_int
        L.orc_is_nan_code.argtypes = [ctypes.c_uint32, c_int]
        L.orc_fmt_max.restype = ctypes.c_double
        L.orc_fmt_max.argtypes = [c_int]
        L.orc_mx_exponent.restype = c_int
        L.orc_mx_exponent.argtypes = [ctypes.c_float, c_int]
        L.orc_mx_tiled_offset.restype = c_i64
        L.orc_mx_tiled_offset.argtypes = [c_i64, c_i64, c_i64, c_i64]
        L.orc_mx_tiled_bytes.restype = c_i64
        L.orc_mx_tiled_bytes.argtypes = [c_i64, c_i64]
        L.orc_bf16_to_f32.restype = ctypes.c_float
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_f32_to_bf16.restype = ctypes.c_uint16
        L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
        L.orc_quantize.restype = c_int
        L.orc_quantize.argtypes = [vp, c_i64, c_i64, c_i64, c_int, c_int, c_int, vp, vp, c_i64, vp, c_int]
        L.orc_dequantize.restype = c_int
        L.orc_dequantize.argtypes = [vp, c_i64, c_i64, c_i64, c_int, c_int, c_int, vp, vp, c_i64, c_int]
        L.orc_gemm.restype = c_int
        L.orc_gemm.argtypes = [vp, c_i64, vp, c_int, c_int, c_int, vp, c_i64, vp, c_int, c_int, c_int,
                               c_i64, c_i64, c_i64, vp, c_i64, vp, c_i64, vp, vp, c_int]
        L.orc_quantize_delayed.restype = c_int
        L.orc_quantize_delayed.argtypes = [vp, c_i64, c_i64, c_int, vp, c_int, c_int, c_int, vp, vp, vp, c_int]
        L.orc_default_threads.restype = c_int
        L.orc_default_threads.argtypes = []
        L.orc_e2m1_decode.restype = ctypes.c_double
        L.orc_e2m1_decode.argtypes = [ctypes.c_uint32]
        L.orc_e2m1_encode_nearest.restype = ctypes.c_uint8
        L.orc_e2m1_encode_nearest.argtypes = [ctypes.c_float]
        L.orc_e2m1_encode_binade.restype = ctypes.c_uint8
        L.orc_e2m1_encode_binade.argtypes = [ctypes.c_float]
        L.orc_e2m1_encoders_disagree.restype = c_i64
        L.orc_e2m1_encoders_disagree.argtypes = [c_u64, c_u64, c_int, ctypes.POINTER(c_u64)]
        L.orc_e2m1_check_codes.restype = c_i64
        L.orc_e2m1_check_codes.argtypes = [c_u64, c_u64, vp, c_int, ctypes.POINTER(c_u64)]
        L.orc_nvfp4_tensor_scale.restype = ctypes.c_float
        L.orc_nvfp4_tensor_scale.argtypes = [ctypes.c_float]
        L.orc_quantize_nvfp4.restype = c_int
        L.orc_quantize_nvfp4.argtypes = [vp, c_i64, c_i64, c_i64, c_int, vp, vp, vp, vp]
        L.orc_dequantize_nvfp4.restype = c_int
        L.orc_dequantize_nvfp4.argtypes = [vp, vp, c_int, ctypes.c_float, c_i64, c_i64, vp]
        L.orc_gemm_nvfp4.restype = c_int
        L.orc_gemm_nvfp4.argtypes = [vp, vp, ctypes.c_float, vp, vp, ctypes.c_float, c_int, c_i64, c_i64, c_i64,
                                     vp, c_i64, vp, c_i64, vp, vp]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return lib().orc_default_threads()


# --------------------------------------------------------------------- codec
def decode(codes, fmt: int) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().orc_decode_array(_p(c), c.size, fmt, _p(out))
    return out


def encode(x, fmt: int) -> np.ndarray:
    """Nearest-value encoder (ties to even, saturating) applied to fp32 inputs."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint8)
    lib().orc_encode_array(_p(f), f.size, fmt, _p(out))
    return out


def encode_nearest(x: float, fmt: int) -> int:
    return int(lib().orc_encode_nearest(float(np.float32(x)), fmt))


def encode_binade(x: float, fmt: int) -> int:
    return int(lib().orc_encode_binade(float(np.float32(x)), fmt))


def encoders_disagree(start: int, count: int, fmt: int, nthreads: int = 0):
    first = ctypes.c_uint64(0)
    bad = lib().orc_encoders_disagree(start, count, fmt, nthreads, ctypes.byref(first))
    return int(bad), int(first.value)


def check_codes(start: int, codes: np.ndarray, fmt: int, nthreads: int = 0):
    """Count entries of ``codes`` that differ from encode(float32 bit pattern start+i)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    first = ctypes.c_uint64(0)
    bad = lib().orc_check_codes(start, c.size, fmt, _p(c), nthreads, ctypes.byref(first))
    return int(bad), int(first.value)


def is_nan_code(code: int, fmt: int) -> bool:
    return bool(lib().orc_is_nan_code(code, fmt))


def fmt_max(fmt: int) -> float:
    return float(lib().orc_fmt_max(fmt))


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x) -> np.ndarray:
    f = np.ascontiguousarray(x, dtype=np.float32).ravel()
    L = lib()
    return np.array([L.orc_f32_to_bf16(float(v)) for v in f], dtype=np.uint16).reshape(np.shape(x))


# ------------------------------------------------------------ scale layouts
def mx_exponent(amax: float, fmt: int) -> int:
    return int(lib().orc_mx_exponent(float(np.float32(amax)), fmt))


def mx_tiled_offset(r: int, j: int, rows: int, ngroups: int) -> int:
    return int(lib().orc_mx_tiled_offset(r, j, rows, ngroups))


def mx_tiled_bytes(rows: int, ngroups: int) -> int:
    return int(lib().orc_mx_tiled_bytes(rows, ngroups))


def scales_shape(rows: int, cols: int, gran: int, sf_layout: int = SF_LINEAR):
    """(numpy dtype, element count) of the scale array of one quantized operand."""
    if gran == TENSOR:
        return np.float32, 1
    if gran == TOKEN:
        return np.float32, rows
    if gran == TILE_1x128:
        return np.float32, (cols // 128) * rows
    if gran == BLOCK_128x128:
        return np.float32, ((rows + 127) // 128) * (cols // 128)
    if gran == CHANNEL:
        return np.float32, cols
    if gran == MX32:
        if sf_layout == SF_TILED:
            return np.uint8, mx_tiled_bytes(rows, cols // 32)
        return np.uint8, rows * (cols // 32)
    raise ValueError(gran)


# -------------------------------------------------------------- quantizers
def quantize(x_bf16: np.ndarray, fmt: int, gran: int, sf_layout: int = SF_LINEAR, static_scale=None,
             nthreads: int = 0):
    """x_bf16: uint16 array [rows, cols] (bf16 bit patterns). Returns (q uint8 [rows, cols], scales)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, cols = x.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    dt, n = scales_shape(rows, cols, gran, sf_layout)
    sc = np.zeros(max(n, 1), dtype=dt)
    ss = None if static_scale is None else np.array([static_scale], dtype=np.float32)
    rc = lib().orc_quantize(_p(x), rows, cols, cols, fmt, gran, sf_layout, _p(ss), _p(q), cols, _p(sc), nthreads)
    if rc != 0:
        raise ValueError("oracle quantize rejected the arguments (rc=%d)" % rc)
    return q, sc[:n]


def quantize_delayed(x_bf16: np.ndarray, fmt: int, history, slot: int, margin: int = 0, nthreads: int = 0):
    """Per-tensor quantization with the scale taken from an amax history.

    Returns (q, scale, new_history) where new_history[slot] = amax(x).
    """
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, cols = x.shape
    h = np.ascontiguousarray(history, dtype=np.float32)
    q = np.empty((rows, cols), dtype=np.uint8)
    s = np.zeros(1, dtype=np.float32)
    nh = np.empty_like(h)
    rc = lib().orc_quantize_delayed(_p(x), rows, cols, fmt, _p(h), h.size, slot, margin, _p(q), _p(s), _p(nh),
                                    nthreads)
    if rc != 0:
        raise ValueError("oracle quantize_delayed rejected the arguments (rc=%d)" % rc)
    return q, s, nh


def dequantize(q: np.ndarray, scales: np.ndarray, fmt: int, gran: int, sf_layout: int = SF_LINEAR,
               nthreads: int = 0) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    rows, cols = q.shape
    dt, n = scales_shape(rows, cols, gran, sf_layout)
    sc = np.ascontiguousarray(scales, dtype=dt)
    out = np.empty((rows, cols), dtype=np.uint16)
    rc = lib().orc_dequantize(_p(q), rows, cols, cols, fmt, gran, sf_layout, _p(sc), _p(out), cols, nthreads)
    if rc != 0:
        raise ValueError("oracle dequantize rejected the arguments")
    return out


# -------------------------------------------------------------------- GEMM
def gemm(a_q, a_scales, a_gran, b_q, b_scales, b_gran, a_fmt=E4M3, b_fmt=E4M3, a_sf=SF_LINEAR,
         b_sf=SF_LINEAR, rows=None, cols=None, nthreads: int = 0):
    """fp64 reference of Out = X_hat @ W_hat^T and the bound sum_k |x_hat * w_hat|.

    a_q: uint8 [M, K]; b_q: uint8 [N, K]. rows / cols select output entries.
    Returns (ref, bound), each float64 [len(rows), len(cols)].
    """
    a = np.ascontiguousarray(a_q, dtype=np.uint8)
    b = np.ascontiguousarray(b_q, dtype=np.uint8)
    M, K = a.shape
    N, K2 = b.shape
    assert K == K2
    adt, _ = scales_shape(M, K, a_gran, a_sf)
    bdt, _ = scales_shape(N, K, b_gran, b_sf)
    sa = np.ascontiguousarray(a_scales, dtype=adt)
    sb = np.ascontiguousarray(b_scales, dtype=bdt)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = M if r is None else r.size
    nc = N if c is None else c.size
    ref = np.empty((nr, nc), dtype=np.float64)
    bound = np.empty((nr, nc), dtype=np.float64)
    rc = lib().orc_gemm(_p(a), K, _p(sa), a_gran, a_sf, a_fmt, _p(b), K, _p(sb), b_gran, b_sf, b_fmt, M, N, K,
                        _p(r), nr, _p(c), nc, _p(ref), _p(bound), nthreads)
    if rc != 0:
        raise ValueError("oracle gemm failed (rc=%d)" % rc)
    return ref, bound


# ---------------------------------------------------------------- NVFP4
# "Low precision: FP8, FP4, and microscaling": blocks of 16, E4M3 microscale
# per block, one fp32 scale per tensor. Element format and scale arithmetic
# are readings stated in oracle.c (NVFP4 section).
def e2m1_decode(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint32).ravel()
    return np.array([lib().orc_e2m1_decode(int(v)) for v in c], dtype=np.float64).reshape(np.shape(codes))


def e2m1_encode_nearest(x: float) -> int:
    return int(lib().orc_e2m1_encode_nearest(float(x)))


def e2m1_encode_binade(x: float) -> int:
    return int(lib().orc_e2m1_encode_binade(float(x)))


def e2m1_encoders_disagree(start: int, count: int, nthreads: int = 0):
    first = ctypes.c_uint64(0)
    bad = lib().orc_e2m1_encoders_disagree(start, count, nthreads, ctypes.byref(first))
    return int(bad), int(first.value)


def e2m1_check_codes(start: int, codes: np.ndarray, nthreads: int = 0):
    """(mismatches, first mismatching fp32 pattern) of E2M1 codes for patterns start.. ."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    first = ctypes.c_uint64(0)
    bad = lib().orc_e2m1_check_codes(start, c.size, _p(c), nthreads, ctypes.byref(first))
    return int(bad), int(first.value)


def nvfp4_tensor_scale(amax: float) -> float:
    return float(lib().orc_nvfp4_tensor_scale(float(amax)))


def quantize_nvfp4(x_bf16: np.ndarray, sf_layout: int = SF_TILED, static_tensor_scale=None):
    """x: uint16 bf16 bits [rows x cols], cols % 16 == 0. Returns (q [rows x cols/2] uint8,
    sf uint8 E4M3 codes (tiled or linear [rows][cols/16]), tensor scale float)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, cols = x.shape
    q = np.zeros((rows, cols // 2), dtype=np.uint8)
    ng = cols // 16
    sf = np.zeros(mx_tiled_bytes(rows, ng) if sf_layout == SF_TILED else rows * ng, dtype=np.uint8)
    st = np.zeros(1, dtype=np.float32)
    stat = None if static_tensor_scale is None else np.array([static_tensor_scale], dtype=np.float32)
    rc = lib().orc_quantize_nvfp4(_p(x), rows, cols, cols, sf_layout, _p(stat), _p(q), _p(sf), _p(st))
    if rc != 0:
        raise ValueError("orc_quantize_nvfp4 failed: %d" % rc)
    return q, sf, float(st[0])


def dequantize_nvfp4(q, sf, tensor_scale: float, cols: int, sf_layout: int = SF_TILED) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    rows = q.shape[0]
    out = np.zeros((rows, cols), dtype=np.uint16)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    rc = lib().orc_dequantize_nvfp4(_p(q), _p(sf), sf_layout, float(tensor_scale), rows, cols, _p(out))
    if rc != 0:
        raise ValueError("orc_dequantize_nvfp4 failed: %d" % rc)
    return out


def gemm_nvfp4(a_q, a_sf, a_ts, b_q, b_sf, b_ts, sf_layout: int = SF_TILED, rows=None, cols=None):
    """fp64 reference and bound of X_hat W_hat^T for NVFP4 operands (packed [M x K/2], [N x K/2])."""
    a_q = np.ascontiguousarray(a_q, dtype=np.uint8)
    b_q = np.ascontiguousarray(b_q, dtype=np.uint8)
    M, K = a_q.shape[0], a_q.shape[1] * 2
    N = b_q.shape[0]
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = M if r is None else len(r)
    nc = N if c is None else len(c)
    ref = np.zeros((nr, nc), dtype=np.float64)
    bound = np.zeros((nr, nc), dtype=np.float64)
    rc = lib().orc_gemm_nvfp4(_p(a_q), _p(np.ascontiguousarray(a_sf, dtype=np.uint8)), float(a_ts), _p(b_q),
                              _p(np.ascontiguousarray(b_sf, dtype=np.uint8)), float(b_ts), sf_layout, M, N, K,
                              _p(r), nr, _p(c), nc, _p(ref), _p(bound))
    if rc != 0:
        raise ValueError("orc_gemm_nvfp4 failed: %d" % rc)
    return ref, bound

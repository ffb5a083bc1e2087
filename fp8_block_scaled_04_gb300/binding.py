"""Thin ctypes binding over libfp8bs.so (argument marshalling only).

Every computation runs in the library's CUDA kernels; torch supplies device
memory (tensors) and the current stream. There is no CPU path: if the library
is not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfp8bs.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "fp8bs.h")

E4M3, E5M2 = 0, 1
TENSOR, TOKEN, TILE_1x128, BLOCK_128x128, MX32, CHANNEL = 0, 1, 2, 3, 4, 5
SF_LINEAR, SF_TCGEN05, SF_TCGEN05_X4 = 0, 1, 2
OK, ERR_INVALID_ARG, ERR_ALIGNMENT, ERR_UNSUPPORTED_SHAPE, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(7)

_lib = None


class Fp8Error(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__("%s failed: %s" % (what, status_string(code)))


CHECK_LIB_PATH = os.path.join(HERE, "libfp8bs_check.so")


def lib():
    """Load libfp8bs.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        _lib = load(LIB_PATH)
    return _lib


def load(path: str):
    """A ctypes handle on a build of the library at `path`, signatures declared."""
    if not os.path.exists(path):
        raise RuntimeError("%s is not built; run __graft_entry__.build()" % path)
    L = ctypes.CDLL(path)
    i64, u64, i32, vp, sz = ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
    L.fp8_status_string.restype = ctypes.c_char_p
    L.fp8_status_string.argtypes = [i32]
    L.fp8_scales_bytes.restype = sz
    L.fp8_scales_bytes.argtypes = [i64, i64, i32, i32]
    L.fp8_quantize_workspace_bytes.restype = sz
    L.fp8_quantize_workspace_bytes.argtypes = [i64, i64, i32]
    L.fp8_quantize.restype = i32
    L.fp8_quantize.argtypes = [vp, i64, i64, i64, i32, i32, i32, vp, vp, i64, vp, vp, sz, vp]
    L.fp8_quantize_tensor_noalloc.restype = i32
    L.fp8_quantize_tensor_noalloc.argtypes = [vp, i64, i64, i64, i32, vp, i64, vp, vp]
    L.fp8_quantize_delayed.restype = i32
    L.fp8_quantize_delayed.argtypes = [vp, i64, i64, i64, i32, vp, i32, i32, i32, vp, i64, vp, vp]
    L.fp8_dequantize.restype = i32
    L.fp8_dequantize.argtypes = [vp, i64, i64, i64, i32, i32, i32, vp, vp, i64, vp]
    L.fp8_gemm_blockscaled.restype = i32
    L.fp8_gemm_blockscaled.argtypes = [vp, vp, i32, vp, vp, i32, i32, i32, vp, i64, i64, i64, vp, vp]
    L.fp8_gemm_blockscaled_quantized_out.restype = i32
    L.fp8_gemm_blockscaled_quantized_out.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, vp, i64, i64, i64, vp, vp]
    L.fp8_gemm_mx.restype = i32
    L.fp8_gemm_mx.argtypes = [vp, vp, vp, vp, i32, i32, vp, i64, i64, i64, vp, vp]
    L.fp8_gemm_mx_x4.restype = i32
    L.fp8_gemm_mx_x4.argtypes = [vp, vp, vp, vp, i32, i32, vp, i64, i64, i64, vp, vp]
    L.fp8_nvfp4_scales_bytes.restype = sz
    L.fp8_nvfp4_scales_bytes.argtypes = [i64, i64, i32]
    L.fp8_quantize_nvfp4.restype = i32
    L.fp8_quantize_nvfp4.argtypes = [vp, i64, i64, i64, i32, vp, vp, i64, vp, vp, vp, sz, vp]
    L.fp8_dequantize_nvfp4.restype = i32
    L.fp8_dequantize_nvfp4.argtypes = [vp, i64, i64, i64, i32, vp, vp, vp, i64, vp]
    L.fp8_gemm_nvfp4.restype = i32
    L.fp8_gemm_nvfp4.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, vp, vp]
    L.fp8_debug_gemm_mx_pairs.restype = i32
    L.fp8_debug_gemm_mx_pairs.argtypes = [vp, vp, vp, vp, i32, i32, vp, i64, i64, i64, vp, vp]
    L.fp8_debug_gemm_mx_single.restype = i32
    L.fp8_debug_gemm_mx_single.argtypes = [vp, vp, vp, vp, i32, i32, vp, i64, i64, i64, vp, vp]
    L.fp8_debug_gemm_blockscaled_pairs.restype = i32
    L.fp8_debug_gemm_blockscaled_pairs.argtypes = [vp, vp, vp, vp, i32, i32, vp, i64, i64, i64, vp, vp]
    L.fp8_debug_encode_e2m1_f32.restype = i32
    L.fp8_debug_encode_e2m1_f32.argtypes = [vp, i64, vp, vp]
    L.fp8_debug_encode_f32.restype = i32
    L.fp8_debug_encode_f32.argtypes = [vp, i64, i32, vp, vp]
    L.fp8_debug_gemm_blockscaled_wait_limit.restype = i32
    L.fp8_debug_gemm_blockscaled_wait_limit.argtypes = [vp, vp, i32, vp, vp, i32, i32, i32, vp, i64, i64, i64, vp,
                                                         u64, vp]
    L.fp8_debug_gemm_mx_wait_limit.restype = i32
    L.fp8_debug_gemm_mx_wait_limit.argtypes = [vp, vp, vp, vp, i32, i32, vp, i64, i64, i64, vp, u64, vp]
    L.fp8_debug_wait_probe.restype = i32
    L.fp8_debug_wait_probe.argtypes = [vp, u64, vp]
    L.fp8_launch_count.restype = u64
    L.fp8_launch_count.argtypes = []
    L.fp8_debug_oob_read.restype = u64
    L.fp8_debug_oob_read.argtypes = []
    L.fp8_debug_checked_build.restype = i32
    L.fp8_debug_checked_build.argtypes = []
    return L


def declared_functions() -> list[str]:
    """Names of the functions include/fp8bs.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8_[a-z0-9_]+)\s*\(", text)))


def status_string(code: int) -> str:
    return lib().fp8_status_string(int(code)).decode()


def launch_count() -> int:
    return int(lib().fp8_launch_count())


def scales_bytes(rows: int, cols: int, gran: int, sf_layout: int = SF_LINEAR) -> int:
    return int(lib().fp8_scales_bytes(rows, cols, gran, sf_layout))


def workspace_bytes(rows: int, cols: int, gran: int) -> int:
    return int(lib().fp8_quantize_workspace_bytes(rows, cols, gran))


def _check(rc: int, what: str):
    if rc != OK:
        raise Fp8Error(rc, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


_default_status = {}


def default_status(device=None):
    """The status word the GEMM wrappers pass when the caller gives none: one zeroed
    int32 per device, allocated on first use. A bounded wait that expires inside a
    kernel writes FP8_ERR_TIMEOUT there (the library never clears it); read it with
    check_status() after the work has completed."""
    import torch

    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    key = dev.index if dev.index is not None else torch.cuda.current_device()
    s = _default_status.get(key)
    if s is None:
        s = torch.zeros(1, dtype=torch.int32, device=torch.device("cuda", key))
        _default_status[key] = s
    return s


def check_status(status=None, device=None):
    """Synchronise the device, then raise Fp8Error if a kernel recorded an error in
    `status` (by default the per-device word the GEMM wrappers use when called
    without one); the word is cleared afterwards. Without this check (or an
    explicit status tensor read by the caller) a timed-out GEMM leaves its output
    partly written and nothing reports it."""
    import torch

    s = default_status(device) if status is None else status
    torch.cuda.synchronize(s.device)
    code = int(s.item())
    if code != OK:
        s.zero_()
        raise Fp8Error(code, "device status")


def _status(status, t):
    return default_status(t.device) if status is None else status


def _stream(stream=None):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


# ---------------------------------------------------------------- quantize
def quantize(x, fmt: int, gran: int, sf_layout: int = SF_LINEAR, static_scale=None, q=None, scales=None,
             workspace=None, stream=None):
    """x: bf16 CUDA tensor [rows, cols] (row stride may exceed cols).

    Returns (q uint8 [rows, cols], scales) where scales is float32 (or uint8 for MX32).
    """
    import torch

    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    dev = x.device
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
    if scales is None:
        nbytes = scales_bytes(rows, cols, gran, sf_layout)
        if gran == MX32:
            scales = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)[:nbytes]
        else:
            scales = torch.empty(max(nbytes // 4, 1), dtype=torch.float32, device=dev)[: nbytes // 4]
    wsb = workspace_bytes(rows, cols, gran)
    if workspace is None and wsb > 0 and (static_scale is None or gran == CHANNEL):
        workspace = torch.empty(wsb, dtype=torch.uint8, device=dev)
    rc = lib().fp8_quantize(_ptr(x), rows, cols, x.stride(0), fmt, gran, sf_layout, _ptr(static_scale), _ptr(q),
                            q.stride(0), _ptr(scales), _ptr(workspace),
                            0 if workspace is None else workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "fp8_quantize")
    return q, scales


def quantize_delayed(x, fmt: int, history, slot: int, margin: int = 0, q=None, scale=None, stream=None):
    """Per-tensor quantization with the scale from an amax history (updated in place at `slot`)."""
    import torch

    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    assert history.dtype == torch.float32 and history.is_contiguous()
    rows, cols = x.shape
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(1, dtype=torch.float32, device=x.device)
    rc = lib().fp8_quantize_delayed(_ptr(x), rows, cols, x.stride(0), fmt, _ptr(history), history.numel(), slot,
                                    margin, _ptr(q), q.stride(0), _ptr(scale), _stream(stream))
    _check(rc, "fp8_quantize_delayed")
    return q, scale


def dequantize(q, scales, fmt: int, gran: int, sf_layout: int = SF_LINEAR, out=None, stream=None):
    import torch

    assert q.dtype == torch.uint8 and q.dim() == 2 and q.stride(1) == 1
    rows, cols = q.shape
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.bfloat16, device=q.device)
    rc = lib().fp8_dequantize(_ptr(q), rows, cols, q.stride(0), fmt, gran, sf_layout, _ptr(scales), _ptr(out),
                              out.stride(0), _stream(stream))
    _check(rc, "fp8_dequantize")
    return out


# ---------------------------------------------------------------- GEMMs
def gemm_blockscaled(a, a_scales, a_gran: int, b, b_scales, b_gran: int, a_fmt: int = E4M3, b_fmt: int = E4M3,
                     out=None, status=None, stream=None):
    """Out[M, N] bf16 = X_hat @ W_hat^T; a: uint8 [M, K], b: uint8 [N, K] (contiguous).

    status: a zeroed int32 CUDA tensor the kernel sets to ERR_TIMEOUT if a bounded
    wait expires; None uses the per-device word of default_status(), which
    check_status() reads. The same holds for every GEMM wrapper here."""
    import torch

    M, K = a.shape
    N, K2 = b.shape
    assert K == K2 and a.is_contiguous() and b.is_contiguous()
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    status = _status(status, a)
    rc = lib().fp8_gemm_blockscaled(_ptr(a), _ptr(a_scales), a_gran, _ptr(b), _ptr(b_scales), b_gran, a_fmt, b_fmt,
                                    _ptr(out), M, N, K, _ptr(status), _stream(stream))
    _check(rc, "fp8_gemm_blockscaled")
    return out


def gemm_blockscaled_quantized_out(a, a_scales, b, b_scales, a_fmt: int = E4M3, b_fmt: int = E4M3,
                                   out_fmt: int = E4M3, q_out=None, q_scales=None, status=None, stream=None):
    """Block-scaled GEMM whose epilogue quantizes the bf16 output at 1x128.

    Returns (q uint8 [M, N], scales float32 [(N/128) * M]) in the 1x128 tile layout.
    """
    import torch

    M, K = a.shape
    N, K2 = b.shape
    assert K == K2 and a.is_contiguous() and b.is_contiguous()
    if q_out is None:
        q_out = torch.empty((M, N), dtype=torch.uint8, device=a.device)
    if q_scales is None:
        q_scales = torch.empty((N // 128) * M, dtype=torch.float32, device=a.device)
    status = _status(status, a)
    rc = lib().fp8_gemm_blockscaled_quantized_out(_ptr(a), _ptr(a_scales), _ptr(b), _ptr(b_scales), a_fmt, b_fmt,
                                                  out_fmt, _ptr(q_out), _ptr(q_scales), M, N, K, _ptr(status),
                                                  _stream(stream))
    _check(rc, "fp8_gemm_blockscaled_quantized_out")
    return q_out, q_scales


def gemm_mx(a, a_sf, b, b_sf, a_fmt: int = E4M3, b_fmt: int = E4M3, out=None, status=None, stream=None,
            sf_layout: int = SF_TCGEN05):
    """MXFP8 GEMM; a_sf / b_sf in the SF_TCGEN05 layout (fp8_gemm_mx) or, with
    sf_layout=SF_TCGEN05_X4, in the staged-four-times layout (fp8_gemm_mx_x4)."""
    import torch

    M, K = a.shape
    N, K2 = b.shape
    assert K == K2 and a.is_contiguous() and b.is_contiguous()
    assert sf_layout in (SF_TCGEN05, SF_TCGEN05_X4)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    status = _status(status, a)
    fn = lib().fp8_gemm_mx if sf_layout == SF_TCGEN05 else lib().fp8_gemm_mx_x4
    rc = fn(_ptr(a), _ptr(a_sf), _ptr(b), _ptr(b_sf), a_fmt, b_fmt, _ptr(out), M, N, K, _ptr(status),
            _stream(stream))
    _check(rc, "fp8_gemm_mx" if sf_layout == SF_TCGEN05 else "fp8_gemm_mx_x4")
    return out


def debug_gemm_mx_kernel(kernel: str, a, a_sf, b, b_sf, a_fmt: int = E4M3, b_fmt: int = E4M3, out=None, status=None,
                         stream=None):
    """fp8_gemm_mx on the named kernel: "pairs" (CTA pairs) or "single" (one CTA per tile)."""
    import torch

    M, K = a.shape
    N, K2 = b.shape
    assert K == K2 and a.is_contiguous() and b.is_contiguous() and kernel in ("pairs", "single")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    status = _status(status, a)
    fn = lib().fp8_debug_gemm_mx_pairs if kernel == "pairs" else lib().fp8_debug_gemm_mx_single
    rc = fn(_ptr(a), _ptr(a_sf), _ptr(b), _ptr(b_sf), a_fmt, b_fmt, _ptr(out), M, N, K, _ptr(status), _stream(stream))
    _check(rc, "fp8_debug_gemm_mx_" + kernel)
    return out


def nvfp4_scales_bytes(rows: int, cols: int, sf_layout: int = SF_TCGEN05) -> int:
    return int(lib().fp8_nvfp4_scales_bytes(rows, cols, sf_layout))


def quantize_nvfp4(x, sf_layout: int = SF_TCGEN05, static_tensor_scale=None, q=None, sf=None, tensor_scale=None,
                   stream=None):
    """NVFP4 quantize of bf16 x [rows x cols]: (codes uint8 [rows x cols/2], E4M3 block scales uint8,
    tensor scale float32 [1]); static_tensor_scale: None (from this tensor's amax) or a device float32 [1]."""
    import torch

    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    dev = x.device
    if q is None:
        q = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
    if sf is None:
        sf = torch.empty(max(1, nvfp4_scales_bytes(rows, cols, sf_layout)), dtype=torch.uint8, device=dev)
    if tensor_scale is None:
        tensor_scale = torch.empty(1, dtype=torch.float32, device=dev)
    ws = None
    if static_tensor_scale is None:
        ws = torch.empty(max(1, workspace_bytes(rows, cols, TENSOR)), dtype=torch.uint8, device=dev)
    rc = lib().fp8_quantize_nvfp4(_ptr(x), rows, cols, x.stride(0), sf_layout, _ptr(static_tensor_scale), _ptr(q),
                                  q.stride(0), _ptr(sf), _ptr(tensor_scale), _ptr(ws),
                                  0 if ws is None else ws.numel(), _stream(stream))
    _check(rc, "fp8_quantize_nvfp4")
    return q, sf, tensor_scale


def dequantize_nvfp4(q, sf, tensor_scale, cols: int, sf_layout: int = SF_TCGEN05, out=None, stream=None):
    import torch

    rows = q.shape[0]
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.bfloat16, device=q.device)
    rc = lib().fp8_dequantize_nvfp4(_ptr(q), rows, cols, q.stride(0), sf_layout, _ptr(sf), _ptr(tensor_scale),
                                    _ptr(out), out.stride(0), _stream(stream))
    _check(rc, "fp8_dequantize_nvfp4")
    return out


def gemm_nvfp4(a, a_sf, a_ts, b, b_sf, b_ts, out=None, status=None, stream=None):
    """NVFP4 GEMM: a [M x K/2], b [N x K/2] packed codes, scales in SF_TCGEN05, tensor scales float32 [1]."""
    import torch

    M, Kh = a.shape
    N, Kh2 = b.shape
    assert Kh == Kh2 and a.is_contiguous() and b.is_contiguous()
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    status = _status(status, a)
    rc = lib().fp8_gemm_nvfp4(_ptr(a), _ptr(a_sf), _ptr(a_ts), _ptr(b), _ptr(b_sf), _ptr(b_ts), _ptr(out), M, N,
                              2 * Kh, _ptr(status), _stream(stream))
    _check(rc, "fp8_gemm_nvfp4")
    return out


def debug_encode_f32(x, fmt: int, out=None, stream=None):
    """RNE-satfinite encode of fp32 values (the quantizers' element step, scale 1)."""
    import torch

    assert x.dtype == torch.float32 and x.is_contiguous()
    if out is None:
        out = torch.empty(x.numel(), dtype=torch.uint8, device=x.device)
    _check(lib().fp8_debug_encode_f32(_ptr(x), x.numel(), fmt, _ptr(out), _stream(stream)), "fp8_debug_encode_f32")
    return out


def debug_gemm_blockscaled_pairs(a, a_scales, b, b_scales, a_fmt: int = E4M3, b_fmt: int = E4M3, out=None,
                                 status=None, stream=None):
    """The 1x128 x 128x128 block-scaled GEMM on the CTA-pair kernel, whatever the shape."""
    import torch

    M, K = a.shape
    N = b.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    status = _status(status, a)
    rc = lib().fp8_debug_gemm_blockscaled_pairs(_ptr(a), _ptr(a_scales), _ptr(b), _ptr(b_scales), a_fmt, b_fmt,
                                                _ptr(out), M, N, K, _ptr(status), _stream(stream))
    _check(rc, "fp8_debug_gemm_blockscaled_pairs")
    return out


def debug_encode_e2m1_f32(x, out=None, stream=None):
    """E2M1 codes (one per byte) of fp32 values: NVFP4's element step with scale 1."""
    import torch

    assert x.dtype == torch.float32 and x.is_contiguous()
    if out is None:
        out = torch.empty(x.numel(), dtype=torch.uint8, device=x.device)
    _check(lib().fp8_debug_encode_e2m1_f32(_ptr(x), x.numel(), _ptr(out), _stream(stream)), "fp8_debug_encode_e2m1_f32")
    return out


def debug_wait_probe(status, timeout_ns: int, stream=None):
    _check(lib().fp8_debug_wait_probe(_ptr(status), int(timeout_ns), _stream(stream)), "fp8_debug_wait_probe")

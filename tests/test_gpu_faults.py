"""Failure handling on the GPU without faulting it: bounded waits report a
status and leave the context usable; bad arguments are refused on the host
before anything is enqueued."""
import pytest
import torch

from fp8_block_scaled_04_gb300 import binding as fb

pytestmark = pytest.mark.gpu


def test_wait_limit_expires_with_status_and_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fb.debug_wait_probe(status, 2_000_000)  # 2 ms on a barrier nothing arrives on
    torch.cuda.synchronize()
    assert int(status.item()) == fb.ERR_TIMEOUT
    # the context still works: a real launch runs and completes
    x = torch.randn(64, 256, device="cuda").to(torch.bfloat16)
    q, s = fb.quantize(x, fb.E4M3, fb.TOKEN)
    torch.cuda.synchronize()
    assert q.shape == (64, 256)


def test_misaligned_pointers_refused_without_launch():
    buf = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    x = torch.zeros((8, 128), dtype=torch.bfloat16, device="cuda")
    n0 = fb.launch_count()
    L = fb.lib()
    import ctypes

    bad = ctypes.c_void_p(buf.data_ptr() + 1)
    rc = L.fp8_quantize(ctypes.c_void_p(x.data_ptr()), 8, 128, 128, 0, 1, 0, None, bad, 128,
                        ctypes.c_void_p(buf.data_ptr() + 2048), None, 0, None)
    assert rc == fb.ERR_ALIGNMENT
    rc = L.fp8_gemm_blockscaled(bad, ctypes.c_void_p(buf.data_ptr()), 2, ctypes.c_void_p(buf.data_ptr()),
                                ctypes.c_void_p(buf.data_ptr()), 3, 0, 0, ctypes.c_void_p(buf.data_ptr()), 16, 16,
                                128, None, None)
    assert rc == fb.ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert fb.launch_count() == n0


def test_bad_shapes_refused():
    a = torch.zeros((16, 130), dtype=torch.uint8, device="cuda")
    s = torch.ones(64, dtype=torch.float32, device="cuda")
    out = torch.empty((16, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fb.Fp8Error) as e:
        fb.gemm_blockscaled(a, s, fb.TILE_1x128, a, s, fb.BLOCK_128x128, out=out)  # K % 128 != 0
    assert e.value.code in (fb.ERR_UNSUPPORTED_SHAPE, fb.ERR_ALIGNMENT)
    b = torch.zeros((24, 128), dtype=torch.uint8, device="cuda")
    a2 = torch.zeros((16, 128), dtype=torch.uint8, device="cuda")
    with pytest.raises(fb.Fp8Error) as e:
        fb.gemm_blockscaled(a2, s, fb.TILE_1x128, b, s, fb.BLOCK_128x128)  # N % 16 != 0
    assert e.value.code == fb.ERR_UNSUPPORTED_SHAPE


# ------------------------------------------------------------ GEMM timeout exit
# The single-CTA GEMM kernels run with every bounded wait limited to 1 ns: the
# first wait that is not already satisfied expires, the kernel records
# FP8_ERR_TIMEOUT, drains its copies and MMAs, frees tensor memory and returns.
# A normal GEMM on the same context afterwards must still match the oracle.
import ctypes  # noqa: E402

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from fp8_block_scaled_04_gb300 import synth  # noqa: E402
from gpu_util import out_f64, within_tolerance  # noqa: E402

_P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
_S = lambda: ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)  # noqa: E731

# (name, M, N, K, a_gran, b_gran): the fold kernel with 256- and 128-wide tiles,
# the operand-swapped decode kernel (no split-K cluster on this path), the
# epilogue-scaled tensor-memory kernel, and the MXFP8 block-scaled kernel
_CASES = [("fold_wide", 2048, 4096, 1024, fb.TILE_1x128, fb.BLOCK_128x128),
          ("fold_narrow", 256, 1024, 2048, fb.TILE_1x128, fb.BLOCK_128x128),
          ("swap", 16, 2048, 2048, fb.TILE_1x128, fb.BLOCK_128x128),
          ("epi", 512, 1024, 1024, fb.TOKEN, fb.TOKEN),
          ("mx", 1024, 1024, 1024, fb.MX32, fb.MX32)]


@pytest.mark.parametrize("name,M,N,K,ga,gb", _CASES, ids=[c[0] for c in _CASES])
def test_gemm_timeout_exit_then_context_usable(name, M, N, K, ga, gb):
    L = fb.lib()
    x = synth.bf16_matrix(M, K, 1.0, 700 + M, 701, 0.01, 30.0)
    w = synth.bf16_matrix(N, K, 0.02, 702 + N)
    lay = fb.SF_TCGEN05 if ga == fb.MX32 else fb.SF_LINEAR
    qa, sa = oracle.quantize(x, fb.E4M3, ga, lay)
    qb, sb = oracle.quantize(w, fb.E4M3, gb, lay)
    a, sad, b, sbd = (torch.from_numpy(t).cuda() for t in (qa, sa, qb, sb))
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes = []
    for _ in range(5):
        status.zero_()
        if ga == fb.MX32:
            rc = L.fp8_debug_gemm_mx_wait_limit(_P(a), _P(sad), _P(b), _P(sbd), 0, 0, _P(out), M, N, K, _P(status), 1,
                                                _S())
        else:
            rc = L.fp8_debug_gemm_blockscaled_wait_limit(_P(a), _P(sad), ga, _P(b), _P(sbd), gb, 0, 0, _P(out), M, N,
                                                         K, _P(status), 1, _S())
        assert rc == fb.OK
        torch.cuda.synchronize()
        codes.append(int(status.item()))
        if codes[-1] == fb.ERR_TIMEOUT:
            break
    assert set(codes) <= {fb.OK, fb.ERR_TIMEOUT} and codes[-1] == fb.ERR_TIMEOUT, codes
    # the context still works: the same GEMM with the production limit matches the oracle
    status.zero_()
    out.zero_()
    if ga == fb.MX32:
        fb.gemm_mx(a, sad, b, sbd, out=out, status=status)
    else:
        fb.gemm_blockscaled(a, sad, ga, b, sbd, gb, out=out, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == fb.OK
    rows = np.unique(np.concatenate([np.arange(0, M, max(1, M // 64)), [M - 1]]))
    kw = dict(a_sf=lay, b_sf=lay) if ga == fb.MX32 else {}
    ref, bound = oracle.gemm(qa, sa, ga, qb, sb, gb, rows=rows, **kw)
    tol = within_tolerance(out_f64(out)[rows], ref, bound)
    assert tol.bad == 0, tol


def test_default_status_word_reports_timeouts():
    """The binding's per-device status word (used when a GEMM wrapper gets no status)
    carries a timeout to check_status(), which raises and clears it."""
    st = fb.default_status()
    st.fill_(fb.ERR_TIMEOUT)  # what an expired wait leaves there
    with pytest.raises(fb.Fp8Error) as e:
        fb.check_status()
    assert e.value.code == fb.ERR_TIMEOUT
    fb.check_status()  # cleared


def test_empty_gemms_launch_nothing_and_k0_is_refused():
    """M = 0 or N = 0 is an empty product: every GEMM entry returns OK and launches
    nothing. K = 0 with M, N > 0 has no scale blocks to fold: refused as a shape."""
    d = "cuda"
    u8 = lambda *s: torch.zeros(s, dtype=torch.uint8, device=d)  # noqa: E731
    f32 = lambda n: torch.ones(n, dtype=torch.float32, device=d)  # noqa: E731
    n0 = fb.launch_count()
    for M, N in ((0, 256), (128, 0), (0, 0)):
        K = 256
        a, b = u8(M, K), u8(N, K)
        out = torch.empty((M, N), dtype=torch.bfloat16, device=d)
        fb.gemm_blockscaled(a, f32(max(1, M * 2)), fb.TILE_1x128, b, f32(max(1, N)), fb.BLOCK_128x128, out=out)
        fb.gemm_blockscaled(a, f32(1), fb.TENSOR, b, f32(1), fb.TENSOR, out=out)
        fb.gemm_mx(a, u8(4096), b, u8(4096), out=out)
        fb.gemm_nvfp4(u8(M, K // 2), u8(4096), f32(1), u8(N, K // 2), u8(4096), f32(1), out=out)
        if N % 128 == 0:
            fb.gemm_blockscaled_quantized_out(a, f32(max(1, M * 2)), b, f32(max(1, N)))
    torch.cuda.synchronize()
    assert fb.launch_count() == n0
    a, b = u8(16, 0), u8(128, 0)
    for call in (lambda: fb.gemm_blockscaled(a, f32(1), fb.TILE_1x128, b, f32(1), fb.BLOCK_128x128),
                 lambda: fb.gemm_blockscaled(a, f32(1), fb.TENSOR, b, f32(1), fb.TENSOR),
                 lambda: fb.gemm_mx(a, u8(512), b, u8(512))):
        with pytest.raises(fb.Fp8Error) as e:
            call()
        assert e.value.code == fb.ERR_UNSUPPORTED_SHAPE
    assert fb.launch_count() == n0

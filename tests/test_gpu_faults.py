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

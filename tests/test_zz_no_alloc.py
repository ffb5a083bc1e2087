"""The allocation-free per-tensor quantize entry point, called through the C ABI.

fp8_quantize_tensor_noalloc serves callers that cannot call cudaMalloc (a host
framework that owns all device memory, or a path that cannot afford
cudaMalloc's implicit synchronisation): it keeps its amax scratch in a static
device array inside the library instead of a caller workspace. Its output must
equal that of fp8_quantize (per-tensor, dynamic), bit for bit, on two calls in a
row -- the second with a smaller amax than the first, so a scratch word left
over from the first call would show.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from fp8_block_scaled_04_gb300 import binding as fb
from fp8_block_scaled_04_gb300 import synth

pytestmark = pytest.mark.gpu


def _dev_bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()


def _noalloc(x, fmt):
    rows, cols = x.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    s = torch.empty(1, dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = fb.lib().fp8_quantize_tensor_noalloc(ctypes.c_void_p(x.data_ptr()), rows, cols, x.stride(0), fmt,
                                              ctypes.c_void_p(q.data_ptr()), q.stride(0),
                                              ctypes.c_void_p(s.data_ptr()), stream)
    assert rc == fb.OK, fb.status_string(rc)
    return q, s


@pytest.mark.parametrize("fmt", [fb.E4M3, fb.E5M2])
def test_noalloc_matches_workspace_entry_point_twice(fmt):
    big = _dev_bf16(synth.bf16_matrix(300, 1024, 1.0, 501, 502, 0.01, 80.0))
    small = _dev_bf16(synth.bf16_matrix(130, 640, 0.001, 503))
    for x in (big, small):  # second call has the smaller amax
        q1, s1 = _noalloc(x, fmt)
        q0, s0 = fb.quantize(x, fmt, fb.TENSOR)
        torch.cuda.synchronize()
        assert torch.equal(q1, q0)
        assert torch.equal(s1.view(torch.int32), s0.view(torch.int32))


def test_noalloc_refuses_bad_arguments_without_launch():
    L = fb.lib()
    n0 = fb.launch_count()
    a = ctypes.c_void_p(0x100000)
    assert L.fp8_quantize_tensor_noalloc(a, 8, 120, 128, 0, a, 128, a, None) == fb.ERR_UNSUPPORTED_SHAPE
    assert L.fp8_quantize_tensor_noalloc(ctypes.c_void_p(0x100001), 8, 128, 128, 0, a, 128, a, None) == \
        fb.ERR_ALIGNMENT
    assert L.fp8_quantize_tensor_noalloc(None, 8, 128, 128, 0, a, 128, a, None) == fb.ERR_INVALID_ARG
    assert fb.launch_count() == n0

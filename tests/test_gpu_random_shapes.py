"""Seeded random shapes through every GEMM kernel family against the oracle: the
shape rule's branches (wide and narrow fold tiles, operand-swapped decode tiles of
16 / 32 / 64 rows, split-K clusters, the tensor-copy and per-lane scale paths),
both MXFP8 kernels and NVFP4, on sizes no hand-picked test names. Entries are
sampled (rows and columns spread over the output, plus the last ones)."""
import functools

import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_04_gb300 import binding as fb
from fp8_block_scaled_04_gb300 import synth
from gpu_util import out_f64, to_dev_bf16, within_tolerance

pytestmark = pytest.mark.gpu


def _shapes(seed, n, k_unit):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        m = int(rng.choice([rng.integers(1, 65), rng.integers(65, 700)]))
        nn = 16 * int(rng.integers(1, 1400))
        k = k_unit * int(rng.integers(1, max(2, 4096 // k_unit)))
        out.append((m, nn, k))
    return out


@functools.lru_cache(maxsize=2)
def _fold_operands(M, N, K):
    return (synth.bf16_matrix(M, K, 1.0, 900 + M, 901 + K, 0.01, 30.0), synth.bf16_matrix(N, K, 0.02, 902 + N))


def _sample(n, count=48):
    return np.unique(np.concatenate([np.linspace(0, n - 1, count).astype(np.int64), [n - 1]]))


@pytest.mark.parametrize("fmt", [fb.E4M3, fb.E5M2])
@pytest.mark.parametrize("M,N,K", _shapes(2024, 12, 128))
def test_fold_gemm_random_shapes(M, N, K, fmt):
    x, w = _fold_operands(M, N, K)
    qa, sa = oracle.quantize(x, fmt, fb.TILE_1x128)
    qb, sb = oracle.quantize(w, fmt, fb.BLOCK_128x128)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fb.gemm_blockscaled(*(torch.from_numpy(v).cuda() for v in (qa, sa)), fb.TILE_1x128,
                              *(torch.from_numpy(v).cuda() for v in (qb, sb)), fb.BLOCK_128x128, fmt, fmt,
                              status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows, cols = _sample(M), _sample(N)
    ref, bound = oracle.gemm(qa, sa, fb.TILE_1x128, qb, sb, fb.BLOCK_128x128, fmt, fmt, rows=rows, cols=cols)
    tol = within_tolerance(out_f64(out)[np.ix_(rows, cols)], ref, bound)
    assert tol.bad == 0, tol


@pytest.mark.parametrize("M,N,K", _shapes(2025, 8, 32))
@pytest.mark.parametrize("kernel", ["single", "pairs"])
def test_mx_gemm_random_shapes(M, N, K, kernel):
    x = synth.bf16_matrix(M, K, 1.0, 910 + M, 911, 0.005, 50.0)
    w = synth.bf16_matrix(N, K, 1.0, 912 + N, 913, 0.005, 50.0)
    qa, sfa = oracle.quantize(x, fb.E4M3, fb.MX32, fb.SF_TCGEN05)
    qb, sfb = oracle.quantize(w, fb.E4M3, fb.MX32, fb.SF_TCGEN05)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fb.debug_gemm_mx_kernel(kernel, *(torch.from_numpy(v).cuda() for v in (qa, sfa, qb, sfb)), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows, cols = _sample(M), _sample(N)
    ref, bound = oracle.gemm(qa, sfa, fb.MX32, qb, sfb, fb.MX32, a_sf=fb.SF_TCGEN05, b_sf=fb.SF_TCGEN05, rows=rows,
                             cols=cols)
    tol = within_tolerance(out_f64(out)[np.ix_(rows, cols)], ref, bound)
    assert tol.bad == 0, tol


@pytest.mark.parametrize("M,N,K", _shapes(2026, 6, 256))
def test_nvfp4_gemm_random_shapes(M, N, K):
    x = synth.bf16_matrix(M, K, 1.0, 920 + M, 921, 0.005, 20.0)
    w = synth.bf16_matrix(N, K, 0.05, 922 + N)
    qa, sfa, ta = oracle.quantize_nvfp4(x, fb.SF_TCGEN05)
    qb, sfb, tb = oracle.quantize_nvfp4(w, fb.SF_TCGEN05)
    dev = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fb.gemm_nvfp4(dev(qa), dev(sfa), dev(np.array([ta], dtype=np.float32).reshape(1)), dev(qb), dev(sfb),
                        dev(np.array([tb], dtype=np.float32).reshape(1)), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows, cols = _sample(M), _sample(N)
    ref, bound = oracle.gemm_nvfp4(qa, sfa, ta, qb, sfb, tb, rows=rows, cols=cols)
    tol = within_tolerance(out_f64(out)[np.ix_(rows, cols)], ref, bound)
    assert tol.bad == 0, tol


_GRAN_UNITS = [(fb.TENSOR, fb.SF_LINEAR, 16), (fb.TOKEN, fb.SF_LINEAR, 16), (fb.CHANNEL, fb.SF_LINEAR, 16),
               (fb.TILE_1x128, fb.SF_LINEAR, 128), (fb.BLOCK_128x128, fb.SF_LINEAR, 128),
               (fb.MX32, fb.SF_LINEAR, 32), (fb.MX32, fb.SF_TCGEN05, 32)]


def _quant_cases(seed, n):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        gran, lay, unit = _GRAN_UNITS[i % len(_GRAN_UNITS)]
        rows = int(rng.choice([rng.integers(1, 130), rng.integers(130, 5000)]))
        cols = unit * int(rng.integers(1, max(2, 20000 // unit)))
        fmt = fb.E4M3 if rng.integers(0, 2) == 0 else fb.E5M2
        cases.append((gran, lay, fmt, rows, cols))
    return cases


@pytest.mark.parametrize("gran,lay,fmt,rows,cols", _quant_cases(2027, 28))
def test_quantize_random_shapes_bit_exact(gran, lay, fmt, rows, cols):
    """Every granularity and scale layout on seeded random shapes (ragged row and column
    tails, one row, many rows): codes and scales bit-exact, dequantized values too."""
    x = synth.bf16_matrix(rows, cols, 1.0, 930 + rows, 931 + cols, 0.01, 40.0)
    q, s = fb.quantize(to_dev_bf16(x), fmt, gran, lay)
    oq, os_ = oracle.quantize(x, fmt, gran, lay)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy().view(np.uint8).reshape(-1), np.ascontiguousarray(os_).view(np.uint8).reshape(-1))
    d = fb.dequantize(q, s, fmt, gran, lay)
    ref = oracle.dequantize(oq, os_, fmt, gran, lay)
    assert np.array_equal(d.view(torch.int16).cpu().numpy().view(np.uint16), ref)

"""Helpers shared by the GPU parity tests (host-side conversions only)."""
import numpy as np
import torch


def to_dev_bf16(x_u16: np.ndarray, device="cuda:0") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x_u16).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_host(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32_bits(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def out_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def half_ulp_bf16(v: np.ndarray) -> np.ndarray:
    """Half a bf16 ulp at |v| (8 significant bits): 2^(e-8) for |v| in [2^e, 2^(e+1))."""
    _, ex = np.frexp(np.abs(v))
    return np.ldexp(1.0, ex - 9)


def within_tolerance(got: np.ndarray, ref: np.ndarray, bound: np.ndarray):
    """Parity rule of the GEMMs.

    |gpu - ref| <= 1e-3 * sum_k |x_hat w_hat| + 1e-6 + half_ulp_bf16(max(|ref|, |gpu|)).
    The first two terms are the stated accumulation tolerance; the last is the
    rounding of the bf16 output itself, which the stated term alone cannot
    absorb when one product dominates the sum (|ref| close to the bound).
    Returns (number of violations, worst (|err| - half ulp) / bound).
    """
    err = np.abs(got - ref)
    hu = half_ulp_bf16(np.maximum(np.abs(ref), np.abs(got)))
    bad = err > 1e-3 * bound + 1e-6 + hu
    worst = float((np.maximum(err - hu, 0.0) / (bound + 1e-30)).max()) if err.size else 0.0
    return int(bad.sum()), worst

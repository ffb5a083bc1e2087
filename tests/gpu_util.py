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


def within_tolerance(got: np.ndarray, ref: np.ndarray, bound: np.ndarray):
    """Parity rule of the GEMMs: |gpu - ref| <= 1e-3 * sum_k |x_hat w_hat| + 1e-6."""
    err = np.abs(got - ref)
    bad = err > 1e-3 * bound + 1e-6
    worst = float((err / (bound + 1e-30)).max()) if err.size else 0.0
    return int(bad.sum()), worst

"""Helpers shared by the GPU parity tests (host-side conversions only)."""
import os

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


class Tolerance:
    """Outcome of the GEMM parity rule on one output (see within_tolerance).

    Unpacks as (bad, worst) for the callers that only need those two numbers.
    """

    def __init__(self, n, bad, worst, half_ulp_used, worst_plain):
        self.n = n                          # elements compared
        self.bad = bad                      # elements outside the full rule
        self.worst = worst                  # max (|err| - half ulp) / bound
        self.half_ulp_used = half_ulp_used  # elements inside the rule only thanks to the half-ulp term
        self.worst_plain = worst_plain      # max |err| / bound, no half-ulp term

    def __iter__(self):
        return iter((self.bad, self.worst))

    def __repr__(self):
        return ("Tolerance(n=%d, bad=%d, worst=%.3g, half_ulp_used=%d, worst_plain=%.3g)"
                % (self.n, self.bad, self.worst, self.half_ulp_used, self.worst_plain))


# every parity check of this session: (test id, Tolerance); printed in the terminal summary
RECORDS = []


def within_tolerance(got: np.ndarray, ref: np.ndarray, bound: np.ndarray) -> Tolerance:
    """Parity rule of the GEMMs.

    |gpu - ref| <= 1e-3 * sum_k |x_hat w_hat| + 1e-6 + half_ulp_bf16(max(|ref|, |gpu|)).
    The first two terms are the stated accumulation tolerance; the last is the
    rounding of the bf16 output itself, which the stated term alone cannot
    absorb when one product dominates the sum (|ref| close to the bound).
    The result also counts the elements that pass only because of the half-ulp
    term and the worst |err| / bound without it, so every test reports how
    often the bf16 rounding term was needed.
    """
    err = np.abs(got - ref)
    stated = 1e-3 * bound + 1e-6
    hu = half_ulp_bf16(np.maximum(np.abs(ref), np.abs(got)))
    bad = err > stated + hu
    needed = (err > stated) & ~bad
    if err.size:
        worst = float((np.maximum(err - hu, 0.0) / (bound + 1e-30)).max())
        worst_plain = float((err / (bound + 1e-30)).max())
    else:
        worst = worst_plain = 0.0
    tol = Tolerance(int(err.size), int(bad.sum()), worst, int(needed.sum()), worst_plain)
    RECORDS.append((os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], tol))
    return tol


GUARD_BYTES = 4096
GUARD_BYTE = 0xA5


class Guarded:
    """A device buffer with GUARD_BYTES of a known byte on each side (a stand-in for
    a memory checker: any store that strays past either end of the buffer changes a
    guard byte). .t is the tensor view handed to the library (16-byte aligned)."""

    def __init__(self, shape, dtype, device="cuda"):
        elt = torch.empty((), dtype=dtype).element_size()
        n = 1
        for s in shape:
            n *= s
        self.nbytes = n * elt
        self.raw = torch.full((GUARD_BYTES + self.nbytes + GUARD_BYTES,), GUARD_BYTE, dtype=torch.uint8, device=device)
        self.t = self.raw[GUARD_BYTES:GUARD_BYTES + self.nbytes].view(dtype).view(*shape)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        lo = self.raw[:GUARD_BYTES]
        hi = self.raw[GUARD_BYTES + self.nbytes:]
        return bool((lo == GUARD_BYTE).all()) and bool((hi == GUARD_BYTE).all())


def x4_layout(sf_tiled):
    """Scales in the tensor-core tiled layout -> the staged-four-times layout
    (each 512-byte block stored four times in a row). Layout plumbing only: the
    bytes are the oracle's, repeated."""
    blocks = np.asarray(sf_tiled, dtype=np.uint8).reshape(-1, 1, 512)
    return np.ascontiguousarray(np.repeat(blocks, 4, axis=1)).reshape(-1)

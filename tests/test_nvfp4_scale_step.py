"""The NVFP4 encoder's fast block-scale step, checked on the CPU as arithmetic.

The encoder needs only the E4M3 code of u = fp32(fp32(amax_b / 6) / s_t). It forms
u' = fp32(amax_b * c), c = fp32(fp32(1/6) / s_t), and keeps u' when its 20 fp32
mantissa bits below E4M3's three are at least 6 units from the rounding midpoint,
u' lies in [2^-6, 440] and amax_b >= 6 * 2^-126 (so that fp32(amax_b / 6) is a normal
number); otherwise it divides. The claim (five roundings of at most
2^-24 relative each keep |u' - u| within 5 units in the last place of u) is checked
here on every positive finite bf16 amax_b for tensor scales around 1 (the midpoint
band), plus random amax_b for tensor scales across the range the dynamic path gives
(s_t = amax_t / 2688). numpy float32 arithmetic is IEEE round-to-nearest; the E4M3
rounding is the oracle's encoder.
"""
import numpy as np

import oracle

F32 = np.float32


AMAX_B_MIN = F32(6.0 * 2.0 ** -126)  # smallest block amax whose amax / 6 is an fp32 normal


def _fast_applies(u_fast, c, amax_b, guard=True):
    d = (u_fast.view(np.uint32) & 0xFFFFF).astype(np.int64) - 0x80000
    normal_c = np.isfinite(c) and abs(float(c)) >= 2.0 ** -126
    m = normal_c & (u_fast >= F32(2.0 ** -6)) & (u_fast <= F32(440.0)) & (np.abs(d) >= 6)
    return m & (amax_b >= AMAX_B_MIN) if guard else m


def _codes(amax_b, s_t, guard=True):
    """(E4M3 code of the two-division u, code of the fast u') where the fast step applies."""
    c = F32(F32(F32(1.0) / F32(6.0)) / s_t)
    with np.errstate(all="ignore"):
        u_exact = (amax_b / F32(6.0)).astype(np.float32) / s_t
        u_fast = (amax_b * c).astype(np.float32)
    m = _fast_applies(u_fast, c, amax_b, guard) & np.isfinite(u_exact)
    if not m.any():
        return np.zeros(0, np.uint8), np.zeros(0, np.uint8)
    return (oracle.encode(u_exact[m].astype(np.float32), oracle.E4M3),
            oracle.encode(u_fast[m].astype(np.float32), oracle.E4M3))


def _check(amax_b, s_t):
    c = F32(F32(F32(1.0) / F32(6.0)) / s_t)
    with np.errstate(all="ignore"):
        u_exact = (amax_b / F32(6.0)).astype(np.float32) / s_t
        u_fast = (amax_b * c).astype(np.float32)
    m = _fast_applies(u_fast, c, amax_b) & np.isfinite(u_exact)
    if not m.any():
        return 0
    a = oracle.encode(u_exact[m].astype(np.float32), oracle.E4M3)
    b = oracle.encode(u_fast[m].astype(np.float32), oracle.E4M3)
    assert np.array_equal(a, b), (float(s_t), u_exact[m][a != b][:4], u_fast[m][a != b][:4])
    return int(m.sum())


def test_every_bf16_amax_near_unit_tensor_scales():
    bits = np.arange(1, 0x7F80, dtype=np.uint32)  # positive finite bf16
    amax_b = (bits << 16).view(np.float32)
    used = 0
    for k in range(-16, 17):
        s_t = F32(1.0 + k * 2.0 ** -23) if k >= 0 else F32(1.0 + k * 2.0 ** -24)
        used += _check(amax_b, s_t)
    assert used > 50000


def test_random_amax_under_dynamic_tensor_scales():
    rng = np.random.default_rng(3)
    bits = np.arange(1, 0x7F80, dtype=np.uint32)
    used = 0
    for _ in range(40):
        amax_t = F32(np.exp(rng.uniform(-20, 20)))
        s_t = F32(amax_t / F32(2688.0))
        # block maxima up to the tensor's, in bf16
        a = (bits[rng.integers(0, len(bits), 50000)] << 16).view(np.float32)
        a = a[a <= amax_t]
        used += _check(a, s_t)
    assert used > 10000


def test_tiny_tensor_scales_and_subnormal_block_maxima():
    """Tensor scales in [5e-40, 5e-37] (static, or from a tensor whose amax is ~1e-36)
    with bf16 block maxima below and around 6 * 2^-126: where the fast step applies it
    gives the two-division code; two witnesses show it would not without the amax_b
    guard."""
    rng = np.random.default_rng(7)
    bits = np.arange(1, 0x7F80, dtype=np.uint32)
    allb = (bits << 16).view(np.float32)
    small = allb[allb < F32(64.0 * 2.0 ** -126)]  # every bf16 up to 64 * 2^-126, subnormals included
    used = 0
    for s_t in np.concatenate([np.geomspace(5e-40, 5e-37, 60), [1.335e-38]]).astype(np.float32):
        used += _check(small, F32(s_t))
    for _ in range(20):
        s_t = F32(np.exp(rng.uniform(np.log(5e-40), np.log(5e-37))))
        used += _check(allb[rng.integers(0, len(allb), 50000)], s_t)
    assert used > 1000
    # Why the amax_b guard is needed: with s_t = fp32 bits 0x000A28A2 (a subnormal,
    # 9.33e-40) and bf16 block maxima 5 * 2^-133 and 20 * 2^-133, fp32(amax_b / 6) is
    # subnormal and the two-division code differs from the fast one (26 vs 27, 42 vs
    # 43); the guard sends both blocks to the divisions.
    s_t = np.array([0x000A28A2], dtype=np.uint32).view(np.float32)[0]
    wit = (np.array([5, 20], dtype=np.uint32) << 16).view(np.float32)
    a, b = _codes(wit, s_t, guard=False)
    assert a.tolist() == [26, 42] and b.tolist() == [27, 43]
    assert _codes(wit, s_t, guard=True)[0].size == 0

"""The INT2 quantizer's code decision, restated in numpy fp32 (every step
IEEE round-to-nearest, as the kernel's __fsub_rn / __frcp_rn / __fmul_rn /
__fdiv_rn), gives the oracle's codes on every element.

The kernel forms y = (x - z) * (1/s), two roundings, instead of the
oracle's single-rounding (x - z) / s. It takes the correctly rounded quotient
only when y lies within 2^-16 of a rounding threshold of the code (0.5, 1.5
or 2.5).  It then reads the code from two bits: sign = y < 1.5, and
magnitude = y <= 0.5 or y > 2.5.  The test checks that this matches
clamp(rint((x - z) / s), 0, 3), ties to even, on millions of elements.  Many
of them sit exactly on a threshold or one ulp either side."""
import numpy as np

from oracle import qevict as QE
from workloads import bf16_bits_to_f32, f32_to_bf16_bits

F = np.float32


def kernel_codes(x, z, s):
    """The kernel's rule; x fp32 values, z and s fp32 (fp16-valued), broadcast."""
    with np.errstate(divide="ignore", invalid="ignore"):
        d = (x - z).astype(F)
        r = np.where(s == 0, F(0), F(1) / s).astype(F)
        y = (d * r).astype(F)
        dc = np.abs(y - F(1.5))
        near = (dc <= F(2.0 ** -16)) | (np.abs(dc - F(1)) <= F(2.0 ** -16))
        y = np.where(near, (d / s).astype(F), y)
    sign = y < F(1.5)
    mag = (y <= F(0.5)) | (y > F(2.5))
    code = np.where(sign, np.where(mag, 0, 1), np.where(mag, 3, 2))
    return np.where(s == 0, 0, code).astype(np.uint8)


def _check(x_groups):
    """x_groups [n][32] fp32 (bf16 values): the oracle's codes and the rule's."""
    codes, scale, zero = QE.quantize_groups(x_groups, axis=1)
    s = scale.astype(F)[:, None]
    z = zero.astype(F)[:, None]
    got = kernel_codes(x_groups, z, s)
    bad = got != codes
    assert not bad.any(), (f"{bad.sum()} codes differ, e.g. x={x_groups[bad][:4]}, "
                           f"s={np.broadcast_to(s, bad.shape)[bad][:4]}")
    return codes


def _bf16(x):
    return bf16_bits_to_f32(f32_to_bf16_bits(np.asarray(x, dtype=F)))


def test_random_groups_of_several_spreads():
    rng = np.random.default_rng(0)
    for scale in (1e-3, 0.37, 1.0, 8.0, 300.0):
        x = _bf16(rng.standard_normal((40000, 32)) * scale)
        _check(x)
        x = _bf16(rng.uniform(-scale, 3 * scale, (40000, 32)))
        _check(x)


def test_groups_with_elements_on_the_thresholds():
    """Each group's min and max fix z and s; its other elements are placed at
    z + (k / 2) s for k = 1, 3, 5 (exact ties of rint) and one bf16 ulp
    either side, as far as bf16 can represent them."""
    rng = np.random.default_rng(1)
    n = 30000
    lo = _bf16(rng.uniform(-4, 4, n))
    hi = _bf16(lo + np.abs(rng.standard_normal(n)) * 3 + 1e-2)
    x = np.empty((n, 32), dtype=F)
    x[:, 0], x[:, 1] = lo, hi
    z = lo.astype(np.float16).astype(F)
    s = ((hi - lo) / F(3)).astype(np.float16).astype(F)
    for j in range(2, 32):
        k = rng.choice([1, 3, 5])
        t = (z + F(k / 2) * s).astype(F)
        tb = f32_to_bf16_bits(t)
        b = (tb.astype(np.int32) + rng.integers(-1, 2, n)) & 0xFFFF   # a bf16 ulp either way
        near = bf16_bits_to_f32(b.astype(np.uint16))
        near = np.where(np.isfinite(near) & (tb & 0x7FFF != 0), near, bf16_bits_to_f32(tb))
        x[:, j] = np.clip(near, lo, hi)
    codes = _check(x)
    assert set(np.unique(codes)) == {0, 1, 2, 3}


def test_constant_and_two_valued_groups():
    x = np.full((4, 32), 2.5, dtype=F)
    x[1] = -1.0
    x[2, ::2], x[2, 1::2] = 0.0, 1.0                 # two values: codes 0 and 3
    x[3] = _bf16(np.linspace(-1, 1, 32))
    codes = _check(x)
    assert not codes[0].any() and not codes[1].any()  # scale 0: every code 0
    assert set(codes[2].tolist()) == {0, 3}

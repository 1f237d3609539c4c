"""The scorer folds the layer-sequential EMA in four layer segments (the
scoring kernel and the fused step alike; eight are modelled too): the first
from the stored score, the others from 0, then chains them in layer order as
m <- (1 - alpha)^n m + c_k (the fold is affine in its start; the host forms
the power in fp64 and rounds it to fp32 once).  Restated in
fp32, with fmaf emulated through fp64 and products and sums rounded to fp32 as
on the device, this is as accurate as a plain sequential fp32 fold.  Both are
compared with the fp64 fold, for every alpha of the workloads and 32 or 36
layers.

The rounding error of any fp32 fold grows with the score: about 4.5e-7 * m.
It is within the 1e-5 score tolerance up to head sums of 16, and reaches
1.5e-5 at 32, the most a layer of 32 summed heads can give (every head on one
token)."""
import numpy as np
import pytest

F = np.float32


def fmaf(a, b, c):
    return F(np.float64(a) * np.float64(b) + np.float64(c))


def segmented(m0, s, alpha, segs=4):
    n = len(s)
    oma = F(1.0) - F(alpha)
    cs = []
    for k in range(segs):
        la, lb = k * n // segs, (k + 1) * n // segs
        c = F(m0) if k == 0 else F(0)
        for layer in range(la, lb):
            c = fmaf(F(alpha), F(s[layer]), F(oma * c))
        cs.append((la, lb, c))
    m = cs[0][2]
    for la, lb, c in cs[1:]:
        decay = 1.0                   # (1 - alpha)^n in fp64, rounded once
        for _ in range(la, lb):
            decay *= float(oma)
        m = fmaf(F(decay), m, c)
    return float(m)


def sequential(m0, s, alpha):
    m = float(m0)
    for x in s:
        m = alpha * float(x) + (1.0 - alpha) * m
    return m


def plain_fp32(m0, s, alpha):
    m, oma = F(m0), F(1.0) - F(alpha)
    for x in s:
        m = fmaf(F(alpha), F(x), F(oma * m))
    return float(m)


@pytest.mark.parametrize("alpha", [0.01, 0.05, 0.15, 0.8])
@pytest.mark.parametrize("n_layers", [32, 36])
@pytest.mark.parametrize("top", [1.0, 4.0, 16.0, 32.0])
@pytest.mark.parametrize("segs", [4, 8])
def test_segmented_fold_is_as_accurate_as_a_sequential_fp32_fold(alpha, n_layers, top, segs):
    rng = np.random.default_rng(n_layers + int(top))
    worst_seg = worst_seq = 0.0
    for trial in range(200):
        s = (rng.uniform(0, top, n_layers) if trial % 5 else np.full(n_layers, top)).astype(F)
        m0 = F(rng.uniform(0, top))
        ref = sequential(m0, s, alpha)
        worst_seg = max(worst_seg, abs(segmented(m0, s, alpha, segs) - ref))
        worst_seq = max(worst_seq, abs(plain_fp32(m0, s, alpha) - ref))
    assert worst_seg <= 1.5 * worst_seq + 2 ** -24 * top, (worst_seg, worst_seq)
    assert worst_seg <= 6e-7 * top                 # fp32 resolution of scores up to `top`
    if top <= 16.0:
        assert worst_seg <= 1e-5


def test_four_layers_in_one_four_or_eight_segments():
    """p4's worked EMA inputs as four layers, folded whole, one layer per
    segment, or in eight segments of which four are empty: all within 1e-7
    of the fp64 fold."""
    s = np.array([0.45, 0.12, 0.30, 0.08], dtype=F)
    for segs in (1, 4, 8):
        got = segmented(F(0), s, 0.05, segs)
        assert abs(got - sequential(0.0, s, 0.05)) <= 1e-7

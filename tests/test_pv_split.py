"""Why the attention kernel feeds P to the P.V tensor-core product as two
bf16 parts.

The fp32 probabilities of a tile become the A operand of a bf16 mma.  Their
bf16 rounding alone (8 significant bits) puts an error of up to 2^-9 on each
weight.  With hi = bf16(p) and lo = bf16(p - hi), the pair keeps about 16
bits.  Restated in numpy, over many 2k-token rows of realistic logits:
- the output error relative to the row's largest output stays below 1e-5
  with the split (3.8e-6 seen);
- with hi alone it reaches 2.9e-3, beyond the 2e-3 output tolerance."""
import numpy as np

F = np.float32


def bf16_rn(x):
    u = np.asarray(x, F).view(np.uint32).astype(np.uint64)
    return (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16).astype(np.uint32).view(F)


def test_split_p_keeps_the_output_an_order_of_magnitude_closer():
    rng = np.random.default_rng(0)
    worst_split = worst_hi = 0.0
    for trial in range(60):
        L, d = 2048, 128
        logits = (rng.standard_normal(L) * (1.0, 2.5, 4.0)[trial % 3]).astype(F)
        v = bf16_rn(rng.standard_normal((L, d)).astype(F)).astype(np.float64)
        p = np.exp2(logits - logits.max()).astype(F)                # unnormalised, <= 1
        ref = (p.astype(np.float64) @ v) / p.astype(np.float64).sum()
        hi = bf16_rn(p)
        lo = bf16_rn((p - hi).astype(F))
        den = p.astype(np.float64).sum()
        out_split = ((hi.astype(np.float64) + lo.astype(np.float64)) @ v) / den
        out_hi = (hi.astype(np.float64) @ v) / den
        scale = np.abs(ref).max()
        worst_split = max(worst_split, np.abs(out_split - ref).max() / scale)
        worst_hi = max(worst_hi, np.abs(out_hi - ref).max() / scale)
    assert worst_split <= 1e-5, worst_split
    assert worst_hi > 2e-3, worst_hi            # hi alone would fail the output tolerance

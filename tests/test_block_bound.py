"""The host's bound on each sequence's live blocks never falls below the true
count.

kvev_paged_step refuses a step before launching when a sequence might need
more pages than it owns.  That needs an upper bound of the live blocks,
kept on the host without reading the device back:
- the prefill's blocks at begin;
- after each step, one more, capped by the blocks a step can keep: the
  budget, the pinned prefill blocks when they are more, or the whole pool
  when decoded tokens are pinned;
- one more for each re-admission.
Restated here, that bound is checked against the oracle's live block count
after every step of random runs, re-admissions and pinned regions included."""
import numpy as np
import pytest

import oracle as O
from oracle import paged as PG


def _bits(x):
    from workloads import f32_to_bf16_bits
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


class HostBound:
    def __init__(self, nb0, budget, pps, pin_blocks=0, decode_pinned=False):
        self.u, self.budget, self.pps = nb0, budget, pps
        self.pin_blocks, self.decode_pinned = pin_blocks, decode_pinned

    def may_step(self):
        return self.u + 1 <= self.pps

    def after_step(self):
        cap = self.budget
        if self.decode_pinned:
            cap = self.pps
        elif self.pin_blocks > cap:
            cap = self.pin_blocks
        self.u = min(self.u + 1, cap)

    def may_readmit(self):
        return self.u + 2 <= self.pps

    def after_readmit(self):
        self.u += 1


@pytest.mark.parametrize("seed", range(6))
def test_bound_covers_the_live_blocks(seed):
    rng = np.random.default_rng(seed)
    page, Ly, Hq, Hkv, d = 4, 1, 2, 1, 8
    nb0 = int(rng.integers(1, 12))
    budget = int(rng.integers(1, 8))
    pps = nb0 + 40
    pinned_mode = seed % 3            # 0: no regions, 1: pinned prefill tokens, 2: pinned decode
    K = _bits(rng.standard_normal((Ly, Hkv, nb0 * page, d)))
    V = _bits(rng.standard_normal((Ly, Hkv, nb0 * page, d)))
    kw = {}
    pin_blocks = 0
    if pinned_mode:
        region = np.zeros(nb0 * page, dtype=np.int64)
        if pinned_mode == 1:
            pins = rng.choice(nb0, size=min(nb0, budget + 2), replace=False)
            region[pins * page] = 1
            pin_blocks = len(pins)
        kw = dict(region=region, pinned_regions=(False, True),
                  decode_region=1 if pinned_mode == 2 else 0)
    seq = PG.PagedSequence.from_prefill(K, V, page, **kw)
    P = O.OracleParams(Ly, Hq, Hkv, d, budget, 0.05, 0.001, O.AGE_SINCE_ACCESS, False)
    host = HostBound(nb0, budget, pps, pin_blocks, pinned_mode == 2)
    for t in range(1, 36):
        if not pinned_mode and t % 9 == 0 and host.may_readmit():
            if PG.readmit(seq, int(rng.integers(0, nb0)), t):
                pass
            host.after_readmit()
            assert len(seq.blocks) <= host.u
        assert host.may_step(), t
        q = _bits(rng.standard_normal((Ly, Hq, d)))
        kn = _bits(rng.standard_normal((Ly, Hkv, d)))
        PG.step(P, seq, t, True, q, kn, kn)
        host.after_step()
        assert len(seq.blocks) <= host.u, (t, len(seq.blocks), host.u)

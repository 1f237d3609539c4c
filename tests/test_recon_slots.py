"""Reconstruction slots of the rotary two-tier mode, restated on the host.

With rotary positions the INT2 windows are attended as bf16 reconstructions
held in 8 K_q pages set aside at the end of each sequence's range, one
8-page slot per INT2 window.  The device keeps a free-slot stack per
sequence:
- kvev_tier_begin frees every slot, the lowest on top;
- a routing event first pushes, in window order, the slots of windows
  leaving the INT2 tier (promoted or evicted), then pops one from the top,
  in window order, for every window entering it (first or later demotion),
  which the reconstruction kernel then fills; the launch is sized for the
  new INT2 count, an upper bound of the entering windows;
- the first step after a checkpoint import gives the e-th INT2 window slot e
  and frees the others.
Restated here and driven by the oracle's tier sequence over long runs, the
stack never runs dry, every INT2 window holds exactly one slot of its own,
and the windows reconstructed at each event are exactly those entering."""
import numpy as np
import pytest

from oracle import qevict as QE

SINKS, RECENT, W = 5, 32, 128


class Slots:
    """The device's slot bookkeeping for one sequence."""

    def __init__(self, k_quant):
        self.n = k_quant                       # slots set aside at begin
        self.free = list(range(self.n - 1, -1, -1))   # stack, top = end: lowest on top
        self.slot = {}                         # window -> slot

    def route(self, old, new):
        """old / new: tier of every window before / after the event.
        Returns the windows listed for reconstruction."""
        for w, (o, t) in enumerate(zip(old, new)):
            if o == QE.QUANT and t != QE.QUANT:
                self.free.append(self.slot.pop(w))
        listed = []
        for w, (o, t) in enumerate(zip(old, new)):
            if o != QE.QUANT and t == QE.QUANT:
                assert self.free, "the slot stack ran dry"
                self.slot[w] = self.free.pop()
                listed.append(w)
        return listed

    def rebuild(self, tiers):
        q = [w for w, t in enumerate(tiers) if t == QE.QUANT]
        self.slot = {w: e for e, w in enumerate(q)}
        self.free = list(range(self.n - 1, len(q) - 1, -1))


@pytest.mark.parametrize("prefill,k_full,k_quant,omega,steps,import_at", [
    (5 + 128 * 6 + 20, 2, 2, 8, 600, 203),
    (5 + 128 * 3 + 127, 1, 3, 3, 500, 150),
    (5 + 128 * 8, 0, 2, 1, 400, 77),         # no bf16 tier, routing every step
    (5 + 128 * 5 + 1, 1, 4, 2, 500, None),   # INT2 capacity above the routed windows at first
    (5 + 40, 2, 1, 5, 700, 400),             # no window at the start
])
def test_slots_follow_the_oracle_tiers(prefill, k_full, k_quant, omega, steps, import_at):
    P = QE.QParams(n_layers=1, n_q_heads=1, n_kv_heads=1, head_dim=32, k_full=k_full,
                   k_quant=k_quant, alpha=0.05, window=W, n_sink=SINKS, n_recent=RECENT,
                   omega=omega, group=32)
    rng = np.random.default_rng(prefill * 7 + steps)
    bits = lambda shape: rng.integers(0x3C00, 0x4000, size=shape, dtype=np.uint16)
    seq = QE.QSequence.from_prefill(P, bits((1, 1, prefill, 32)), bits((1, 1, prefill, 32)))
    slots = Slots(k_quant)
    entered = 0
    for t in range(1, steps + 1):
        if t == import_at:   # a resumed run: slots anew from the INT2 list
            slots.rebuild(seq.tiers())
        old = seq.tiers()
        QE.step(P, seq, t, bits((1, 1, 32)), bits((1, 1, 32)), bits((1, 1, 32)))
        new = seq.tiers()
        if t % omega == 0:
            old = old + [QE.UNROUTED] * (len(new) - len(old))   # a window formed this step
            listed = slots.route(old, new)
            entering = [w for w, (o, n) in enumerate(zip(old, new))
                        if o != QE.QUANT and n == QE.QUANT]
            assert listed == entering, t
            assert len(listed) <= new.count(QE.QUANT) <= k_quant, t   # the launch bound
            entered += len(listed)
        q = [w for w, x in enumerate(new) if x == QE.QUANT]
        assert sorted(slots.slot) == q, t                      # every INT2 window has a slot
        held = sorted(slots.slot.values())
        assert len(set(held)) == len(held) and all(0 <= s < k_quant for s in held), t
        assert sorted(held + slots.free) == list(range(k_quant)), t   # no slot lost
    assert entered > 0

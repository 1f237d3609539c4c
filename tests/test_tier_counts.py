"""The host's copy of the two-tier window counts follows the oracle.

Before each launch kvev_tier_step derives, on the host, the counts that size
its launches:
- formed windows, and tokens in the tail;
- the first window not yet routed;
- windows in the bf16 and INT2 tiers after a routing event.
Restated here, those counts must equal the ones read off the oracle's
windows after every step of long runs.  The runs use the workload's
geometry (5 sinks, 32 recent tokens, windows of 128) and several capacities
and routing intervals."""
import numpy as np
import pytest

from oracle import qevict as QE

SINKS, RECENT, W = 5, 32, 128


class HostCounts:
    """The host bookkeeping of kvev_tier_begin / kvev_tier_step."""

    def __init__(self, prefill, k_full, k_quant, omega):
        hist = prefill - SINKS
        self.nw, self.tl = hist // W, hist % W
        self.first_u = self.nf = self.nq = 0
        self.len = prefill
        self.k_full, self.k_quant, self.omega = k_full, k_quant, omega

    def step(self, t):
        nw, tl = self.nw, self.tl + 1
        if tl == W:
            nw, tl = nw + 1, 0
        L = self.len + 1
        if t % self.omega == 0:
            horizon = L - RECENT
            aged_total = (horizon - SINKS) // W if horizon >= SINKS + W else 0
            n_aged = max(0, min(nw, aged_total) - self.first_u)
            n_cand = self.nf + self.nq + n_aged
            nf2 = min(self.k_full, n_cand)
            nq2 = min(self.k_quant, n_cand - nf2)
            self.first_u += n_aged
            self.nf, self.nq = nf2, nq2
        self.nw, self.tl, self.len = nw, tl, L


@pytest.mark.parametrize("prefill,k_full,k_quant,omega,steps", [
    (5 + 128 * 6 + 20, 2, 2, 8, 600),
    (5 + 128 * 3 + 127, 1, 3, 3, 500),
    (5 + 40, 3, 1, 5, 700),            # no window yet at the start
    (5 + 128 * 8, 0, 2, 1, 400),       # no bf16 tier, routing every step
    (5 + 128 * 4 + 1, 10, 10, 8, 400), # capacity above the window count
])
def test_host_counts_follow_the_oracle(prefill, k_full, k_quant, omega, steps):
    P = QE.QParams(n_layers=1, n_q_heads=1, n_kv_heads=1, head_dim=32, k_full=k_full,
                   k_quant=k_quant, alpha=0.05, window=W, n_sink=SINKS, n_recent=RECENT,
                   omega=omega, group=32)
    rng = np.random.default_rng(prefill + steps)
    bits = lambda shape: rng.integers(0x3C00, 0x4000, size=shape, dtype=np.uint16)   # bf16 in [0.0078, 2)
    seq = QE.QSequence.from_prefill(P, bits((1, 1, prefill, 32)), bits((1, 1, prefill, 32)))
    host = HostCounts(prefill, k_full, k_quant, omega)
    for t in range(1, steps + 1):
        QE.step(P, seq, t, bits((1, 1, 32)), bits((1, 1, 32)), bits((1, 1, 32)))
        host.step(t)
        tiers = seq.tiers()
        assert host.nw == len(seq.windows), t
        assert host.tl == seq.K_tail.shape[2], t
        assert host.first_u == sum(x != QE.UNROUTED for x in tiers), t
        assert host.nf == tiers.count(QE.FULL) and host.nq == tiers.count(QE.QUANT), t
        assert host.len == seq.L

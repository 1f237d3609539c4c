"""The compaction's reused-prefix rule, restated on row labels, keeps the cache
exact over long random runs.

The rule, as the compaction applies it:
- Two buffers take turns being live.
- The count vp[step parity] says how many leading rows the other buffer still
  shares with the live one.
- A step that evicts writes retained row R[j] to row j of the other buffer,
  except rows below min(vp_in, first_moved). Those already match, because
  R[j] = j below first_moved. That buffer then becomes live.
- The next count is first_moved.
- A step that evicts nothing (the cache within the budget) copies nothing
  and carries the count over to the next parity.
- A reset (kvev_init_state, kvev_import_state) sets both counts to 0.

The restatement tracks which token each row of both buffers holds, so one row
left uncopied by mistake shows up as a wrong label."""
import numpy as np
import pytest


def run(rng, L0, budget, steps, reset_every=0, evict_tail_prob=0.2):
    cap = max(L0, budget) + steps + 2
    buf = [np.full(cap, -1, dtype=np.int64), np.full(cap, -2, dtype=np.int64)]
    buf[0][:L0] = np.arange(L0)                # token ids of the prefill
    live, n, next_tok = 0, L0, L0
    vp = [0, 0]
    for step in range(1, steps + 1):
        if reset_every and step % reset_every == 0:
            vp = [0, 0]                          # init_state / import_state
        buf[live][n] = next_tok                  # append the new token at row n
        want = list(buf[live][:n + 1])
        next_tok += 1
        L = n + 1
        vp_in = vp[step & 1]
        if L <= budget:                          # nothing evicted
            vp[(step + 1) & 1] = vp_in
            n = L
            assert list(buf[live][:n]) == want
            continue
        if rng.random() < evict_tail_prob:       # evict only trailing rows
            keep = np.arange(budget)
        else:
            keep = np.sort(rng.choice(L, size=budget, replace=False))
        moved = np.nonzero(keep != np.arange(budget))[0]
        first_moved = int(moved[0]) if len(moved) else budget
        skip = min(vp_in, first_moved)
        dst = buf[live ^ 1]
        dst[skip:budget] = buf[live][keep[skip:]]
        vp[(step + 1) & 1] = first_moved
        live ^= 1
        n = budget
        assert list(buf[live][:n]) == [want[k] for k in keep], f"step {step}"


@pytest.mark.parametrize("seed", range(6))
def test_random_runs_stay_exact(seed):
    rng = np.random.default_rng(seed)
    run(rng, L0=int(rng.integers(1, 60)), budget=int(rng.integers(1, 40)), steps=400)


def test_runs_that_grow_into_the_budget_and_reset():
    rng = np.random.default_rng(7)
    run(rng, L0=3, budget=20, steps=300, reset_every=37)     # identity steps first
    run(rng, L0=50, budget=50, steps=300, evict_tail_prob=0.6)


def test_a_wrong_count_is_caught():
    """Carrying the old count over an evicting step (instead of first_moved)
    leaves stale rows; the restatement sees them."""
    cap, budget = 80, 16
    a = np.arange(cap)
    b = np.full(cap, -1)
    b[:budget] = a[:budget]                      # the other buffer shares 16 rows
    keep = np.delete(np.arange(budget + 1), 5)   # token 5 evicted: rows 5.. shift
    first_moved = int(np.nonzero(keep != np.arange(budget))[0][0])
    skip_wrong = budget                          # vp_in instead of min(vp_in, first_moved)
    dst = b.copy()
    dst[skip_wrong:budget] = a[keep[skip_wrong:]]
    assert first_moved < budget and list(dst[:budget]) != list(a[keep])

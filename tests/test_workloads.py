"""The seeded input generators keep the recipe the design states: bf16
rounding to nearest-even, per-step draws that do not depend on the order in
which steps are drawn, outlier key channels, heavy-hitter rows, and a query
pulled toward the mean key of a needle set that is re-drawn every P steps."""
import numpy as np
import pytest

from workloads import (Geometry, Workload, bf16_bits_to_f32, f32_to_bf16_bits,
                       llama8b_workload, paged_workload, region_labels, tiny_workload)


def test_bf16_rounding_is_nearest_even():
    one = 1.0
    ulp = 2.0 ** -7                       # bf16 spacing at 1
    x = np.array([one, one + ulp / 2, one + 3 * ulp / 2, one + ulp / 2 + 2 ** -20, -2.5],
                 dtype=np.float32)
    got = f32_to_bf16_bits(x)
    assert got[0] == 0x3F80
    assert got[1] == 0x3F80               # tie: down to the even mantissa
    assert got[2] == 0x3F82               # tie: up to the even mantissa
    assert got[3] == 0x3F81               # above the tie: up
    assert got[4] == 0xC020
    assert np.array_equal(bf16_bits_to_f32(f32_to_bf16_bits(bf16_bits_to_f32(got))),
                          bf16_bits_to_f32(got))   # bf16 values round to themselves


def test_step_draws_do_not_depend_on_order():
    a = Workload(Geometry(2, 8, 2, 64, 2), 100, seed=7, outliers=2, needle=4, needle_period=3)
    b = Workload(Geometry(2, 8, 2, 64, 2), 100, seed=7, outliers=2, needle=4, needle_period=3)
    late = b.step_inputs(5)
    for t in (1, 2, 3, 4):
        a.step_inputs(t)
    for x, y in zip(a.step_inputs(5), late):
        assert np.array_equal(x, y)
    c = Workload(Geometry(2, 8, 2, 64, 2), 100, seed=8, outliers=2, needle=4, needle_period=3)
    assert not np.array_equal(c.step_inputs(5)[0], late[0])


def test_outlier_channels_and_heavy_rows():
    wl = Workload(Geometry(1, 4, 1, 64, 1), 4096, seed=3, outliers=4, outlier_sigma=8.0,
                  heavy=8, heavy_scale=4.0)
    k, v = wl.prefill()
    kf = bf16_bits_to_f32(k[0, 0, 0]).astype(np.float64)          # [L0][d]
    normal = np.setdiff1d(np.arange(wl.L0), wl.heavy_positions)
    std = kf[normal].std(axis=0)
    out = wl.outlier_channels
    assert len(out) == 4 and np.all(np.abs(std[out] - 8.0) < 0.5)
    rest = np.setdiff1d(np.arange(64), out)
    assert np.all(np.abs(std[rest] - 1.0) < 0.06)
    assert abs(bf16_bits_to_f32(v[0, 0, 0]).std() - 1.0) < 0.01
    # heavy rows are the same draw scaled by 4 (exactly, before the bf16 rounding)
    plain = Workload(Geometry(1, 4, 1, 64, 1), 4096, seed=3, outliers=4, outlier_sigma=8.0)
    kp = bf16_bits_to_f32(plain.prefill()[0][0, 0, 0])
    hp = wl.heavy_positions
    assert np.array_equal(bf16_bits_to_f32(k[0, 0, 0])[hp], kp[hp] * 4.0)


def test_needle_is_redrawn_every_period_and_pulls_the_query():
    wl = Workload(Geometry(2, 8, 2, 64, 1), 300, seed=5, needle=16, needle_period=4,
                  needle_weight=0.5)
    assert np.array_equal(wl.needle_positions(1), wl.needle_positions(4))
    assert not np.array_equal(wl.needle_positions(4), wl.needle_positions(5))
    pos = wl.needle_positions(2)
    assert len(np.unique(pos)) == 16 and pos.min() >= 0 and pos.max() < 300
    # q = N(0,1) draw + 0.5 * the mean needle key of the query head's KV head
    plain = Workload(Geometry(2, 8, 2, 64, 1), 300, seed=5)
    q = bf16_bits_to_f32(wl.step_inputs(2)[0]).astype(np.float64)     # [b][Ly][Hq][d]
    q0 = bf16_bits_to_f32(plain.step_inputs(2)[0]).astype(np.float64)
    k = bf16_bits_to_f32(wl.prefill()[0]).astype(np.float64)          # [Ly][b][g][L0][d]
    mean = k[:, 0][:, :, pos, :].mean(axis=2)                         # [Ly][g][d]
    want = q0[0] + 0.5 * np.repeat(mean, 4, axis=1)
    # q and the plain draw q0 are each a bf16 rounding (unit roundoff 2^-8)
    assert np.all(np.abs(q[0] - want) <= 2.0 ** -8 * (np.abs(q[0]) + np.abs(q0[0])) + 1e-6)
    # a query without the pull, or with the full mean, misses by far more
    for w in (0.0, 1.0):
        other = q0[0] + w * np.repeat(mean, 4, axis=1)
        assert np.abs(q[0] - other).max() > 0.05


def test_named_workloads_have_the_stated_shapes():
    t = tiny_workload()
    assert (t.geom, t.L0, len(t.heavy_positions)) == (Geometry(1, 8, 2, 64, 1), 512, 8)
    ll = llama8b_workload(prefill_len=64, n_layers=2)
    assert (ll.geom.n_q_heads, ll.geom.n_kv_heads, ll.geom.head_dim) == (32, 8, 128)
    assert (len(ll.outlier_channels), ll.needle, ll.needle_period) == (4, 16, 50)
    assert llama8b_workload().L0 == 32768 and llama8b_workload().geom.n_layers == 32
    pg = paged_workload(prefill_len=64, n_layers=2, batch=2)
    assert (pg.needle, pg.needle_period) == (16, 200)
    lab = region_labels(16384)
    assert np.array_equal(np.bincount(lab), [819, 819, 1638, 4915, 4915, 3278])
    assert np.all(np.diff(lab.astype(int)) >= 0)                      # contiguous spans in order


@pytest.mark.parametrize("step", [0, -1])
def test_steps_are_numbered_from_one(step):
    with pytest.raises(ValueError):
        tiny_workload().step_inputs(step)


def test_rotary_keys_keep_position_zero_and_pair_norms():
    """With rope_base the cache holds rotated keys: position 0 is the drawn
    key itself (angle 0), every (j, j + d/2) pair keeps its length up to the
    bf16 rounding, and the table is cos / sin of p * base^(-2 j / d)."""
    from workloads import Geometry, Workload, bf16_bits_to_f32
    g = Geometry(1, 4, 1, 64, 1)
    plain = Workload(g, 40, seed=4)
    rot = Workload(g, 40, seed=4, rope_base=10000.0)
    kp = bf16_bits_to_f32(plain.prefill()[0]).astype(np.float64)
    kr = bf16_bits_to_f32(rot.prefill()[0]).astype(np.float64)
    assert np.array_equal(kp[..., 0, :], kr[..., 0, :])
    np_, nr = kp[..., :32] ** 2 + kp[..., 32:] ** 2, kr[..., :32] ** 2 + kr[..., 32:] ** 2
    assert np.allclose(nr, np_, rtol=2e-2, atol=1e-3)
    t = rot.rope_table(41)
    assert t.shape == (41, 32, 2) and t.dtype == np.float32
    assert t[7, 5, 0] == np.float32(np.cos(7 * 10000.0 ** (-10 / 64)))
    assert t[7, 5, 1] == np.float32(np.sin(7 * 10000.0 ** (-10 / 64)))

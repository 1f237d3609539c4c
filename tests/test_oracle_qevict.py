"""Pins for the two-tier (QEvict) window-routing oracle and its INT2 codec."""
import numpy as np
import pytest

from oracle import qevict as QE
from workloads import f32_to_bf16_bits


def _bits(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _params(**kw):
    base = dict(n_layers=1, n_q_heads=1, n_kv_heads=1, head_dim=32, k_full=1, k_quant=1,
                alpha=0.05, window=32, n_sink=1, n_recent=2, omega=1, group=32)
    base.update(kw)
    return QE.QParams(**base)


def test_tier_capacities_worked_example():
    """Sec. 4.5: B_hist 100 MB, q = 0.70, 1 MB full and ~0.131 MB INT2 per
    window give K_f = 30 and K_q = 534."""
    assert QE.capacities(100.0, 0.70, 1.0, 0.131) == (30, 534)


def test_int2_footprint_per_token_layer():
    """Llama-8B geometry: bf16 K+V is 4096 B per token-layer; the INT2 tier
    holds 512 B of codes plus 256 B of fp16 scale/zero (groups of 32)."""
    assert QE.int2_bytes_per_token_layer(8, 128) == 768
    assert QE.int2_bytes_per_token_layer(8, 128, group=64) == 640


def test_codec_exact_on_representable_groups():
    """Values zero + code * scale with fp16-exact zero and scale come back
    bit for bit; the group's min codes to 0 and its max to 3."""
    x = np.array([[1.0, 1.5, 2.0, 2.5] * 8], dtype=np.float32)      # one group of 32
    codes, scale, zero = QE.quantize_groups(x, axis=1)
    assert float(zero[0]) == 1.0 and float(scale[0]) == 0.5
    assert codes[0].tolist() == [0, 1, 2, 3] * 8
    assert np.array_equal(QE.dequantize(codes, scale, zero, axis=1), x)


def test_codec_error_bound_and_constant_groups():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((64, 32)).astype(np.float32) * 3
    codes, scale, zero = QE.quantize_groups(x, axis=1)
    assert codes.min() >= 0 and codes.max() <= 3
    xh = QE.dequantize(codes, scale, zero, axis=1)
    s = scale.astype(np.float32)[:, None]
    slack = np.abs(zero.astype(np.float32) - x.min(axis=1))[:, None] + 1e-6 * np.abs(x)
    assert np.all(np.abs(x - xh) <= 0.5 * s + slack + 1e-6)
    c = np.full((2, 32), 0.75, np.float32)                            # max = min: scale 0
    codes, scale, zero = QE.quantize_groups(c, axis=1)
    assert np.all(scale == 0) and np.all(codes == 0)
    assert np.array_equal(QE.dequantize(codes, scale, zero, axis=1), c)


def test_keys_per_channel_values_per_token():
    """Keys constant along tokens within a channel and values constant along
    channels within a token quantize with scale 0 and come back exactly;
    the other orientation would spread each group over distinct values."""
    W, d = 64, 64
    k = np.tile(np.arange(d, dtype=np.float32) / 8, (W, 1))           # varies by channel
    v = np.tile(np.arange(W, dtype=np.float32)[:, None] / 8, (1, d))  # varies by token
    led = QE.quantize_window(_bits(k)[None, None], _bits(v)[None, None], group=32)
    assert np.all(led["ks"] == 0) and np.all(led["vs"] == 0)
    kd, vd = QE.dequantize_window(led)
    assert np.array_equal(kd[0, 0], k) and np.array_equal(vd[0, 0], v)


def test_window_partition():
    """Sinks [0, 5), windows of 128 from position 5, the rest is the tail:
    131072 tokens make 1023 windows and a 123-token tail."""
    P = _params(window=128, n_sink=5)
    z = np.zeros((1, 1, 5 + 128 * 3 + 10, 32), np.uint16)
    seq = QE.QSequence.from_prefill(P, z, z)
    assert len(seq.windows) == 3 and seq.K_tail.shape[2] == 10 and seq.K_sink.shape[2] == 5
    assert (131072 - 5) // 128 == 1023 and (131072 - 5) % 128 == 123
    # a window needs all of its 128 positions after the sinks: one short of
    # two windows leaves one window and a 127-token tail
    for L0, nw, tail in ((5 + 128 * 2 - 1, 1, 127), (5 + 128, 1, 0), (5 + 127, 0, 127)):
        z = np.zeros((1, 1, L0, 32), np.uint16)
        seq = QE.QSequence.from_prefill(P, z, z)
        assert (len(seq.windows), seq.K_tail.shape[2]) == (nw, tail)
        assert [seq.window_end(P, w) for w in seq.windows] == [5 + 128 * (j + 1) for j in range(nw)]


def test_attention_is_the_scaled_softmax_over_gqa_groups():
    """The tier oracle's own attention: two keys give the logistic of the
    logit difference q.(k1 - k2) / sqrt(d); query heads 2h, 2h + 1 read KV
    head h (Hq = 4, Hkv = 2); the output is the probability-weighted sum of
    the values."""
    d = 16
    q = np.zeros((4, d), np.float32)
    q[:, 0] = [1.0, 2.0, 3.0, -1.0]
    K = np.zeros((2, 2, d), np.float32)
    K[0, 0, 0], K[0, 1, 0] = 2.0, -2.0             # KV head 0: logit gap 4 q0 / 4
    K[1, 0, 0], K[1, 1, 0] = -1.0, 3.0             # KV head 1: logit gap -4 q0 / 4
    V = np.zeros((2, 2, d), np.float32)
    V[:, 0, 1], V[:, 1, 1] = 10.0, -6.0
    p, out = QE.attention_f64(q, K, V)
    gap = np.array([1.0, 2.0, -3.0, 1.0])          # (l0 - l1) per query head
    p0 = 1.0 / (1.0 + np.exp(-gap))
    assert np.allclose(p[:, 0], p0, rtol=1e-14, atol=0)
    assert np.allclose(p.sum(axis=1), 1.0, rtol=1e-15, atol=0)
    assert np.allclose(out[:, 1], 10.0 * p0 - 6.0 * (1.0 - p0), rtol=1e-13, atol=0)
    assert not out[:, 0].any() and not out[:, 2:].any()


def test_window_score_is_a_layer_sequential_ema_of_head_mean_mass():
    """Uniform attention (zero keys): every token gets 1/n in every head, so
    a window's per-layer mass is W/n and after one step over Ly layers its
    score is (1 - (1 - alpha)^Ly) W / n."""
    P = _params(n_layers=3, n_q_heads=2, n_kv_heads=1, alpha=0.2, omega=100)
    z = np.zeros((3, 1, 1 + 32 * 2 + 3, 32), np.uint16)
    seq = QE.QSequence.from_prefill(P, z, z)
    zq = np.zeros((3, 2, 32), np.uint16)
    zk = np.zeros((3, 1, 32), np.uint16)
    res = QE.step(P, seq, 1, zq, zk, zk)
    n = 1 + 64 + 4
    want = (1 - 0.8 ** 3) * 32 / n
    assert res["m"][0] == pytest.approx(want, rel=1e-12)
    assert res["m"][1] == pytest.approx(want, rel=1e-12)


def test_cumulative_window_score_sums_every_layer_and_step():
    """Eq. (1) as the cumulative mode reads it: with uniform attention a
    window's per-layer mass at a step over n cached tokens is W/n, so after
    steps 1..3 (n = 69, 70, 71) over Ly layers its score is
    Ly W (1/69 + 1/70 + 1/71): nothing decays."""
    P = _params(n_layers=3, n_q_heads=2, n_kv_heads=1, alpha=0.2, omega=100, cumulative=True)
    z = np.zeros((3, 1, 1 + 32 * 2 + 3, 32), np.uint16)
    seq = QE.QSequence.from_prefill(P, z, z)
    zq = np.zeros((3, 2, 32), np.uint16)
    zk = np.zeros((3, 1, 32), np.uint16)
    for t in (1, 2, 3):
        res = QE.step(P, seq, t, zq, zk, zk)
    want = 3 * 32 * (1 / 69 + 1 / 70 + 1 / 71)
    assert res["m"][0] == pytest.approx(want, rel=1e-12)
    assert res["m"][1] == pytest.approx(want, rel=1e-12)


def _seq_with_scores(P, scores, tail=3):
    nw = len(scores)
    rng = np.random.default_rng(1)
    K = _bits(rng.standard_normal((1, 1, P.n_sink + P.window * nw + tail, P.head_dim)))
    seq = QE.QSequence.from_prefill(P, K, K.copy())
    for w, m in zip(seq.windows, scores):
        w.m = m
    return seq


def test_routing_top_k_full_next_k_quantized_rest_evicted():
    """Eq. (5): rank candidates by score (ties: lower index first); the top
    K_f are Full, the next K_q Quantized, the rest Evicted; a window not yet
    aged out of the recent region is no candidate."""
    P = _params(k_full=2, k_quant=1, n_recent=34)
    seq = _seq_with_scores(P, [0.1, 0.5, 0.3, 0.3, 0.9, 0.0, 0.7], tail=3)
    # L = 1 + 7*32 + 3 = 228, horizon 194: window 6 (ends at 225) is not aged;
    # windows 2 and 3 tie and the lower index takes the one quantized slot
    QE.route(P, seq)
    assert seq.tiers() == ["E", "F", "Q", "E", "F", "E", "U"]
    QE.route(P, seq)                                # evicted windows never come back
    assert seq.tiers()[0] == "E" and seq.tiers()[3] == "E" and seq.tiers()[5] == "E"
    assert seq.windows[2].ledger is not None and seq.windows[2].K is None


def test_routing_runs_at_the_end_of_every_omega_th_step():
    """This build's reading of the routing time (the page gives Omega, not
    where in a step routing falls): an event at the end of each step t with
    t mod Omega = 0, taking effect from the next step.  Omega = 3, one
    candidate window, no capacity for it: it is evicted after step 3 and
    attended until then."""
    P = _params(k_full=0, k_quant=0, n_recent=1, omega=3)
    rng = np.random.default_rng(5)
    K = _bits(rng.standard_normal((1, 1, P.n_sink + P.window + 2, P.head_dim)))
    seq = QE.QSequence.from_prefill(P, K, K.copy())
    routed = []
    for t in range(1, 7):
        q, kn = (_bits(rng.standard_normal(shape)) for shape in ((1, 1, 32), (1, 1, 32)))
        res = QE.step(P, seq, t, q, kn, kn)
        routed.append(res["routed"])
        attended = (res["owner"] == 0).any()
        assert attended == (t <= 3)
    assert routed == [False, False, True, False, False, True]
    assert seq.tiers() == ["E"]


def test_ledger_is_reused_across_migrations():
    """A window is quantized on its first demotion only; promoted, it holds
    the bf16 rounding of its dequantized values; demoted again it keeps the
    ledger entry of the first demotion."""
    P = _params(k_full=1, k_quant=1, n_recent=1)
    seq = _seq_with_scores(P, [0.2, 0.8], tail=1)
    QE.route(P, seq)                                # window 0 -> Q (first quantization)
    led = seq.windows[0].ledger
    first = {k: v.copy() for k, v in led.items() if isinstance(v, np.ndarray)}
    assert seq.windows[0].K is None                 # the full-precision copy is dropped
    seq.windows[0].m, seq.windows[1].m = 0.9, 0.1
    QE.route(P, seq)                                # promote 0, demote 1
    w0 = seq.windows[0]
    kd, vd = QE.dequantize_window(w0.ledger)
    assert w0.tier == "F" and np.array_equal(w0.K, _bits(kd)) and np.array_equal(w0.V, _bits(vd))
    seq.windows[0].m, seq.windows[1].m = 0.1, 0.9
    QE.route(P, seq)                                # demote 0 again: same codes
    assert seq.windows[0].ledger is led             # the ledger entry itself is reused
    for k in first:
        assert np.array_equal(seq.windows[0].ledger[k], first[k])


def test_evicted_window_no_longer_attended_and_quantized_one_is():
    """A window whose keys would take nearly all attention stops affecting
    the output once evicted; a quantized window with fp16-exact values is
    attended exactly as its dequantized values say."""
    P = _params(k_full=0, k_quant=1, n_recent=1, omega=1)
    d = 32
    K = np.zeros((1, 1, 1 + 64 + 1, d), np.float32)
    V = np.zeros_like(K)
    K[0, 0, 1:33, 0] = 20.0                         # window 0: dominant keys
    V[0, 0, 1:33, 1] = 7.0
    V[0, 0, 33:65, 2] = np.tile([0.75, 1.5, 3.0, 6.0], 8)   # window 1: val/3 fp16-exact
    seq = QE.QSequence.from_prefill(P, _bits(K), _bits(V))
    seq.windows[0].m, seq.windows[1].m = 0.0, 1.0
    QE.route(P, seq)
    assert seq.tiers() == ["E", "Q"]
    q = np.zeros((1, 1, d), np.float32)
    q[0, 0, 0] = 1.0
    z = np.zeros((1, 1, d), np.float32)
    res = QE.step(P, seq, 3, _bits(q), _bits(z), _bits(z))
    out = res["out"][0, 0]
    # accessible: sink (0), window 1 (32 tokens), tail token, new token: all logits 0
    n = 1 + 32 + 2
    assert out[1] == pytest.approx(0.0, abs=1e-15)
    assert out[2] == pytest.approx(np.tile([0.75, 1.5, 3.0, 6.0], 8).sum() / n, rel=1e-12)


# ---- rotary positions (Sec. 4.4: pre-rotation quantization, rotation re-applied)
def _table(n_pos, half, cos, sin):
    t = np.zeros((n_pos, half, 2), np.float32)
    t[..., 0], t[..., 1] = cos, sin
    return t


def test_quarter_turn_quantizes_the_swapped_keys():
    """With every angle a quarter turn (cos 0, sin 1) the key rotated back is
    (x_{j+d/2}, -x_j): exact in fp32.  So the ledger of a window quantized
    with that table holds exactly the codes, scales and zeros of the same
    window with its key halves swapped and the second half negated,
    quantized without rotation; the values are untouched."""
    P = _params(k_full=0, k_quant=1, n_recent=1)
    Pr = _params(k_full=0, k_quant=1, n_recent=1,
                 rope=_table(1 + 32 + 8, 16, 0.0, 1.0))
    rng = np.random.default_rng(3)
    K = _bits(rng.standard_normal((1, 1, 1 + 32 + 1, 32)))
    V = _bits(rng.standard_normal((1, 1, 1 + 32 + 1, 32)))
    kf = (K.astype(np.uint32) << 16).view(np.float32)
    swapped = np.concatenate([kf[..., 16:], -kf[..., :16]], axis=-1)
    seq_r = QE.QSequence.from_prefill(Pr, K, V)
    seq_p = QE.QSequence.from_prefill(P, _bits(swapped), V)
    QE.route(Pr, seq_r)
    QE.route(P, seq_p)
    a, b = seq_r.windows[0].ledger, seq_p.windows[0].ledger
    for k in ("kq", "vq"):
        assert np.array_equal(a[k], b[k])
    for k in ("ks", "kz", "vs", "vz"):
        assert np.array_equal(a[k].view(np.uint16), b[k].view(np.uint16))


def test_quarter_turn_promotion_rotates_the_dequantized_keys_forward():
    """Promoted under a quarter turn, the bf16 key is the forward rotation
    (-x_{j+d/2}, x_j) of the dequantized pre-rotation key: with the ledger
    of the swapped keys (previous pin) that is the plain promotion with the
    halves swapped back and negated."""
    Pr = _params(k_full=1, k_quant=1, n_recent=1, rope=_table(1 + 64 + 8, 16, 0.0, 1.0))
    seq = _seq_with_scores(Pr, [0.2, 0.8], tail=1)
    QE.route(Pr, seq)                        # window 0 -> Q
    seq.windows[0].m, seq.windows[1].m = 0.9, 0.1
    QE.route(Pr, seq)                        # promote window 0
    w0 = seq.windows[0]
    kd, vd = QE.dequantize_window(w0.ledger)            # no rotation
    fwd = np.concatenate([-kd[..., 16:], kd[..., :16]], axis=-1)
    assert w0.tier == "F"
    assert np.array_equal(w0.K, _bits(fwd)) and np.array_equal(w0.V, _bits(vd))


def test_rotation_round_trip_and_pair_norms():
    """Any angle: back then forward returns the key within fp32 rounding,
    and each (j, j + d/2) pair keeps its length."""
    rng = np.random.default_rng(5)
    ang = rng.uniform(0, 2 * np.pi, (64, 16))
    cs = np.stack([np.cos(ang), np.sin(ang)], axis=-1).astype(np.float32)
    x = rng.standard_normal((3, 64, 32)).astype(np.float32)
    y = QE.rotate(x, cs)
    back = QE.rotate(y, cs, back=True)
    assert np.abs(back - x).max() <= 1e-6 * np.abs(x).max()
    n0 = x[..., :16] ** 2 + x[..., 16:] ** 2
    n1 = y[..., :16].astype(np.float64) ** 2 + y[..., 16:].astype(np.float64) ** 2
    assert np.allclose(n1, n0, rtol=1e-6)


def test_identity_table_routes_and_quantizes_as_without_rotation():
    """cos 1, sin 0 everywhere: the same tiers and ledgers as without a
    table, and the same promoted pages."""
    P = _params(k_full=1, k_quant=1, n_recent=1)
    Pr = _params(k_full=1, k_quant=1, n_recent=1, rope=_table(1 + 64 + 8, 16, 1.0, 0.0))
    seq_p = _seq_with_scores(P, [0.2, 0.8], tail=1)
    seq_r = _seq_with_scores(Pr, [0.2, 0.8], tail=1)
    for m in ((0.2, 0.8), (0.9, 0.1)):
        for s_ in (seq_p, seq_r):
            s_.windows[0].m, s_.windows[1].m = m
        QE.route(P, seq_p)
        QE.route(Pr, seq_r)
        assert seq_p.tiers() == seq_r.tiers()
    for a, b in zip(seq_p.windows, seq_r.windows):
        if a.K is not None:
            assert np.array_equal(a.K, b.K) and np.array_equal(a.V, b.V)
        if a.ledger is not None:
            assert np.array_equal(a.ledger["kq"], b.ledger["kq"])


def test_reconstructed_int2_window_is_attended_in_bf16():
    """With a table, attention sees an INT2 window as its reconstruction in
    bf16.  All keys 0 give every token the same weight, so the output is the
    mean of the values: a value group holding 0 and 1 has scale
    fp16(1/3) = 0.333251953125 and dequantizes to 0, s, 2 s, 3 s, which bf16
    rounds to 0, 0.333984375, 0.66796875, 1.0; without a table the fp32
    values are attended."""
    d = 32
    K = np.zeros((1, 1, 1 + 32 + 1, d), np.float32)
    V = np.zeros_like(K)
    V[0, 0, 1:33, :] = np.tile([0.0, 1.0], 16)[None, :]    # every value group spans [0, 1]
    V[0, 0, 1:33, 0] = np.tile([0.0, 1.0 / 3, 2.0 / 3, 1.0], 8)
    out = {}
    for name, rope in (("plain", None), ("rope", _table(64, 16, 1.0, 0.0))):
        P = _params(k_full=0, k_quant=1, n_recent=1, rope=rope)
        seq = QE.QSequence.from_prefill(P, _bits(K), _bits(V))
        QE.route(P, seq)
        assert seq.tiers() == ["Q"]
        z = np.zeros((1, 1, d), np.float32)
        out[name] = QE.step(P, seq, 2, _bits(z), _bits(z), _bits(z))["out"][0, 0, 0]
    led_codes = [0, 1, 2, 3] * 8                    # channel 0 per token: 0, 1/3, 2/3, 1
    s32 = np.float32(np.float16(np.float32(1.0) / np.float32(3.0)))
    deq = np.array([np.float32(c) * s32 for c in led_codes], np.float32)
    bf = {0: 0.0, 1: 0.333984375, 2: 0.66796875, 3: 1.0}
    n = 1 + 32 + 2                                  # sink, window, tail token, new token
    assert out["rope"] == pytest.approx(sum(bf[c] for c in led_codes) / n, rel=1e-12)
    assert out["plain"] == pytest.approx(float(deq.astype(np.float64).sum()) / n, rel=1e-12)


def test_reconstructed_keys_are_bf16_in_the_logits():
    """Key channel 0 of an INT2 window spans [0, 1] (scale fp16(1/3), codes
    0-3); the query reads only that channel.  With a table the logits use the
    bf16 reconstruction 0, 0.333984375, 0.66796875, 1.0 of the dequantized
    keys, and the values (code 3 of scale fp16(1/3)) are bf16(0.999755859375)
    = 1.0; every other token has key 0 and value 0.  Closed form: out_1 =
    sum_i e^(8 k_i / sqrt(32)) / (sum_i e^(8 k_i / sqrt(32)) + 3)."""
    d = 32
    K = np.zeros((1, 1, 1 + 32 + 1, d), np.float32)
    V = np.zeros_like(K)
    K[0, 0, 1:33, 0] = np.tile([0.0, 1.0 / 3, 2.0 / 3, 1.0], 8)
    V[0, 0, 1:33, 1] = 1.0
    P = _params(k_full=0, k_quant=1, n_recent=1, rope=_table(64, 16, 1.0, 0.0))
    seq = QE.QSequence.from_prefill(P, _bits(K), _bits(V))
    QE.route(P, seq)
    q = np.zeros((1, 1, d), np.float32)
    q[0, 0, 0] = 8.0
    z = np.zeros((1, 1, d), np.float32)
    out = QE.step(P, seq, 2, _bits(q), _bits(z), _bits(z))["out"][0, 0, 1]
    k = np.tile([0.0, 0.333984375, 0.66796875, 1.0], 8)
    w = np.exp(8.0 * k / np.sqrt(32.0))
    assert out == pytest.approx(w.sum() / (w.sum() + 3.0), rel=1e-12)

"""The oracle's pins catch plausible mistakes.

Each case plants ONE mistake in a scratch copy of the oracle: a dropped term,
a swapped operand, a wrong sign, index or comparison. It then runs the
CPU pin files on that copy, and at least one pin must fail.  The mistakes are
planted in the oracle only, on the CPU; nothing here touches the CUDA library.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PIN_FILES = ["test_oracle_pins.py", "test_oracle_scorers.py", "test_oracle_diagnostics.py",
             "test_oracle_paged.py", "test_oracle_memdecay.py", "test_oracle_qevict.py"]

# (oracle file, text, replacement, the mistake it models)
MUTANTS = [
    # token-granular oracle (C)
    ("kvev_oracle.c", "return alpha * new_score + (1.0 - alpha) * score;",
     "return (1.0 - alpha) * new_score + alpha * score;", "EMA weights swapped"),
    ("kvev_oracle.c", "double scale = 1.0 / sqrt((double)d);", "double scale = 1.0 / (double)d;",
     "logit scale 1/d"),
    ("kvev_oracle.c", "p[i] = dot * scale;", "p[i] = dot;", "logit scale dropped"),
    ("kvev_oracle.c", "for (int64_t i = 0; i < L; ++i) p[i] /= sum;", "", "softmax not normalised"),
    ("kvev_oracle.c", "out[h * d + c] += p[i] * bf16_to_double(vr[c]);",
     "out[h * d + c] += p[i] * bf16_to_double(vr[(c + 1) % d]);", "value channel off by one"),
    ("kvev_oracle.c", "memcpy(V + dst, v_new + ((int64_t)l * Hkv + g) * d",
     "memcpy(V + dst, k_new + ((int64_t)l * Hkv + g) * d", "new key appended as the value"),
    ("kvev_oracle.c", "if (x->pr < y->pr) return -1;", "if (x->pr > y->pr) return -1;",
     "highest priority kept"),
    ("kvev_oracle.c", "return (x->idx < y->idx) ? -1 : (x->idx > y->idx);",
     "return (x->idx > y->idx) ? -1 : (x->idx < y->idx);", "ties to the higher index"),
    ("kvev_oracle.c", "keys[i].pr = (pinned && pinned[i]) ? -INFINITY : pr[i];",
     "keys[i].pr = pr[i];", "pinning ignored"),
    ("kvev_oracle.c", "if (np > n) n = np;", "", "pinned units cut at the budget"),
    ("kvev_oracle.c", "qsort(kept, (size_t)n, sizeof(int64_t), kvo_idx_cmp);", "",
     "retained list not in slot order"),
    ("kvev_oracle.c", "double decay = (steps == 0) ? 0.0 : 1.0 - exp(-beta * (double)steps);",
     "double decay = 1.0 - exp(-beta * (double)steps);", "age 0 not protected at beta = inf"),
    ("kvev_oracle.c", "return (1.0 - score) * decay;", "return score * decay;",
     "priority without 1 - score"),
    ("kvev_oracle.c", "acc = mean_attn >= 2.0 / (double)L;", "acc = mean_attn >= 1.0 / (double)L;",
     "access threshold 1/L"),
    ("kvev_oracle.c", "acc = mean_attn >= 2.0 / (double)L;", "acc = mean_attn > 2.0 / (double)L;",
     "access threshold exclusive"),
    ("kvev_oracle.c", "double mean_attn = ssum[i] / ((double)Ly * (double)Hq);",
     "double mean_attn = ssum[i] / (double)Hq;", "access mass not averaged over layers"),
    ("kvev_oracle.c", "new_m = acc / (double)L_prev;", "new_m = 0.0;",
     "new token scores 0 off refresh steps"),
    ("kvev_oracle.c", "new_m = acc / (double)L_prev;", "new_m = acc / (double)L;",
     "mean momentum over the wrong count"),
    ("kvev_oracle.c", "if (P->pool_mean) s /= (double)Hq;", ";", "head mean ignored"),
    ("kvev_oracle.c", "if (!refresh) continue;", ";", "EMA on non-refresh steps"),
    ("kvev_oracle.c", "t_ins[L_prev] = t;", "t_ins[L_prev] = 0;", "new token's insertion step 0"),
    ("kvev_oracle.c", "t_ref[L_prev] = t;", "t_ref[L_prev] = 0;", "new token's clock 0"),
    ("kvev_oracle.c", "pos[L_prev] = new_pos;", "pos[L_prev] = L_prev;", "logical position lost"),
    ("kvev_oracle.c", "if (acc) t_ref[i] = t;", "if (acc) t_ins[i] = t;",
     "access resets the insertion step"),
    ("kvev_oracle.c", "int64_t age = t - (P->age_mode ? t_ref[i] : t_ins[i]);",
     "int64_t age = t - (P->age_mode ? t_ins[i] : t_ref[i]);", "age modes swapped"),
    ("kvev_oracle.c", "m_out[j] = m_upd[retained[j]];", "m_out[j] = m[retained[j]];",
     "compaction keeps the pre-step scores"),
    ("kvev_oracle.c", "t_ref_out[j] = t_ref[retained[j]];", "t_ref_out[j] = t_ins[retained[j]];",
     "compaction mixes the clocks"),
    ("kvev_oracle.c", "pos_out[j] = pos[retained[j]];", "pos_out[j] = pos[j];",
     "compaction drops the position map"),
    ("kvev_oracle.c", "memcpy(K_out + dst, K + src, sizeof(uint16_t) * d);",
     "memcpy(K_out + dst, V + src, sizeof(uint16_t) * d);", "compaction copies V into K"),
    ("kvev_oracle.c", "ssum[i] += s;", "ssum[i] += s / (double)Hq;", "access mass scaled twice"),
    # aggregation and weighting variants
    ("kvev_oracle.c", "? m_upd[i] + s", "? s", "cumulative forgets the state"),
    ("kvev_oracle.c", "mean /= (double)L;", ";", "VNorm not normalised by the mean norm"),
    ("kvev_oracle.c", "wg[i] = sqrt(ss);", "wg[i] = ss;", "VNorm on the squared norm"),
    ("kvev_oracle.c", "vw[(int64_t)(h * Hkv / Hq) * L + i]", "vw[i]",
     "VNorm factors of KV head 0 for every head"),
    ("kvev_oracle.c", "if (vnorm) s = sw;", ";", "VNorm factors unused"),
    ("kvev_oracle.c", "acc += hh / log((double)L);", "acc += hh;", "entropy not normalised"),
    ("kvev_oracle.c", "return acc / (double)Hq;", "return acc;", "entropy summed over heads"),
    ("kvev_oracle.c", "    s *= lw;", ";", "entropy weight unused"),
    ("kvev_oracle.c", "if (L <= 1) return 1.0;", "if (L <= 1) return 0.0;",
     "a single token's entropy weight 0"),
    # ranking diagnostics
    ("diagnostics.py", "key=lambda i: (-raw[i], i)", "key=lambda i: (-raw[i], -i)",
     "raw top-B ties to the higher slot"),
    ("diagnostics.py", "key=lambda i: (-raw[i], i)", "key=lambda i: (raw[i], i)",
     "raw top-B keeps the lowest scores"),
    ("diagnostics.py", "len(a & b) / len(union)", "len(a & b) / max(len(a), 1)",
     "Jaccard over one set's size"),
    ("diagnostics.py", "held = set(int(p) for p in held_pos) | {int(new_pos)}",
     "held = set(int(p) for p in held_pos)", "new token counted as missed"),
    ("diagnostics.py", "if s >= self.sustain:", "if s > self.sustain:",
     "revival needs a longer span"),
    ("diagnostics.py", '"kept_and_prev_kept": len(E - {L - 1})', '"kept_and_prev_kept": len(E)',
     "new token counted as previously kept"),
]
MUTANTS += [
    # block-granular oracle
    ("paged.py", "s_blk = np.array([s_tok[owner == j].max()", "s_blk = np.array([s_tok[owner == j].mean()",
     "block score is the mean, not the max"),
    ("paged.py", "m0 = float(np.mean([b.m for b in seq.blocks]))", "m0 = 0.0",
     "new block scores 0 off refresh steps"),
    ("paged.py", "m = seq.table.get(lid, 0.0) if persist else 0.0", "m = 0.0",
     "re-admission resets the score"),
    ("paged.py", "blk = Block(lid, seq.backing_K[lid].copy(), seq.backing_V[lid].copy(), m, 0, t)",
     "blk = Block(lid, seq.backing_K[lid].copy(), seq.backing_V[lid].copy(), m, 0, 0)",
     "re-admission is no access"),
    ("paged.py", "while pos < len(seq.blocks) and seq.blocks[pos].lid < lid:",
     "while pos < len(seq.blocks):", "re-admitted block appended at the end"),
    ("paged.py", "tok_acc = tok_sum / (Ly * Hq) >= 2.0 / L", "tok_acc = tok_sum / (Ly * Hq) >= 1.0 / L",
     "block access threshold 1/L"),
    ("paged.py", "accessed = np.array([tok_acc[owner == j].any()",
     "accessed = np.array([tok_acc[owner == j].all()", "block access needs every token"),
    ("paged.py", "seq.table[seq.blocks[j].lid] = seq.blocks[j].m", "seq.table[seq.blocks[j].lid] = 0.0",
     "evicted score not stored"),
    ("paged.py", "m = np.array([O.ema(m[j], s_blk[j], P.alpha)", "m = np.array([O.ema(s_blk[j], m[j], P.alpha)",
     "EMA operands swapped"),
    ("paged.py", "        ob.t_ref = t\n", "        pass\n", "append into the open block is no access"),
    ("paged.py", "kept = O.select(pr, P.budget, pinned=pinned)", "kept = O.select(pr, P.budget)",
     "block pinning ignored"),
    ("paged.py", "return np.array([any(self.pinned_regions[r] for r in b.region)",
     "return np.array([all(self.pinned_regions[r] for r in b.region)",
     "block pinned only if all its tokens are"),
    ("paged.py", "ob.region = np.append(ob.region, seq.decode_region)",
     "ob.region = np.append(ob.region, 0)", "decoded token joining a block loses its label"),
    # MemDecay oracle
    ("memdecay.py", "a = P.rho * a + (1.0 - P.rho) * A_bar", "a = (1.0 - P.rho) * a + P.rho * A_bar",
     "importance EWMA weights swapped"),
    ("memdecay.py", "accessed = A_bar >= P.tau_scale / L", "accessed = A_bar > P.tau_scale / L",
     "tau exclusive"),
    ("memdecay.py", "A_bar = mass / (Ly * Hq)", "A_bar = mass / Hq", "mass not averaged over layers"),
    ("memdecay.py", "t_ref = np.where(accessed, t, t_ref)", "t_ref = np.where(accessed, t_ref, t)",
     "clock reset inverted"),
    ("memdecay.py", "+ P.attn_weight * a", "+ a", "attention weight dropped"),
    ("memdecay.py", "np.exp(-lam * (t - ", "np.exp(lam * (t - ", "decay sign"),
    ("memdecay.py", "S = np.array([s[owner == j].mean()", "S = np.array([s[owner == j].max()",
     "page score is the max"),
    ("memdecay.py", "heap = [(float(S[j]), -j)", "heap = [(float(S[j]), j)", "ties evict the lower page"),
    ("memdecay.py", "while total > budget and heap:", "while total >= budget and heap:",
     "evicts down to below the budget"),
    ("memdecay.py", "pinned = np.array([any(P.pinned[r]", "pinned = np.array([all(P.pinned[r]",
     "page pinned only if all its tokens are"),
    ("memdecay.py", "np.array([P.decode_region]), np.zeros(1),\n                                np.array([t],",
     "np.array([P.decode_region]), np.zeros(1),\n                                np.array([0],",
     "new page's token clock 0"),
    ("memdecay.py", "pg.t_ref = np.append(pg.t_ref, t)", "pg.t_ref = np.append(pg.t_ref, 0)",
     "token joining a partial page has clock 0"),
    ("memdecay.py", "if not seq.pages or seq.pages[-1].n == seq.page:", "if True:",
     "every token opens a page"),
    ("memdecay.py", "mass += p.sum(axis=0)", "mass += p.max(axis=0)", "max over heads"),
    # two-tier oracle
    ("qevict.py", "return int(np.floor((1.0 - q) * b_hist / m_full)), int(np.floor(q * b_hist / m_quant))",
     "return int(np.floor(q * b_hist / m_full)), int(np.floor((1.0 - q) * b_hist / m_quant))",
     "tier capacities swapped"),
    ("qevict.py", "scale = ((mx - mn) / np.float32(3.0)).astype(np.float16)",
     "scale = ((mx - mn) / np.float32(4.0)).astype(np.float16)", "scale over 4 levels"),
    ("qevict.py", "r = np.rint((x - z32) / s32)", "r = np.floor((x - z32) / s32)", "codes truncated"),
    ("qevict.py", "codes = np.clip(r, 0, 3).astype(np.uint8)", "codes = np.clip(r, 0, 2).astype(np.uint8)",
     "codes clipped at 2"),
    ("qevict.py", "kq, ks, kz = quantize_groups(k, axis=3)", "kq, ks, kz = quantize_groups(k, axis=4)",
     "keys grouped per token"),
    ("qevict.py", "return (codes.astype(np.float32) * s + z)", "return (codes.astype(np.float32) * s)",
     "zero point dropped"),
    ("qevict.py", "cand.sort(key=lambda w: (-w.m, w.wid))", "cand.sort(key=lambda w: (w.m, w.wid))",
     "lowest scores kept"),
    ("qevict.py", "cand.sort(key=lambda w: (-w.m, w.wid))", "cand.sort(key=lambda w: (-w.m, -w.wid))",
     "ties to the higher window"),
    ("qevict.py", "            if w.ledger is None:                 # first demotion: quantize once\n",
     "            if True:\n", "re-quantized on every demotion"),
    ("qevict.py", "seq.window_end(P, w) <= horizon", "seq.window_end(P, w) <= seq.L",
     "recent windows routed"),
    ("qevict.py", "m = P.alpha * s + (1.0 - P.alpha) * m", "m = (1.0 - P.alpha) * s + P.alpha * m",
     "window EMA weights swapped"),
    ("qevict.py", "tok = p.sum(axis=0) / Hq", "tok = p.sum(axis=0)", "head sum instead of mean"),
    ("qevict.py", "            m = m + s\n", "            m = s\n", "cumulative score forgets"),
    ("qevict.py", "routed = t % P.omega == 0", "routed = t % P.omega == 1", "routing one step early"),
    ("qevict.py", "lg = (k64 @ q[heads].astype(np.float64).T).T / np.sqrt(d)",
     "lg = (k64 @ q[heads].astype(np.float64).T).T / d", "tier attention scale 1/d"),
    ("qevict.py", "codes = 2 * n_kv_heads * head_dim * 2 // 8", "codes = n_kv_heads * head_dim * 2 // 8",
     "value codes left out of the footprint"),
    ("qevict.py", "nw = (L0 - ns) // W", "nw = L0 // W", "windows counted from position 0"),
    # rotary positions
    ("qevict.py", "        ya = (a * c).astype(np.float32) + (b * s).astype(np.float32)\n",
     "        ya = (a * c).astype(np.float32) - (b * s).astype(np.float32)\n",
     "rotation back with the forward sine"),
    ("qevict.py", "    a, b = x[..., :h], x[..., h:]", "    a, b = x[..., 0::2], x[..., 1::2]",
     "rotation pairs adjacent channels"),
    ("qevict.py", "k, v = dequantize_window(w.ledger, cs=window_cs(P, w.wid))",
     "k, v = dequantize_window(w.ledger)", "promoted keys not rotated forward"),
    ("qevict.py", "w.ledger = quantize_window(w.K, w.V, P.group, window_cs(P, w.wid))",
     "w.ledger = quantize_window(w.K, w.V, P.group)", "keys quantized after rotation"),
    ("qevict.py", "                k = _bits_to_f32(_f32_to_bf16_bits(k))\n",
     "                k = k\n", "reconstructed keys not rounded to bf16"),
    ("qevict.py", "                v = _bits_to_f32(_f32_to_bf16_bits(v))\n",
     "                v = v\n", "reconstructed values not rounded to bf16"),
]


def _scratch_copy(dst, with_lib):
    ignore = shutil.ignore_patterns("__pycache__", "*.tmp", *(() if with_lib else ("*.so",)))
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(dst, "oracle"), ignore=ignore)
    shutil.copytree(os.path.join(ROOT, "workloads"), os.path.join(dst, "workloads"),
                    ignore=shutil.ignore_patterns("__pycache__"))
    os.makedirs(os.path.join(dst, "tests"))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))
    for f in ["conftest.py"] + PIN_FILES:
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))


@pytest.mark.parametrize("src,old,new,what", MUTANTS, ids=[m[3] for m in MUTANTS])
def test_a_planted_mistake_fails_a_pin(tmp_path, src, old, new, what):
    from oracle import build

    build()                                           # the unmutated library, reused by Python mutants
    _scratch_copy(str(tmp_path), with_lib=not src.endswith(".c"))
    path = tmp_path / "oracle" / src
    text = path.read_text()
    assert text.count(old) == 1, f"the text to mutate is not unique in {src}: {old!r}"
    path.write_text(text.replace(old, new))
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *("tests/" + f for f in PIN_FILES)],
                       cwd=str(tmp_path), env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 1, f"no pin failed with '{what}':\n{r.stdout[-2000:]}{r.stderr[-2000:]}"

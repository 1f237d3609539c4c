#!/usr/bin/env python
"""Benchmark of the GB300 decode-time KV-eviction pass.

Workload (one "step" = one whole eviction pass): Llama-3.1-8B attention
geometry (32 layers, 32 query / 8 KV heads, head_dim 128, bf16), batch 1, a
32768-token prefilled cache plus the appended token (L = 32769), budget 3277
(10%), EMA alpha 0.05, beta 0.001, access-clock ages, full refresh: append,
split-K attention with probability capture, combine, scoring (probabilities,
head sum, 32-layer EMA, priority), selection, compaction.  Each timed step
re-runs decode step 1 on the untouched prefill buffer (compaction writes the
other ping-pong buffer), after resetting the per-token state on the device.

Metric: algorithmic K/V bytes per step (every live row read once by the
attention, plus the retained rows read and written by the compaction) over
the device step time, in GB/s; the same over the end-to-end time of the
host-buffer entry point (kvev_step_host) is the "e2e" figure.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kvev|reference]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the pass has no cross-GPU exchange at batch 1); the value is the sum over
ranks of the bytes processed over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "eviction decode-step us & KV GB/s vs HBM peak (Llama-8B shape, 32k ctx, 10%)"
WORKLOAD = dict(workload="llama3.1-8b-shape eviction step, 32k ctx, 10% budget",
                n_layers=32, n_q_heads=32, n_kv_heads=8, head_dim=128, batch=1,
                prefill=32768, budget=3277, alpha=0.05, beta=0.001,
                age="since last access", refresh="full", step=1)
PAGED = dict(workload="paged block eviction with score persistence, 64 x 8192 tokens, "
                      "25% of blocks",
             n_layers=32, n_q_heads=32, n_kv_heads=8, head_dim=128, batch=64, prefill=8192,
             page=16, budget_blocks=128, alpha=0.05, beta=0.001, age="since last access",
             refresh="full", needle_blocks=4, needle_period=200, readmit="needle blocks at "
             "t = 1 + 200k, k >= 1", persistence=True)
MEMDECAY = dict(workload="region-aware (MemDecay) page eviction, 32 x 16384 tokens, 30% budget",
                n_layers=36, n_q_heads=16, n_kv_heads=2, head_dim=128, batch=32, prefill=16384,
                page=16, budget_tokens=4915, regions="system 5% (pinned), plan 5%, user 10%, "
                "tool 30%, retrieved 30%, scratchpad 20%; half-lives 160/80/60/30/40/15 steps",
                rho=0.9, attn_weight=0.5, tau="2/|K_t|", refresh="full (observation every step)")
TIERS = dict(workload="two-tier (QEvict) windows, 4 x 131072 tokens, 5% bf16 + 20% INT2",
             n_layers=32, n_q_heads=32, n_kv_heads=8, head_dim=128, batch=4, prefill=131072,
             window=128, sinks=5, recent=32, k_full=51, k_quant=204, omega=8, alpha=0.05,
             int2="keys per channel / values per token, groups of 32, fp16 scale and zero",
             needle="16 positions re-drawn every 64 steps")
# decode steps of the workloads the headline line carries (the block run
# reaches the re-admission at t = 201; the two-tier run 32 routing events)
WORKLOAD_STEPS = {"paged": 256, "memdecay": 128, "tiers": 256}
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def kv_bytes(n_layers, n_kv, d, L, budget, batch=1):
    """(algorithmic bytes of one step, of which attention reads)."""
    row = 2 * d * 2 * n_kv * n_layers          # K and V of one token, all layers/heads
    attn = L * row * batch
    comp = (2 * min(L, budget) * row * batch) if L > budget else 0
    return attn + comp, attn


def slowest_ms(ms: float, dist, device: str = "cuda") -> float:
    """The largest per-rank time (the job ends when its slowest rank does);
    `ms` itself without a process group."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: every replica processes `units_per_rank` per
    step (weak scaling), the step lasting the slowest rank's `ms`."""
    return world * units_per_rank / (ms * 1e-3)


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def code_sha256(text: str) -> str:
    """Hash of a CUDA source's code: comments dropped and whitespace runs
    collapsed, so a comment edit keeps a DRAM record while any change of the
    code voids it."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':                                   # string literal: kept as is
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    code = " ".join("".join(out).split())
    return hashlib.sha256(code.encode()).hexdigest()


def _traffic_record(key: str, kernel_file: str):
    """The committed ncu DRAM record `key`, if it was taken on the current
    code of `kernel_file`; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)[key]
        src = open(os.path.join(ROOT, "decoding_kv_cache_split_gb300", "csrc", kernel_file),
                   encoding="utf-8").read()
        if rec.get("code_sha256") != code_sha256(src):
            return None
        return rec
    except Exception:
        return None


def ncu_traffic(kernel_file: str, units: float):
    """Per-launch DRAM bytes of the attention kernel from the committed ncu
    summary, if it was taken on the current source; else None."""
    rec = _traffic_record("attention", kernel_file)
    return None if rec is None else float(rec["bytes_per_token_layer"]) * units


def traffic_ratio(key: str, kernel_file: str):
    """DRAM bytes over algorithmic bytes of a smaller ncu capture of the same
    kernel (applied to the bench's launches by the units they process)."""
    rec = _traffic_record(key, kernel_file)
    return None if rec is None else float(rec["ratio_to_algorithmic"])


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        self.proc.wait()
        sm, smax, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    smax = float(f[2])
                    power.append(float(f[3]))
                except ValueError:
                    continue
                for name, val in zip(names, f[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": ["no samples"]}
        busy = [s for s, p in zip(sm, power) if p > 1.5 * min(power)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def to_dev(bits, torch):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def cpu_baseline(wl, n_layers_sample: int, min_seconds: float = 10.0, max_reps: int = 32):
    """The fp64 oracle (single thread) on the first `n_layers_sample` layers
    of the same step, repeated until about `min_seconds` of CPU work (at most
    `max_reps` times; the step rewrites the same slots, so each repetition
    does the same work); returns (GB/s, total seconds, sample description)."""
    import oracle as O
    L0, W = wl.L0, WORKLOAD
    kv = [wl.prefill_layer(layer) for layer in range(n_layers_sample)]
    K = np.stack([k[0] for k, _ in kv])          # [layers][Hkv][L0][d] of sequence 0
    V = np.stack([v[0] for _, v in kv])
    del kv
    st = O.SequenceState.from_prefill(K, V, L0, L0 + 2)
    del K, V
    q, kn, vn = wl.step_inputs(1)
    P = O.OracleParams(n_layers_sample, W["n_q_heads"], W["n_kv_heads"], W["head_dim"],
                       W["budget"], W["alpha"], W["beta"], O.AGE_SINCE_ACCESS)
    total, reps = 0.0, 0
    while reps < 1 or (total < min_seconds and reps < max_reps):
        t0 = time.perf_counter()
        O.step(P, st, 1, True, q[0, :n_layers_sample], kn[0, :n_layers_sample],
               vn[0, :n_layers_sample], L0, want_probs=False)
        total += time.perf_counter() - t0
        reps += 1
    nbytes, _ = kv_bytes(n_layers_sample, W["n_kv_heads"], W["head_dim"], L0 + 1, W["budget"])
    return nbytes * reps / total / 1e9, total, (
        f"step 1 of the same workload restricted to its first {n_layers_sample} of "
        f"{W['n_layers']} layers (all {L0 + 1} tokens), timed {reps} times")


def reference_arm(args, rank, world):
    """The oracle, timed on the host cores on a bounded sample per step."""
    if rank != 0:
        return
    import oracle as O
    from workloads import llama8b_workload
    W = WORKLOAD
    # sample: one layer, a token prefix sized so that warmup + steps fit ~2 min
    per_step_s = max(0.05, 120.0 / max(1, args.steps + args.warmup))
    tokens = int(min(W["prefill"], max(512, per_step_s / 25e-6)))
    wl = llama8b_workload(0, prefill_len=tokens, n_layers=1)
    K, V = wl.prefill()
    st = O.SequenceState.from_prefill(K[:, 0], V[:, 0], tokens, tokens + 2)
    q, kn, vn = wl.step_inputs(1)
    budget = max(1, (tokens * W["budget"]) // W["prefill"])
    P = O.OracleParams(1, W["n_q_heads"], W["n_kv_heads"], W["head_dim"], budget, W["alpha"],
                       W["beta"], O.AGE_SINCE_ACCESS)

    n_cores, model = host_cpu()
    used = O.set_threads(n_cores)

    def one():
        O.step(P, st, 1, True, q[0], kn[0], vn[0], tokens, want_probs=False)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    nbytes, _ = kv_bytes(1, W["n_kv_heads"], W["head_dim"], tokens + 1, budget)
    val = nbytes / dt / 1e9
    sample = (f"1 of 32 layers, {tokens}-token prefill + 1, budget {budget} "
              f"(same geometry, alpha, beta, access clock); the attention's query heads on "
              f"{used} threads")
    line = {"impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(W, sample=sample),
            "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": used,
                             "kind": "oracle", "cpu": model, "sample": sample},
            "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def replay_mode(fh, ctx, ep, step_in, step_ms, alpha, name, period, L0, B, row, k0, v0,
                stream):
    """Replays one refresh-mode run (outside the timed region; the run is
    deterministic) reading the state back after every step, and returns each
    step's algorithmic bytes: the attention over the live tokens plus the
    read and write of the rows the compaction shifts (those at and after the
    first slot the step evicted).  With `fh`, also writes a JSONL record per
    step: the timed step's duration, bytes and GB/s, whether it refreshed
    the scores, and the retained-set churn (the share of the previous step's
    retained tokens, by original position, that this step evicted)."""
    import torch
    from decoding_kv_cache_split_gb300 import kvev
    ep.k[0].copy_(k0)
    ep.v[0].copy_(v0)
    ep.cache.cur = 0
    kvev.kvev_begin(ctx, L0)
    kvev.kvev_init_state(ctx, ep.state, stream)
    prev, step_bytes = None, []
    kvev.kvev_profile(ctx, True)          # per-kernel events of steps 2.. (synchronised steps)
    for t, ins in enumerate(step_in, start=1):
        if t == 2:
            kvev.kvev_profile_read(ctx)    # drop step 1
        L = kvev.kvev_length(ctx) + 1                 # live tokens after the append
        kvev.kvev_step(ctx, *ins, ep.cache, ep.state, t, ep.out, ep.retained, ep.n_retained,
                       stream)
        kvev.kvev_sync(ctx)
        n = int(ep.n_retained[0].item())
        ret = ep.retained[0, :n].cpu()
        moved = (ret != torch.arange(n, dtype=ret.dtype)).nonzero()
        first_gap = int(moved[0]) if len(moved) else n       # rows below it did not move
        nbytes = L * row + 2 * (n - first_gap) * row
        step_bytes.append(nbytes)
        if fh is not None:
            kept = set(ep.pos[0, :n].cpu().tolist())
            churn = None if prev is None else len(prev - kept) / max(1, len(prev))
            refresh = (name == "full" or (name == "lazy8" and (t - 1) % period == 0)
                       or (name == "frozen" and t == 1))
            fh.write(json.dumps({"alpha": alpha, "mode": name, "step": t,
                                 "us": round(step_ms[t - 1] * 1e3, 2), "bytes": nbytes,
                                 "GBps": round(nbytes / (step_ms[t - 1] * 1e-3) / 1e9, 1),
                                 "refresh": refresh, "live": L, "kept": n,
                                 "churn": None if churn is None else round(churn, 6),
                                 "first_moved_row": first_gap}) + "\n")
            prev = kept
    prof = kvev.kvev_profile_read(ctx)
    kvev.kvev_profile(ctx, False)
    n = max(1, len(step_in) - 1)
    kernels = {k: round(v[0] / n * 1e3, 2) for k, v in prof.items()}
    return step_bytes, kernels


def fused_mode_run(ctx, ep, step_in, L0, k0, v0, stream, mode=None):
    """The refresh-mode run again with a fused refresh step (`mode`, default
    all three phases): step 1 and the mean of steps 2.. in us (CUDA events
    between steps)."""
    import torch
    from decoding_kv_cache_split_gb300 import kvev
    try:
        kvev.kvev_set_fused_step(ctx, kvev.KVEV_FUSED_ALL if mode is None else mode)
    except kvev.KvevError as err:
        return {"unavailable": str(err)}
    ep.k[0].copy_(k0)
    ep.v[0].copy_(v0)
    ep.cache.cur = 0
    kvev.kvev_begin(ctx, L0)
    kvev.kvev_init_state(ctx, ep.state, stream)
    n = len(step_in)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    torch.cuda.synchronize()
    evs[0].record(stream)
    for t in range(1, n + 1):
        kvev.kvev_step(ctx, *step_in[t - 1], ep.cache, ep.state, t, ep.out, ep.retained,
                       ep.n_retained, stream)
        evs[t].record(stream)
    torch.cuda.synchronize()
    kvev.kvev_sync(ctx)
    kvev.kvev_set_fused_step(ctx, kvev.KVEV_FUSED_OFF)
    st = [evs[t - 1].elapsed_time(evs[t]) for t in range(1, n + 1)]
    return {"step1_us": round(st[0] * 1e3, 1),
            "steady_us": round(sum(st[1:]) / max(1, n - 1) * 1e3, 1)}


def diagnostics_run(fh, ctx, ep, step_in, L0, k0, v0, stream, alpha, name):
    """One more replay of a refresh-mode run with the device's ranking
    diagnostics on (kvev_set_diagnostics): per scoring step the raw top-B set
    R (the attention summed over heads and layers, before aggregation)
    against the retained set E.  Returns the means over the scoring steps
    after the first of: raw/EMA Jaccard |R & E| / |R | E|, raw churn (Jaccard
    distance of consecutive raw sets), EMA churn (of consecutive retained
    sets, every step) and the share of R evicted; with `fh`, a JSONL record
    per step with the counters."""
    import torch
    from decoding_kv_cache_split_gb300 import kvev
    cnt = torch.zeros((1, kvev.KVEV_DIAG_FIELDS), dtype=torch.int32, device="cuda")
    kvev.kvev_set_diagnostics(ctx, cnt, None)
    ep.k[0].copy_(k0)
    ep.v[0].copy_(v0)
    ep.cache.cur = 0
    kvev.kvev_begin(ctx, L0)
    kvev.kvev_init_state(ctx, ep.state, stream)
    jac, raw_churn, ema_churn, raw_ev = [], [], [], []
    prev_kept = None
    for t, ins in enumerate(step_in, start=1):
        kvev.kvev_step(ctx, *ins, ep.cache, ep.state, t, ep.out, ep.retained, ep.n_retained,
                       stream)
        kvev.kvev_sync(ctx)
        c = dict(zip(kvev.DIAG_NAMES, cnt[0].cpu().tolist()))
        if prev_kept is not None:
            ee = c["kept_and_prev_kept"]
            ema_churn.append(1 - ee / max(1, c["n_kept"] + prev_kept - ee))
        prev_kept = c["n_kept"]
        rec = {"alpha": alpha, "mode": name, "step": t, "diag": c}
        if c["refreshed"] and c["n_raw"]:
            j = c["raw_and_kept"] / (c["n_raw"] + c["n_kept"] - c["raw_and_kept"])
            rec["raw_ema_jaccard"] = round(j, 6)
            if t > 1:
                jac.append(j)
                raw_ev.append(1 - c["raw_and_kept"] / c["n_raw"])
            if c["n_prev_raw"]:
                rr = c["raw_and_prev_raw"]
                ch = 1 - rr / (c["n_raw"] + c["n_prev_raw"] - rr)
                raw_churn.append(ch)
                rec["raw_churn"] = round(ch, 6)
        if fh is not None:
            fh.write(json.dumps(rec) + "\n")
    kvev.kvev_set_diagnostics(ctx, None, None)
    mean = lambda x: round(sum(x) / len(x), 6) if x else None
    return {"raw_ema_jaccard": mean(jac), "raw_churn": mean(raw_churn),
            "ema_churn": mean(ema_churn), "raw_top_evicted": mean(raw_ev),
            "scoring_steps": len(jac) + 1}


def steady_graph_us(ctx, ep, step_in, L0, k0, v0, stream, warmup, n_capture=8, reps=25):
    """Steady steps replayed from a CUDA graph: decode steps 2..9 of a run
    are captured once (their kernels, with the sizes and buffers of those
    steps) and the graph is replayed; returns the time per step in us.  The
    replays redo the same eight steps' work on the evolving state (same
    sizes: the cache stays at the budget), which is what the timing needs."""
    import torch
    from decoding_kv_cache_split_gb300 import kvev
    ep.k[0].copy_(k0)
    ep.v[0].copy_(v0)
    ep.cache.cur = 0
    kvev.kvev_begin(ctx, L0)
    kvev.kvev_init_state(ctx, ep.state, stream)
    kvev.kvev_step(ctx, *step_in[0], ep.cache, ep.state, 1, ep.out, ep.retained, ep.n_retained,
                   stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream()
        for t in range(2, 2 + n_capture):
            kvev.kvev_step(ctx, *step_in[t - 1], ep.cache, ep.state, t, ep.out, ep.retained,
                           ep.n_retained, cs)
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    kvev.kvev_sync(ctx)
    del g
    return round(e0.elapsed_time(e1) / (reps * n_capture) * 1e3, 2)


def finish_dist(world):
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kvev", choices=["kvev", "reference"])
    ap.add_argument("--cpu-layers", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--log-steps", default=None,
                    help="write a JSONL record per step of the refresh-mode runs to this file")
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the CUDA-graph replay timing of the headline pass")
    ap.add_argument("--mode-steps", type=int, default=256,
                    help="decode steps of each (alpha, refresh mode) run reported under 'modes' "
                         "(0: skip)")
    ap.add_argument("--layers", type=int, default=WORKLOAD["n_layers"],
                    help="smaller cases for profiling; the headline uses 32")
    ap.add_argument("--prefill", type=int, default=WORKLOAD["prefill"])
    ap.add_argument("--workload", default="llama8b-32k",
                    choices=["llama8b-32k", "paged", "memdecay", "tiers"],
                    help="the headline token-granular step, or the block-granular run")
    ap.add_argument("--batch", type=int, default=PAGED["batch"],
                    help="paged workload: sequences (profiling cases only)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="the headline line only: skip the block, region-aware and two-tier "
                         "workloads it carries under 'workloads'")
    ap.add_argument("--omega", type=int, default=TIERS["omega"],
                    help="two-tier workload: routing interval")
    ap.add_argument("--no-sweep", action="store_true",
                    help="two-tier workload: skip the routing-interval sweep")
    ap.add_argument("--rope", action="store_true",
                    help="two-tier workload: the whole run in rotary mode (rope base 10000; "
                         "INT2 windows attended as bf16 reconstructions)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return

    if args.workload in ("paged", "memdecay"):
        bench_paged(args, rank, world, local_rank, md=args.workload == "memdecay")
        finish_dist(world)
        return
    if args.workload == "tiers":
        bench_tiers(args, rank, world, local_rank, omega=args.omega,
                    omega_sweep=() if args.no_sweep else (1, 32), rotary=not args.no_sweep)
        finish_dist(world)
        return

    import torch
    dist = init_dist(world, local_rank)
    kvev = load_kvev()
    from workloads import llama8b_workload

    W = dict(WORKLOAD)
    if args.layers != W["n_layers"] or args.prefill != W["prefill"]:
        W.update(workload=f"profiling case: {args.layers} layers, {args.prefill}-token prefill",
                 n_layers=args.layers, prefill=args.prefill,
                 budget=-(-args.prefill // 10))
    L0, B = W["prefill"], W["budget"]
    max_ctx = L0 + 64
    wl = llama8b_workload(0, prefill_len=L0, n_layers=W["n_layers"])
    ep = kvev.EvictionPass(W["n_layers"], W["n_q_heads"], W["n_kv_heads"], W["head_dim"],
                           W["batch"], max_ctx, B, W["alpha"], W["beta"],
                           age_mode=kvev.KVEV_AGE_SINCE_ACCESS)
    for layer in range(W["n_layers"]):
        k, v = wl.prefill_layer(layer)
        ep.k[0][layer, :, :, :L0].copy_(torch.from_numpy(k.view(np.int16)).view(torch.bfloat16))
        ep.v[0][layer, :, :, :L0].copy_(torch.from_numpy(v.view(np.int16)).view(torch.bfloat16))
    q, kn, vn = wl.step_inputs(1)
    qd, knd, vnd = to_dev(q, torch), to_dev(kn, torch), to_dev(vn, torch)
    stream = torch.cuda.current_stream()

    def one_step():
        ep.begin(L0, stream)
        ep.step(qd, knd, vnd, stream)

    for _ in range(args.warmup):
        one_step()
    kvev.kvev_sync(ep.ctx)

    # ---------------------------------------------------------- device timing
    # Headline region: the pass back to back, no per-kernel events (an event
    # between kernels would stop each kernel's launch from overlapping the
    # previous one's tail).
    n0 = kvev.kvev_launch_count(ep.ctx)
    clocks = ClockSampler(local_rank)
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        one_step()
    e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    kvev.kvev_sync(ep.ctx)
    launches = kvev.kvev_launch_count(ep.ctx) - n0
    ms = e0.elapsed_time(e1) / args.steps
    ms = slowest_ms(ms, dist)

    # The same pass captured once in a CUDA graph (re-setting the context's host
    # state, the state reset and step 1 against the untouched prefill) and
    # replayed: launch overhead off the host, same outputs bit for bit.
    graph_us = None
    if not args.no_graph:
        ref_out = ep.out.clone()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            ep.begin(L0, torch.cuda.current_stream())
            ep.step(qd, knd, vnd, torch.cuda.current_stream())
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        kvev.kvev_sync(ep.ctx)
        graph_us = g0.elapsed_time(g1) / args.steps * 1e3
        assert torch.equal(ep.out, ref_out), "graph replay differs from the eager step"
        del g

    # The same pass with the fused refresh step (attention, combine and scoring
    # in one cooperative launch), timed the same way; its output is compared
    # with the three-launch pass's.
    fused = {}
    for fname, fmode in (("all", kvev.KVEV_FUSED_ALL),
                         ("attn_combine", kvev.KVEV_FUSED_ATTN_COMBINE)):
        try:
            kvev.kvev_set_fused_step(ep.ctx, fmode)
            ref_out = ep.out.clone()
            for _ in range(args.warmup):
                one_step()
            torch.cuda.synchronize()
            f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            f0.record(stream)
            for _ in range(args.steps):
                one_step()
            f1.record(stream)
            torch.cuda.synchronize()
            kvev.kvev_sync(ep.ctx)
            fus_ms = f0.elapsed_time(f1) / args.steps
            fused[fname] = {
                "us_per_step": round(fus_ms * 1e3, 2),
                "GBps": round(kv_bytes(W["n_layers"], W["n_kv_heads"], W["head_dim"], L0 + 1,
                                       B)[0] / (fus_ms * 1e-3) / 1e9, 2),
                "same_output_bits": bool(torch.equal(ep.out, ref_out))}
        except kvev.KvevError as err:
            fused[fname] = {"unavailable": str(err)}
        finally:
            kvev.kvev_set_fused_step(ep.ctx, kvev.KVEV_FUSED_OFF)

    # Per-kernel region: CUDA events around every launch, on the launching stream.
    kvev.kvev_profile(ep.ctx, True)
    kvev.kvev_profile_read(ep.ctx)          # reset accumulators
    n_prof = max(10, min(args.steps, 200))
    for _ in range(n_prof):
        one_step()
    kvev.kvev_sync(ep.ctx)
    prof = kvev.kvev_profile_read(ep.ctx)
    kvev.kvev_profile(ep.ctx, False)
    nbytes, attn_bytes = kv_bytes(W["n_layers"], W["n_kv_heads"], W["head_dim"], L0 + 1, B)
    value = job_rate(nbytes, world, ms) / 1e9

    # -------------------------------------------------- end to end (host API)
    # the user's call: host buffers in, the bf16 attention output (the type a
    # caller feeds to the next bf16 projection) and the retained list back
    kvev.kvev_set_output(ep.ctx, kvev.KVEV_OUT_BF16)
    qh = torch.from_numpy(q.view(np.int16)).pin_memory()
    knh = torch.from_numpy(kn.view(np.int16)).pin_memory()
    vnh = torch.from_numpy(vn.view(np.int16)).pin_memory()
    outh = torch.empty((1, W["n_layers"], W["n_q_heads"], W["head_dim"]),
                       dtype=torch.bfloat16).pin_memory()
    reth = torch.empty((1, B), dtype=torch.int32).pin_memory()
    nreth = torch.empty((1,), dtype=torch.int32).pin_memory()
    h2d = qh.numel() * 2 + knh.numel() * 2 + vnh.numel() * 2
    d2h = outh.numel() * 2 + reth.numel() * 4 + nreth.numel() * 4

    def one_e2e(step_no=1):
        ep.begin(L0, stream)
        kvev.kvev_step_host(ep.ctx, qh, knh, vnh, ep.cache, ep.state, step_no, outh, reth, nreth,
                            stream)

    for _ in range(args.warmup):
        one_e2e()
    n_e2e = max(10, min(args.steps, 500))
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        one_e2e()
    torch.cuda.synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / n_e2e
    e2e_ms = slowest_ms(e2e_ms, dist)
    e2e_val = job_rate(nbytes, world, e2e_ms) / 1e9
    assert int(nreth[0]) == B
    kvev.kvev_set_output(ep.ctx, kvev.KVEV_OUT_F32)

    # ------------------------------------- refresh modes x alphas (steady state)
    # Every (alpha, mode) run starts from the prefill at step 1 and decodes
    # --mode-steps steps; steady = steps 2.. (about B + 1 live tokens each).
    modes = []
    step_log = open(args.log_steps, "w") if args.log_steps and rank == 0 else None
    if args.mode_steps > 0 and args.layers == WORKLOAD["n_layers"]:
        k0, v0 = ep.k[0].clone(), ep.v[0].clone()
        n_ms = args.mode_steps
        step_in = [tuple(to_dev(x, torch) for x in wl.step_inputs(t)) for t in range(1, n_ms + 1)]
        row = 2 * W["head_dim"] * 2 * W["n_kv_heads"] * W["n_layers"]
        for alpha in (0.01, 0.05, 0.15):
            ctx = kvev.kvev_create(ep.layout, B, 1, alpha, W["beta"])
            kvev.kvev_configure(ctx, kvev.KVEV_AGE_SINCE_ACCESS, kvev.KVEV_POOL_SUM)
            for name, mode, period in (("full", kvev.KVEV_REFRESH_FULL, 1),
                                       ("lazy8", kvev.KVEV_REFRESH_LAZY, 8),
                                       ("frozen", kvev.KVEV_REFRESH_FROZEN, 1)):
                kvev.kvev_refresh_mode(ctx, mode, period)
                ep.k[0].copy_(k0)
                ep.v[0].copy_(v0)
                ep.cache.cur = 0
                kvev.kvev_begin(ctx, L0)
                kvev.kvev_init_state(ctx, ep.state, stream)
                evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_ms + 1)]
                torch.cuda.synchronize()
                evs[0].record(stream)
                for t in range(1, n_ms + 1):
                    kvev.kvev_step(ctx, *step_in[t - 1], ep.cache, ep.state, t, ep.out,
                                   ep.retained, ep.n_retained, stream)
                    evs[t].record(stream)
                torch.cuda.synchronize()
                kvev.kvev_sync(ctx)
                st = [evs[t - 1].elapsed_time(evs[t]) for t in range(1, n_ms + 1)]
                steady = sum(st[1:]) / max(1, n_ms - 1)
                sb, kern = replay_mode(step_log, ctx, ep, step_in, st, alpha, name, period, L0,
                                       B, row, k0, v0, stream)
                steady_bytes = sum(sb[1:]) / max(1, n_ms - 1)   # attention + shifted rows
                rec = {"alpha": alpha, "mode": name, "step1_us": round(st[0] * 1e3, 1),
                       "steady_us": round(steady * 1e3, 1),
                       "steady_GBps": round(steady_bytes / (steady * 1e-3) / 1e9, 1),
                       "steady_frac_measured": round(steady_bytes / (steady * 1e-3) / 1e9
                                                     / measured_peak()[0], 4),
                       "steady_bytes": int(steady_bytes),
                       "steady_kernels_us": kern}
                if alpha == 0.05 and not args.no_graph:
                    rec["steady_graph_us"] = steady_graph_us(ctx, ep, step_in, L0, k0, v0,
                                                             stream, args.warmup)
                if alpha == 0.05:   # the same run with the fused refresh steps
                    rec["fused"] = {
                        "all": fused_mode_run(ctx, ep, step_in, L0, k0, v0, stream,
                                              kvev.KVEV_FUSED_ALL),
                        "attn_combine": fused_mode_run(ctx, ep, step_in, L0, k0, v0, stream,
                                                       kvev.KVEV_FUSED_ATTN_COMBINE)}
                if name != "frozen":   # Score-Free scores once: no ranking to trace
                    rec["diagnostics"] = diagnostics_run(step_log, ctx, ep, step_in, L0, k0,
                                                         v0, stream, alpha, name)
                modes.append(rec)
            kvev.kvev_destroy(ctx)
        del k0, v0, step_in
    if step_log is not None:
        step_log.close()

    # --------------------------------------------------------------- roofline
    peak, peak_kind = measured_peak()
    # the attention of one step may be split into launches over groups of
    # layers: the algorithmic bytes of a step over its attention time per step
    att_ms, att_n = prof.get("attention", (0.0, 0))
    att_per_step = att_ms / n_prof
    attn_achieved = attn_bytes / (att_per_step * 1e-3) / 1e9 if att_per_step > 0 else None
    tokens_layers = (L0 + 1) * W["n_layers"]
    traffic = ncu_traffic("attn.cu", tokens_layers)
    kernels_us = {k: round(v[0] / n_prof * 1e3, 2) for k, v in prof.items()}   # per step
    kernels_us["launches_per_step"] = {k: v[1] // n_prof for k, v in prof.items()}
    kernels_us["profiled_steps"] = n_prof

    line = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            import oracle as O
            n_cores, model = host_cpu()
            O.set_threads(1)
            val1, secs1, _ = cpu_baseline(wl, min(args.cpu_layers, W["n_layers"]))
            used = O.set_threads(n_cores)
            valn, secsn, sample = cpu_baseline(wl, min(args.cpu_layers, W["n_layers"]))
            cpu = {"value": round(valn, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
                   "cpu": model, "sample": sample + f"; the attention's query heads on {used} "
                   "threads (OpenMP)", "seconds": round(secsn, 2),
                   "single_thread": {"value": round(val1, 4), "cores": 1,
                                     "seconds": round(secs1, 2)}}
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "us_per_step": round(ms * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(W, parallelism=f"replicas{world}",
                           l2="inputs larger than L2 (4.3 GB of K/V per step)"),
            "frac_of_peak": {"measured": round(value / world / peak, 4),
                             "nominal_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
                             "peak_kind": peak_kind},
            "kv_tokens_per_s": round(world * (L0 + 1) / (ms * 1e-3), 1),
            "roofline": {"bound": "hbm", "kernel": "attention (all launches of a step)",
                         "achieved": round(attn_achieved, 2) if attn_achieved else None,
                         "peak": peak, "unit": "GB/s",
                         "frac": round(attn_achieved / peak, 4) if attn_achieved else None,
                         "traffic": traffic, "algorithmic_bytes": attn_bytes,
                         "peak_kind": f"{peak_kind} (copy bandwidth)"},
            "kernels_us": kernels_us,
            "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "ms_per_step": round(e2e_ms, 4),
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "output": "bf16",
                    "call": "kvev_step_host"},
            "graph": ({"us_per_step": round(graph_us, 2), "replays": args.steps} if graph_us else None),
            "fused_step": fused,
            "gpu_launches": launches,
            "clocks": clk,
            "cpu_baseline": cpu,
            "modes": modes,
        }
    ep.close()
    del ep
    torch.cuda.empty_cache()

    # ------------------------------ the other workloads, each at its own size
    # (block-granular with re-admission, region-aware, two-tier INT2); their
    # step counts are fixed so that the run stays within a few minutes
    if not args.no_workloads and args.layers == WORKLOAD["n_layers"] and \
            args.prefill == WORKLOAD["prefill"]:
        subs = []
        for name, fn in (("paged", lambda: bench_paged(args, rank, world, local_rank,
                                                        steps=WORKLOAD_STEPS["paged"],
                                                        quiet=True)),
                         ("memdecay", lambda: bench_paged(args, rank, world, local_rank, md=True,
                                                           steps=WORKLOAD_STEPS["memdecay"],
                                                           quiet=True)),
                         ("tiers", lambda: bench_tiers(args, rank, world, local_rank,
                                                       steps=WORKLOAD_STEPS["tiers"],
                                                       quiet=True))):
            rec = fn()
            if rec is not None:
                rec = {k: v for k, v in rec.items() if k not in ("metric", "n_gpus", "warmup")}
                rec["name"] = name
                subs.append(rec)
        if line is not None:
            line["workloads"] = subs
    if line is not None:
        print(json.dumps(line), flush=True)
    finish_dist(world)


def init_dist(world, local_rank):
    """The process group under torchrun (None for one process) and the device."""
    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        if not dist.is_initialized():
            dist.init_process_group("nccl")
        return dist
    torch.cuda.set_device(0)
    return None


def load_kvev():
    from decoding_kv_cache_split_gb300 import build as kbuild
    if not os.path.exists(kbuild.LIB):
        kbuild.build()
    from decoding_kv_cache_split_gb300 import kvev
    return kvev


def host_cpu():
    """(logical CPUs, CPU model) of this host, for the CPU-baseline legs."""
    model = None
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if model is None:
        import platform
        model = platform.processor() or platform.machine()
    return os.cpu_count() or 1, model


def timed_reps(fn, min_seconds: float, max_reps: int, prepare=None):
    """Run fn until about min_seconds of wall time (at least once); returns
    (repetitions, seconds).  With `prepare`, each repetition runs
    fn(prepare()) and only fn is timed (a fresh copy of a state, say)."""
    total, reps = 0.0, 0
    while reps < 1 or (total < min_seconds and reps < max_reps):
        arg = prepare() if prepare is not None else None
        t0 = time.perf_counter()
        fn(arg) if prepare is not None else fn()
        total += time.perf_counter() - t0
        reps += 1
    return reps, total


def cpu_baseline_block(kind, W, seq_K, seq_V, inputs1, labels=None, min_seconds=10.0):
    """The oracle of a block workload (oracle/paged.py or oracle/memdecay.py)
    on one sequence of the batch, decode step 1 over its whole prefill,
    repeated to about `min_seconds`; the sequences are independent, so one
    sequence's time is the per-sequence cost of the batch.  Threads: the
    oracle's attention runs its query heads on all host cores."""
    import oracle as O
    q, kn, vn = inputs1
    Ly, d = W["n_layers"], W["head_dim"]
    if kind == "memdecay":
        import math
        from oracle import memdecay as MD
        from workloads import DECODE_REGION, REGION_HALF_LIVES, REGION_PINNED
        lam = tuple(math.log(2.0) / h for h in REGION_HALF_LIVES)
        P = MD.MDParams(Ly, W["n_q_heads"], W["n_kv_heads"], d, W["budget_tokens"],
                        base=(1.0,) * len(lam), lam=lam, pinned=REGION_PINNED,
                        decode_region=DECODE_REGION)
        seq0 = MD.MDSequence.from_prefill(seq_K, seq_V, labels, W["page"])
        fn = lambda s: MD.step(P, s, 1, True, q, kn, vn)
    else:
        from oracle import paged as PG
        P = O.OracleParams(Ly, W["n_q_heads"], W["n_kv_heads"], d, W["budget_blocks"],
                           W["alpha"], W["beta"], O.AGE_SINCE_ACCESS, False)
        seq0 = PG.PagedSequence.from_prefill(seq_K, seq_V, W["page"])
        fn = lambda s: PG.step(P, s, 1, True, q, kn, vn)
    threads = O.set_threads(os.cpu_count() or 1)
    # each repetition steps a fresh copy of the prefill state (the copy untimed)
    reps, secs = timed_reps(fn, min_seconds, 64, prepare=seq0.copy)
    row = 2 * d * 2 * W["n_kv_heads"] * Ly
    nbytes = (W["prefill"] + 1) * row
    cores, model = host_cpu()
    return {"value": round(nbytes * reps / secs / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle", "cpu": model, "seconds": round(secs, 2),
            "sample": f"decode step 1 of sequence 0 of {W['batch']} ({W['prefill']} + 1 tokens, "
                      f"all {Ly} layers), timed {reps} times; sequences are independent"}


def bench_paged(args, rank, world, local_rank, md=False, steps=None, quiet=False):
    """Block-granular runs.  Block workload: 64 sequences of 8192 tokens in
    16-token blocks, budget 128 blocks; step 1 evicts from 513 to 128 blocks
    per sequence, later steps attend over ~2049 tokens per sequence; the
    needle blocks are re-admitted (scores restored) when the needle is
    re-drawn.  Region-aware (md): Qwen2.5-3B geometry, 32 sequences of 16384
    region-labelled tokens, MemDecay page scores, budget 4915 tokens.  Timed:
    K consecutive decode steps after step 1 (readmissions included); step 1
    alone is timed separately (re-run on the untouched prefill pages).
    Returns the JSON record (rank 0) or None."""
    import torch
    dist = init_dist(world, local_rank)
    kvev = load_kvev()
    from workloads.device import PagedDeviceWorkload

    W = dict(MEMDECAY if md else PAGED)
    if args.layers != WORKLOAD["n_layers"] or args.batch != PAGED["batch"] or \
            args.prefill != WORKLOAD["prefill"]:
        pre = args.prefill if args.prefill != WORKLOAD["prefill"] else W["prefill"]
        W.update(workload=f"profiling case: {args.layers} layers, {args.batch} x {pre} tokens",
                 n_layers=args.layers, batch=args.batch, prefill=pre)
        if md:
            W.update(budget_tokens=max(1, (3 * pre) // 10))
        else:
            W.update(budget_blocks=max(1, pre // W["page"] // 4))
    Ly, b, P = W["n_layers"], W["batch"], W["page"]
    nb0 = -(-W["prefill"] // P)
    pps = nb0 + 8
    labels = None
    if md:
        import math
        from workloads import (DECODE_REGION, REGION_HALF_LIVES, REGION_PINNED,
                               region_labels)
        wl = PagedDeviceWorkload(0, n_layers=Ly, n_q_heads=W["n_q_heads"],
                                 n_kv_heads=W["n_kv_heads"], batch=b, prefill=W["prefill"],
                                 page=P, needle_blocks=0)
        table = kvev.region_table([1.0] * len(REGION_HALF_LIVES),
                                  [math.log(2.0) / h for h in REGION_HALF_LIVES], REGION_PINNED,
                                  score_kind=kvev.KVEV_SCORE_MEMDECAY, rho=W["rho"],
                                  attn_weight=W["attn_weight"], tau_scale=2.0,
                                  decode_region=DECODE_REGION)
        pp = kvev.PagedEvictionPass(Ly, W["n_q_heads"], W["n_kv_heads"], W["head_dim"], b, pps,
                                    P, W["budget_tokens"], 0.05, 0.001, regions=table)
        wl.fill(torch, pp.k_pool, pp.v_pool, pps)
        labels = region_labels(W["prefill"])
        lab = np.zeros(nb0 * P, np.uint8)
        lab[:W["prefill"]] = labels
        lab_t = torch.from_numpy(lab).cuda()
        for s_ in range(b):
            pp.region[s_ * pps * P:s_ * pps * P + nb0 * P].copy_(lab_t)
    else:
        wl = PagedDeviceWorkload(0, n_layers=Ly, batch=b, prefill=W["prefill"], page=P,
                                 needle_blocks=W["needle_blocks"],
                                 needle_period=W["needle_period"])
        pp = kvev.PagedEvictionPass(Ly, W["n_q_heads"], W["n_kv_heads"], W["head_dim"], b, pps,
                                    P, W["budget_blocks"], W["alpha"], W["beta"], n_backing=nb0,
                                    table_len=nb0, age_mode=kvev.KVEV_AGE_SINCE_ACCESS)
        wl.fill(torch, pp.k_pool, pp.v_pool, pps, pp.backing_k, pp.backing_v)
    n_steps = steps if steps is not None else args.steps
    last = max(n_steps + 1, args.warmup)
    inputs = [wl.step_inputs(torch, t, pp.backing_k) for t in range(1, last + 1)]
    readmits = {}
    for t in range(1 + W.get("needle_period", last + 1), last + 1, W.get("needle_period", 1)):
        nd = wl.needle(t)
        readmits[t] = [(s, int(x)) for s in range(b) for x in nd[s]]
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()

    def run_step(t):
        for (s, lid) in readmits.get(t, ()):
            pp.readmit(s, lid, True, stream)
        q, kn, vn = inputs[t - 1]
        pp.step(q, kn, vn, stream)

    # warm-up: the first W steps of a run
    pp.begin(W["prefill"], stream)
    for t in range(1, args.warmup + 1):
        run_step(t)
    kvev.kvev_sync(pp.ctx)

    # timed: steps 2 .. K+1 of a fresh run
    pp.begin(W["prefill"], stream)
    run_step(1)
    n0 = kvev.kvev_launch_count(pp.ctx)
    clocks = ClockSampler(local_rank)
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for t in range(2, n_steps + 2):
        run_step(t)
    e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    kvev.kvev_sync(pp.ctx)
    launches = kvev.kvev_launch_count(pp.ctx) - n0
    ms = e0.elapsed_time(e1) / n_steps
    ms = slowest_ms(ms, dist)

    # replay with per-kernel events; count the live tokens each step attends
    row = 2 * W["head_dim"] * 2 * W["n_kv_heads"] * Ly        # bytes of one token, all layers
    kvev.kvev_profile(pp.ctx, True)
    pp.begin(W["prefill"], stream)
    run_step(1)
    kvev.kvev_sync(pp.ctx)
    kvev.kvev_profile_read(pp.ctx)

    def live_tokens():
        nb, lens = pp.n_blocks.cpu().numpy(), pp.len.cpu().numpy()
        return int(sum(lens[s, :nb[s]].sum() for s in range(b)))

    tokens_after = live_tokens()               # after step 1's compaction
    attn_tokens = 0
    readmit_blocks = 0
    for t in range(2, n_steps + 2):
        if t in readmits:                          # readmitted blocks are attended too
            before = live_tokens()
            for (s, lid) in readmits[t]:
                pp.readmit(s, lid, True, stream)
            kvev.kvev_sync(pp.ctx)
            readmit_blocks += (live_tokens() - before) // P
            tokens_after = live_tokens()
        q, kn, vn = inputs[t - 1]
        pp.step(q, kn, vn, stream)
        kvev.kvev_sync(pp.ctx)
        attn_tokens += tokens_after + b            # previous live tokens + the new ones
        tokens_after = live_tokens()
    prof = kvev.kvev_profile_read(pp.ctx)
    kvev.kvev_profile(pp.ctx, False)
    attn_bytes_total = attn_tokens * row
    # pages never move; a re-admission copies one block (all layers) from the backing tier
    nbytes_total = attn_bytes_total + readmit_blocks * P * row * 2
    att_ms = prof.get("attention", (0.0, 0))[0]
    value = world * nbytes_total / n_steps / (ms * 1e-3) / 1e9
    attn_achieved = attn_bytes_total / (att_ms * 1e-3) / 1e9 if att_ms > 0 else None
    kernels_us = {k: round(v[0] / n_steps * 1e3, 2) for k, v in prof.items()}
    kernels_us["launches_per_step"] = {k: round(v[1] / n_steps, 2) for k, v in prof.items()}

    # step 1 alone: every sequence's whole prefill, eviction to the budget
    n1 = 10
    pp.begin(W["prefill"], stream)
    run_step(1)
    torch.cuda.synchronize()
    step1_ms = 0.0
    for _ in range(n1):   # events around the step only (kvev_paged_begin may synchronize)
        pp.begin(W["prefill"], stream)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        run_step(1)
        s1.record(stream)
        torch.cuda.synchronize()
        step1_ms += s0.elapsed_time(s1) / n1
    kvev.kvev_sync(pp.ctx)
    step1_bytes = b * (W["prefill"] + 1) * row

    # end to end: host inputs (pinned) in, the bf16 output and the kept ids
    # back, every step
    kvev.kvev_set_output(pp.ctx, kvev.KVEV_OUT_BF16)
    out_dev = torch.empty(pp.out.shape, dtype=torch.bfloat16, device="cuda")
    n_e2e = min(n_steps, 64)
    host_in = [tuple(x.view(torch.int16).cpu().pin_memory() for x in inputs[t - 1])
               for t in range(2, n_e2e + 2)]
    dev_in = [torch.empty_like(x) for x in inputs[0]]
    out_h = torch.empty(pp.out.shape, dtype=torch.bfloat16).pin_memory()
    ret_h = torch.empty(pp.retained_lid.shape, dtype=torch.int32).pin_memory()
    nret_h = torch.empty(pp.n_retained.shape, dtype=torch.int32).pin_memory()
    h2d = sum(x.numel() * 2 for x in host_in[0])
    d2h = out_h.numel() * 2 + ret_h.numel() * 4 + nret_h.numel() * 4
    pp.begin(W["prefill"], stream)
    run_step(1)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i, t in enumerate(range(2, n_e2e + 2)):
        for d, h in zip(dev_in, host_in[i]):
            d.view(torch.int16).copy_(h, non_blocking=True)
        for (s, lid) in readmits.get(t, ()):
            pp.readmit(s, lid, True, stream)
        pp.step_no += 1
        kvev.kvev_paged_step(pp.ctx, *dev_in, pp.cache, pp.state, pp.step_no, out_dev,
                             pp.retained_lid, pp.n_retained, stream)
        out_h.copy_(out_dev, non_blocking=True)
        ret_h.copy_(pp.retained_lid, non_blocking=True)
        nret_h.copy_(pp.n_retained, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / n_e2e
    kvev.kvev_sync(pp.ctx)
    kvev.kvev_set_output(pp.ctx, kvev.KVEV_OUT_F32)
    e2e_val = world * (attn_bytes_total / n_steps) / (e2e_ms * 1e-3) / 1e9
    # DRAM bytes per launch: the algorithmic bytes times the ratio of an ncu
    # capture of the same kernel on a smaller block workload (the region-aware
    # workload runs another instantiation: none)
    ratio = traffic_ratio("attention_paged", "attn.cu")
    paged_traffic = round(attn_bytes_total / n_steps * ratio) if ratio and not md else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        seq_pages = slice(0, nb0)
        src_k = pp.k_pool[seq_pages] if md else pp.backing_k[0, :nb0]
        src_v = pp.v_pool[seq_pages] if md else pp.backing_v[0, :nb0]
        bits = lambda x: x.view(torch.int16).cpu().numpy().view(np.uint16)
        Kh = bits(src_k).transpose(1, 2, 0, 3, 4).reshape(Ly, W["n_kv_heads"], -1, W["head_dim"])
        Vh = bits(src_v).transpose(1, 2, 0, 3, 4).reshape(Ly, W["n_kv_heads"], -1, W["head_dim"])
        Kh = np.ascontiguousarray(Kh[:, :, :W["prefill"]])
        Vh = np.ascontiguousarray(Vh[:, :, :W["prefill"]])
        q1, kn1, vn1 = inputs[0]
        cpu = cpu_baseline_block("memdecay" if md else "paged", W, Kh, Vh,
                                 (bits(q1[0]), bits(kn1[0]), bits(vn1[0])), labels)
        del Kh, Vh

    peak, peak_kind = measured_peak()
    line = None
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": n_steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "us_per_step": round(ms * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (device Philox)",
            "config": dict(W, parallelism=f"replicas{world}", timed="decode steps 2..K+1",
                           l2="inputs larger than L2 (>= 5 GB of K/V per step)"),
            "frac_of_peak": {"measured": round(value / world / peak, 4),
                             "nominal_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
                             "peak_kind": peak_kind},
            "kv_tokens_per_s": round(world * attn_tokens / n_steps / (ms * 1e-3), 1),
            "step1": {"us": round(step1_ms * 1e3, 2), "bytes": step1_bytes,
                      "GB/s": round(step1_bytes / (step1_ms * 1e-3) / 1e9, 2),
                      "frac_measured": round(step1_bytes / (step1_ms * 1e-3) / 1e9 / peak, 4)},
            "readmitted_blocks": readmit_blocks,
            "roofline": {"bound": "hbm", "kernel": "attention (block table)",
                         "achieved": round(attn_achieved, 2) if attn_achieved else None,
                         "peak": peak, "unit": "GB/s",
                         "frac": round(attn_achieved / peak, 4) if attn_achieved else None,
                         "traffic": paged_traffic, "algorithmic_bytes": attn_bytes_total // n_steps,
                         "peak_kind": f"{peak_kind} (copy bandwidth)"},
            "kernels_us": kernels_us,
            "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "ms_per_step": round(e2e_ms, 4),
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "output": "bf16", "steps": n_e2e},
            "gpu_launches": launches,
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        if not quiet:
            print(json.dumps(line), flush=True)
    pp.close()
    del pp, inputs
    torch.cuda.empty_cache()
    return line


def bench_tiers(args, rank, world, local_rank, steps=None, omega=None, quiet=False,
                omega_sweep=(1, 32), sweep_steps=96, rotary=True):
    """Two-tier run: 4 sequences of 131072 tokens in 128-token windows, K_f
    51 bf16 windows, K_q 204 INT2 windows, routing every omega = 8 steps.
    Timed: K consecutive decode steps from step 1 of a fresh run (steps 1-7
    attend the whole prefill, the first routing event quantizes 204 windows
    per sequence, later steps attend ~6.6k bf16 and ~26k INT2 tokens per
    sequence); the steady state (steps after the first event) is reported
    beside it, with the memory the tiers hold (bf16 pages, INT2 ledger) per
    step, and short runs at other routing intervals (omega_sweep) and in
    rotary mode (rotary: INT2 windows attended as bf16 reconstructions with
    keys rotated forward, rebuilt after each routing event).  Returns the
    JSON record (rank 0) or None."""
    import torch
    dist = init_dist(world, local_rank)
    kvev = load_kvev()
    from workloads.device import TierDeviceWorkload

    W = dict(TIERS)
    if omega is not None:
        W["omega"] = int(omega)
    rope_main = bool(getattr(args, "rope", False))
    if rope_main:   # the rotary record below would repeat the main run
        rotary = False
    if args.layers != WORKLOAD["n_layers"] or args.prefill != WORKLOAD["prefill"]:
        pre = args.prefill if args.prefill != WORKLOAD["prefill"] else W["prefill"]
        W.update(workload=f"profiling case: {args.layers} layers, {W['batch']} x {pre} tokens",
                 n_layers=args.layers, prefill=pre)
    if rope_main:
        W["workload"] += ", rotary positions (rope base 10000)"
    Ly, b, L0 = W["n_layers"], W["batch"], W["prefill"]
    n_steps = steps if steps is not None else args.steps
    max_ctx = L0 + max(n_steps, args.warmup, sweep_steps) + 16
    wl = TierDeviceWorkload(0, n_layers=Ly, batch=b, prefill=L0)
    # bf16 pages: prefill, promotions and, in rotary mode, the reconstructions
    pps = wl.n_pages + 16 + 8 * W["k_full"] + (8 * W["k_quant"] if rotary or rope_main else 0)
    rope_main_table = None
    if rope_main:
        from workloads import rope_table
        rope_main_table = rope_table(max_ctx, W["head_dim"], 10000.0)
    tp = kvev.TierEvictionPass(Ly, W["n_q_heads"], W["n_kv_heads"], W["head_dim"], b, max_ctx,
                               pps, W["k_full"], W["k_quant"], W["omega"], W["alpha"],
                               rope=rope_main_table)
    wl.fill(torch, tp.k_pool, tp.v_pool, pps)
    last = max(n_steps, args.warmup, sweep_steps if omega_sweep else 0)
    inputs = [wl.step_inputs(torch, t, tp.k_pool, pps) for t in range(1, last + 1)]
    # the prefill pages are reused once windows are routed: keep a copy to restart from
    k0, v0 = tp.k_pool.clone(), tp.v_pool.clone()
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()

    def restart(om=None):
        tp.k_pool.copy_(k0)
        tp.v_pool.copy_(v0)
        kvev.kvev_set_tiers(tp.ctx, W["k_full"], W["k_quant"], om or W["omega"])
        tp.begin(L0, stream)

    restart()
    for t in range(1, args.warmup + 1):
        tp.step(*inputs[t - 1], stream)
    kvev.kvev_sync(tp.ctx)

    # timed: steps 1..K of a fresh run, with an event after every step
    restart()
    torch.cuda.synchronize()
    n0 = kvev.kvev_launch_count(tp.ctx)
    clocks = ClockSampler(local_rank)
    clocks.start()
    if dist:
        dist.barrier()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_steps + 1)]
    evs[0].record(stream)
    for t in range(1, n_steps + 1):
        tp.step(*inputs[t - 1], stream)
        evs[t].record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    kvev.kvev_sync(tp.ctx)
    launches = kvev.kvev_launch_count(tp.ctx) - n0
    step_ms = [evs[t - 1].elapsed_time(evs[t]) for t in range(1, n_steps + 1)]
    ms = sum(step_ms) / n_steps
    ms = slowest_ms(ms, dist)

    # replay with per-kernel events, counting what each step attends and the
    # memory the tiers hold after it
    row_bf16 = 2 * W["head_dim"] * 2 * W["n_kv_heads"] * Ly       # bytes per token, all layers
    row_int2 = 768 * W["n_kv_heads"] // 8 * Ly
    ledger_entry = kvev.TIER_LEDGER_BYTES * Ly * W["n_kv_heads"]  # one window, all layers
    kvev.kvev_profile(tp.ctx, True)
    restart()
    kvev.kvev_profile_read(tp.ctx)
    per_step, mem = [], []
    for t in range(1, n_steps + 1):
        tiers = tp.tier.cpu().numpy()
        tl = tp.tail_len.cpu().numpy()
        bf = sum(int(((tiers[s_] == kvev.KVEV_TIER_UNROUTED) | (tiers[s_] == kvev.KVEV_TIER_FULL)).sum())
                 * 128 for s_ in range(b))
        qn = int((tiers == kvev.KVEV_TIER_QUANT).sum()) * 128
        tok_bf = bf + b * (5 + int(tl.max()) + 1)      # + sinks and tail (with the new token)
        per_step.append((tok_bf, qn))
        tp.step(*inputs[t - 1], stream)
        kvev.kvev_sync(tp.ctx)
        tiers = tp.tier.cpu().numpy()
        n_bf_win = int(((tiers == kvev.KVEV_TIER_UNROUTED) | (tiers == kvev.KVEV_TIER_FULL)).sum())
        n_led = int(tp.has_codes.cpu().numpy().astype(bool).sum())
        mem.append((n_bf_win * 128 * row_bf16, n_led * ledger_entry,
                    int((tiers == kvev.KVEV_TIER_QUANT).sum())))
    prof = kvev.kvev_profile_read(tp.ctx)
    kvev.kvev_profile(tp.ctx, False)
    bytes_step = [tb * row_bf16 + tq * row_int2 for tb, tq in per_step]
    total_bytes = sum(bytes_step)
    # DRAM bytes per step of the two attention kernels: their algorithmic bytes
    # times the ratios of ncu captures of the same kernels on smaller cases
    r_bf, r_q = traffic_ratio("attention_paged", "attn.cu"), traffic_ratio("attention_int2",
                                                                          "attn_int2.cu")
    tier_traffic = (round(sum(tb * row_bf16 * r_bf + tq * row_int2 * r_q
                              for tb, tq in per_step) / n_steps)
                    if r_bf and r_q else None)
    value = world * total_bytes / (sum(step_ms) * 1e-3) / 1e9
    first = W["omega"]                     # steps after the first routing event
    steady_ms = sum(step_ms[first:]) / max(1, n_steps - first)
    steady_bytes = sum(bytes_step[first:]) / max(1, n_steps - first)
    att_ms = prof.get("attention", (0.0, 0))[0]
    attn_achieved = total_bytes / (att_ms * 1e-3) / 1e9 if att_ms > 0 else None
    kernels_us = {k: round(v[0] / n_steps * 1e3, 2) for k, v in prof.items()}
    kernels_us["launches_per_step"] = {k: round(v[1] / n_steps, 2) for k, v in prof.items()}
    full_bf16 = b * (L0 + n_steps) * row_bf16
    memory = {"bf16_window_bytes_end": mem[-1][0], "ledger_bytes_end": mem[-1][1],
              "ledger_bytes_max": max(m[1] for m in mem),
              "quant_windows_end": mem[-1][2],
              "ledger_bytes_per_step": [m[1] for m in mem[::max(1, len(mem) // 32)]],
              "full_bf16_cache_bytes": full_bf16,
              "note": "bf16 bytes of unrouted and Full windows (sinks and tail aside) and the "
                      "INT2 ledger (codes kept for every window ever quantized), summed over "
                      "sequences, after each step"}

    # end to end over the same steps 1..K: pinned host q/k/v in, the bf16
    # output and the tiers back, every step
    n_e2e = n_steps
    host_in = [tuple(x.view(torch.int16).cpu().pin_memory() for x in inputs[t - 1])
               for t in range(1, n_e2e + 1)]
    dev_in = [torch.empty_like(x) for x in inputs[0]]
    kvev.kvev_set_output(tp.ctx, kvev.KVEV_OUT_BF16)
    out_dev = torch.empty(tp.out.shape, dtype=torch.bfloat16, device="cuda")
    out_h = torch.empty(tp.out.shape, dtype=torch.bfloat16).pin_memory()
    tier_h = torch.empty(tp.tier.shape, dtype=torch.uint8).pin_memory()
    h2d = sum(x.numel() * 2 for x in host_in[0])
    d2h = out_h.numel() * 2 + tier_h.numel()
    restart()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(n_e2e):
        for d_, h_ in zip(dev_in, host_in[i]):
            d_.view(torch.int16).copy_(h_, non_blocking=True)
        tp.step_no += 1
        kvev.kvev_tier_step(tp.ctx, *dev_in, tp.cache, tp.state, tp.step_no, out_dev, stream)
        out_h.copy_(out_dev, non_blocking=True)
        tier_h.copy_(tp.tier, non_blocking=True)
        stream.synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / n_e2e
    kvev.kvev_sync(tp.ctx)
    kvev.kvev_set_output(tp.ctx, kvev.KVEV_OUT_F32)
    del host_in
    e2e_val = world * (sum(bytes_step[:n_e2e]) / n_e2e) / (e2e_ms * 1e-3) / 1e9

    # routing interval sweep: the same run with routing every omega' steps,
    # timed over steps 1..sweep_steps (mean step and the steps after the
    # first routing event)
    sweep = []
    for om in (omega_sweep or ()):
        if om == W["omega"]:
            continue
        restart(om)
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(sweep_steps + 1)]
        ev[0].record(stream)
        for t in range(1, sweep_steps + 1):
            tp.step(*inputs[t - 1], stream)
            ev[t].record(stream)
        torch.cuda.synchronize()
        kvev.kvev_sync(tp.ctx)
        sm = [ev[t - 1].elapsed_time(ev[t]) for t in range(1, sweep_steps + 1)]
        sweep.append({"omega": om, "steps": sweep_steps,
                      "mean_us": round(sum(sm) / len(sm) * 1e3, 1),
                      "after_first_route_us": round(sum(sm[om:]) / max(1, len(sm) - om) * 1e3, 1),
                      "quant_windows_end": int((tp.tier.cpu().numpy() == kvev.KVEV_TIER_QUANT).sum()),
                      "ledger_bytes_end": int(tp.has_codes.cpu().numpy().astype(bool).sum()) * ledger_entry})
    # rotary mode over the same steps: its cost does not depend on the key
    # values, so the drawn keys stand in for rotated ones
    rot = None
    if rotary:
        from workloads import rope_table
        table = torch.from_numpy(rope_table(max_ctx, W["head_dim"], 10000.0)).to("cuda")
        kvev.kvev_set_rope(tp.ctx, table, max_ctx)
        restart()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(sweep_steps + 1)]
        ev[0].record(stream)
        for t in range(1, sweep_steps + 1):
            tp.step(*inputs[t - 1], stream)
            ev[t].record(stream)
        torch.cuda.synchronize()
        kvev.kvev_sync(tp.ctx)
        kvev.kvev_set_rope(tp.ctx, None, 0)
        sm = [ev[t - 1].elapsed_time(ev[t]) for t in range(1, sweep_steps + 1)]
        om = W["omega"]
        # the first routing event quantizes and reconstructs K_q windows per
        # sequence; later ones reconstruct only the windows entering the tier
        after = range(om + 1, sweep_steps + 1)
        routes = [sm[t - 1] for t in after if t % om == 0]
        plain = [sm[t - 1] for t in after if t % om != 0]
        rot = {"steps": sweep_steps, "omega": om, "rope_base": 10000.0,
               "mean_us": round(sum(sm) / len(sm) * 1e3, 1),
               "after_first_route_us": round(sum(sm[om:]) / max(1, len(sm) - om) * 1e3, 1),
               "first_route_step_us": round(sm[om - 1] * 1e3, 1),
               "route_step_us": round(sum(routes) / max(1, len(routes)) * 1e3, 1),
               "plain_step_us": round(sum(plain) / max(1, len(plain)) * 1e3, 1),
               "note": "INT2 windows attended as bf16 reconstructions (keys rotated forward), "
                       "made at the routing event where a window enters the INT2 tier"}
        del table
    restart()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_tiers(tp, wl, W, inputs[0])

    peak, peak_kind = measured_peak()
    line = None
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": n_steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "us_per_step": round(ms * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 + int2", "data": "synthetic (device Philox)",
            "config": dict(W, parallelism=f"replicas{world}", timed="decode steps 1..K",
                           l2="inputs larger than L2 (>= 5 GB of K/V per step)"),
            "frac_of_peak": {"measured": round(value / world / peak, 4),
                             "nominal_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
                             "peak_kind": peak_kind},
            "steady": {"us": round(steady_ms * 1e3, 2), "bytes": int(steady_bytes),
                       "GB/s": round(steady_bytes / (steady_ms * 1e-3) / 1e9, 2),
                       "frac_measured": round(steady_bytes / (steady_ms * 1e-3) / 1e9 / peak, 4)},
            "first_steps_us": [round(x * 1e3, 1) for x in step_ms[:first + 1]],
            "memory": memory,
            "omega_sweep": sweep,
            "rotary": rot,
            "roofline": {"bound": "hbm", "kernel": "attention (bf16 pages + INT2 windows)",
                         "achieved": round(attn_achieved, 2) if attn_achieved else None,
                         "peak": peak, "unit": "GB/s",
                         "frac": round(attn_achieved / peak, 4) if attn_achieved else None,
                         "traffic": tier_traffic, "algorithmic_bytes": int(total_bytes / n_steps),
                         "peak_kind": f"{peak_kind} (copy bandwidth)"},
            "kernels_us": kernels_us,
            "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "ms_per_step": round(e2e_ms, 4),
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "output": "bf16"},
            "gpu_launches": launches,
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        if not quiet:
            print(json.dumps(line), flush=True)
    tp.close()
    del tp, inputs, k0, v0
    torch.cuda.empty_cache()
    return line


def cpu_baseline_tiers(tp, wl, W, inputs1, n_layers_sample=2, min_seconds=10.0):
    """The two-tier oracle (oracle/qevict.py) on sequence 0 of the batch,
    its first `n_layers_sample` layers, decode step 1 over the whole bf16
    prefill, repeated to about `min_seconds`."""
    import torch

    import oracle as O
    from oracle import qevict as QE
    Ly, d, Hkv = n_layers_sample, W["head_dim"], W["n_kv_heads"]
    L0 = W["prefill"]
    bits = lambda x: x.view(torch.int16).cpu().numpy().view(np.uint16)
    kp = bits(tp.k_pool[0:wl.n_pages, :Ly])
    vp = bits(tp.v_pool[0:wl.n_pages, :Ly])

    def tokens(p):
        rest = p[1:].transpose(1, 2, 0, 3, 4).reshape(Ly, Hkv, -1, d)[:, :, :L0 - 5]
        return np.ascontiguousarray(np.concatenate([p[0, :, :, :5], rest], axis=2))

    K, V = tokens(kp), tokens(vp)
    del kp, vp
    P = QE.QParams(Ly, W["n_q_heads"], Hkv, d, W["k_full"], W["k_quant"], alpha=W["alpha"],
                   omega=W["omega"])
    seq0 = QE.QSequence.from_prefill(P, K, V)
    q, kn, vn = (bits(x[0, :Ly]) for x in inputs1)
    import copy
    threads = O.set_threads(os.cpu_count() or 1)
    # each repetition steps a fresh copy of the prefill state (the copy untimed)
    reps, secs = timed_reps(lambda s: QE.step(P, s, 1, q, kn, vn), min_seconds, 32,
                            prepare=lambda: copy.deepcopy(seq0))
    nbytes = (L0 + 1) * 2 * d * 2 * Hkv * Ly
    cores, model = host_cpu()
    return {"value": round(nbytes * reps / secs / 1e9, 4), "unit": "GB/s",
            "cores": cores, "kind": "oracle", "cpu": model, "seconds": round(secs, 2),
            "sample": f"decode step 1 of sequence 0 of {W['batch']}, its first {Ly} of "
                      f"{W['n_layers']} layers ({L0} + 1 tokens), timed {reps} times; numpy "
                      f"fp64 on the host's BLAS threads"}


if __name__ == "__main__":
    main()

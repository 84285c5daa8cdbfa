"""Benchmark of the decode-step token-selection path on GB300.

One step takes a 49 x 248,320 fp32 verify batch (Gumbel-perturbed Zipf(1.1)
log-probabilities, seed 2) through the whole selection path via the C ABI:
  sel_argmax, sel_topk (k = 20), sel_sample (T 0.7, top_k 40, top_p 0.9,
  min_p 0.05, one uniform per row), and spec_accept in both rules over the
  same 49 rows read as 7 sequences x (6 drafts + 1 bonus) target rows, with
  draft rows = target + N(0, 0.25) and draft tokens drawn from q.
value = verify-batch rows taken through that path per second (49 per step
and rank). Inputs are resident in HBM before the timed region; every launch
reads a copy of the batch that no launch has touched within the previous
>= 487 MB of traffic (more than 3.7 x the 129 MB L2), so each read comes
from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
  python bench.py --profile-steps P    # P untimed eager steps (for ncu), then exit

With --impl reference the CPU oracle (the plain, double-precision C
implementation the tests check against) runs a bounded sample of the same
step on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

ROWS, V = 49, 248_320
K_TOPK = 20
SPEC_S, SPEC_K = 7, 6
POLICY = dict(temperature=0.7, top_k=40, top_p=0.9, min_p=0.05)
ROW_BYTES = V * 4
WORKLOAD = "batched verify selection 49 x 248,320 fp32"
METRIC = "logits rows/s and achieved HBM GB/s (% of GB300 peak) at V=248k, rows=1-49"
N_COPIES = 11         # rotating copies of the batch: 11 x 48.7 MB = 535 MB >= 4 x L2
OP_REPS = 110         # launches per op in the per-op timed regions (a multiple of N_COPIES)
N_GRAPHS = 5 * N_COPIES  # captured step graphs; step s replays graph s % N_GRAPHS
STEPS_PER_GRAPH = 5      # steps captured together for the timed loop


NOMINAL_HBM_GBS = 8000.0  # the ~8 TB/s HBM3e figure the target is stated against


def fracs(gbs: float, peak: float) -> dict:
    """Fractions of the measured copy peak and of the nominal HBM figure."""
    return {"frac_of_peak": round(gbs / peak, 4), "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4)}


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def build_inputs():
    from sampling_row_fp32_gb300 import synth
    x, _ = synth.workload_verify_batch(ROWS, V)
    si = synth.spec_inputs(S=SPEC_S, K=SPEC_K, V=V, target=x.reshape(SPEC_S, SPEC_K + 1, V))
    u = synth.uniforms(4, ROWS)
    return x, si, u


def gpu_arm(args, rank, world, local_rank):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from sampling_row_fp32_gb300 import binding as B

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    x, si, u = build_inputs()

    # resident inputs: rotating copies of the batch and of the draft rows
    xs = [torch.from_numpy(x).to(dev) for _ in range(N_COPIES)]
    drafts = [torch.from_numpy(si.draft).to(dev) for _ in range(2)]
    tok = torch.from_numpy(si.draft_tokens.view(np.int32)).to(dev)
    ua = torch.from_numpy(si.u_acc).to(dev)
    uf = torch.from_numpy(si.u_fin).to(dev)
    ud = torch.from_numpy(u).to(dev)
    ids = torch.empty(ROWS, dtype=torch.int32, device=dev)
    tv = torch.empty(ROWS, K_TOPK, dtype=torch.float32, device=dev)
    ti = torch.empty(ROWS, K_TOPK, dtype=torch.int32, device=dev)
    sid = torch.empty(ROWS, dtype=torch.int32, device=dev)
    sp = torch.empty(ROWS, dtype=torch.float32, device=dev)
    acc = torch.empty(SPEC_S, dtype=torch.int32, device=dev)
    emi = torch.empty(SPEC_S, SPEC_K + 1, dtype=torch.int32, device=dev)
    acc2 = torch.empty(SPEC_S, dtype=torch.int32, device=dev)
    emi2 = torch.empty(SPEC_S, SPEC_K + 1, dtype=torch.int32, device=dev)
    ws_a = B.workspace(B.SEL_OP_ARGMAX, ROWS, V, device=dev)
    ws_t = B.workspace(B.SEL_OP_TOPK, ROWS, V, K_TOPK, device=dev)
    ws_s = B.workspace(B.SEL_OP_SAMPLE, ROWS, V, POLICY["top_k"], device=dev)
    ws_r = B.workspace(B.SEL_OP_SPEC, SPEC_S, V, SPEC_K, device=dev)
    ws_g = B.workspace(B.SEL_OP_SPEC, SPEC_S, V, SPEC_K, device=dev)
    prm = B.SampleParams(POLICY["temperature"], POLICY["top_k"], POLICY["top_p"], POLICY["min_p"],
                         B.SEL_ORDER_TEMP_FIRST)
    rej = B.SpecParams(1.0, B.SPEC_MODE_REJECTION)
    arg = B.SpecParams(1.0, B.SPEC_MODE_ARGMAX)
    OPS = ["argmax", "topk", "sample", "spec_rejection", "spec_argmax"]
    # the copy each op of step s reads: consecutive reads walk the N_COPIES
    # copies in turn, so a copy is read again only after 10 others (487 MB)
    def copy_for(step, op):
        return xs[(5 * step + op) % N_COPIES]

    def target_view(t):
        return t.view(SPEC_S, SPEC_K + 1, V)

    def run_op(step, op):  # on the current stream
        if op == 0:
            B.sel_argmax(copy_for(step, 0), ids, ws_a)
        elif op == 1:
            B.sel_topk(copy_for(step, 1), K_TOPK, tv, ti, ws_t)
        elif op == 2:
            B.sel_sample(copy_for(step, 2), prm, ud, sid, sp, ws_s)
        elif op == 3:
            B.spec_accept(target_view(copy_for(step, 3)), drafts[step % 2], tok, rej, ua, uf, acc, emi, ws_r)
        else:
            B.spec_accept(target_view(copy_for(step, 4)), None, tok, arg, None, None, acc2, emi2, ws_g)

    # argmax, top-k, sample and the argmax rule: a main launch and a finishing
    # launch each; the rejection rule: phase 1, the decision with the draw's
    # chunk sums, and the draw's find launch
    launches_per_step = len(STEP_LAUNCHES)
    bytes_per_op = [ROWS * ROW_BYTES, ROWS * ROW_BYTES, ROWS * ROW_BYTES,
                    None, ROWS * ROW_BYTES]

    # eager warm-up (also the first launches of every kernel)
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for s in range(max(args.warmup, 1)):
            for op in range(5):
                run_op(s, op)
    torch.cuda.synchronize()
    # residual re-read of the rejection rule: the rejecting position's target
    # and draft rows, or the bonus row when all positions accept
    n_acc = acc.cpu().numpy()
    resid_rows = int(sum(2 if a < SPEC_K else 1 for a in n_acc))
    bytes_per_op[3] = (SPEC_S * (2 * SPEC_K + 1) + resid_rows) * ROW_BYTES

    if args.profile_steps:
        # untimed eager steps for a profiler, nothing else
        with torch.cuda.stream(stream):
            for s in range(args.profile_steps):
                for op in range(5):
                    run_op(s, op)
        torch.cuda.synchronize()
        return None

    # Each step is replayed from a CUDA graph of its five calls (11 launches),
    # so the host's launch cost does not gap the GPU. Step s (warm-up steps
    # first) replays graph s % N_GRAPHS, which keeps the copy rotation.
    n_graphs = N_GRAPHS
    graphs = []
    for gi in range(n_graphs):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for op in range(5):
                run_op(gi, op)
        graphs.append(g)
    # The timed loop replays runs of STEPS_PER_GRAPH consecutive steps from
    # one graph (steps s0 .. s0 + 4 for s0 a multiple of 5), so a graph
    # launch's own latency is paid once per run; steps outside a whole run
    # replay their single-step graph.
    multi = []
    for gi in range(n_graphs // STEPS_PER_GRAPH):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for s in range(gi * STEPS_PER_GRAPH, (gi + 1) * STEPS_PER_GRAPH):
                for op in range(5):
                    run_op(s, op)
        multi.append(g)

    def replay_steps(first, count):
        s, end = first, first + count
        while s < end:
            if s % STEPS_PER_GRAPH == 0 and s + STEPS_PER_GRAPH <= end:
                multi[(s % n_graphs) // STEPS_PER_GRAPH].replay()
                s += STEPS_PER_GRAPH
            else:
                graphs[s % n_graphs].replay()
                s += 1

    # per-op timing: one graph of OP_REPS launches of each op (same input
    # rotation), bracketed by events on the launching stream
    op_graphs = []
    for op in range(5):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(OP_REPS):
                run_op(r, op)
        op_graphs.append(g)
    with torch.cuda.stream(stream):
        for s in range(args.warmup):
            graphs[s % n_graphs].replay()
        for g in multi:
            g.replay()
        for g in op_graphs:
            g.replay()
    torch.cuda.synchronize()

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.25)  # let the sampler start
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        replay_steps(args.warmup, args.steps)
        t_end.record(stream)
    torch.cuda.synchronize()
    # per-op timed regions, right after the steps (same clocks)
    per_op_us = []
    for op in range(5):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            op_graphs[op].replay()
            b.record(stream)
        torch.cuda.synchronize()
        per_op_us.append(a.elapsed_time(b) * 1e3 / OP_REPS)
    extra = extra_ops(B, dev, xs, drafts, tok, stream)
    # keep the same load running briefly so the clock sampler sees it even
    # when the timed region is shorter than its period
    tail_until = time.time() + 0.6
    s = args.warmup + args.steps
    while time.time() < tail_until:
        with torch.cuda.stream(stream):
            for _ in range(8):
                graphs[s % n_graphs].replay()
                s += 1
        torch.cuda.synchronize()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([total_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())

    # end to end through the same C-ABI calls with host buffers: pinned input
    # copied to the device, the five calls, results copied back, every step
    e2e = e2e_leg(args, B, dev, x, si, u, prm, rej, arg, ws_a, ws_t, ws_s, ws_r, ws_g)

    peak, peak_kind = measured_peak()
    step_s = total_ms / 1e3 / args.steps
    rows_per_s = ROWS * world / step_s
    step_bytes = sum(bytes_per_op)
    dom = int(np.argmax(per_op_us))
    dom_gbs = bytes_per_op[dom] / (per_op_us[dom] * 1e-6) / 1e9
    ops = {OPS[i]: dict({"us": round(per_op_us[i], 3), "bytes": bytes_per_op[i],
                         "gbs": round(bytes_per_op[i] / (per_op_us[i] * 1e-6) / 1e9, 1)},
                        **fracs(bytes_per_op[i] / (per_op_us[i] * 1e-6) / 1e9, peak))
           for i in range(5)}
    traffic = load_traffic(OPS[dom])
    line = {
        "metric": METRIC,
        "value": round(rows_per_s, 1),
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded Gumbel-perturbed Zipf(1.1) logits; no dataset)",
        "config": dict(workload_config(),
                       l2=f"inputs rotate over {N_COPIES} resident copies of the batch (535 MB); each "
                          "launch reads a copy untouched for >= 487 MB of traffic (L2 is 129 MB)",
                       parallelism=f"replicas x{world} (independent rows)"),
        "step_gbs": round(step_bytes / step_s / 1e9, 1),
        "ops": ops,
        "roofline": {"bound": "hbm", "kernel": OPS[dom], "achieved": round(dom_gbs, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(dom_gbs / peak, 4),
                     "frac_of_nominal": round(dom_gbs / NOMINAL_HBM_GBS, 4), "nominal_gbs": NOMINAL_HBM_GBS,
                     "traffic": traffic},
        "gpu_launches": launches_per_step * args.steps,
        "timing": f"steps replayed from CUDA graphs of {STEPS_PER_GRAPH} consecutive steps; per-op times "
                  f"from {OP_REPS} graph-replayed launches of each op between events on the launching stream",
        "clocks": clk,
        "e2e": e2e,
        "extra_ops": extra,
        "configs": named_configs(B, dev, stream),
        "rows_sweep": rows_sweep(B, dev, stream),
        "spec_sweep": spec_sweep(B, dev, stream),
    }
    return line


def full_row_search_rows() -> int:
    """Rows of the verify batch whose top-p nucleus (at the step's T and
    top_p, over the whole row) holds more than the 64 candidates, so that the
    cut search decides them (computed in double on the host)."""
    from sampling_row_fp32_gb300 import synth
    x, _ = synth.workload_verify_batch(ROWS, V)
    z = x.astype(np.float64) / POLICY["temperature"]
    z -= z.max(axis=1, keepdims=True)
    w = np.exp(z)
    w /= w.sum(axis=1, keepdims=True)
    c = np.cumsum(-np.sort(-w, axis=1), axis=1)
    return int((((c < POLICY["top_p"]).sum(axis=1) + 1) > 64).sum())


TYPICAL_P = 0.9  # the full-row typical line: T as the step's, typical_p 0.9, no other filter


def full_row_typical_search_rows() -> int:
    """Rows of the verify batch whose locally typical window (at the step's
    T, typical_p TYPICAL_P, over the whole row) reaches past the 64 most
    probable tokens, so that the cut search decides them (double, host)."""
    from sampling_row_fp32_gb300 import synth
    x, _ = synth.workload_verify_batch(ROWS, V)
    n = 0
    for r in range(ROWS):
        z = x[r].astype(np.float64) / POLICY["temperature"]
        z -= z.max()
        p = np.exp(z)
        p /= p.sum()
        lp = np.log(p, where=p > 0, out=np.full_like(p, -np.inf))
        h = -(p[p > 0] * lp[p > 0]).sum()
        score = np.abs(-lp - h)
        order = np.lexsort((np.arange(p.size), score))
        k = int(np.searchsorted(np.cumsum(p[order]), TYPICAL_P) + 1)
        rank = np.empty(p.size, dtype=np.int64)
        rank[np.lexsort((np.arange(p.size), -p))] = np.arange(p.size)
        n += int(rank[order[:k]].max() >= 64)
    return n


def extra_ops(B, dev, xs, drafts, tok, stream):
    """The calls beyond the step, on the same batch and copy rotation, each
    timed over OP_REPS graph-replayed launches: the EOG-excluding argmax (8
    ids), sampling with the step's policy plus top-n-sigma 1.0 and typical_p
    0.8, full-row sampling (top_k = 0, the step's T, top_p and min_p),
    sampler-match acceptance (7 x 6, the step's policy), the closed-form
    diagnostics (7 x 6), a two-shard top-k (k = 20 per shard on each half
    of the vocabulary, then the merge), and full-row locally typical sampling
    (top_k = 0, the step's T, typical_p TYPICAL_P)."""
    import torch
    peak, _ = measured_peak()
    ids = torch.empty(ROWS, dtype=torch.int32, device=dev)
    exd = torch.tensor([0, 5, 1000, 4096, 77_777, 151_643, 151_645, 248_000], dtype=torch.int32, device=dev)
    ws_a = B.workspace(B.SEL_OP_ARGMAX, ROWS, V, device=dev)
    prm = B.SampleParams(POLICY["temperature"], POLICY["top_k"], POLICY["top_p"], POLICY["min_p"],
                         B.SEL_ORDER_TEMP_FIRST)
    ud = torch.rand(SPEC_S, SPEC_K + 1, device=dev)
    acc = torch.empty(SPEC_S, dtype=torch.int32, device=dev)
    emi = torch.empty(SPEC_S, SPEC_K + 1, dtype=torch.int32, device=dev)
    ws_m = B.workspace(B.SEL_OP_SPEC_SAMPLER, ROWS, V, POLICY["top_k"], device=dev)
    smin = torch.empty(SPEC_S, SPEC_K, device=dev)
    sprod = torch.empty(SPEC_S, SPEC_K, device=dev)
    ws_d = B.workspace(B.SEL_OP_SPEC_DIAG, SPEC_S, V, SPEC_K, device=dev)
    from sampling_row_fp32_gb300 import shards as sh
    offs = sh.shard_offsets(V, 2, min_size=K_TOPK)
    halves = [[x[:, offs[g]:offs[g + 1]].contiguous() for g in range(2)] for x in xs]
    sv = [torch.empty(ROWS, K_TOPK, device=dev) for _ in range(2)]
    si = [torch.empty(ROWS, K_TOPK, dtype=torch.int32, device=dev) for _ in range(2)]
    ws_s = [B.workspace(B.SEL_OP_TOPK, ROWS, offs[g + 1] - offs[g], K_TOPK, device=dev) for g in range(2)]
    gv = torch.empty(ROWS, 2, K_TOPK, device=dev)
    gi = torch.empty(ROWS, 2, K_TOPK, dtype=torch.int32, device=dev)
    mv = torch.empty(ROWS, K_TOPK, device=dev)
    mi = torch.empty(ROWS, K_TOPK, dtype=torch.int32, device=dev)

    def tview(t):
        return t.view(SPEC_S, SPEC_K + 1, V)

    def sharded(r):
        for g in range(2):
            B.sel_topk(halves[r % N_COPIES][g], K_TOPK, sv[g], si[g], ws_s[g])
            gv[:, g].copy_(sv[g])
            gi[:, g].copy_(si[g])
        B.sel_merge_shards(gv, gi, offs, mv, mi)

    prm_f = B.SampleParams(POLICY["temperature"], POLICY["top_k"], POLICY["top_p"], POLICY["min_p"],
                           B.SEL_ORDER_TEMP_FIRST, 1.0, 0.8)
    sid = torch.empty(ROWS, dtype=torch.int32, device=dev)
    spr = torch.empty(ROWS, dtype=torch.float32, device=dev)
    uu = torch.rand(ROWS, device=dev)
    ws_f = B.workspace(B.SEL_OP_SAMPLE, ROWS, V, POLICY["top_k"], device=dev)
    prm_full = B.SampleParams(POLICY["temperature"], 0, POLICY["top_p"], POLICY["min_p"], B.SEL_ORDER_TEMP_FIRST)
    prm_last = B.SampleParams(POLICY["temperature"], POLICY["top_k"], POLICY["top_p"], POLICY["min_p"],
                              B.SEL_ORDER_TEMP_LAST)
    ws_full = B.workspace(B.SEL_OP_SAMPLE, ROWS, V, 0, device=dev)
    prm_typ = B.SampleParams(POLICY["temperature"], 0, 1.0, 0.0, B.SEL_ORDER_TEMP_FIRST, 0.0, TYPICAL_P)
    ws_typ = B.workspace(B.SEL_OP_SAMPLE, ROWS, V, 0, device=dev)
    typ_rows = full_row_typical_search_rows()
    calls = {
        "argmax_excluding_8": (lambda r: B.sel_argmax_excluding(xs[r % N_COPIES], exd, ids, ws_a), ROWS * ROW_BYTES),
        # full-row sampling reads every row twice (candidates and sums, then
        # the draw); a row whose cut lies past the 64 candidates is read once
        # more by the cut search (staged in shared memory, whose passes then
        # read no more of it): counted too
        "sample_full_row": (lambda r: B.sel_sample(xs[r % N_COPIES], prm_full, uu, sid, spr, ws_full),
                            (2 * ROWS + full_row_search_rows()) * ROW_BYTES),
        "sample_full_row_typical": (lambda r: B.sel_sample(xs[r % N_COPIES], prm_typ, uu, sid, spr, ws_typ),
                                    (2 * ROWS + typ_rows) * ROW_BYTES),
        "sample_nsigma1_typical08": (lambda r: B.sel_sample(xs[r % N_COPIES], prm_f, uu, sid, spr, ws_f),
                                     ROWS * ROW_BYTES),
        # the step's policy with the filters on the untempered distribution
        # and the temperature in the draw only
        "sample_temp_last": (lambda r: B.sel_sample(xs[r % N_COPIES], prm_last, uu, sid, spr, ws_f),
                             ROWS * ROW_BYTES),
        "spec_sampler_match": (lambda r: B.spec_accept_sampler(tview(xs[r % N_COPIES]), tok, prm, ud, acc, emi, ws_m),
                               ROWS * ROW_BYTES),
        "spec_diagnostics": (lambda r: B.spec_diagnostics(tview(xs[r % N_COPIES]), drafts[r % 2], 1.0, smin, sprod,
                                                          ws_d),
                             (SPEC_S * (2 * SPEC_K + 1) + 2 * SPEC_S * SPEC_K) * ROW_BYTES),
        "topk_two_shards": (sharded, ROWS * ROW_BYTES),
    }
    out = {}
    for name, (fn, nbytes) in calls.items():
        with torch.cuda.stream(stream):
            for r in range(3):
                fn(r)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(OP_REPS):
                fn(r)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / OP_REPS
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = dict({"us": round(us, 3), "bytes": nbytes, "gbs": round(gbs, 1)}, **fracs(gbs, peak))
    out["sample_full_row"]["cut_search_rows"] = full_row_search_rows()
    with torch.cuda.stream(stream):
        B.sel_sample(xs[0], prm_full, uu, sid, spr, ws_full)
    torch.cuda.synchronize()
    out["sample_full_row"]["failed_rows"] = int((B.ids_to_numpy(sid) == 0xFFFFFFFF).sum())
    out["sample_full_row_typical"]["cut_search_rows"] = typ_rows
    with torch.cuda.stream(stream):
        B.sel_sample(xs[0], prm_typ, uu, sid, spr, ws_typ)
    torch.cuda.synchronize()
    out["sample_full_row_typical"]["failed_rows"] = int((B.ids_to_numpy(sid) == 0xFFFFFFFF).sum())
    return out


SWEEP_ROWS = (1, 2, 4, 8, 16, 32, 49)
SWEEP_REPS = 110


def rows_sweep(B, dev, stream):
    """The metric's range: argmax, top-k (k = 20) and sampling (the step's
    policy) on 1 .. 49 rows of V = 248,320, timed like the step's ops. The
    verify batch's rows are repeated through a buffer of about 630 MB, and
    call i reads the block of rows that starts i rows-sizes further on, so a
    block is read again only after at least ~480 MB of other reads (L2 is
    129 MB). Below a few MB a call these are bound by launch latency."""
    import torch
    from sampling_row_fp32_gb300 import synth
    peak, _ = measured_peak()
    x, _ = synth.workload_verify_batch(ROWS, V)
    reps = 13
    big = torch.from_numpy(np.ascontiguousarray(x)).to(dev).repeat(reps, 1)  # reps * 49 rows
    total_rows = big.shape[0]
    u = torch.from_numpy(synth.uniforms(5, total_rows)).to(dev)
    prm = B.SampleParams(POLICY["temperature"], POLICY["top_k"], POLICY["top_p"], POLICY["min_p"],
                         B.SEL_ORDER_TEMP_FIRST)
    out = {"workload": f"rows of the verify batch, V = {V:,}; argmax, top-k k = {K_TOPK}, sampling "
                       f"(T {POLICY['temperature']}, top_k {POLICY['top_k']}, top_p {POLICY['top_p']}, "
                       f"min_p {POLICY['min_p']})",
           "rows": list(SWEEP_ROWS), "argmax": [], "topk": [], "sample": []}
    for r in SWEEP_ROWS:
        n_blocks = total_rows // r
        ids = torch.empty(r, dtype=torch.int32, device=dev)
        tv = torch.empty(r, K_TOPK, device=dev)
        ti = torch.empty(r, K_TOPK, dtype=torch.int32, device=dev)
        sid = torch.empty(r, dtype=torch.int32, device=dev)
        sp = torch.empty(r, device=dev)
        ws_a = B.workspace(B.SEL_OP_ARGMAX, r, V, device=dev)
        ws_t = B.workspace(B.SEL_OP_TOPK, r, V, K_TOPK, device=dev)
        ws_s = B.workspace(B.SEL_OP_SAMPLE, r, V, POLICY["top_k"], device=dev)

        def blk(i):
            b = (i % n_blocks) * r
            return big[b:b + r]

        calls = {
            "argmax": lambda i: B.sel_argmax(blk(i), ids, ws_a),
            "topk": lambda i: B.sel_topk(blk(i), K_TOPK, tv, ti, ws_t),
            "sample": lambda i: B.sel_sample(blk(i), prm, u[(i % n_blocks) * r:(i % n_blocks) * r + r], sid, sp,
                                             ws_s),
        }
        for op, fn in calls.items():
            with torch.cuda.stream(stream):
                for i in range(3):
                    fn(i)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(SWEEP_REPS):
                    fn(i)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                g.replay()
                a.record(stream)
                g.replay()
                b.record(stream)
            torch.cuda.synchronize()
            us = a.elapsed_time(b) * 1e3 / SWEEP_REPS
            nbytes = r * V * 4
            gbs = nbytes / (us * 1e-6) / 1e9
            out[op].append(dict({"rows": r, "us": round(us, 3), "rows_per_s": round(r / (us * 1e-6), 1),
                                 "gbs": round(gbs, 1)}, **fracs(gbs, peak)))
            del g
    del big
    torch.cuda.synchronize()
    return out


SPEC_SWEEP = ((1, 1), (1, 4), (1, 8), (2, 4), (4, 4))


def spec_sweep(B, dev, stream):
    """Speculative acceptance on small batches (S sequences x K drafts) at
    V = 248,320, both rules, timed like the step's ops: each call reads one
    of several resident copies of its inputs (at least ~500 MB between two
    reads of a copy, or 64 copies). Latency-bound: a few MB a call."""
    import torch
    from sampling_row_fp32_gb300 import synth
    out = {"workload": f"S sequences x K drafts, V = {V:,}, T = 1, draft = target + N(0, 0.7^2)", "cases": []}
    for S, K in SPEC_SWEEP:
        si = synth.spec_inputs(S=S, K=K, V=V, seed_target=S + K, seed_draft=7, seed_u=9, sigma_noise=0.7)
        n = int(min(64, max(2, 500e6 // (si.target.nbytes + si.draft.nbytes))))
        t = torch.from_numpy(si.target).to(dev).unsqueeze(0).repeat(n, 1, 1, 1)
        d = torch.from_numpy(si.draft).to(dev).unsqueeze(0).repeat(n, 1, 1, 1)
        tok = torch.from_numpy(si.draft_tokens.view(np.int32)).to(dev)
        ua = torch.from_numpy(si.u_acc).to(dev)
        uf = torch.from_numpy(si.u_fin).to(dev)
        acc = torch.empty(S, dtype=torch.int32, device=dev)
        emi = torch.empty(S, K + 1, dtype=torch.int32, device=dev)
        ws = B.workspace(B.SEL_OP_SPEC, S, V, K, device=dev)
        rej = B.SpecParams(1.0, B.SPEC_MODE_REJECTION)
        arg = B.SpecParams(1.0, B.SPEC_MODE_ARGMAX)
        case = {"S": S, "K": K}
        for name, fn in (("rejection_us", lambda i: B.spec_accept(t[i % n], d[i % n], tok, rej, ua, uf, acc, emi, ws)),
                         ("argmax_us", lambda i: B.spec_accept(t[i % n], None, tok, arg, None, None, acc, emi, ws))):
            with torch.cuda.stream(stream):
                for i in range(3):
                    fn(i)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(SWEEP_REPS):
                    fn(i)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                g.replay()
                a.record(stream)
                g.replay()
                b.record(stream)
            torch.cuda.synchronize()
            case[name] = round(a.elapsed_time(b) * 1e3 / SWEEP_REPS, 3)
            del g
        out["cases"].append(case)
        del t, d
    torch.cuda.synchronize()
    return out


def named_configs(B, dev, stream):
    """The other named workloads, each timed like the step's ops: graph-replayed
    calls between events, every call reading a copy of its input that at
    least ~480 MB of other reads have passed since (L2 is 129 MB). The one-row
    argmax and the three-row top-k move under 3 MB a call: they are bound by
    launch latency, so their HBM fractions are reported but mean little."""
    import torch
    from sampling_row_fp32_gb300 import synth
    peak, _ = measured_peak()
    out = {}

    def timed(fn, n_copies, reps):
        with torch.cuda.stream(stream):
            for r in range(3):
                fn(r % n_copies)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(reps):
                fn(r % n_copies)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / reps

    def record(name, what, us, rows, nbytes, note=None):
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = dict({"workload": what, "us": round(us, 3), "rows_per_s": round(rows / (us * 1e-6), 1),
                          "bytes": nbytes, "gbs": round(gbs, 1)}, **fracs(gbs, peak))
        if note:
            out[name]["note"] = note

    def copies(a: np.ndarray, n: int):
        t = torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        big = torch.empty((n,) + tuple(t.shape), dtype=t.dtype, device=dev)
        big.copy_(t.unsqueeze(0).expand_as(big))
        return big

    latency = "latency-bound: under 3 MB a call, so the HBM fraction is not the figure of merit"
    # greedy argmax, 1 x 202,048, three planted maxima
    x1, _ = synth.workload_argmax_planted()
    n1 = 640
    c1 = copies(x1, n1)
    ids1 = torch.empty(1, dtype=torch.int32, device=dev)
    ws1 = B.workspace(B.SEL_OP_ARGMAX, 1, x1.shape[1], device=dev)
    us = timed(lambda r: B.sel_argmax(c1[r], ids1, ws1), n1, n1)
    record("argmax_1x202048", "greedy argmax, 1 x 202,048 fp32, 3 planted maxima", us, 1, x1.nbytes, latency)
    del c1
    # exact top-k, k = 84, 3 x 248,320 with a peaked head
    x2, k2 = synth.workload_topk_peaked()
    n2 = 180
    c2 = copies(x2, n2)
    tv2 = torch.empty(3, k2, device=dev)
    ti2 = torch.empty(3, k2, dtype=torch.int32, device=dev)
    ws2 = B.workspace(B.SEL_OP_TOPK, 3, x2.shape[1], k2, device=dev)
    us = timed(lambda r: B.sel_topk(c2[r], k2, tv2, ti2, ws2), n2, n2)
    record("topk84_3x248320", "exact top-k k = 84, 3 x 248,320 fp32, peaked head", us, 3, x2.nbytes, latency)
    del c2
    # filtered sampling, 64 x 202,048, T 0.7, top_k 40, top_p 0.9, min_p 0.05
    x4, u4, pol = synth.workload_sample()
    n4 = 11
    c4 = copies(x4, n4)
    ud4 = torch.from_numpy(u4).to(dev)
    sid4 = torch.empty(64, dtype=torch.int32, device=dev)
    sp4 = torch.empty(64, device=dev)
    prm4 = B.SampleParams(pol.temperature, pol.top_k, pol.top_p, pol.min_p, B.SEL_ORDER_TEMP_FIRST)
    ws4 = B.workspace(B.SEL_OP_SAMPLE, 64, x4.shape[1], pol.top_k, device=dev)
    us = timed(lambda r: B.sel_sample(c4[r], prm4, ud4, sid4, sp4, ws4), n4, 10 * n4)
    record("sample_64x202048", "sampling 64 x 202,048 fp32, T 0.7, top_k 40, top_p 0.9, min_p 0.05",
           us, 64, x4.nbytes)
    del c4
    # speculative acceptance, 8 sequences x 8 drafts, V = 151,936, both rules
    si = synth.workload_spec()
    S5, K5 = si.draft_tokens.shape
    V5 = si.target.shape[2]
    n5 = 7
    ct = copies(si.target, n5)
    cd = copies(si.draft, n5)
    tok5 = torch.from_numpy(si.draft_tokens.view(np.int32)).to(dev)
    ua5 = torch.from_numpy(si.u_acc).to(dev)
    uf5 = torch.from_numpy(si.u_fin).to(dev)
    acc5 = torch.empty(S5, dtype=torch.int32, device=dev)
    emi5 = torch.empty(S5, K5 + 1, dtype=torch.int32, device=dev)
    ws5 = B.workspace(B.SEL_OP_SPEC, S5, V5, K5, device=dev)
    rej = B.SpecParams(si.temperature, B.SPEC_MODE_REJECTION)
    arg = B.SpecParams(si.temperature, B.SPEC_MODE_ARGMAX)
    row5 = V5 * 4
    us = timed(lambda r: B.spec_accept(ct[r], cd[r], tok5, rej, ua5, uf5, acc5, emi5, ws5), n5, 10 * n5)
    n_acc = B.ids_to_numpy(acc5)
    resid = int(sum(2 if a < K5 else 1 for a in n_acc))
    record("spec_rejection_8x8", "speculative acceptance, rejection rule, 8 x 8 drafts, V = 151,936",
           us, S5, (S5 * (2 * K5 + 1) + resid) * row5)
    us = timed(lambda r: B.spec_accept(ct[r], None, tok5, arg, None, None, acc5, emi5, ws5), n5, 10 * n5)
    record("spec_argmax_8x8", "speculative acceptance, argmax rule, 8 x 8 drafts, V = 151,936",
           us, S5, S5 * (K5 + 1) * row5)
    del ct, cd
    torch.cuda.synchronize()
    return out


# The launches of one eager step, in order, with the op each belongs to and
# a piece of its kernel name (ncu prints "...<1, 0>" for template flags).
STEP_LAUNCHES = [
    ("argmax", "argmax_kernel"), ("argmax", "argmax_finish_kernel"),
    ("topk", "topk_kernel"), ("topk", "topk_finish_kernel<0"),
    ("sample", "topk_kernel"), ("sample", "topk_finish_kernel<1"),
    ("spec_rejection", "spec_phase1_kernel"), ("spec_rejection", "spec_decide_draw_cl_kernel"),
    ("spec_argmax", "argmax_kernel"), ("spec_argmax", "spec_argmax_finish_kernel"),
]
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic.json")


def sources_fingerprint() -> str:
    """sha256 over the kernel sources and the public header: counters taken
    from another fingerprint describe other kernels."""
    import hashlib
    h = hashlib.sha256()
    dirs = [os.path.join(ROOT, "sampling_row_fp32_gb300", "csrc"), os.path.join(ROOT, "include")]
    for d in dirs:
        for f in sorted(os.listdir(d)):
            if f.endswith((".cu", ".cuh", ".h")):
                h.update(f.encode())
                with open(os.path.join(d, f), "rb") as fh:
                    h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(op_name):
    """DRAM bytes (read + write) per call of the op, from the committed ncu
    counters, or None when they were taken on other kernel sources."""
    try:
        with open(TRAFFIC_JSON) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("sources") != sources_fingerprint():
        return None
    return t.get("ops", {}).get(op_name)


def write_traffic(csv_path):
    """Turn an ncu CSV of dram__bytes_read.sum / dram__bytes_write.sum per
    launch (whole eager steps, from the first launch of a step) into
    profiles/traffic.json: mean bytes per call of each op, stamped with the
    current sources' fingerprint."""
    import csv
    import collections
    rows = list(csv.reader(open(csv_path)))
    hdr_i = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
    hdr = rows[hdr_i]
    ki, mi, vi, ui, idi = (hdr.index(c) for c in ("Kernel Name", "Metric Name", "Metric Value",
                                                     "Metric Unit", "ID"))
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    per_launch = collections.defaultdict(float)
    names = {}
    for r in rows[hdr_i + 1:]:
        if len(r) <= vi or r[mi] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        per_launch[r[idi]] += float(r[vi].replace(",", "")) * scale[r[ui]]
        names[r[idi]] = r[ki]
    # whole steps of STEP_LAUNCHES, in launch order; each launch's name must
    # match its slot
    ids = sorted(per_launch, key=int)
    n = len(STEP_LAUNCHES)
    steps = len(ids) // n
    if steps == 0:
        raise SystemExit(f"{csv_path}: fewer than {n} launches")
    sums = collections.defaultdict(float)
    for st in range(steps):
        for j, (op, pat) in enumerate(STEP_LAUNCHES):
            lid = ids[st * n + j]
            if pat not in names[lid]:
                raise SystemExit(f"launch {lid} is {names[lid]!r}, expected {pat!r}: not aligned to a step")
            sums[op] += per_launch[lid]
    ops = {op: round(v / steps) for op, v in sums.items()}
    out = {"sources": sources_fingerprint(), "unit": "bytes per call (dram read + write)",
           "source_csv": os.path.basename(csv_path), "ops": ops}
    with open(TRAFFIC_JSON, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    return out


def e2e_leg(args, B, dev, x, si, u, prm, rej, arg, ws_a, ws_t, ws_s, ws_r, ws_g):
    """The step through the public calls with host buffers: every step copies
    its inputs from pinned host memory to the device, runs the five calls and
    copies every output back. Two device input sets alternate, so the copy of
    step s + 1 (on its own stream) runs while step s computes; a step's calls
    wait for its own copy, and a copy waits until the calls that last read its
    buffers are done. The link (about 210 GB/s host to device on this machine)
    bounds the rate."""
    import torch
    hx = torch.from_numpy(x).pin_memory()
    hd = torch.from_numpy(si.draft).pin_memory()
    htok = torch.from_numpy(si.draft_tokens.view(np.int32)).pin_memory()
    hua = torch.from_numpy(si.u_acc).pin_memory()
    huf = torch.from_numpy(si.u_fin).pin_memory()
    hu = torch.from_numpy(u).pin_memory()
    host_in = (hx, hd, htok, hua, huf, hu)
    dev_in = [[torch.empty_like(h, device=dev) for h in host_in] for _ in range(2)]
    outs_d = [torch.empty(ROWS, dtype=torch.int32, device=dev), torch.empty(ROWS, K_TOPK, device=dev),
              torch.empty(ROWS, K_TOPK, dtype=torch.int32, device=dev),
              torch.empty(ROWS, dtype=torch.int32, device=dev), torch.empty(ROWS, device=dev),
              torch.empty(SPEC_S, dtype=torch.int32, device=dev),
              torch.empty(SPEC_S, SPEC_K + 1, dtype=torch.int32, device=dev),
              torch.empty(SPEC_S, dtype=torch.int32, device=dev),
              torch.empty(SPEC_S, SPEC_K + 1, dtype=torch.int32, device=dev)]
    outs_h = [torch.empty_like(o, device="cpu").pin_memory() for o in outs_d]
    stream = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream(device=dev)
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in outs_d)
    freed = [None, None]  # per input set: the event after the calls that read it

    def step(sidx):
        buf = dev_in[sidx % 2]
        with torch.cuda.stream(copy_stream):
            if freed[sidx % 2] is not None:
                copy_stream.wait_event(freed[sidx % 2])
            for h, d in zip(host_in, buf):
                d.copy_(h, non_blocking=True)
            copied = torch.cuda.Event()
            copied.record(copy_stream)
        stream.wait_event(copied)
        dx, dd, dtok, dua, duf, du = buf
        B.sel_argmax(dx, outs_d[0], ws_a, stream)
        B.sel_topk(dx, K_TOPK, outs_d[1], outs_d[2], ws_t, stream)
        B.sel_sample(dx, prm, du, outs_d[3], outs_d[4], ws_s, stream)
        tv = dx.view(SPEC_S, SPEC_K + 1, V)
        B.spec_accept(tv, dd, dtok, rej, dua, duf, outs_d[5], outs_d[6], ws_r, stream)
        B.spec_accept(tv, None, dtok, arg, None, None, outs_d[7], outs_d[8], ws_g, stream)
        done = torch.cuda.Event()
        done.record(stream)
        freed[sidx % 2] = done
        for d, h in zip(outs_d, outs_h):
            h.copy_(d, non_blocking=True)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    n = max(args.steps, 1)
    # the timed region starts before the first step's copy
    a.record(copy_stream)
    stream.wait_event(a)
    for i in range(n):
        step(i)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / n
    return {"value": round(ROWS / (ms / 1e3), 1), "unit": "rows/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 5),
            "pipelined": "two input sets: the copy of step s + 1 overlaps the calls of step s"}


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle on a bounded sample of the step
# ---------------------------------------------------------------------------

REF_ROWS = 7  # one spec sequence (6 drafts + bonus) and 7 rows for the other ops


def oracle_step(orc, x, si, u):
    xs = x[:REF_ROWS]
    orc.argmax(xs)
    orc.topk(xs, K_TOPK)
    orc.sample(xs, u[:REF_ROWS], POLICY["temperature"], POLICY["top_k"], POLICY["top_p"], POLICY["min_p"])
    orc.spec_accept(si.target[:1], si.draft[:1], si.draft_tokens[:1], 1.0, 0, si.u_acc[:1], si.u_fin[:1])
    orc.spec_accept(si.target[:1], None, si.draft_tokens[:1], 1.0, 1)


def oracle_step_rows(orc, x, si, u, pool):
    """The whole step on the oracle, row-parallel: each of the 49 rows (argmax,
    top-k, sampling) and each spec sequence (both rules) is one task on the
    thread pool. The oracle's C calls release the GIL and keep no state."""
    def row_task(r):
        xr = x[r:r + 1]
        orc.argmax(xr)
        orc.topk(xr, K_TOPK)
        orc.sample(xr, u[r:r + 1], POLICY["temperature"], POLICY["top_k"], POLICY["top_p"], POLICY["min_p"])

    def seq_task(q):
        sl = slice(q, q + 1)
        orc.spec_accept(si.target[sl], si.draft[sl], si.draft_tokens[sl], 1.0, 0, si.u_acc[sl], si.u_fin[sl])
        orc.spec_accept(si.target[sl], None, si.draft_tokens[sl], 1.0, 1)

    futs = [pool.submit(row_task, r) for r in range(ROWS)] + [pool.submit(seq_task, q) for q in range(SPEC_S)]
    for f in futs:
        f.result()


def cpu_baseline(steps=20, par_steps=3):
    """The oracle as it stands on the host: single-threaded on a bounded
    sample of the step, and row-parallel over all host cores on whole steps.
    The reported value is the row-parallel one (cores = its threads)."""
    import concurrent.futures as cf
    import oracle
    orc = oracle.default()
    x, si, u = build_inputs()
    oracle_step(orc, x, si, u)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_step(orc, x, si, u)
    single = REF_ROWS / ((time.perf_counter() - t0) / steps)
    cores = os.cpu_count() or 1
    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        oracle_step_rows(orc, x, si, u, pool)
        t0 = time.perf_counter()
        for _ in range(par_steps):
            oracle_step_rows(orc, x, si, u, pool)
        par = ROWS / ((time.perf_counter() - t0) / par_steps)
    return {"value": round(par, 3), "unit": "rows/s", "cores": cores, "kind": "oracle",
            "sample": f"{par_steps} whole steps ({ROWS} rows: argmax, top-k, sampling; {SPEC_S} spec "
                      f"sequences in both rules), one row or sequence per task on {cores} threads",
            "single_thread": {"value": round(single, 3), "cores": 1,
                              "sample": f"{REF_ROWS} of the {ROWS} rows per step and one spec sequence, "
                                        f"{steps} steps"}}


def workload_config():
    """The workload both arms run (the GPU arm adds how its inputs are laid out)."""
    return {"workload": WORKLOAD, "rows": ROWS, "V": V, "topk_k": K_TOPK, "sample": POLICY,
            "spec": {"sequences": SPEC_S, "drafts": SPEC_K, "T": 1.0, "rules": ["rejection", "argmax"]}}


def reference_arm(args, rank, world):
    if rank != 0:
        return None
    import oracle
    orc = oracle.default()
    x, si, u = build_inputs()
    for _ in range(args.warmup):
        oracle_step(orc, x, si, u)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(orc, x, si, u)
    dt = time.perf_counter() - t0
    v = REF_ROWS * args.steps / dt
    return {"impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded Gumbel-perturbed Zipf(1.1) logits; no dataset)",
            "config": workload_config(),
            "cpu_baseline": {"value": round(v, 3), "unit": "rows/s", "cores": 1, "kind": "oracle",
                             "sample": f"{REF_ROWS} of {ROWS} rows and one spec sequence per step"},
            "e2e": {"value": round(v, 3), "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="run this many untimed eager steps (for ncu) and exit")
    ap.add_argument("--traffic-from", default=None,
                    help="write profiles/traffic.json from an ncu CSV of dram bytes and exit")
    args = ap.parse_args()
    if args.traffic_from:
        print(json.dumps(write_traffic(args.traffic_from)))
        return
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))

    if args.impl == "reference":
        line = reference_arm(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = gpu_arm(args, rank, world, local_rank)
    if line is None:  # --profile-steps
        print("profile steps done", flush=True)
        return
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline() if world == 1 else None
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

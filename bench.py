"""Decode-step benchmark of the verify -> select -> sparse-draft hot path.

One step = 1 verification attention (k+1 rows, Collect-2 capture) + 1 KV
selection + k sparse draft attentions, on one seeded synthetic GQA layer.
The headline workload is the batch-8 Llama-3-8B-shaped layer with contexts
drawn in [16K, 64K]; the 32K and 128K single-sequence layers are measured in
the same run and reported under "workloads".

Cold L2 for every step kernel, as in a real model where other layers evict
it: before the verify call a buffer larger than L2 is written and another is
read, and before each draft call one is read (reading last leaves L2 holding
clean, unrelated lines, so a timed kernel does not pay for write-backs of the
flush's own dirty data).

Two device timings (CUDA events on the launching stream):
  value       the step as it runs in a stream: the whole cold step (flushes
              and step kernels) is captured once as a CUDA graph and
              replayed K times, and the same graph with the step kernels left
              out (flushes only) is replayed K times; value = mean time per
              replay of the first minus that of the second.  Stage figures
              ("stages_graph_us") are the full graph minus the graph without
              that stage.
  stages_us   every call of K eagerly launched cold steps bracketed by its
              own event pair; their sum is "events_us_per_step".  An event
              pair around a call adds its own ~2 us, so this is an upper
              bound; the verify segment is the roofline's kernel time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-cpu-baseline] [--no-extra]

Under torchrun each rank runs an independent replica on its own GPU (the path
shards by sequence with no exchange); the max over ranks is reported.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "llama8b_b8_16k_64k"
EXTRA_WORKLOADS = ("llama8b_32k", "qwen14b_128k")
METRIC = "us_per_decode_step"
METRIC_DESC = "µs per decode step (verify+select+sparse draft) and HBM GB/s vs peak"


def algorithmic_bytes(spec, capture_mode=1):
    """Bytes the method must move per step (bf16 = 2 B): every K and V row read
    once in verify, the capture written once and read once by select, the
    selected rows plus tail gathered by every draft step, and Q/O/indices."""
    B, R, Hq, Hkv, d, k = (spec.batch, spec.n_rows, spec.num_q_heads, spec.num_kv_heads,
                           spec.head_dim, spec.n_drafts)
    kv_row = Hkv * d * 2 * 2
    verify_kv = sum((L + R) * kv_row for L in spec.prefix_lens)
    qo = 2 * B * R * Hq * d * 2
    if capture_mode == 1:
        cap = sum(B_L * Hkv * 4 for B_L in spec.prefix_lens)
    else:
        cap = sum(L * Hq * 2 * 4 for L in spec.prefix_lens)
    n_sel = [min(L, spec.n_sel_max) for L in spec.prefix_lens]
    idx = sum(n_sel) * 4
    draft = sum(sum((n + t) * kv_row for n in n_sel) for t in range(1, k + 1))
    draft_qo = k * 2 * B * Hq * d * 2
    verify = verify_kv + qo + cap
    select = cap + idx
    drafts = draft + draft_qo + k * idx
    return {"verify": verify, "select": select, "drafts": drafts,
            "step": verify + select + drafts, "verify_kv": verify_kv}


def rank_env():
    """(rank, world size, local rank) from the torchrun environment."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def reduce_max(values, world, device=None):
    """Each value's maximum over the ranks (the slowest rank sets the job's
    time); a no-op for one rank.  Every rank gets the result."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def speedup_projection(alpha, k, t_draft, t_verify, t_select, t_dense):
    """Projected speedup of self-speculative decoding over dense decoding,
    attention only, from measured per-call times (µs).

    A Sparse Glimpse of the Whole, "What carries the argument": speedup
    S = (alpha k + 1) / (k gamma + 1), gamma = cost of a draft step relative
    to a verification.  Here gamma = t_draft / (t_verify + t_select).  With
    the accepted prefix rule (a draft counts only if every earlier one was
    accepted) the tokens per iteration are E[a + 1] = (1 - alpha^(k+1)) /
    (1 - alpha) instead of alpha k + 1; that variant is also given, with the
    iteration cost measured against one dense one-row decode step t_dense."""
    gamma = t_draft / (t_verify + t_select)
    s_pages = (alpha * k + 1) / (k * gamma + 1)
    tokens = (1 - alpha ** (k + 1)) / (1 - alpha) if alpha != 1 else k + 1
    iteration = k * t_draft + t_verify + t_select
    return {"alpha": alpha, "k": k, "gamma": gamma, "S_formula": s_pages,
            "tokens_per_iteration_prefix_rule": tokens,
            "S_measured_prefix_rule": tokens * t_dense / iteration,
            "t_dense_decode_us": t_dense}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def verify_traffic(workload):
    """Per-launch DRAM bytes of the verify kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    src = os.path.join(ROOT, "self_speculative_sparse_vg_gb300", "csrc", "verify.cu")
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    path = os.path.join(ROOT, "profiles", f"verify_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ": " in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(": ", 1)
            fields[k.strip()] = v.strip()
    if fields.get("verify.cu sha256[:16]") != digest:
        return None
    try:
        return int(fields["dram bytes per launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the GPU works."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", str(gpu_index)], stdout=self.file,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.file.name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons),
                "window": "every GPU phase of the run: warm-up, timed steps, studies, "
                          "the other workloads"}


# ----------------------------------------------------------------- oracle arm
# The float64 oracle, as it stands, on one decode step of a workload: per
# (sequence, KV head) unit, the verify of the unit's query heads over its
# prefix, its selection and the k draft steps.  Run in a fresh process
# without CUDA; with several cores the units are spread over a fork pool (one
# BLAS thread per worker).  A step times all units, or a sample of them when
# a full step does not fit the budget, scaled to the full step by the units'
# prefix lengths (the oracle's cost grows with the length).
_ORACLE_CODE = """
import sys, os, time, json
sys.path.insert(0, {root!r})
import multiprocessing as mp
import numpy as np
from oracle import vg_oracle as O
from self_speculative_sparse_vg_gb300.workloads import WORKLOADS, make_inputs
s = WORKLOADS[{workload!r}]
inp = make_inputs(s)
B, Hkv, g = s.batch, s.num_kv_heads, s.group
q = inp.q_verify.double().numpy()
k = [x.double().numpy() for x in inp.k_dense]
v = [x.double().numpy() for x in inp.v_dense]
dq = inp.draft_q.double().numpy()
del inp
units = [(b, h) for b in range(B) for h in range(Hkv)]
weight = [s.prefix_lens[b] + s.n_rows for b, h in units]


def unit(i):
    b, h = units[i]
    qs = q[b:b + 1, :, h * g:(h + 1) * g]
    ks, vs = [k[b][h:h + 1]], [v[b][h:h + 1]]
    lens = [s.prefix_lens[b]]
    out, rows = O.verify_attention(qs, ks, vs, lens, s.softmax_scale)
    sel = O.select_kv(O.group_sum(rows, 1), O.CAPTURE_GROUP_SUM, lens, g, 1, s.top_k,
                      s.n_sink, s.n_recent, False)
    for t in range(1, s.n_drafts + 1):
        O.sparse_draft_attention(dq[t - 1][b:b + 1, h * g:(h + 1) * g], ks, vs, sel, False,
                                 lens, [lens[0] + t], s.softmax_scale)
    return i


cores = {cores} or len(os.sched_getaffinity(0))
n_steps, budget = {n_steps}, {budget}
t0 = time.perf_counter()
unit(0)                                                   # calibration (not reported)
t_w = (time.perf_counter() - t0) / weight[0]
full = t_w * sum(weight) / cores                          # estimated wall time of a step
per_step = len(units)
if full * n_steps > budget:                               # a sample of the units per step
    per_step = max(1, int(len(units) * budget / (n_steps * full)))
    per_step = max(min(cores, len(units)), per_step // cores * cores)
pool = mp.get_context("fork").Pool(cores) if cores > 1 else None
times, nxt = [], 0
for _ in range(n_steps):
    sel = [(nxt + j) % len(units) for j in range(per_step)]
    nxt += per_step
    t0 = time.perf_counter()
    if pool is None:
        for i in sel:
            unit(i)
    else:
        pool.map(unit, sel, chunksize=1)
    wall = time.perf_counter() - t0
    times.append(wall * sum(weight) / sum(weight[i] for i in sel) * 1e6)
if pool is not None:
    pool.close()
print(json.dumps({{"step_us": times, "units_per_step": per_step, "units": len(units),
                  "cores": cores}}))
"""


def host_info():
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return {"cpu_model": model, "nproc": len(os.sched_getaffinity(0)),
            "machine": os.uname().machine}


def time_oracle(workload, n_steps, cores, budget_s):
    """Run the oracle timing in a fresh process; cores 0 = all of them."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = _ORACLE_CODE.format(root=ROOT, workload=workload, n_steps=n_steps, cores=cores,
                               budget=budget_s)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=3600)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def _sample_text(res, workload, spec, n_steps):
    part = ("every (sequence, KV head) unit" if res["units_per_step"] == res["units"] else
            f"{res['units_per_step']} of the {res['units']} (sequence, KV head) units, scaled "
            f"to the full step by prefix length")
    return (f"{n_steps} step(s) of {workload}, each {part}: verify of the unit's query heads "
            f"over its prefix, its selection, {spec.n_drafts} draft steps; float64 numpy, "
            f"{res['cores']} worker process(es) of one thread")


def cpu_baseline(workload):
    """The float64 oracle (as it stands) on one decode step of the workload:
    on all of the host's cores (the reported figure) and on one thread."""
    from self_speculative_sparse_vg_gb300.workloads import WORKLOADS
    spec = WORKLOADS[workload]
    par = time_oracle(workload, 1, 0, 30.0)
    one = time_oracle(workload, 1, 1, 30.0)
    return {"value": par["step_us"][0], "unit": "us", "cores": par["cores"], "kind": "oracle",
            "sample": _sample_text(par, workload, spec, 1),
            "single_thread": {"value": one["step_us"][0], "unit": "us", "cores": 1,
                              "sample": _sample_text(one, workload, spec, 1)},
            "host": host_info()}


REFERENCE_BUDGET_S = 150.0  # wall time of the timed oracle steps of the reference arm


def run_reference(args, rank, world):
    """The float64 oracle as it stands, timed on the host's cores (a fork pool
    over the (sequence, KV head) units), on the workload of `--workload`.
    Each of the warm-up + timed steps is a full decode step, or a bounded
    sample of its units scaled to the full step when the run would not end
    within REFERENCE_BUDGET_S.  Under torchrun rank 0 alone runs."""
    if rank != 0:
        return
    from self_speculative_sparse_vg_gb300.workloads import WORKLOADS
    spec = WORKLOADS[args.workload]
    n = args.warmup + args.steps
    res = time_oracle(args.workload, n, 0, REFERENCE_BUDGET_S)
    val = statistics.mean(res["step_us"][args.warmup:])
    cb = {"value": val, "unit": "us", "cores": res["cores"], "kind": "oracle",
          "sample": _sample_text(res, args.workload, spec, n), "host": host_info()}
    print(json.dumps({"impl": "reference", "metric": METRIC, "value": val, "unit": "us",
                      "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                      "ms_per_step": val / 1e3, "higher_is_better": False, "scaling": "weak",
                      "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                      "config": _config(spec, args.gpus), "cpu_baseline": cb,
                      "e2e": {"value": val, "unit": "us", "h2d_bytes_per_step": 0,
                              "d2h_bytes_per_step": 0}}))


def run_stack(args, rank, world, local):
    """The 32-layer decode loop: µs of attention kernels per draft/verify
    iteration (k drafts x 32 layers, verify + select x 32 layers), summed from
    CUDA events around every call.  Each layer's K/V (1.3 GB) is far larger
    than L2, so every call starts cold without a flush."""
    import dataclasses
    import torch
    from self_speculative_sparse_vg_gb300.stack import DecodeStack
    from self_speculative_sparse_vg_gb300.workloads import STACKS
    spec = dataclasses.replace(STACKS[args.workload], iterations=args.warmup + args.steps)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    st = DecodeStack(spec, dev)
    sampler = ClockSampler(local) if rank == 0 else None
    st.seed_selection()
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()
    iters, nbytes = [], []
    kv_row = spec.num_kv_heads * spec.head_dim * 2 * 2
    R, k = spec.n_drafts + 1, spec.n_drafts
    for _ in range(args.steps):
        lens = st.lens.cpu().tolist()
        st.timing = []
        st.step()
        torch.cuda.synchronize()
        tot = {"verify": 0.0, "select": 0.0, "draft": 0.0}
        for kind, a, b in st.timing:
            tot[kind] += a.elapsed_time(b) * 1e3
        iters.append(tot)
        n_sel = [min(L, spec.n_sel_max) for L in lens]
        per_layer = (sum((L + R) * kv_row + L * spec.num_kv_heads * 4 * 2 for L in lens) +
                     sum(sum((n + t) * kv_row for n in n_sel) for t in range(1, k + 1)))
        nbytes.append(per_layer * spec.layers)
    st.timing = None
    clocks = sampler.stop() if sampler else None
    assert int(st.flag.item()) == 0, "device error flag set"
    step_us = [sum(t.values()) for t in iters]
    value = statistics.mean(step_us)
    (value,) = reduce_max([value], world, dev)
    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    gbs = statistics.mean(nbytes) / (value * 1e-6) / 1e9
    print(json.dumps({
        "metric": "us_per_decode_iteration_attention", "mode": "stack", "value": value,
        "unit": "us", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": value / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; see workloads.py)",
        "config": {"workload": spec.name, "layers": spec.layers, "batch": spec.batch,
                   "prefix_lens_at_start": list(spec.prefix_lens), "n_drafts": k,
                   "top_k": spec.top_k, "n_sink": spec.n_sink, "n_recent": spec.n_recent,
                   "l2": "no flush: each layer's K/V (1.3 GB) exceeds L2"},
        "stages_us": {key: statistics.mean(t[key] for t in iters) for key in iters[0]},
        "algorithmic_bytes_per_iteration": statistics.mean(nbytes),
        "hbm_gbs": gbs, "hbm_frac": gbs / peak, "peak_kind": peak_kind,
        "gpu_launches": args.steps * spec.layers * st.launches_per_iteration(),
        "clocks": clocks}))


def _config(spec, n):
    return {"workload": spec.name, "batch": spec.batch, "num_q_heads": spec.num_q_heads,
            "num_kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim,
            "prefix_lens": list(spec.prefix_lens) if spec.batch <= 8 else "many",
            "n_drafts": spec.n_drafts, "top_k": spec.top_k, "n_sink": spec.n_sink,
            "n_recent": spec.n_recent, "selection": "per_head" if spec.per_head else "head_avg",
            "capture": "group_sum", "kv": "paged bf16, page 16",
            "l2": "flushed before verify (write then read 1.5x L2) and before every draft "
                  "step (read 1.5x L2); inputs of each timed kernel start cold",
            "replicas": n}


# ------------------------------------------------------------------ GPU arm
class Flusher:
    """Buffers larger than L2: a write then a read before a step, a read
    before each draft step."""

    def __init__(self, dev):
        import torch
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.w = torch.empty(int(1.5 * l2), dtype=torch.uint8, device=dev)
        self.r = torch.ones(int(1.5 * l2) // 4, dtype=torch.float32, device=dev)
        self.out = torch.empty((), dtype=torch.float32, device=dev)

    def read(self):
        import torch
        torch.sum(self.r, dim=0, out=self.out)

    def full(self, i=1):
        self.w.fill_(i & 0xFF)
        self.read()


def _events(n):
    import torch
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def cold_graphs(st, fl, dev):
    """CUDA graphs of one cold step and of its variants: "full" (flushes and
    every step kernel), "flush" (flushes only), and "no_verify",
    "no_select", "no_drafts" (one stage left out; the kernels left in read
    what the previous replays wrote, which is the same data)."""
    import torch
    k = st.spec.n_drafts
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    graphs = {}

    def body(skip):
        fl.full(1)
        if skip not in ("verify", "all"):
            st.verify(side)
        if skip not in ("select", "all"):
            st.select(side)
        for t in range(1, k + 1):
            fl.read()
            if skip not in ("drafts", "all"):
                st.draft(t, side)

    with torch.cuda.stream(side):
        body(None)  # bind the side stream's call arguments outside capture
        torch.cuda.synchronize()
        for name, skip in (("full", None), ("flush", "all"), ("no_verify", "verify"),
                           ("no_select", "select"), ("no_drafts", "drafts")):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                body(skip)
            graphs[name] = g
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    return graphs


def time_graph(g, reps, barrier):
    """Mean µs per replay of `reps` replays (3 untimed first), an event pair
    around each replay on the current stream."""
    import torch
    stream = torch.cuda.current_stream()
    for _ in range(3):
        g.replay()
    barrier()
    marks = []
    for _ in range(reps):
        a, b = _events(2)
        a.record(stream)
        g.replay()
        b.record(stream)
        marks.append((a, b))
    barrier()
    return statistics.mean(a.elapsed_time(b) * 1e3 for a, b in marks)


def measure(spec, inp, st, fl, steps, warmup, barrier, dev):
    """Cold-step timings of one workload: the graph figure and the
    per-call event figures."""
    import torch
    k = spec.n_drafts
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        fl.full(i)
        st.run()
    barrier()
    graphs = cold_graphs(st, fl, dev)
    T = {}
    for name in ("full", "flush", "no_verify", "no_select", "no_drafts"):
        T[name] = time_graph(graphs[name], steps, barrier)
    del graphs
    # every call with its own event pair
    marks = []
    for i in range(steps):
        fl.full(i)
        e = _events(3 + 2 * k)
        e[0].record(stream)
        st.verify()
        e[1].record(stream)
        st.select()
        e[2].record(stream)
        for t in range(1, k + 1):
            fl.read()
            e[1 + 2 * t].record(stream)
            st.draft(t)
            e[2 + 2 * t].record(stream)
        marks.append(e)
    barrier()
    assert int(st.error_flag.item()) == 0, "device error flag set"
    ver = statistics.mean(m[0].elapsed_time(m[1]) * 1e3 for m in marks)
    sel = statistics.mean(m[1].elapsed_time(m[2]) * 1e3 for m in marks)
    dra = statistics.mean(sum(m[1 + 2 * t].elapsed_time(m[2 + 2 * t]) * 1e3
                              for t in range(1, k + 1)) for m in marks)
    return {"graph_full_us": T["full"], "graph_flush_us": T["flush"],
            "value": T["full"] - T["flush"],
            "stages_graph_us": {"verify": T["full"] - T["no_verify"],
                                "select": T["full"] - T["no_select"],
                                "drafts_total": T["full"] - T["no_drafts"],
                                "draft_each": (T["full"] - T["no_drafts"]) / max(k, 1)},
            "stages_us": {"verify": ver, "select": sel, "drafts_total": dra,
                          "draft_each": dra / max(k, 1)},
            "events_us_per_step": ver + sel + dra}


def summarize(spec, m, peak, peak_kind, launches):
    nb = algorithmic_bytes(spec)
    v = m["value"]
    achieved = nb["verify"] / (m["stages_us"]["verify"] * 1e-6) / 1e9
    return {
        "value": v,
        "hbm_gbs_step": nb["step"] / (v * 1e-6) / 1e9,
        "hbm_frac_step": nb["step"] / (v * 1e-6) / 1e9 / peak,
        "gap_to_0.70_us": v - nb["step"] / (0.70 * peak * 1e9) * 1e6,
        "graph_full_us": m["graph_full_us"], "graph_flush_us": m["graph_flush_us"],
        "stages_graph_us": m["stages_graph_us"],
        "stages_us": m["stages_us"],
        "events_us_per_step": m["events_us_per_step"],
        "hbm_frac_step_events": nb["step"] / (m["events_us_per_step"] * 1e-6) / 1e9 / peak,
        "stages_bytes": nb,
        "launches_per_step": launches,
        "roofline": {"kernel": "verify_kernel (+ split merge)", "bound": "hbm",
                     "achieved": achieved, "peak": peak,
                     "peak_kind": f"{peak_kind} hbm_gbs (copy, burst)", "unit": "GB/s",
                     "frac": achieved / peak, "traffic": verify_traffic(spec.name),
                     "time": "mean event time of the verify call (cold L2) over the timed steps"},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    args = ap.parse_args()
    assert args.warmup >= 3

    rank, world, local = rank_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import torch.distributed as dist
    from self_speculative_sparse_vg_gb300 import vg
    from self_speculative_sparse_vg_gb300.step import DecodeStep
    from self_speculative_sparse_vg_gb300.workloads import STACKS, WORKLOADS, make_inputs

    if args.workload in STACKS:
        if world > 1:
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        run_stack(args, rank, world, local)
        if world > 1:
            dist.destroy_process_group()
        return

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    spec = WORKLOADS[args.workload]
    names = [n for n in EXTRA_WORKLOADS if n != args.workload] if not args.no_extra else []
    # inputs are drawn on the CPU before the GPU phase starts
    inputs = {n: make_inputs(WORKLOADS[n]) for n in [args.workload] + names}
    steps_of = {n: st for n, st in ((n, DecodeStep.create(inputs[n], dev)) for n in inputs)}
    fl = Flusher(dev)
    k = spec.n_drafts
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(local) if rank == 0 else None
    st = steps_of[args.workload]

    # ---------------- the headline workload: K cold steps
    m = measure(spec, inputs[args.workload], st, fl, args.steps, args.warmup, barrier, dev)

    # ---------------- hot: the step back to back, no flushes, replayed as a
    # CUDA graph so that host launch cost is not in the number
    graph = torch.cuda.CUDAGraph()
    cap_stream = torch.cuda.Stream(dev)
    cap_stream.wait_stream(stream)
    with torch.cuda.stream(cap_stream):
        st.run(cap_stream)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=cap_stream):
            st.run(cap_stream)
    stream.wait_stream(cap_stream)
    barrier()
    hot_us = time_graph(graph, min(args.steps, 200), barrier)
    del graph

    # ---------------- end to end through the C ABI with host buffers: every
    # step copies its inputs (verify and draft queries, one pinned buffer) to
    # the device and reads its results (attention outputs; indices and
    # counts) back.  Device-timed: event pairs around [H2D, verify, select],
    # each draft call and [D2H]; the L2 flushes between them are left out.
    in_h = torch.empty(st.io_in.shape, dtype=st.io_in.dtype).pin_memory()
    in_h.copy_(st.io_in.cpu())
    out_h = torch.empty(st.io_out.shape, dtype=st.io_out.dtype).pin_memory()
    sel_h = torch.empty(st.io_sel.shape, dtype=st.io_sel.dtype).pin_memory()
    h2d = in_h.numel() * in_h.element_size()
    d2h = out_h.numel() * out_h.element_size() + sel_h.numel() * sel_h.element_size()
    e2e_marks = []
    n_e2e = min(args.steps, 200)
    for i in range(n_e2e + args.warmup):
        fl.full(i)
        e = _events(4 + 2 * k)
        e[0].record(stream)
        st.io_in.copy_(in_h, non_blocking=True)
        st.verify()
        st.select()
        e[1].record(stream)
        for t in range(1, k + 1):
            fl.read()
            e[2 * t].record(stream)
            st.draft(t)
            e[2 * t + 1].record(stream)
        e[2 * k + 2].record(stream)
        out_h.copy_(st.io_out, non_blocking=True)
        sel_h.copy_(st.io_sel, non_blocking=True)
        e[2 * k + 3].record(stream)
        if i >= args.warmup:
            e2e_marks.append(e)
    barrier()
    e2e_us = statistics.mean(
        sum(m_[2 * j].elapsed_time(m_[2 * j + 1]) for j in range(k + 2)) * 1e3 for m_ in e2e_marks)
    ix_h = sel_h[:st.indices.numel()].view(st.indices.shape)
    assert torch.equal(ix_h, st.indices.cpu())

    # ---------------- capture rules (Figure 6 analogue) and dense decode
    # Verify alone under each capture mode, cold L2 each time; the Collect-2
    # vs Collect-All selections are compared on the same inputs.  A one-row
    # verify without capture is the dense decode step of the projection.
    def time_verify(rows, mode, capture, ws, reps=30):
        q = st.q_verify[:, :rows].contiguous()
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
        ts = []
        for i in range(reps + 3):
            fl.full(i)
            a, b_ = _events(2)
            a.record(stream)
            vg.verify_attention(st.kv, q, st.prefix_lens, spec.max_prefix, spec.softmax_scale,
                                out, mode, capture, 0, ws, st.error_flag)
            b_.record(stream)
            if i >= 3:
                ts.append((a, b_))
        torch.cuda.synchronize()
        return statistics.median(x.elapsed_time(y) * 1e3 for x, y in ts)

    B_, R_ = spec.batch, spec.n_rows
    cap_rows = torch.zeros(B_, spec.num_q_heads, 2, spec.max_prefix, device=dev)
    cap_all = torch.zeros_like(st.capture)
    ws1 = vg.zero_workspace(vg.verify_workspace_bytes(B_, 1, spec.num_q_heads, spec.num_kv_heads,
                                                      spec.head_dim, spec.max_prefix), dev)
    capture_study = {
        "verify_us_no_capture": time_verify(R_, vg.CAPTURE_NONE, None, st.ws_verify),
        "verify_us_collect2_group_sum": time_verify(R_, vg.CAPTURE_GROUP_SUM, st.capture,
                                                    st.ws_verify),
        "verify_us_collect2_rows": time_verify(R_, vg.CAPTURE_ROWS, cap_rows, st.ws_verify),
        "verify_us_collect_all": time_verify(R_, vg.CAPTURE_ALL_SUM, cap_all, st.ws_verify),
    }
    t_dense = time_verify(1, vg.CAPTURE_NONE, None, ws1)
    idx2, cnt2 = st.indices.clone(), st.counts.clone()
    vg.select_kv(st.capture, vg.CAPTURE_GROUP_SUM, st.prefix_lens, spec.num_q_heads,
                 spec.num_kv_heads, spec.max_prefix, spec.top_k, spec.n_sink, spec.n_recent,
                 st.per_head, idx2, cnt2, st.error_flag, workspace=st.ws_select)
    idxa, cnta = st.indices.clone(), st.counts.clone()
    vg.select_kv(cap_all, vg.CAPTURE_ALL_SUM, st.prefix_lens, spec.num_q_heads,
                 spec.num_kv_heads, spec.max_prefix, spec.top_k, spec.n_sink, spec.n_recent,
                 st.per_head, idxa, cnta, st.error_flag, workspace=st.ws_select)
    torch.cuda.synchronize()
    inter = tot = 0
    for b_ in range(B_):
        for r_ in range(idx2.shape[1]):
            s2 = set(idx2[b_, r_, :int(cnt2[b_, r_])].tolist())
            sa = set(idxa[b_, r_, :int(cnta[b_, r_])].tolist())
            inter += len(s2 & sa)
            tot += len(s2)
    capture_study["selection_overlap_collect2_vs_all"] = inter / max(tot, 1)
    del cap_rows, cap_all, ws1

    # ---------------- sparse verification (merged schedule): each row keeps
    # 7 % of the prefix blocks, rows sharing three quarters of them
    from self_speculative_sparse_vg_gb300.workloads import make_block_selection
    blocks, counts = make_block_selection(spec, 0.07, 11)
    bl_d, ct_d = blocks.to(dev), counts.to(dev)
    out_sv = torch.empty(st.q_verify.shape, dtype=torch.bfloat16, device=dev)
    ws_sv = vg.zero_workspace(vg.sparse_verify_workspace_bytes(
        B_, R_, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.max_prefix,
        blocks.shape[-1]), dev)
    sv_t = []
    for i in range(33):
        fl.full(i)
        a, b_ = _events(2)
        a.record(stream)
        vg.sparse_verify_attention(st.kv, st.q_verify, st.prefix_lens, spec.max_prefix,
                                   spec.softmax_scale, bl_d, ct_d, out_sv, workspace=ws_sv,
                                   error_flag=st.error_flag)
        b_.record(stream)
        if i >= 3:
            sv_t.append((a, b_))
    torch.cuda.synchronize()
    union = rows_sum = 0
    for b_i, L in enumerate(spec.prefix_lens):
        tail = set(range(L // 16, (L + R_ + 15) // 16))
        u = set(tail)
        for i in range(R_):
            row_blocks = set(blocks[b_i, i, :int(counts[b_i, i])].tolist())
            u |= row_blocks
            rows_sum += len(row_blocks | tail)
        union += len(u)
    page_bytes = spec.num_kv_heads * 16 * spec.head_dim * 2 * 2
    sparse_study = {
        "sparse_verify_us": statistics.median(x.elapsed_time(y) * 1e3 for x, y in sv_t),
        "dense_verify_us": capture_study["verify_us_no_capture"],
        "row_block_fraction": 0.07, "union_pages": union, "row_pages_summed": rows_sum,
        "pages_loaded_per_row_page": union / max(rows_sum, 1),
        "union_bytes": union * page_bytes}
    del ws_sv, out_sv
    assert int(st.error_flag.item()) == 0, "device error flag set"

    # ---------------- the other workloads: the same cold-step timings
    others = {}
    for n in names:
        s_o = WORKLOADS[n]
        mo = measure(s_o, inputs[n], steps_of[n], fl, min(args.steps, 50), 3, barrier, dev)
        others[n] = (s_o, mo)
    clocks = sampler.stop() if sampler else None

    flat = [m["value"], e2e_us, hot_us, m["stages_us"]["verify"]]
    for n in names:
        flat += [others[n][1]["value"], others[n][1]["stages_us"]["verify"]]
    red = reduce_max(flat, world, dev)
    m["value"], e2e_val, hot_val, m["stages_us"]["verify"] = red[:4]
    for i, n in enumerate(names):
        others[n][1]["value"], others[n][1]["stages_us"]["verify"] = red[4 + 2 * i:6 + 2 * i]
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peaks()
    head = summarize(spec, m, peak, peak_kind, st.launches_per_step())
    res = {
        "metric": METRIC, "metric_desc": METRIC_DESC, "value": head["value"], "unit": "us",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": head["value"] / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; see workloads.py)",
        "config": _config(spec, world),
        "timing": "value: cold step as a replayed CUDA graph (flushes + step kernels) minus "
                  "the same graph with flushes only, mean over the timed replays; stages_us: "
                  "event pair around every eagerly launched call",
    }
    res.update({key: val for key, val in head.items() if key != "value"})
    res.update({
        "hot_us_per_step": hot_val,
        "e2e": {"value": e2e_val, "unit": "us", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "timing": "device events around [H2D + verify + select], each draft call and "
                          "[D2H], issued through the C ABI from Python; L2 flushes between "
                          "them excluded; host-side completion not included"},
        "gpu_launches": args.steps * st.launches_per_step(),
        "capture_rules": capture_study,
        "sparse_verification": sparse_study,
        # per-call event times throughout (the dense decode step is timed
        # the same way)
        "projection": speedup_projection(0.7, k, head["stages_us"]["draft_each"],
                                         head["stages_us"]["verify"],
                                         head["stages_us"]["select"], t_dense),
        "workloads": {n: summarize(others[n][0], others[n][1], peak, peak_kind,
                                   steps_of[n].launches_per_step()) for n in names},
        "clocks": clocks,
    })
    if not args.no_cpu_baseline:
        try:
            res["cpu_baseline"] = cpu_baseline(spec.name)
        except Exception as exc:  # reported, never fatal
            res["cpu_baseline"] = {"error": str(exc)[-300:]}
    print(json.dumps(res))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

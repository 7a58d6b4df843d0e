"""Benchmark of the prefix-shared KV attention hot path on one GB300 (or N replicas).

One *step* is the whole hot path over one batch of the chosen synthetic workload:
kv_store of the step's new tokens, then the attention call(s) (extend and/or decode,
with the shared-prefix cascade), then the partial-state merge.  Inputs are resident in HBM
when the timed region starts; the L2 is flushed (512 MiB write) between timed steps, outside
the per-step CUDA events.  ``e2e`` repeats the measurement through the same C-ABI calls with
every step's inputs copied from pinned host memory and its output copied back inside the
timed region, the copies of neighbouring steps overlapping each step's kernels (three device
buffer sets, one copy stream each way).  ``unflushed`` repeats the device-resident steps back
to back with no flush between them; ``kv_store`` gives the store's GB/s on its bytes read and
written.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5] [--impl ours|reference]
                    [--page-size P] [--workload chunked_prefill|serving] [--no-graph] [--no-cascade]
                    [--no-cpu-baseline] [--no-more-configs] [--pool-slots S] [--chunked-gather]
                    [--kv-layout interleaved|separate]

The default run (few-shot extend, configuration 2) also measures the decode workloads and the
mixed fp8 step (configurations 3-5) after the headline and reports them under
``more_configs``; the oracle leg (``cpu_baseline``) is at the same time the parity check of
every output it covers (``parity``).

--impl reference times the oracle (plain float64 CPU code) on the host cores on bounded
samples of the same workload.  Under torchrun each rank runs an independent replica (the
path shards by request group with no exchange); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention tokens/s (extend+decode) and achieved HBM GB/s vs roofline, 1 GB300"
DEFAULT_CONFIG = 2


# ----------------------------------------------------------------------------------------
# helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms from start() to stop(); each
    sample carries the host time it arrived, so a summary covers any interval of the run."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []   # (host time, csv line)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.proc = None

    def summary(self, t0=None, t1=None):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, ln in list(self.lines):
            if (t0 is not None and t < t0) or (t1 is not None and t > t1):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}

    def clocks(self, timed, window):
        """The clock record of a measurement: the samples inside its timed region, and when
        those are fewer than three (a short region), the samples of the whole measurement
        window around it (warm-up, timed steps and the other timed variants: the same load)."""
        s = self.summary(*timed)
        if s["samples"] >= 3:
            return s
        w = self.summary(*window)
        w["timed_region_samples"] = s["samples"]
        w["window"] = "the measurement's warm-up, timed and end-to-end steps (the timed region alone is short)"
        return w


_SAMPLER = None


def sampler():
    """The run's clock sampler (started on first use, before any measurement)."""
    global _SAMPLER
    if _SAMPLER is None:
        import torch
        _SAMPLER = ClockSampler(torch.cuda.current_device() if torch.cuda.is_available() else 0).start()
        time.sleep(0.3)   # nvidia-smi's first samples arrive before the first measurement
    return _SAMPLER


def max_over_ranks(seconds, device):
    """Each rank's timings -> their elementwise maximum over all ranks (the slowest replica
    sets the job's time); with no process group, the rank's own timings."""
    import torch
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return [float(x) for x in seconds]
    t = torch.tensor([float(x) for x in seconds], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t]


def job_throughput(world, steps, units_per_step, seconds):
    """Whole-job rate: every replica processes ``units_per_step`` per step (weak scaling)."""
    return world * steps * units_per_step / seconds


def kernel_hash(kind):
    # the sources of every kernel the measured region runs (decode also runs the extend kernel),
    # and the planner, which decides what those kernels read
    srcs = {"extend": ("attn_extend.cu", "plan.cpp"), "decode": ("attn_decode.cu", "attn_extend.cu", "plan.cpp"),
            "store": ("kv_store.cu",)}
    h = hashlib.sha256()
    for f in srcs[kind] + ("common.cuh",):
        with open(os.path.join(ROOT, "prefix_shared_kv_token_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kind, workload):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current source."""
    path = os.path.join(ROOT, "profiles", f"{kind}_{workload}.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("source_hash") == kernel_hash(kind):
            return float(d["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def workload_facts(w):
    """Algorithmic work of one step: query tokens, unmasked-pair FLOPs, unique KV bytes."""
    hq, hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
    elem = 1 if w.dtype == "fp8_e4m3" else 2
    facts = {}
    for kind in ("extend", "decode"):
        reqs = [r for r in w.requests if r.kind == kind]
        if not reqs:
            continue
        pairs = 0
        segs = set()
        for r in reqs:
            L = w.context_len(r)
            if kind == "extend":
                p = L - r.n_new
                pairs += sum(p + i + 1 for i in range(r.n_new))
            else:
                pairs += L
            segs.update(r.path)
        unique_tokens = sum(len(w.segments[s].tokens) for s in segs)
        nq = sum(r.n_new if kind == "extend" else 1 for r in reqs)
        facts[kind] = {
            "queries": nq,
            "flops": 4.0 * d * hq * pairs,
            "kv_bytes": float(unique_tokens * hkv * d * elem * 2),
            "qo_bytes": float(nq * hq * d * 2 * 2),
            "new_tokens": sum(r.n_new for r in reqs),
        }
    return facts


def load_workload(args):
    """The configuration's workload; --pool-slots only shrinks the pool (same tokens/values
    up to the slot permutation), for profiler captures that must stay a few GB."""
    import workloads as W
    if args.workload == "chunked_prefill":
        # 16 prompts of 8,192 tokens prefilled in 1,024-token chunks (one call per chunk)
        return W.chunked_prefill(seed=6, **({"num_slots": args.pool_slots} if args.pool_slots else {}))
    if not args.pool_slots:
        return W.config(args.config)
    gen = {1: W.tiny_decode, 2: W.fewshot_extend, 3: W.batched_decode, 4: W.multiturn_decode, 5: W.tot_mixed}
    return gen[args.config](seed=args.config, num_slots=args.pool_slots)


# ----------------------------------------------------------------------------------------
# our arm


def run_serving(args):
    """Multi-step serving of a 256-request few-shot stream (8 groups x 32 requests sharing a
    1,800-token prefix, unique 50-150-token questions, 32-64 generated tokens, all waiting from
    step 0 in an interleaved group order) with at most 64 running on a 16,384-slot pool (the
    stream needs ~52k slots even with sharing), once admitting longest-cached-prefix first and
    once first-come-first-served.  A step is one
    serving step (admissions + prefill + one decode token per running request); the timed
    region is the whole run.  value = prompt + generated tokens served per second of device
    time (CUDA events around every kv_store + attention call)."""
    import torch
    import workloads as W
    from prefix_shared_kv_token_gb300.serving import ServingSim
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    warm = W.serving_stream(seed=70, n_groups=2, per_group=4, shared=300, unique=(10, 20), out=(2, 3))
    ServingSim(warm, capacity=4096).run()
    stream = W.serving_stream(seed=7, per_step=256)
    served = sum(len(r.prompt) + r.out_len for r in stream.requests)
    cap = args.pool_slots or 16384
    res = {}
    smp = sampler()
    ts0 = time.perf_counter()
    for policy in ("lpm", "fcfs"):
        sim = ServingSim(stream, capacity=cap, policy=policy, max_running=64, prefill_budget=16384,
                         page_size=args.page_size)
        t0 = time.perf_counter()
        sim.run()
        st = sim.summary()
        st["wall_s"] = round(time.perf_counter() - t0, 3)
        st["served_tokens_per_s_device"] = round(served / (st["device_ms"] / 1e3), 1)
        st["served_tokens_per_s_wall"] = round(served / st["wall_s"], 1)
        res[policy] = {k: (round(v, 4) if isinstance(v, float) else v) for k, v in st.items()}
    lpm = res["lpm"]
    return {
        "metric": METRIC, "value": lpm["served_tokens_per_s_device"], "unit": "tokens/s", "n_gpus": 1,
        "steps": lpm["steps"], "warmup": 1, "ms_per_step": round(lpm["device_ms"] / lpm["steps"], 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "serving_stream", "requests": len(stream.requests), "pool_slots": cap,
                   "page_size": args.page_size,
                   "max_running": 64, "prefill_budget": 16384, "heads_q_kv": "32/8", "head_dim": 128,
                   "l2": "not flushed (a serving run; steps follow each other)"},
        "e2e": {"value": lpm["served_tokens_per_s_wall"], "unit": "tokens/s (host + device wall clock)"},
        "serving": res,
        "lpm_over_fcfs": {"device_time": round(res["fcfs"]["device_ms"] / lpm["device_ms"], 3),
                          "hit_rate": [lpm["hit_rate"], res["fcfs"]["hit_rate"]]},
        "clocks": smp.summary(ts0, time.perf_counter()),
    }


def measure(w, args, dev, steps, world, e2e=True):
    """Build the workload's calls in a fresh pool and time ``steps`` steps of them (after
    ``args.warmup`` untimed steps): per-step CUDA events on the launching stream, the L2
    flushed between steps outside the events, clocks sampled meanwhile.  With ``e2e`` also the
    pipelined end-to-end steps, the serial end-to-end steps and the unflushed steps.  Returns
    (fields of the JSON line, the calls)."""
    import torch
    import prefix_shared_kv_token_gb300 as pkv
    from prefix_shared_kv_token_gb300.runtime import PrefixCache, run_e2e_pipelined

    facts = workload_facts(w)
    pc = PrefixCache(w, device=str(dev), page_size=args.page_size, kv_layout=args.kv_layout)
    if w.name == "chunked_prefill":
        # one extend call per chunk, over the chunks before it: stored with its chunk and read
        # from a context buffer (default), or stored separately and gathered from the pool
        calls = pc.prepare_chunked(fused=not getattr(args, "chunked_gather", False))
        plan_ms = None
    else:
        pc.populate()
        kinds = [k for k in ("extend", "decode") if any(r.kind == k for r in w.requests)]
        popts = {"span_sms": args.span_sms} if getattr(args, "span_sms", 0) else None
        calls = [pc.prepare(kind, cascade=not args.no_cascade, opts=popts if kind == "decode" else None)
                 for kind in kinds]
        # host planning of one step (tree match + lock, slots, tables, cascade, plan), which a
        # server repeats for every new batch; measured after the calls above are built
        plan_ms = (sum(pc.host_step_ms(k, reps=3, cascade=not args.no_cascade) for k in kinds)
                   if args.page_size == 1 else None)
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def step():
        for c in calls:
            c.store()
        for c in calls:
            c.attend()

    smp = sampler()
    win0 = time.perf_counter()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    # a decode call's launches (gathers, span pass, decode kernel, merge) are replayed from a
    # CUDA graph captured once, as a decode loop reusing its plan does; an extend call stays
    # a plain call (its kernel-only timing events are recorded inside the library)
    for c in calls:
        if c.kind == "decode" and not args.no_graph:
            c.capture_attend()
    torch.cuda.synchronize()
    for c in calls:
        if pkv.get_device_error(c.workspace) != 0:
            raise RuntimeError("device error word set during warm-up")

    # timed region: per-step events (store, attention per call) on the launching stream
    K = steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 + 2 * len(calls))] for _ in range(K)]
    # the extend call's tensor-core kernel alone (after its key gather, before its merge)
    kev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in calls]
           for _ in range(K)]
    for a, b in (pair for step_ in kev for pair in step_):
        a.record(stream)
        b.record(stream)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(K):
        flush.zero_()
        e = ev[k]
        e[0].record(stream)
        for c in calls:
            c.store()
        e[1].record(stream)
        for i, c in enumerate(calls):
            if c.kind == "extend":
                pkv.set_kernel_events(*kev[k][i])
            e[2 + 2 * i].record(stream)
            c.replay_attend() if c.graph is not None else c.attend()
            e[3 + 2 * i].record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    wall = t1 - t0
    if world > 1:
        torch.distributed.barrier()
    step_ms = [ev[k][0].elapsed_time(ev[k][-1]) for k in range(K)]
    store_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]
    attn_ms = {}
    for i, c in enumerate(calls):   # per kind: all of the step's calls of that kind
        t = [ev[k][2 + 2 * i].elapsed_time(ev[k][3 + 2 * i]) for k in range(K)]
        attn_ms[c.kind] = [x + y for x, y in zip(attn_ms[c.kind], t)] if c.kind in attn_ms else t
    # per step: the extend kernels of all the step's extend calls
    ext_kernel_ms = [sum(a.elapsed_time(b) for (a, b), c in zip(kev[k], calls) if c.kind == "extend")
                     for k in range(K)] if any(c.kind == "extend" for c in calls) else None
    for c in calls:
        if pkv.get_device_error(c.workspace) != 0:
            raise RuntimeError("device error word set during the timed steps")

    tokens_per_step = sum(c.num_queries for c in calls)
    t_total = max_over_ranks([sum(step_ms) / 1e3], dev)[0]
    value = job_throughput(world, K, tokens_per_step, t_total)

    # roofline of the dominant kernel
    pk = peaks()
    dominant = max(attn_ms, key=lambda k: float(np.mean(attn_ms[k])))
    fx = facts[dominant]
    if dominant == "extend":
        # algorithmic flops / the extend kernel's own duration (events on its launch stream)
        dur = float(np.mean(ext_kernel_ms)) / 1e3
        achieved = fx["flops"] / dur / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved / pk["bf16_tflops"], 4), "kernel": "extend_kernel",
                "algorithmic_per_launch": fx["flops"], "kernel_ms": round(dur * 1e3, 4)}
    else:
        # unique KV + Q/O bytes / the whole decode call (every kernel of it moves those bytes)
        dur = float(np.mean(attn_ms[dominant])) / 1e3
        achieved = (fx["kv_bytes"] + fx["qo_bytes"]) / dur / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / pk["hbm_gbs"], 4), "kernel": "attn_decode (all its kernels)",
                "algorithmic_per_launch": fx["kv_bytes"] + fx["qo_bytes"], "kernel_ms": round(dur * 1e3, 4),
                "frac_of_8tbs_nominal": round(achieved / 8000.0, 4)}
    # the committed ncu captures are of the token pool
    traffic = profiled_traffic(dominant, w.name) if args.page_size == 1 else None
    roof["traffic"] = traffic
    roof["peak_source"] = pk["source"] + " (burst)"

    launches_per_step = sum(c.launches() for c in calls)
    # kv_store: bf16 K and V rows read, pool rows written (bf16 or e4m3), slot indices read
    elem = 1 if w.dtype == "fp8_e4m3" else 2
    store_bytes = sum((c.k_new.numel() + c.v_new.numel()) * (2 + elem) + c.out_cache_loc.numel() * 4 for c in calls)
    # a fused or context-buffer call stores its new rows inside the attention call: the store
    # events then hold no kernel and give no store time of their own
    separate_store = [c for c in calls if c.ctx is None and not c.fused]
    inside = len(separate_store) < len(calls)
    sep_bytes = sum((c.k_new.numel() + c.v_new.numel()) * (2 + elem) + c.out_cache_loc.numel() * 4
                    for c in separate_store)
    out = {
        "value": round(value, 1), "ms_per_step": round(t_total * 1e3 / K, 4), "steps": K,
        "tokens_per_step": tokens_per_step, "roofline": roof, "gpu_launches": K * launches_per_step,
        "kernel_ms": {**({"kv_store": round(float(np.mean(store_ms)), 4)} if separate_store else {}),
                      **{f"attn_{k}": round(float(np.mean(v)), 4) for k, v in attn_ms.items()},
                      **({"attn_decode_median": round(float(np.median(attn_ms["decode"])), 4)}
                         if "decode" in attn_ms else {})},
        "kv_store": {"bytes_per_step": int(store_bytes),
                     "gbs": (round(sep_bytes / (float(np.mean(store_ms)) / 1e3) / 1e9, 1)
                             if separate_store and not inside else None),
                     **({"note": "the new rows are stored inside the attention call (fused store); its time is "
                                 "part of attn_extend"} if inside else {})},
        "wall_s": round(wall, 4), "clocks": smp.clocks((t0, t1), (win0, time.perf_counter())),
        "host_plan_ms_per_step": None if plan_ms is None else round(plan_ms, 3),
    }
    for kind, fx_ in facts.items():
        out[f"{kind}_queries"] = fx_["queries"]
    if not e2e:
        return out, calls
    win_mid = time.perf_counter()

    # end-to-end: same calls, inputs from pinned host memory, output back to the host.
    # Pipelined (step k+1's inputs copy in and step k-1's output copies out while step k
    # computes; three device buffer sets, so the two copies never wait on each other), with a
    # 256 MiB L2 flush before every step's kernels inside the timed span; and, for reference,
    # fully serialised steps.
    for c in calls:
        c.pin_host()
    sets = [c.e2e_sets(3) for c in calls]
    e2e_flush = flush[:(256 << 20) // 4]
    run_e2e_pipelined(sets, args.warmup, e2e_flush)
    if world > 1:
        torch.distributed.barrier()
    e2e_total_ms = run_e2e_pipelined(sets, K, e2e_flush)
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for k in range(K):
        flush.zero_()
        e2e_ev[k][0].record(stream)
        for c in calls:
            c.run_e2e()
        e2e_ev[k][1].record(stream)
    torch.cuda.synchronize()
    # the same device-resident steps back to back without the L2 flush (shared spans and
    # the previous step's tables may still be in L2): reported beside the flushed figure
    uev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for k in range(K):
        uev[k][0].record(stream)
        for c in calls:
            c.store()
        for c in calls:
            c.replay_attend() if c.graph is not None else c.attend()
        uev[k][1].record(stream)
    torch.cuda.synchronize()
    unflushed_ms = [a.elapsed_time(b) for a, b in uev]
    e2e_serial_ms = [a.elapsed_time(b) for a, b in e2e_ev]
    t_e2e = max_over_ranks([e2e_total_ms / 1e3], dev)[0]
    e2e_value = job_throughput(world, K, tokens_per_step, t_e2e)
    h2d = sum(c.h2d_bytes() for c in calls)
    d2h = sum(c.d2h_bytes() for c in calls)
    e2e_ms = t_e2e * 1e3 / K
    out["e2e"] = {
        "value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
        "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 4),
        "mode": "pipelined: step k+1's H2D and step k-1's D2H overlap step k's kernels (3 device "
                "buffer sets); a 256 MiB L2 flush precedes each step's kernels inside the span",
        "serial_ms_per_step": round(float(np.mean(e2e_serial_ms)), 4),
        # a new batch every step also costs its host planning; if it does not overlap the
        # previous step's device work, a step takes e2e + planning:
        "host_plan_ms_per_step": out["host_plan_ms_per_step"],
        "value_with_host_plan_serial": (None if plan_ms is None else
                                        round(job_throughput(world, 1, tokens_per_step,
                                                             (e2e_ms + plan_ms) / 1e3), 1)),
    }
    if out["clocks"].get("window"):   # the window grew by the end-to-end and unflushed steps
        out["clocks"] = smp.clocks((t0, t1), (win0, time.perf_counter()))
    out["unflushed"] = {"ms_per_step": round(float(np.mean(unflushed_ms)), 4),
                        "value": round(job_throughput(world, K, tokens_per_step, sum(unflushed_ms) / 1e3), 1),
                        "note": "same steps without the L2 flush between them"}
    return out, calls


def run_ours(args, rank, world):
    import torch
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = load_workload(args)
    m, calls = measure(w, args, dev, args.steps, world, e2e=True)
    cfg = {"workload": w.name, "config_id": None if args.workload else args.config, "requests": len(w.requests),
           "heads_q_kv": f"{w.num_q_heads}/{w.num_kv_heads}", "head_dim": w.head_dim, "pool_dtype": w.dtype,
           "pool_slots": w.num_slots, "page_size": args.page_size, "kv_layout": args.kv_layout,
           "cascade": not args.no_cascade,
           "decode_launch": "plain" if args.no_graph else "CUDA graph replay of the call's launches",
           "l2": "flushed between timed steps (512 MiB write outside the step events)",
           "tokens_per_step": m["tokens_per_step"]}
    if w.name == "chunked_prefill":
        cfg["chunks"] = "separate stores, gather per chunk" if args.chunked_gather else \
            "stored into and read from a context buffer"
    for kind in ("extend", "decode"):
        if f"{kind}_queries" in m:
            cfg[f"{kind}_queries"] = m[f"{kind}_queries"]
    out = {
        "metric": METRIC, "value": m["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": m["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "bf16 (fp8_e4m3 pool)",
        "data": "synthetic", "config": cfg, "e2e": m["e2e"], "roofline": m["roofline"],
        "gpu_launches": m["gpu_launches"], "kernel_ms": m["kernel_ms"], "kv_store": m["kv_store"],
        "unflushed": m["unflushed"], "wall_s": m["wall_s"], "clocks": m["clocks"],
    }
    return out, w, calls


def run_more_configs(args, world, ids=(3, 4, 5), steps=200):
    """The decode workloads (and the mixed fp8 step) measured in the same run as the headline,
    each in its own pool (freed before the next): per call the device time, tokens/s and the
    roofline -- unique K/V + q/o bytes over the decode call against the measured copy peak
    and against 8 TB/s -- with its clocks and, on rank 0, every output checked against the
    oracle.  ``steps`` timed steps each (a longer region than the headline's, so the clock
    sampler sees it)."""
    import torch
    import workloads as W
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    res = {}
    sub = argparse.Namespace(**vars(args))
    sub.workload, sub.pool_slots = "", 0
    for k in ids:
        sub.config = k
        w = W.config(k)
        m, calls = measure(w, sub, dev, steps, world, e2e=False)
        entry = {"workload": w.name, "steps": steps, "ms_per_step": m["ms_per_step"],
                 "tokens_per_step": m["tokens_per_step"], "value": m["value"], "unit": "tokens/s",
                 "kernel_ms": m["kernel_ms"], "roofline": m["roofline"], "clocks": m["clocks"],
                 "host_plan_ms_per_step": m["host_plan_ms_per_step"]}
        if "decode" in workload_facts(w):
            fx = workload_facts(w)["decode"]
            t = m["kernel_ms"]["attn_decode"] / 1e3
            byts = fx["kv_bytes"] + fx["qo_bytes"]
            entry["decode"] = {"ms_per_call": m["kernel_ms"]["attn_decode"],
                               "ms_per_call_median": m["kernel_ms"].get("attn_decode_median"),
                               "tokens_per_s": round(fx["queries"] / t, 1),
                               "unique_bytes": byts, "achieved_gbs": round(byts / t / 1e9, 1),
                               "frac_of_measured_peak": round(byts / t / 1e9 / peaks()["hbm_gbs"], 4),
                               "frac_of_8tbs_nominal": round(byts / t / 1e9 / 8000.0, 4),
                               "traffic": profiled_traffic("decode", w.name)}
        if int(os.environ.get("RANK", 0)) == 0:
            entry["parity"] = oracle_parity(w, calls, budget_s=60.0)["parity"]
        res[f"config_{k}"] = entry
        del calls, m
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------------------
# the oracle on the host cores


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
        return int(n)
    except Exception:
        return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def oracle_sample(w, budget_s, start=0):
    """Run the oracle over requests (round robin from `start`) until `budget_s` of CPU work;
    returns (query tokens, seconds, requests used)."""
    from oracle import step as ostep
    t0 = time.perf_counter()
    toks, used, i = 0, 0, start
    n = len(w.requests)
    while used < n:
        r = w.requests[i % n]
        ostep.request_output(w, r)
        toks += r.n_new if r.kind == "extend" else 1
        used += 1
        i += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return toks, time.perf_counter() - t0, used


PARITY_TOL = {"bf16": 1e-2, "fp8_e4m3": 5e-2}


def oracle_parity(w, calls, budget_s=60.0):
    """The oracle over the workload's requests in order, until `budget_s` of CPU work, each
    request's outputs compared element by element with the GPU's (the calls' last outputs).
    Returns {"parity": {...}, "cpu": (query tokens, seconds, requests)}: the max-abs error
    against the tolerance over every compared output, and the oracle's own timing."""
    from oracle import step as ostep
    rows = {}   # request id -> (call, first output row)
    for c in calls:
        got = c.o.float().cpu().numpy()
        r0 = 0
        for r in c.requests:
            n = r.n_new if c.kind == "extend" else 1
            rows[r.rid] = (got, r0, n)
            r0 += n
    t0 = time.perf_counter()
    err, compared, toks, used = 0.0, 0, 0, 0
    total = sum(n for _, _, n in rows.values())
    finite = True
    for r in w.requests:
        if r.rid not in rows:
            continue
        want, _ = ostep.request_output(w, r)
        got, r0, n = rows[r.rid]
        g = got[r0:r0 + n]
        finite &= bool(np.all(np.isfinite(g)))
        err = max(err, float(np.max(np.abs(g - want))))
        compared += n
        toks += n
        used += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    secs = time.perf_counter() - t0
    tol = PARITY_TOL[w.dtype]
    return {"parity": {"max_abs_err": round(err, 6), "tol": tol, "outputs_compared": compared,
                       "outputs_total": total, "elements_compared": compared * w.num_q_heads * w.head_dim,
                       "pass": bool(finite and err <= tol and compared == total)},
            "cpu": (toks, secs, used)}


def cpu_baseline(w, calls=None, budget_s=12.0):
    """The oracle timed on the host cores over a bounded sample of the workload; with the
    GPU calls, the same oracle run is also the parity check of every output it covers."""
    if calls is not None:
        res = oracle_parity(w, calls, budget_s=max(budget_s, 60.0))
        toks, secs, used = res["cpu"]
        parity = res["parity"]
    else:
        toks, secs, used = oracle_sample(w, budget_s)
        parity = None
    cb = {"value": round(toks / secs, 2), "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
          "sample": f"{used} of {len(w.requests)} requests ({toks} query tokens) of {w.name}, float64 numpy, "
                    f"{secs:.1f} s"}
    return cb, parity


def run_reference(args, rank, world):
    w = load_workload(args)
    per_step = 2.0
    for k in range(args.warmup):
        oracle_sample(w, 0.2, start=k)
    toks_total, secs_total, used_total = 0, 0.0, 0
    for k in range(args.steps):
        toks, secs, used = oracle_sample(w, per_step, start=k * 7)
        toks_total += toks
        secs_total += secs
        used_total += used
    value = toks_total / secs_total
    cb = {"value": round(value, 2), "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
          "sample": f"{args.steps} steps x ~{per_step:.0f} s, {used_total} requests ({toks_total} query tokens) "
                    f"of {w.name}, float64 numpy"}
    return {"metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(secs_total * 1e3 / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "config_id": None if args.workload else args.config,
                       "requests": len(w.requests)},
            "impl": "reference", "cpu_baseline": cb,
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------------------


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cascade", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--span-sms", type=int, default=0,
                    help="decode: SMs left to the tensor-core span pass, run beside the decode kernel (0: after it)")
    ap.add_argument("--kv-layout", default="interleaved", choices=["interleaved", "separate"],
                    help="pool layout: a slot's K and V rows adjacent (default) or two dense arrays")
    ap.add_argument("--chunked-gather", action="store_true",
                    help="chunked_prefill: separate stores and a gather of the whole context per chunk "
                         "(instead of chunks stored into and read from a context buffer)")
    ap.add_argument("--no-more-configs", action="store_true",
                    help="skip the decode and mixed workloads (configurations 3-5) measured after the headline")
    ap.add_argument("--pool-slots", type=int, default=0)
    ap.add_argument("--no-graph", action="store_true", help="launch decode calls directly instead of from a CUDA graph")
    ap.add_argument("--page-size", type=int, default=1,
                    help="1: token pool; P > 1: paged pool, whole P-token blocks shared, page-table batches")
    ap.add_argument("--workload", default="", choices=["", "chunked_prefill", "serving"],
                    help="chunked_prefill: long prompts prefilled chunk by chunk; serving: a multi-step "
                         "serving run, longest-prefix-first against first-come-first-served (instead of --config)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)))
        return

    if args.workload == "serving":
        if rank == 0:
            print(json.dumps(run_serving(args)))
        return

    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    out, w, calls = run_ours(args, rank, world)
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"], out["parity"] = cpu_baseline(w, calls)
    del calls
    if not args.no_more_configs and not args.workload and args.config == DEFAULT_CONFIG and args.page_size == 1:
        out["more_configs"] = run_more_configs(args, world)
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    try:
        main()
    finally:
        if _SAMPLER is not None:
            _SAMPLER.stop()

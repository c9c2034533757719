"""Benchmark: load-balanced paged-KV decode attention on GB300.

One step = one pass of the hot path over one decode batch: plan (task map) ->
persistent decode -> combine, on the mixed-length workload (batch 32, KV lengths
log-uniform 128-32768, 64 q / 8 KV heads, head_dim 128, page 64, bf16, 148
persistent CTAs).  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference] [--workload NAME]

value: achieved KV GB/s over the whole step (algorithmic KV bytes / step time),
summed over ranks; us_per_step is the same measurement as time.  The workloads'
KV (0.5-9.9 GB) is larger than L2 (126 MB), so steps run back to back without an
L2 flush; inputs smaller than 2 x L2 get a 2 x L2 write-flush before every step,
outside the timed events (config.l2 says which).  N > 1 runs independent replicas (one per GPU, no data-path collective).
--impl reference times the fp64 CPU oracle on the host cores instead.
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "decode attention µs/step and KV GB/s (% of GB300 HBM peak) on mixed-length batches"
NOMINAL_HBM_GBS = 7900.0
FALLBACK_HBM_GBS = 6800.0
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, tagged with host time."""

    def __init__(self, uuid: str | None):
        self.samples = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        window = "timed"
        if not inside:  # timed region shorter than the sampling period: nearest samples
            inside = [s for t, s in self.samples if t0 - 1.0 <= t <= t1 + 1.0]
            window = "timed+-1s"
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in inside:
            try:
                sm.append(float(s[1]))
                mx.append(float(s[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, s[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "window": window}


# The sources each profiled kernel is built from; a committed capture records their combined
# digest, and its counters are used only while the sources are unchanged.
KERNEL_SOURCES = {
    "decode": ("attention.cu", "engine.cuh", "ptx.cuh", "common.h"),
    "multi": ("attention_tc.cu", "engine.cuh", "ptx.cuh", "common.h"),
    "plan": ("plan.cu", "ptx.cuh", "common.h"),
    "combine": ("combine.cu", "ptx.cuh", "common.h"),
    "prologue": ("prologue.cu", "ptx.cuh", "common.h"),
}


def sources_digest(kind: str) -> str:
    """sha256 over the concatenated sources of one kernel family (csrc/, in the listed order)."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "load_balanced_paged_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profile_traffic(workload: str, nbytes: int):
    """DRAM traffic per decode launch from the committed ncu summary of this workload's
    decode kernel (profiles/decode_<workload>[_small].md), scaled by KV bytes when the
    capture was a smaller case of the same workload; None once the kernel's sources differ
    from the ones captured."""
    import re
    sha = sources_digest("decode")
    for suffix in ("", "_small"):
        path = os.path.join(ROOT, "profiles", f"decode_{workload}{suffix}.md")
        if not os.path.exists(path):
            continue
        text = open(path).read()
        m_sha = re.search(r"sources sha256 `([0-9a-f]{64})`", text)
        m_tr = re.search(r"traffic_bytes_per_launch: (\d+)", text)
        m_alg = re.search(r"algorithmic_bytes_per_launch: (\d+)", text)
        if not (m_sha and m_tr and m_alg) or m_sha.group(1) != sha:
            return None, f"{os.path.basename(path)}: stale or incomplete"
        tr, alg = int(m_tr.group(1)), int(m_alg.group(1))
        note = os.path.basename(path) + ("" if alg == nbytes else f", scaled by KV bytes {nbytes}/{alg}")
        return int(round(tr * nbytes / alg)), note
    return None, "no committed capture for this workload"


def flush_buffer(device):
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    return torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=device)


def kv_bytes(inp):
    return workloads.kv_bytes(inp["seq_lens"].cpu().numpy(), inp["num_kv_heads"], inp["kv_dtype"])


def replica_max(value: float, world: int, device) -> float:
    """Max over ranks (replicas are independent; the only cross-rank step is this timing
    reduction after the timed region)."""
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job KV GB/s: the bytes all replicas processed per step over the slowest rank's step."""
    return world * bytes_per_rank / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------------------- our arm

def stats_us(ms) -> dict:
    """Mean, median and 90th percentile of per-replay times (ms in, us out)."""
    a = np.asarray(ms, dtype=np.float64) * 1e3
    return {"mean": round(float(a.mean()), 2), "median": round(float(np.median(a)), 2),
            "p90": round(float(np.percentile(a, 90)), 2), "reps": int(a.size)}


class Timer:
    """Device timing of captured kernel sequences on one stream (CUDA events on that stream),
    with an optional 2 x L2 write-flush before every replay (outside the events)."""

    def __init__(self, stream, flush):
        self.stream = stream
        self.flush = flush

    def flush_l2(self, k):
        if self.flush is not None:
            self.flush.fill_(float(k))

    def graphs_of(self, fns):
        """One CUDA graph per function (each a captured kernel launch)."""
        gs = []
        for f in fns:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                f()
            gs.append(g)
        torch.cuda.synchronize()
        return gs

    def per_kernel(self, fns, steps, warmup):
        """Per-kernel device times: the kernels captured in ONE graph with event-record nodes
        between them (no launch gaps counted), replayed `steps` times.  Returns ms
        [steps, len(fns)]."""
        for _ in range(warmup):
            for f in fns:
                f()
        try:
            evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(fns) + 1)]
        except TypeError:  # torch without external events: one graph per kernel, events between
            return self._separate(fns, steps)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            evs[0].record()
            for i, f in enumerate(fns):
                f()
                evs[i + 1].record()
        torch.cuda.synchronize()
        per = []
        for k in range(steps):
            self.flush_l2(k)
            g.replay()
            self.stream.synchronize()
            per.append([evs[i].elapsed_time(evs[i + 1]) for i in range(len(fns))])
        return np.array(per)

    def _separate(self, fns, steps):
        gs = self.graphs_of(fns)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(fns) + 1)] for _ in range(steps)]
        for k in range(steps):
            self.flush_l2(k)
            ev[k][0].record(self.stream)
            for i, g in enumerate(gs):
                g.replay()
                ev[k][i + 1].record(self.stream)
        self.stream.synchronize()
        return np.array([[ev[k][i].elapsed_time(ev[k][i + 1]) for i in range(len(fns))] for k in range(steps)])

    def whole(self, fns, steps):
        """The kernels captured as ONE graph (a production decode step) timed as a unit, each
        replay between its own pair of events.  Returns ms [steps]."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for f in fns:
                f()
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for k in range(steps):
            self.flush_l2(k)
            ev[k][0].record(self.stream)
            g.replay()
            ev[k][1].record(self.stream)
        self.stream.synchronize()
        return np.array([ev[k][0].elapsed_time(ev[k][1]) for k in range(steps)])


def l2_policy(args, nbytes: int, device):
    """Inputs larger than L2 need no flush between steps (a write-flush would leave L2 dirty and
    bill the next step for ~L2-size of write-backs); small inputs are flushed."""
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    do_flush = args.l2 == "flush" or (args.l2 == "auto" and nbytes < 2 * l2)
    note = ("flushed (2 x L2 write) before every timed step" if do_flush else
            f"inputs larger than L2 ({nbytes / 1e6:.0f} MB of KV vs {l2 / 1e6:.0f} MB L2), no flush")
    return do_flush, note


def workload_config(w, B: int, C: int, m: int, nbytes: int, l2_note: str, world: int) -> dict:
    """The `config` object of a bench line (the reference arm prints the same one)."""
    return {"workload": w.description, "name": w.name, "batch": B, "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": 128, "page_size": 64, "persistent_ctas": C,
            "min_tiles_per_split": m, "kv_bytes_per_step": nbytes, "l2": l2_note,
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"}


class Step:
    """One decode step of a workload through the binding: plan -> decode -> combine."""

    def __init__(self, dsa, inp, w, C: int, m: int, device):
        self.dsa, self.inp, self.w, self.C, self.m = dsa, inp, w, C, m
        self.B, self.hq, self.hkv = int(inp["seq_lens"].shape[0]), w.num_q_heads, w.num_kv_heads
        self.G = self.hq // self.hkv
        self.tm = dsa.TaskMap(self.B, self.hkv, C, device)
        self.po, self.pl = dsa.partial_buffers(self.tm.max_descs, self.G, device)
        self.out = torch.empty(self.B, self.hq, 128, dtype=torch.bfloat16, device=device)
        self.out_lse = torch.empty(self.B, self.hq, dtype=torch.float32, device=device)
        self.kw = dict(q_scale=inp["q_scale"], k_scale=inp["k_scale"], v_scale=inp["v_scale"])
        self.counters = self.tm.unit_counters()

    def plan(self):
        self.dsa.plan(self.inp["seq_lens"], self.hkv, self.C, self.m, task_map=self.tm)

    def decode(self, cta_times=None):
        i = self.inp
        self.dsa.decode(i["q"], i["k_pages"], i["v_pages"], i["block_table"], i["seq_lens"], self.tm, i["sm_scale"],
                        partial_o=self.po, partial_lse=self.pl, cta_times=cta_times, **self.kw)

    def combine(self):
        self.dsa.combine(self.tm, self.po, self.pl, self.hq, out=self.out, out_lse=self.out_lse)

    def decode_fused(self):
        i = self.inp
        self.dsa.decode_fused(i["q"], i["k_pages"], i["v_pages"], i["block_table"], i["seq_lens"], self.tm,
                              i["sm_scale"], out=self.out, out_lse=self.out_lse, partial_o=self.po,
                              partial_lse=self.pl, unit_counters=self.counters, **self.kw)

    def check(self, what):
        torch.cuda.synchronize()
        status = self.dsa.get_status(self.tm)
        if status != 0:
            raise RuntimeError(f"device status {status} on {what}")


def bench_static(dsa, step: Step, timer: Timer, reps: int, device, t_dec_comb: float, t_step: float) -> dict:
    """Both static split-KV forms on the step's inputs (decode + its combine, one CUDA graph
    replayed like the dynamic step), with how evenly each static grid's CTAs finish (one
    untimed launch with per-CTA timestamps).  t_dec_comb / t_step: the dynamic decode + combine
    and plan + decode + combine graphs' median replay times (ms)."""
    inp, B, hq, hkv, G = step.inp, step.B, step.hq, step.hkv, step.G
    static = {}
    max_len = int(inp["seq_lens"].max().item())
    for label, mode, param in (("static_16_splits", 0, 16), ("static_4096_chunk", 1, 4096)):
        S = dsa.static_num_splits(mode, param, max_len)
        spo, spl = dsa.partial_buffers(B * hkv * S, G, device)
        sst = torch.zeros(1, dtype=torch.int32, device=device)

        def sdec(mode=mode, param=param, spo=spo, spl=spl, sst=sst, cta_times=None):
            dsa.static_splitkv(mode, param, max_len, inp["q"], inp["k_pages"], inp["v_pages"],
                               inp["block_table"], inp["seq_lens"], hkv, inp["sm_scale"], partial_o=spo,
                               partial_lse=spl, status=sst, cta_times=cta_times, **step.kw)

        def scomb(S=S, spo=spo, spl=spl):
            dsa.static_combine(S, spo, spl, B, hq, hkv, out=step.out, out_lse=step.out_lse)

        sp = timer.per_kernel([sdec, scomb], reps, 3)
        whole = timer.whole([sdec, scomb], reps)
        if dsa.read_status(sst) != 0:
            raise RuntimeError(f"{label}: device status set")
        s_ms = float(np.median(whole))
        static[label] = {"splits": S, "us_per_step": round(s_ms * 1e3, 2), "us": stats_us(whole),
                         "breakdown_us": {"decode": round(float(np.median(sp[:, 0])) * 1e3, 2),
                                          "combine": round(float(np.median(sp[:, 1])) * 1e3, 2)},
                         "speedup_of_dynamic": round(s_ms / t_dec_comb, 3),
                         "speedup_of_dynamic_with_plan": round(s_ms / t_step, 3)}
        st_times = torch.zeros(B * hkv * S, 2, dtype=torch.int64, device=device)
        sdec(cta_times=st_times)
        static[label]["balance"] = cta_balance(st_times)
        del spo, spl
    return static


def measure_workload(dsa, device, name: str, args, rank: int, world: int, reps: int, seed_offset: int = 0):
    """The step of one workload: whole-step replays (mean / median / p90), per-kernel times,
    both static forms, the persistent bins' balance and the clocks seen meanwhile."""
    w = workloads.WORKLOADS[name]
    inp = workloads.make_workload(name, device=device, seed=w.seed + seed_offset, max_requests=args.requests)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    C = w.num_ctas(sms)
    step = Step(dsa, inp, w, C, args.min_tiles, device)
    nbytes = kv_bytes(inp)
    do_flush, l2_note = l2_policy(args, nbytes, device)
    timer = Timer(torch.cuda.current_stream(device), flush_buffer(device) if do_flush else None)
    fns = [step.plan, step.decode, step.combine]
    timer.per_kernel(fns, 1, args.warmup)  # warm-up + correctness gate (status word must be clean)
    step.check(f"the {name} workload")
    clocks = ClockSampler(gpu_uuid(device))
    time.sleep(0.3)
    t0 = time.time()
    whole = timer.whole(fns, reps)
    whole_dc = timer.whole([step.decode, step.combine], reps)  # the map built above serves every replay
    per = timer.per_kernel(fns, reps, 0)
    t1 = time.time()
    clocks.stop()
    step.check(f"the {name} workload (timed)")
    t_plan, t_dec, t_comb = (float(x) for x in per.mean(axis=0))
    t_step = float(whole.mean())
    static = bench_static(dsa, step, timer, reps, device, float(np.median(whole_dc)), float(np.median(whole)))
    dyn_times = torch.zeros(C, 2, dtype=torch.int64, device=device)
    step.decode(cta_times=dyn_times)
    peak, _ = measured_peaks()
    dec_gbs = nbytes / (t_dec * 1e-3) / 1e9
    step_gbs = nbytes / (t_step * 1e-3) / 1e9
    rec = {"config": workload_config(w, step.B, C, args.min_tiles, nbytes, l2_note, world),
           "step": "plan -> decode -> combine, one CUDA graph", "step_us": stats_us(whole),
           "decode_combine_us": stats_us(whole_dc),
           "breakdown_us": {k: stats_us(per[:, i]) for i, k in enumerate(("plan", "decode", "combine"))},
           "decode_GB/s": round(dec_gbs, 1), "decode_frac_of_hbm_peak": round(dec_gbs / peak, 4),
           "decode_frac_of_hbm_peak_median": round(nbytes / (float(np.median(per[:, 1])) * 1e-3) / 1e9 / peak, 4),
           "step_GB/s": round(step_gbs, 1), "step_frac_of_hbm_peak": round(step_gbs / peak, 4),
           "static": static, "balance": cta_balance(dyn_times),
           "clocks": clocks.summary(t0, t1)}
    rec["decode_traffic_bytes"], rec["decode_traffic_source"] = profile_traffic(name, nbytes)
    if w.kv_dtype == "fp8":
        # multi-token verify steps over E4M3 K/V (q_len 2: mma.sync kernel; 6: tensor-memory kernel)
        rec["multi_token"] = bench_multi(dsa, device, inp, w, sms, args.min_tiles, timer, max(10, min(reps, 30)),
                                         nbytes, t_step)
    rec["gate"] = {"decode_ge_70pct_of_peak": rec["decode_frac_of_hbm_peak"] >= 0.70,
                   "faster_than_both_static_forms": all(v["speedup_of_dynamic"] > 1.0 for v in static.values())}
    return rec, step, timer, (t_plan, t_dec, t_comb)


def gpu_uuid(device):
    u = torch.cuda.get_device_properties(device).uuid
    return u and "GPU-" + str(u)


def bench_ours(args, device, rank, world):
    import load_balanced_paged_gb300 as dsa

    name = args.workload
    reps = max(50, min(args.steps, 500))
    head, step, timer, (t_plan, t_dec, t_comb) = measure_workload(dsa, device, name, args, rank, world, reps,
                                                                  seed_offset=rank)
    w, inp, C, m, B, hq = step.w, step.inp, step.C, step.m, step.B, step.hq
    nbytes = head["config"]["kv_bytes_per_step"]
    fns = [step.plan, step.decode, step.combine]
    timer.per_kernel([step.plan, step.decode_fused], 1, args.warmup)
    step.check("the fused step")

    # ---- the timed region of the contract: exactly K steps of the captured graph
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(gpu_uuid(device))
    time.sleep(0.3)
    t_wall0 = time.time()
    step_ms = timer.whole(fns, args.steps)
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.stop()
    clk = clocks.summary(t_wall0, t_wall1)
    total_ms = replica_max(float(step_ms.sum()), world, device)
    ms_per_step = total_ms / args.steps

    fused_ms = timer.whole([step.plan, step.decode_fused], reps)
    per_f = timer.per_kernel([step.plan, step.decode_fused], reps, 0)
    step.check("the fused step (timed)")
    nrep = max(10, min(args.steps, 200))
    prologue = bench_prologue(dsa, device, w, B, timer, nrep)
    # the same chain writing an E4M3 cache (the FP8 workload's heads), whatever the headline's dtype
    wf = workloads.WORKLOADS["fp8"]
    prologue_e4m3 = prologue if w.kv_dtype == "fp8" else bench_prologue(dsa, device, wf, B, timer, nrep)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    # multi-token steps use one bin per SM: the tensor-memory kernel holds one CTA per SM
    multi = bench_multi(dsa, device, inp, w, sms, m, timer, nrep, nbytes, ms_per_step)
    layouts = bench_layouts(dsa, device, inp, w, C, m, timer, nrep, nbytes, t_dec)
    chain = bench_chain(dsa, device, inp, w, C, m, timer, nrep)

    # end to end through the public API with host buffers (pinned), copies inside the timed region
    host = {k: inp[k].cpu().pin_memory() for k in ("q", "q_scale", "k_pages", "v_pages", "k_scale", "v_scale",
                                                   "block_table", "seq_lens") if inp[k] is not None}
    out_h = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    lse_h = torch.empty(step.out_lse.shape, dtype=step.out_lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        for k, t in host.items():
            inp[k].copy_(t, non_blocking=True)
        step.plan()
        step.decode()
        step.combine()
        out_h.copy_(step.out, non_blocking=True)
        lse_h.copy_(step.out_lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    step.check("the end-to-end step")
    stream = timer.stream
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    e1.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    # the same with the KV pool resident, as in a serving loop where each layer's prologue
    # appends the new tokens to the cache on the device: only the step's query, lengths and
    # block table (and E4M3 Q scales) come from pinned host memory, the output goes back
    small = {k: t for k, t in host.items() if k in ("q", "q_scale", "block_table", "seq_lens")}
    h2d_small = sum(t.numel() * t.element_size() for t in small.values())

    def e2e_step_resident():
        for k, t in small.items():
            inp[k].copy_(t, non_blocking=True)
        step.plan()
        step.decode()
        step.combine()
        out_h.copy_(step.out, non_blocking=True)
        lse_h.copy_(step.out_lse, non_blocking=True)

    for _ in range(3):
        e2e_step_resident()
    step.check("the end-to-end step with the KV pool resident")
    e0.record(stream)
    for _ in range(max(e2e_steps, 50)):
        e2e_step_resident()
    e1.record(stream)
    e1.synchronize()
    e2e_res_ms = e0.elapsed_time(e1) / max(e2e_steps, 50)

    # the other four workloads, each measured the same way (the headline stays `name`)
    others = {}
    if not args.no_other_workloads:
        del host, out_h, lse_h
        for other in workloads.WORKLOADS:
            if other == name:
                continue
            rec, ostep, _, _ = measure_workload(dsa, device, other, args, rank, world, reps, seed_offset=rank)
            others[other] = rec
            del ostep
            torch.cuda.empty_cache()

    peak, peak_src = measured_peaks()
    achieved = nbytes / (t_dec * 1e-3) / 1e9
    traffic, traffic_src = profile_traffic(name, nbytes)
    res = {
        "metric": METRIC,
        "value": round(aggregate_gbs(nbytes, world, ms_per_step), 2),
        "unit": "GB/s",
        "us_per_step": round(ms_per_step * 1e3, 2),
        "us_per_step_stats": stats_us(step_ms),
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.kv_dtype == "bf16" else "e4m3",
        "data": "synthetic (seeded; lengths, page permutation and N(0,1) values drawn as in workloads.py)",
        "config": head["config"],
        "step": "dsa_plan -> dsa_decode -> dsa_combine, one CUDA graph, programmatic dependent launch",
        "breakdown_us": {"plan": round(t_plan * 1e3, 2), "decode": round(t_dec * 1e3, 2),
                         "combine": round(t_comb * 1e3, 2)},
        "breakdown_us_stats": head["breakdown_us"],
        "step_us_stats": head["step_us"],
        "fused_combine": {"us_per_step": round(float(fused_ms.mean()) * 1e3, 2),
                          "decode_fused_us": round(float(per_f[:, 1].mean()) * 1e3, 2),
                          "note": "dsa_plan -> dsa_decode_fused (combine inside the persistent kernel)"},
        "pct_of_nominal_8tbs": round(100 * nbytes / (ms_per_step * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 1),
        "static": head["static"],
        "prologue": prologue,
        "prologue_e4m3": prologue_e4m3,
        "multi_token": multi,
        "page_layouts": layouts,
        "layer_chain": chain,
        "balance": head["balance"],
        "workloads": others,
        "roofline": {"bound": "hbm", "kernel": "attn_kernel (persistent decode, dsa_decode)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_src,
                     "algorithmic_bytes": nbytes, "traffic": traffic, "traffic_source": traffic_src},
        "e2e": {"value": round(world * nbytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "us_per_step": round(e2e_ms * 1e3, 1), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "kv_resident": {"value": round(world * nbytes / (e2e_res_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                                "us_per_step": round(e2e_res_ms * 1e3, 2), "h2d_bytes_per_step": h2d_small,
                                "d2h_bytes_per_step": d2h,
                                "note": "KV pool resident on the device; the step's query, lengths and block "
                                        "table copied from pinned host memory, output and LSE read back, "
                                        "kernels launched eagerly through the public API"}},
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
        "clocks_headline_workload": head["clocks"],
    }
    return res, inp, nbytes


def prologue_bytes(n_tokens: int, hq: int, hkv: int, fp8: bool, rot: int = 128) -> int:
    """Algorithmic bytes of dsa_prologue: per token its qkv row, position, slot and cos/sin
    row read once; its Q and K/V rows (and FP8 scales) written once."""
    rd = (hq + 2 * hkv) * 128 * 2 + 4 + 4 + rot * 4
    wr = (hq + 2 * hkv) * 128 * (1 if fp8 else 2) + ((hq + 2 * hkv) * 4 if fp8 else 0)
    return n_tokens * (rd + wr)


def bench_prologue(dsa, device, w, batch: int, timer, steps: int) -> dict:
    """dsa_prologue (QK-Norm, RoPE, Hadamard, encoding, cache write) for the decode batch of
    this workload and for a 16384-token prefill chunk of the same heads and dtypes."""
    fp8 = w.kv_dtype == "fp8"
    res = {"chain": "RMSNorm(Q, K) -> RoPE neox, rotary_dim 128 -> Hadamard(Q, K) -> "
                    + ("E4M3 + per-(token, head) scale" if fp8 else "bf16") + " -> paged cache write"}
    peak, _ = measured_peaks()
    for label, n in (("decode_batch", batch), ("prefill_16k", 16384)):
        num_pages = (n + 63) // 64 + 1
        pin = workloads.make_prologue_inputs(n, w.num_q_heads, w.num_kv_heads, num_pages, seed=1, device=device,
                                             skip_fraction=0.0)
        shape = (num_pages, w.num_kv_heads, 64, 128)
        dt = torch.uint8 if fp8 else torch.bfloat16
        kp, vp = torch.zeros(shape, dtype=dt, device=device), torch.zeros(shape, dtype=dt, device=device)
        ks = torch.zeros(shape[:3], dtype=torch.float32, device=device) if fp8 else None
        vs = torch.zeros(shape[:3], dtype=torch.float32, device=device) if fp8 else None
        q = torch.empty(n, w.num_q_heads, 128, dtype=dt, device=device)
        qs = torch.empty(n, w.num_q_heads, dtype=torch.float32, device=device) if fp8 else None
        st = torch.zeros(1, dtype=torch.int32, device=device)

        def run(pin=pin, kp=kp, vp=vp, ks=ks, vs=vs, q=q, qs=qs, st=st):
            dsa.prologue(pin["qkv"], w.num_q_heads, w.num_kv_heads, pin["slot_mapping"], kp, vp, ks, vs,
                         positions=pin["positions"], cos_sin=pin["cos_sin"], q_norm_weight=pin["q_norm_weight"],
                         k_norm_weight=pin["k_norm_weight"], hadamard=True, q_dtype=dt, q_out=q, q_scale=qs,
                         status=st)

        ms = float(timer.per_kernel([run], steps, 3).mean())
        if dsa.read_status(st) != 0:
            raise RuntimeError(f"prologue {label}: device status set")
        nb = prologue_bytes(n, w.num_q_heads, w.num_kv_heads, fp8)
        gbs = nb / (ms * 1e-3) / 1e9
        res[label] = {"tokens": n, "us": round(ms * 1e3, 2), "algorithmic_bytes": nb, "GB/s": round(gbs, 1),
                      "frac_of_hbm_peak": round(gbs / peak, 4)}
    return res


def bench_multi(dsa, device, inp, w, C: int, m: int, timer, steps: int, nbytes: int, single_ms: float) -> dict:
    """Multi-token verify steps (q_len query tokens per request, causal within the draft) on
    this workload's KV, C bins: plan -> dsa_decode_multi -> dsa_combine_multi in one graph.  The KV
    stream is read once per step whatever q_len is; `vs_q_len_one_token_steps` compares with
    q_len separate one-token steps (q_len x the one-token step time).  bf16 K/V runs on the
    tensor-memory kernel, E4M3 K/V (with E4M3 Q and per-row Q scales) on the mma.sync one."""
    fp8 = w.kv_dtype == "fp8"
    B, hq, hkv = int(inp["seq_lens"].shape[0]), w.num_q_heads, w.num_kv_heads
    G = hq // hkv
    gen = torch.Generator(device=device)
    gen.manual_seed(5)
    peak, _ = measured_peaks()
    res = {}
    for q_len in (2, 6):
        qf = torch.randn(B, q_len, hq, 128, generator=gen, device=device)
        q, qs = workloads._quantize_e4m3(qf) if fp8 else (qf.to(torch.bfloat16), None)
        tm = dsa.TaskMap(B, hkv, C, device)
        po, pl = dsa.partial_buffers(2 * tm.max_descs, q_len * G, device)  # at most 2 slots per descriptor
        out = torch.empty(B, q_len, hq, 128, dtype=torch.bfloat16, device=device)
        out_lse = torch.empty(B, q_len, hq, dtype=torch.float32, device=device)

        def plan(tm=tm):
            dsa.plan(inp["seq_lens"], hkv, C, m, task_map=tm)

        def dec(q=q, qs=qs, q_len=q_len, tm=tm, po=po, pl=pl):
            dsa.decode_multi(q_len, q, inp["k_pages"], inp["v_pages"], inp["block_table"], inp["seq_lens"], tm,
                             inp["sm_scale"], partial_o=po, partial_lse=pl, q_scale=qs, k_scale=inp["k_scale"],
                             v_scale=inp["v_scale"])

        def comb(q_len=q_len, tm=tm, po=po, pl=pl, out=out, out_lse=out_lse):
            dsa.combine_multi(q_len, tm, po, pl, hq, out=out, out_lse=out_lse)

        per = timer.per_kernel([plan, dec, comb], steps, 3)
        if dsa.get_status(tm) != 0:
            raise RuntimeError(f"multi-token q_len {q_len}: device status set")
        t_plan, t_dec, t_comb = (float(x) for x in per.mean(axis=0))
        step = t_plan + t_dec + t_comb
        gbs = nbytes / (t_dec * 1e-3) / 1e9
        # QK and PV over every (token, KV head): 512 B of bf16 K/V, 264 B of E4M3 K/V + scales
        flops = 4.0 * q_len * G * 128 * (nbytes / (264 if fp8 else 512))
        res[f"q_len_{q_len}"] = {
            "rows_per_unit": q_len * G, "us_per_step": round(step * 1e3, 2),
            "breakdown_us": {"plan": round(t_plan * 1e3, 2), "decode": round(t_dec * 1e3, 2),
                             "combine": round(t_comb * 1e3, 2)},
            "decode_kv_GB/s": round(gbs, 1), "decode_frac_of_hbm_peak": round(gbs / peak, 4),
            "decode_TFLOP/s": round(flops / (t_dec * 1e-3) / 1e12, 1),
            "vs_q_len_one_token_steps": round(q_len * single_ms / step, 2)}
    return res


def bench_chain(dsa, device, inp, w, C: int, m: int, timer, steps: int, n_layers: int = 4) -> dict:
    """A step of n_layers layers behind one plan: per layer the fused prologue (Q and the new
    token of each request into the cache), the decode and the combine, one CUDA graph.  The
    chained form starts each layer's KV gather (every layer but the first) while its prologue
    runs (dsa_decode_chained); the plain form waits for the prologue (dsa_decode)."""
    fp8 = w.kv_dtype == "fp8"
    B, hq, hkv = int(inp["seq_lens"].shape[0]), w.num_q_heads, w.num_kv_heads
    lens = inp["seq_lens"].cpu().numpy()
    pin = workloads.make_prologue_inputs(B, hq, hkv, inp["num_pages"], seed=7, device=device, skip_fraction=0.0,
                                         max_position=int(lens.max()) + 1)
    bt = inp["block_table"].cpu().numpy()
    pos = lens - 1
    pin["positions"] = torch.from_numpy(pos.astype(np.int32)).to(device)
    pin["slot_mapping"] = torch.from_numpy(
        np.array([bt[b, p // 64] * 64 + p % 64 for b, p in enumerate(pos)], np.int32)).to(device)
    qdt = torch.uint8 if fp8 else torch.bfloat16
    q = torch.empty(B, hq, 128, dtype=qdt, device=device)
    qs = torch.empty(B, hq, dtype=torch.float32, device=device) if fp8 else None
    tm = dsa.TaskMap(B, hkv, C, device)
    po, pl = dsa.partial_buffers(tm.max_descs, hq // hkv, device)
    out = torch.empty(B, hq, 128, dtype=torch.bfloat16, device=device)
    kw = dict(q_scale=qs, k_scale=inp["k_scale"], v_scale=inp["v_scale"])

    def step(chained):
        dsa.plan(inp["seq_lens"], hkv, C, m, task_map=tm)
        for layer in range(n_layers):
            dsa.prologue(pin["qkv"], hq, hkv, pin["slot_mapping"], inp["k_pages"], inp["v_pages"], inp["k_scale"],
                         inp["v_scale"], positions=pin["positions"], cos_sin=pin["cos_sin"],
                         q_norm_weight=pin["q_norm_weight"], k_norm_weight=pin["k_norm_weight"], hadamard=True,
                         q_dtype=qdt, q_out=q, q_scale=qs)
            args = (q, inp["k_pages"], inp["v_pages"], inp["block_table"], inp["seq_lens"], tm, inp["sm_scale"])
            if chained and layer > 0:
                dsa.decode_chained(1, *args, partial_o=po, partial_lse=pl, **kw)
            else:
                dsa.decode(*args, partial_o=po, partial_lse=pl, **kw)
            dsa.combine(tm, po, pl, hq, out=out)

    res = {"layers": n_layers, "step": "plan, then per layer: dsa_prologue -> decode -> dsa_combine; one CUDA graph"}
    for label, chained in (("plain", False), ("chained", True)):
        for _ in range(3):
            step(chained)
        torch.cuda.synchronize()
        if dsa.get_status(tm) != 0:
            raise RuntimeError(f"layer chain ({label}): device status set")
        ms = timer.whole([lambda chained=chained: step(chained)], steps)
        res[f"{label}_us"] = stats_us(ms)
    res["saved_us_per_chained_layer"] = round((res["plain_us"]["median"] - res["chained_us"]["median"]) /
                                              (n_layers - 1), 2)
    return res


def cta_balance(times: torch.Tensor) -> dict:
    """Per-CTA [start, end] timer readings (ns) of one launch: the span from the first start
    to the last end, and the idle tail = (last end - median end) / span, the share of the
    launch during which at least half of the CTAs had already finished."""
    t = times.cpu().numpy().astype(np.int64)
    t = t[t[:, 1] > 0]
    if t.size == 0:
        return {}
    start, end = t[:, 0], t[:, 1]
    span = float(end.max() - start.min())
    return {"ctas": int(t.shape[0]), "span_us": round(span / 1e3, 2),
            "idle_tail": round(float(end.max() - np.median(end)) / span, 4) if span > 0 else 0.0,
            "end_spread_us": round(float(end.max() - end.min()) / 1e3, 2)}


def bench_layouts(dsa, device, inp, w, C: int, m: int, timer, steps: int, nbytes: int, base_ms: float) -> dict:
    """The decode kernel on the same lengths and C bins with the KV held in pages of 16 / 32 /
    64 tokens, HND or NHD (dsa_decode_ex): a 64-token tile is then loaded as 64 / P boxes."""
    B, hq, hkv = int(inp["seq_lens"].shape[0]), w.num_q_heads, w.num_kv_heads
    lens = inp["seq_lens"].cpu().numpy()
    peak, _ = measured_peaks()
    tm = dsa.TaskMap(B, hkv, C, device)
    dsa.plan(inp["seq_lens"], hkv, C, m, task_map=tm)
    po, pl = dsa.partial_buffers(tm.max_descs, hq // hkv, device)
    res = {}
    for page, layout in ((64, "NHD"), (32, "HND"), (32, "NHD"), (16, "HND"), (16, "NHD")):
        li = workloads.make_inputs(lens, hq, hkv, w.kv_dtype, w.seed, device, page_size=page, kv_layout=layout)

        def dec(li=li, layout=layout):
            dsa.decode(inp["q"], li["k_pages"], li["v_pages"], li["block_table"], li["seq_lens"], tm,
                       inp["sm_scale"], partial_o=po, partial_lse=pl, q_scale=inp.get("q_scale"),
                       k_scale=li.get("k_scale"), v_scale=li.get("v_scale"), kv_layout=layout)

        per = timer.per_kernel([dec], steps, 3)
        if dsa.get_status(tm) != 0:
            raise RuntimeError(f"page {page} {layout}: device status set")
        t = float(per.mean())
        gbs = nbytes / (t * 1e-3) / 1e9
        res[f"P{page}_{layout}"] = {"decode_us": round(t * 1e3, 2), "kv_GB/s": round(gbs, 1),
                                    "frac_of_hbm_peak": round(gbs / peak, 4),
                                    "time_vs_P64_HND": round(t / base_ms, 3)}
        del li
    return res


# ---------------------------------------------------------------------------- CPU oracle

def oracle_problem(inp, requests):
    """Host copy (exact bytes) of the listed requests with their pages renumbered."""
    import oracle

    def np_bytes(t):
        t = t.detach().cpu().contiguous()
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()

    lens = inp["seq_lens"][requests].cpu().numpy()
    npages = [(int(n) + 63) // 64 for n in lens]
    idx = torch.cat([inp["block_table"][b, :n] for b, n in zip(requests, npages)]).long()
    pools = {k: (None if inp[k] is None else np_bytes(inp[k].index_select(0, idx)))
             for k in ("k_pages", "v_pages", "k_scale", "v_scale")}
    bt = np.full((len(requests), max(max(npages), 1)), -1, np.int32)
    off = 0
    for i, n in enumerate(npages):
        bt[i, :n] = np.arange(off, off + n)
        off += n
    qs = None if inp["q_scale"] is None else np_bytes(inp["q_scale"][requests])
    return oracle.Problem(np_bytes(inp["q"][requests]), pools["k_pages"], pools["v_pages"], bt, lens,
                          inp["num_q_heads"], inp["num_kv_heads"], inp["sm_scale"], q_scale=qs,
                          k_scale=pools["k_scale"], v_scale=pools["v_scale"]), lens


def oracle_seconds_per_token(inp, threads: int) -> float:
    """Oracle time per token of one request (all its KV heads), measured on the request of
    median length (the shortest would fold the per-call cost into every token)."""
    lens = inp["seq_lens"].cpu().numpy()
    b = int(np.argsort(lens)[len(lens) // 2])
    prob, _ = oracle_problem(inp, [b])
    t0 = time.perf_counter()
    prob.attention(n_threads=threads)
    return (time.perf_counter() - t0) / max(int(lens[b]), 1)


def cpu_oracle_rate(inp, budget_s: float, rng_seed: int = 0, threads: int = 0, per_token: float | None = None,
                    fit: bool = False):
    """Time the oracle (all host threads, or `threads`) on a bounded sample of requests;
    returns (GB/s of KV processed, threads, description).  Requests are taken in a seeded
    random order until the estimated time fills the budget; with `fit`, a request that would
    overrun it is skipped instead (at least one request: the shortest if none fits), so that
    small budgets stay small."""
    import oracle
    lens = inp["seq_lens"].cpu().numpy()
    rng = np.random.default_rng(rng_seed)
    order = rng.permutation(len(lens))
    threads = threads or oracle.default_threads()
    if per_token is None:
        per_token = oracle_seconds_per_token(inp, threads)
    # the oracle runs one thread per (request, KV head) unit
    eff = min(threads, inp["num_kv_heads"] * len(lens))
    chosen, est = [], 0.0
    for b in order:
        t = per_token * lens[b] * inp["num_kv_heads"] / eff
        if fit and est + t > budget_s:
            continue
        chosen.append(int(b))
        est += t
        if est >= budget_s:
            break
    if not chosen:
        chosen = [int(np.argmin(lens))]
    prob, sl = oracle_problem(inp, chosen)
    t0 = time.perf_counter()
    prob.attention(n_threads=threads)
    dt = time.perf_counter() - t0
    nbytes = workloads.kv_bytes(sl, inp["num_kv_heads"], inp["kv_dtype"])
    desc = (f"{len(chosen)} of {len(lens)} requests ({int(sl.sum())} of {int(lens.sum())} tokens), "
            f"fp64 oracle, {dt:.1f} s")
    return nbytes / dt / 1e9, threads, desc


# ---------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixed", choices=list(workloads.WORKLOADS))
    ap.add_argument("--min-tiles", type=int, default=4)
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="measure only --workload (the default also measures the other four)")
    ap.add_argument("--requests", type=int, default=None, help="keep only the first N requests (profiling)")
    ap.add_argument("--l2", choices=["auto", "flush", "none"], default="auto",
                    help="auto: flush L2 between steps only when the KV bytes are below 2 x L2")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        bench_reference(args)
        return

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    res, inp, nbytes = bench_ours(args, device, rank, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, desc = cpu_oracle_rate(inp, args.cpu_budget)
        v1, _, desc1 = cpu_oracle_rate(inp, args.cpu_budget / 3, threads=1)
        res["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                               "sample": desc, **host_cpu(),
                               "one_thread": {"value": round(v1, 4), "sample": desc1}}
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def host_cpu() -> dict:
    """Model string and hardware thread count of the host CPU the oracle runs on."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"cpu_model": model or platform.processor() or platform.machine(),
            "hardware_concurrency": os.cpu_count(), "cpu_arch": platform.machine()}


def bench_reference(args):
    """The fp64 CPU oracle as the reference arm: W + K steps, each a bounded sample.  Its
    `config` is the one our arm prints for the same workload."""
    import oracle
    name = args.workload
    w = workloads.WORKLOADS[name]
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    inp = workloads.make_workload(name, device=dev, max_requests=args.requests)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if dev.type == "cuda":
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        _, l2_note = l2_policy(args, kv_bytes(inp), dev)
    else:
        sms, l2_note = 152, "no GPU visible"
    config = workload_config(w, int(inp["seq_lens"].shape[0]), w.num_ctas(sms), args.min_tiles, kv_bytes(inp),
                             l2_note, world)
    # about 150 s of oracle work over the whole run, whatever K and W are
    per_step = 150.0 / (args.steps + args.warmup)
    per_token = oracle_seconds_per_token(inp, oracle.default_threads())
    rates = []
    desc = ""
    for k in range(args.warmup + args.steps):
        v, cores, desc = cpu_oracle_rate(inp, per_step, rng_seed=k, per_token=per_token, fit=True)
        if k >= args.warmup:
            rates.append(v)
    v = float(np.mean(rates))
    nbytes = kv_bytes(inp)
    us = nbytes / (v * 1e9) * 1e6
    res = {"metric": METRIC, "value": round(v, 4), "unit": "GB/s", "us_per_step": round(us, 1),
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded, as in workloads.py)",
           "config": config,
           "impl": "reference",
           "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": oracle.default_threads(),
                            "kind": "oracle", "sample": f"per step: {desc}", **host_cpu()},
           "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()

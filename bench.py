"""Benchmark of the KDA decode / speculative-verify step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload NAME]

A step is one call of the library (one kernel launch) over one batch of the
workload: by default decode_b256_h32 (B=256 requests, H=32 heads, 8192
(request, head) items, 1 GiB of FP32 state pages read + written per step).
Inputs are seeded synthetic tensors resident in HBM before the timed region.
The state pages one step touches (512 MiB) exceed the 129 MB L2, so no L2
flush is inserted between steps.

Prints ONE JSON line (rank 0).  Under torchrun each rank runs its own batch of
the same shape on its own GPU (weak scaling, no collective on the data path);
timing is the max over ranks.

--impl reference times the CPU oracle on the host cores (the only comparison
implementation that exists for this path), on a bounded sample of the same
workload; rank 0 alone runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KDA decode (req,head) items/s + achieved HBM GB/s vs ~8 TB/s at B=256,H=32"
UNIT = "items/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCE = os.path.join(ROOT, "linear_attention_recurrent_kda_gb300", "csrc",
                             "kda_step.cu")
OPROJ_SOURCE = os.path.join(ROOT, "linear_attention_recurrent_kda_gb300", "csrc",
                            "kda_oproj.cu")
RECOVER_SOURCE = os.path.join(ROOT, "linear_attention_recurrent_kda_gb300", "csrc",
                              "kda_recover.cu")


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def shard_workload(workload, rank: int):
    """Rank r's batch: same shape, its own seed (independent requests)."""
    return workload.with_(seed=workload.seed + 7919 * rank)


def max_over_ranks(values, dist, device):
    """Element-wise max of a list of floats over all ranks (timing only)."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sha(source: str = None):
    with open(source or KERNEL_SOURCE, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def ncu_traffic(workload: str, kernel: str = "kda_step", source: str = None):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, or None when absent or taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.ncu.json")
    try:
        with open(path) as f:
            p = json.load(f)
    except Exception:
        return None
    if p.get("source_sha256") != kernel_sha(source):
        return None
    return p.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (100 ms)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, line in self.samples:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        window = [p for ts, p in rows if t0 <= ts <= t1]
        if not window:
            return None
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in window if num(p[1]) is not None]
        mx = [num(p[2]) for p in window if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i - 5] for p in window for i in range(5, 9)
                          if p[i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(window)}


def run_reference(args, workload):
    """The CPU oracle timed on the host cores over a bounded item sample."""
    import numpy as np
    import oracle
    from linear_attention_recurrent_kda_gb300.workloads import make_inputs
    from tests.hostdata import to_oracle
    inp = to_oracle(make_inputs(workload))
    threads = args.oracle_threads or oracle.max_threads()
    rng = np.random.default_rng(0)
    order = rng.permutation(workload.items).astype(np.int32)
    m = min(64, workload.items)
    t = time.perf_counter()
    oracle.run(inp, mode="f32", items=np.sort(order[:m]), in_place=True,
               threads=threads)
    per_item = (time.perf_counter() - t) / m
    # size each step so the whole run stays near one minute of CPU time
    n = int(max(16, min(1024, 60.0 / (max(args.steps, 1) * per_item))))
    n = min(n, workload.items)
    items = np.sort(order[:n])
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.run(inp, mode="f32", items=items, in_place=True, threads=threads)
        times.append(time.perf_counter() - t)
    per_step = sum(times) / len(times)
    value = n / per_step
    sample = (f"{n} of {workload.items} items per step (seeded), full per-item "
              f"step incl. state page read/write, {threads} OpenMP threads")
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "impl": "reference",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step * 1e3 * workload.items / n,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload.name, "batch": workload.batch,
                   "heads": workload.heads, "tokens": workload.tokens,
                   "items": workload.items},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def cpu_baseline(workload, budget_s=12.0, threads=0):
    import numpy as np
    import oracle
    from linear_attention_recurrent_kda_gb300.workloads import make_inputs
    from tests.hostdata import to_oracle
    inp = to_oracle(make_inputs(workload))
    threads = threads or oracle.max_threads()
    rng = np.random.default_rng(1)
    n = min(workload.items, 1024)
    items = np.sort(rng.choice(workload.items, size=n, replace=False)).astype(np.int32)
    done, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        oracle.run(inp, mode="f32", items=items, in_place=True, threads=threads)
        done += n
    dt = time.perf_counter() - t0
    return {"value": done / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{done} items ({n}-item seeded sample of {workload.name}, "
                      f"repeated) in {dt:.1f} s"}


def run_recover(args):
    """Times kda_recover on a record-mode workload (single GPU): one record
    verify produces the records, then each step replays accepted ~ U{1..T}
    tokens of every item in place (checkpoint page -> same slot)."""
    import torch
    from linear_attention_recurrent_kda_gb300.api import kda_recover, step_from_inputs
    from linear_attention_recurrent_kda_gb300.workloads import WORKLOADS, make_inputs
    name = args.workload if WORKLOADS[args.workload].record else "verify_q8_record_b64_h64"
    w = WORKLOADS[name]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    host = make_inputs(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    B, H, T = w.batch, w.heads, w.tokens
    out = torch.empty((B * T, H * 128), dtype=torch.bfloat16, device=dev)
    ru = torch.empty((B, H, T, 128), dtype=torch.float32, device=dev)
    rk = torch.empty((B, H, T, 256), dtype=torch.bfloat16, device=dev)
    step_from_inputs(d, out, rec_u=ru, rec_kg=rk)()
    src = torch.tensor([int(host["slots"][r, int(host["accepted"][r]) - 1])
                        for r in range(B)], dtype=torch.int32, device=dev)
    acc = torch.randint(1, T + 1, (B,), generator=torch.Generator().manual_seed(3),
                        dtype=torch.int32).to(dev)

    sched = torch.zeros(2, dtype=torch.int32, device=dev)

    def call():
        kda_recover(state=d["state"], src_slots=src, dst_slots=src, accepted=acc,
                    rec_u=ru, rec_kg=rk, a_log=d["a_log"], dt_bias=d["dt_bias"],
                    lower_bound=w.lower_bound, sched=sched)

    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    live = int((src > 0).sum()) * H
    acc_live = int(acc[src > 0].sum()) * H
    nbytes = live * 2 * 128 * 128 * 4 + acc_live * (128 * 4 + 256 * 2) + B * 12
    peak, kind = measured_peak()
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": "KDA record replay (req,head) items/s", "op": "recover",
        "value": live / (ms * 1e-3), "unit": "items/s", "ms_per_step": ms,
        "steps": args.steps, "config": {"workload": name, "items_live": live,
                                        "replayed_tokens": acc_live},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                     "frac": gbs / peak, "peak_source": f"{kind} hbm_gbs",
                     "traffic": ncu_traffic(name, "kda_recover", RECOVER_SOURCE),
                     "algorithmic_bytes_per_launch": nbytes}}), flush=True)


def run_oproj(args):
    """Times kda_oproj (the output-projection consumer epilogue) on the TP16,
    256-row, hidden 7168, 8-block workload (single GPU).  Its inputs (~95 MB)
    fit in L2, so a 256 MiB buffer is written between launches and only the
    launches are timed (CUDA events around each one on the launching stream).
    The prefix is updated in place every step, as the layer does."""
    import torch
    from linear_attention_recurrent_kda_gb300.api import kda_oproj
    from linear_attention_recurrent_kda_gb300.workloads import (OPROJ_WORKLOADS,
                                                                make_oproj_inputs)
    w = OPROJ_WORKLOADS["oproj_tp16_t256_h7168_nb8"]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    host = make_oproj_inputs(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    out = torch.empty((w.tokens, w.hidden), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        kda_oproj(partials=d["partials"], prefix=d["prefix"], output=out,
                  out_norm=d["out_norm"], blocks=d["blocks"], norm=d["norm"],
                  query=d["query"], has_delta=w.has_delta, eps=w.eps,
                  out_eps=w.out_eps, stream=stream)

    steps = min(args.steps, 2000)
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    t_w0 = time.time()
    while time.time() - t_w0 < 1.0:          # untimed soak: clock samples under load
        for _ in range(50):
            flush.zero_()
            call()
        torch.cuda.synchronize()
    for e0, e1 in ev:
        flush.zero_()
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    t_w1 = time.time()
    sampler.stop()
    ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps
    row = w.hidden * 2
    rows = w.tp + w.nb + (1 if w.has_delta else 0) + 2   # reads + prefix/output writes
    nbytes = w.tokens * rows * row + 3 * row
    peak, kind = measured_peak()
    gbs = nbytes / (ms * 1e-3) / 1e9
    line = {
        "metric": "output-projection consumer epilogue rows/s", "op": "oproj",
        "value": w.tokens / (ms * 1e-3), "unit": "rows/s", "ms_per_step": ms,
        "steps": steps, "warmup": max(args.warmup, 3), "higher_is_better": True,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "tp": w.tp, "tokens": w.tokens,
                   "hidden": w.hidden, "nb": w.nb, "has_delta": w.has_delta,
                   "l2": "inputs fit in L2: a 256 MiB buffer is written between "
                         "launches; only the launches are timed"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                     "frac": gbs / peak, "peak_source": f"{kind} hbm_gbs",
                     "traffic": ncu_traffic(w.name, "kda_oproj", OPROJ_SOURCE),
                     "algorithmic_bytes_per_launch": nbytes},
        "clocks": dict(sampler.summary(t_w0, t_w1) or {}, window="soak+timed"),
        "gpu_launches": steps,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = oproj_cpu_baseline(w, host, ms)
    print(json.dumps(line), flush=True)


def run_pattern(args):
    """The decode workload's page traffic alone (kda_probe_page_copy: every
    page read into shared memory and written back in place, the step's
    schedule, no arithmetic), with the step's two stages and with three, and
    with contiguous ranges only (no shared items): the bandwidth ceiling of
    that access pattern, beside the measured copy peak."""
    import torch
    from linear_attention_recurrent_kda_gb300.probe import kda_probe_page_copy
    from linear_attention_recurrent_kda_gb300.workloads import WORKLOADS, make_inputs

    from linear_attention_recurrent_kda_gb300.accounting import step_bytes
    w = WORKLOADS[args.workload or "decode_b256_h32"]
    if w.record:                           # record mode writes no page: nothing to probe
        w = WORKLOADS["decode_b256_h32"]
    host = make_inputs(w)
    dev = torch.device("cuda", 0)
    state, slots = host["state"].to(dev), host["slots"].to(dev)
    accepted = host["accepted"].to(dev) if w.tokens > 1 else None
    live = w.items if w.tokens > 1 else int((host["slots"] > 0).sum()) * w.heads
    nbytes = step_bytes(w, host)["state"]
    stream = torch.cuda.Stream(device=dev)
    peak, peak_kind = measured_peak()
    sched = torch.zeros(2, dtype=torch.int32, device=dev)
    res = {}
    for key, stages, sc in (("two", 2, sched), ("three", 3, sched), ("ranges", 2, None)):
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                kda_probe_page_copy(state=state, slots=slots, accepted=accepted,
                                    tokens=w.tokens, stages=stages, sched=sc, stream=stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                kda_probe_page_copy(state=state, slots=slots, accepted=accepted,
                                    tokens=w.tokens, stages=stages, sched=sc, stream=stream)
            e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / args.steps
        res[key] = (ms, nbytes / (ms * 1e-3) / 1e9)
    ms2, gbs2 = res["two"]
    line = {
        "metric": "step page access pattern (read, then every page write, no arithmetic)",
        "value": gbs2, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms2, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name + " pages", "stages": 2, "live_items": live,
                   "schedule": "contiguous ranges, then shared items (the step's)",
                   "l2": "inputs larger than L2 (1 GiB of pages per step); no flush"},
        "roofline": {"bound": "hbm", "achieved": gbs2, "peak": peak, "unit": "GB/s",
                     "frac": gbs2 / peak, "traffic": None,
                     "peak_source": f"{peak_kind} hbm_gbs", "algorithmic_bytes_per_launch": nbytes},
        "three_stages": {"ms_per_step": res["three"][0], "achieved": res["three"][1],
                         "frac": res["three"][1] / peak},
        "ranges_only": {"ms_per_step": res["ranges"][0], "achieved": res["ranges"][1],
                        "frac": res["ranges"][1] / peak},
        "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)


def oproj_cpu_baseline(w, host, gpu_ms):
    """The oracle (FP32 mode, page order) on the host cores, on the first 64
    rows of the same inputs, scaled to rows/s."""
    import oracle
    n = min(64, w.tokens)

    def bits(t):
        return None if t is None else t[:n].contiguous().view(torch_int16()).numpy().view("uint16")

    args = dict(partials=host["partials"][:, :n].contiguous().view(torch_int16()).numpy()
                .view("uint16"), prefix=bits(host["prefix"]),
                out_norm=host["out_norm"].view(torch_int16()).numpy().view("uint16"),
                blocks=bits(host["blocks"]),
                norm=host["norm"].view(torch_int16()).numpy().view("uint16"),
                query=host["query"].view(torch_int16()).numpy().view("uint16"),
                has_delta=w.has_delta, eps=w.eps, out_eps=w.out_eps, mode="f32")
    oracle.oproj(**args)
    t0 = time.time()
    reps = 0
    while time.time() - t0 < 10.0:
        oracle.oproj(**args)
        reps += 1
    sec = (time.time() - t0) / reps
    return {"value": n / sec, "unit": "rows/s", "cores": oracle.max_threads(),
            "kind": "oracle", "sample": f"first {n} of {w.tokens} rows, FP32 mode, "
                                        f"{reps} repetitions"}


def torch_int16():
    import torch
    return torch.int16


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="decode_b256_h32")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-threads", type=int, default=0,
                    help="OpenMP threads of the CPU oracle (reference arm and "
                         "cpu_baseline); 0 = every host core")
    ap.add_argument("--op", default="step",
                    choices=["step", "recover", "oproj", "pattern"],
                    help="step: the decode/verify step (default); recover: the "
                         "record replay after a record-mode verify; oproj: the "
                         "output-projection consumer epilogue; pattern: the decode "
                         "workload's page traffic alone (bandwidth ceiling probe)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from linear_attention_recurrent_kda_gb300.workloads import WORKLOADS
    workload = WORKLOADS[args.workload]
    rank, world, local = dist_env()

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, workload)), flush=True)
        return
    if args.op == "recover":
        run_recover(args)
        return
    if args.op == "pattern":
        return run_pattern(args)
    if args.op == "oproj":
        run_oproj(args)
        return

    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    from linear_attention_recurrent_kda_gb300.accounting import (
        RECURRENCE_FLOP_PER_TOKEN_ITEM, recurrence_flop, step_bytes)
    from linear_attention_recurrent_kda_gb300.api import step_from_inputs
    from linear_attention_recurrent_kda_gb300.workloads import make_inputs

    w = shard_workload(workload, rank)
    host = make_inputs(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    B, H, T = w.batch, w.heads, w.tokens
    out = torch.empty((B * T, H * 128), dtype=torch.bfloat16, device=dev)
    rec_u = rec_kg = None
    if w.record:
        rec_u = torch.empty((B, H, T, 128), dtype=torch.float32, device=dev)
        rec_kg = torch.empty((B, H, T, 256), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    step = step_from_inputs(d, out, rec_u=rec_u, rec_kg=rec_kg)
    nbytes = step_bytes(w, host)

    def barrier():
        if pg is not None:
            pg.barrier()

    sampler = ClockSampler(local)
    sampler.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step(stream)
        stream.synchronize()
        # extra untimed soak so clock samples exist around a short timed region
        t_soak = time.time()
        soak = 0
        while time.time() - t_soak < 1.0:
            for _ in range(200):
                step(stream)
            stream.synchronize()
            soak += 200

        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier()
        torch.cuda.synchronize(dev)
        t_host0 = time.time()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            step(stream)
            ends[i].record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        t_host1 = time.time()
    sampler.stop()
    total_ms = t0.elapsed_time(t1)
    kern_ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps
    ms_step = total_ms / args.steps
    if pg is not None:
        ms_step, kern_ms = max_over_ranks([ms_step, kern_ms], pg, dev)
    clocks = sampler.summary(t_host0 - 0.15, t_host1 + 0.15)
    clock_window = "timed"
    if clocks is None:
        clocks = sampler.summary(t_soak, t_host1 + 0.15)
        clock_window = "soak+timed (timed region shorter than the 100 ms sample period)"

    # ---- end to end: pinned host inputs -> device, the call, output -> host.
    # Every step copies its inputs up and its result down; consecutive steps are
    # double-buffered over a copy-in and a copy-out stream, so step i+1's
    # upload and step i's download overlap the kernels (the state and conv
    # pools stay resident; each kernel still waits for its own inputs).
    per_step_in = ["x", "f_a", "beta", "gate", "slots"] + (["accepted"] if T > 1 else [])
    pinned = {k: host[k].pin_memory() for k in per_step_in}
    h2d = sum(pinned[k].numel() * pinned[k].element_size() for k in per_step_in)
    bufs = []
    for b in range(2):
        db = dict(d)
        for k in per_step_in:
            db[k] = torch.empty_like(d[k])
        ob = torch.empty_like(out)
        hb = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        bufs.append((db, ob, hb, step_from_inputs(db, ob, rec_u=rec_u, rec_kg=rec_kg)))
    d2h = bufs[0][2].numel() * bufs[0][2].element_size()
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_used = [torch.cuda.Event() for _ in range(2)]   # kernel done with buffer b
    ev_out = [torch.cuda.Event() for _ in range(2)]    # download of buffer b done
    e2e_steps = max(1, min(args.steps, 500))

    def e2e_run(n):
        for i in range(n):
            b = i & 1
            db, ob, hb, st = bufs[b]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_used[b])
                for k in per_step_in:
                    db[k].copy_(pinned[k], non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])
            st(stream)
            ev_used[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_used[b])
                hb.copy_(ob, non_blocking=True)
                ev_out[b].record(s_out)

    for sx in (s_in, s_out):
        sx.wait_stream(stream)
    e2e_run(4)
    torch.cuda.synchronize(dev)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    stream.wait_event(e0)
    s_out.wait_event(e0)
    e2e_run(e2e_steps)
    s_out.wait_stream(stream)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    if pg is not None:
        (e2e_ms,) = max_over_ranks([e2e_ms], pg, dev)

    items = w.items * world
    value = items / (ms_step * 1e-3)
    peak, peak_kind = measured_peak()
    achieved = nbytes["total"] / (kern_ms * 1e-3) / 1e9
    state_gbs = nbytes["state"] / (kern_ms * 1e-3) / 1e9
    traffic = ncu_traffic(w.name if rank == 0 else workload.name)
    # Decode and verify: the same pages moved with no arithmetic
    # (kda_probe_page_copy, the step's two stages), timed after the step's
    # region: the ceiling of this access pattern, beside the copy peak.
    pattern = None
    if not w.record:
        from linear_attention_recurrent_kda_gb300.probe import kda_probe_page_copy
        pslots = d["slots"].view(-1).contiguous() if T == 1 else d["slots"]
        pacc = d["accepted"] if T > 1 else None
        psched = torch.zeros(2, dtype=torch.int32, device=dev)

        def probe():
            kda_probe_page_copy(state=d["state"], slots=pslots, accepted=pacc, tokens=T,
                                sched=psched, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(3):
                probe()
            p0 = torch.cuda.Event(enable_timing=True)
            p1 = torch.cuda.Event(enable_timing=True)
            p0.record(stream)
            for _ in range(20):
                probe()
            p1.record(stream)
        torch.cuda.synchronize(dev)
        p_ms = p0.elapsed_time(p1) / 20
        p_gbs = nbytes["state"] / (p_ms * 1e-3) / 1e9
        pattern = {"ms": p_ms, "state_gbs": p_gbs, "frac": p_gbs / peak,
                   "step_state_frac_of_pattern": state_gbs / p_gbs}
    # FP32 pipe: the recurrence's flop against the derived non-tensor FP32 peak
    # (SMs x 128 FP32 lanes x 2 flop per FMA x the maximum SM clock).
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    max_mhz = float((clocks or {}).get("sm_max_mhz") or 2070.0)
    fp32_peak = sms * 128 * 2 * max_mhz * 1e6 / 1e12
    fp32_tf = recurrence_flop(w, host) / (kern_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload.name, "batch": B, "heads": H, "tokens": T,
                   "items_per_gpu": w.items, "state_io": "fp32 pages, bf16 activations",
                   "l2": "inputs larger than L2: 512 MiB of state pages touched per "
                         "step vs 129 MB L2; no flush",
                   "parallelism": f"replica x{world} (independent batches)"},
        "tokens_per_s": items * T / (ms_step * 1e-3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": nbytes["total"],
                     "state_bytes_per_launch": nbytes["state"],
                     "state_gbs": state_gbs, "state_frac": state_gbs / peak,
                     "kernel_ms": kern_ms, "access_pattern_ceiling": pattern},
        "fp32_pipe": {"achieved": fp32_tf, "peak": fp32_peak, "unit": "TFLOP/s",
                      "frac": fp32_tf / fp32_peak,
                      "flop_per_token_item": RECURRENCE_FLOP_PER_TOKEN_ITEM,
                      "peak_source": f"derived: {sms} SMs x 128 FP32 lanes x 2 flop x "
                                     f"{max_mhz:.0f} MHz"},
        "clocks": dict(clocks or {}, window=clock_window),
        "e2e": {"value": items / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms},
        "gpu_launches": args.steps,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(workload, threads=args.oracle_threads)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()

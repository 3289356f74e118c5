#!/usr/bin/env python3
"""Throughput of the batched speculative-decoding verifier step on GB300.

One step = one pass of the whole hot path over one batch: spec_verify (per-position kernel +
per-request selection), spec_compact and spec_choose_gamma, enqueued as one spec_verify_round
call (the per-position kernel, then one kernel for the selection, the compaction and the gamma
choice), on the workload
"B=64 ragged K_i ~ U{0..7}, V=128256, bf16 Zipf logits, T=0.7" (synthetic, seeded). Four
input sets of ~131 MB each (larger than the 126 MB L2) rotate between steps.

Prints one JSON line. `value` is verified rows/s (sum_i (K_i+1) per step over the step time)
for the whole job; `roofline` reports the per-position kernel's achieved HBM bandwidth
(algorithmic bytes: every target and draft logit once) against the measured copy bandwidth.

--impl reference times the float64 CPU oracle on this host's cores instead (a deliberately
slow program: a reported baseline, not a target).

Multi-GPU: one process per GPU under torchrun; requests are independent, so every rank runs
its own replica of the batch (weak scaling, no data-path collective); the step time is the
maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_verification_43_gb300 import workloads as W  # noqa: E402

METRIC = "verified rows/sec (Σ(K_i+1) over V) and achieved HBM GB/s vs GB300 peak"
UNIT = "rows/s"
WORKLOAD = "c3"
GAMMA_COST = 0.05  # relative draft cost c used by the gamma controller each step
KERNEL_SAMPLE = 8  # the per-position kernel is bracketed by CUDA events on every 8th timed step
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "stream_kernel_c3_traffic.json")
CSRC = os.path.join(ROOT, "speculative_decoding_verification_43_gb300", "csrc")
# the per-position kernel's sources: a committed ncu traffic figure counts only while they match
KERNEL_SRCS = ("spec_verify.cu", "spec_kernels.cuh", "spec_math.cuh",
               "spec_device.cuh")


def parse():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--input-sets", type=int, default=4)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def job_value(world: int, rows_per_step: int, steps: int, ms_total_max: float) -> float:
    """Whole-job throughput: every rank verifies its own batch each step (weak scaling); the
    slowest rank's time (the max over ranks) bounds the job."""
    return world * rows_per_step * steps / (ms_total_max / 1e3)


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed loop runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.gpu = self._gpu_id(device_index)

    @staticmethod
    def _gpu_id(device_index):
        try:
            u = str(torch.cuda.get_device_properties(device_index).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            ids = [v for v in vis.split(",") if v.strip()]
            return ids[device_index] if device_index < len(ids) else str(device_index)

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower().startswith("active")})
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------ shared helpers

def measured_peak():
    try:
        d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def code_of(src: str) -> str:
    """A C++/CUDA source without its comments and blank lines: what the compiler sees."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def kernel_hash(read=None):
    """Hash of the per-position kernel's code (comments excluded): a recorded ncu figure counts
    only while the code it was taken on is unchanged."""
    read = read or (lambda f: open(os.path.join(CSRC, f)).read())
    h = hashlib.sha256()
    for f in KERNEL_SRCS:
        h.update(code_of(read(f)).encode())
    return h.hexdigest()[:16]


def recorded_traffic(bytes_per_launch):
    """DRAM bytes per launch from the committed ncu capture, if it was taken on this kernel."""
    try:
        d = json.load(open(PROFILE_TRAFFIC))
    except Exception:
        return None
    if d.get("kernel_src_sha256_16") != kernel_hash():
        return None
    return d.get("dram_bytes_per_launch")


def kernel_label(wl, rows):
    """The per-position kernel the library launches for this workload, and its grid."""
    from speculative_decoding_verification_43_gb300 import api
    plan = api.verify_plan(wl.B, wl.V, rows, wl.dtype)
    if plan is None:
        return "none"
    name, c, n = plan
    return f"{name}<{'bf16' if wl.dtype == torch.bfloat16 else 'f32'}>, {n} clusters of {c}"


def workload_config(wl, rows, logit_bytes):
    return {
        "workload": f"{wl.name}: {wl.note}",
        "B": wl.B, "V": wl.V, "input_dtype": "bf16" if wl.dtype == torch.bfloat16 else "f32",
        "rows_per_step": rows, "logit_bytes_per_step": logit_bytes,
        "step": "spec_verify_round: spec_verify + spec_compact (P=4096, page 16) + spec_choose_gamma in one call",
        "l2": "inputs larger than L2: 4 rotating input sets of ~131 MB each (L2 126 MB)",
    }


def _host_round(rd):
    return dict(target=W.to_numpy_logits(rd.target), draft=W.to_numpy_logits(rd.draft),
                row_off=rd.row_off.cpu().numpy(), toks=rd.draft_tokens.cpu().numpy(),
                u=rd.uniforms.cpu().numpy(), temp=rd.temperature.cpu().numpy())


def oracle_rows(h, reqs):
    """Oracle inputs of the sub-batch [(request, positions kept)]."""
    ro = h["row_off"]
    t_rows, d_rows, off, temps = [], [], [0], []
    for i, k in reqs:
        r0 = int(ro[i])
        t_rows.extend(range(r0, r0 + k + 1))
        d_rows.extend(range(r0 - i, r0 - i + k))
        off.append(off[-1] + k + 1)
        temps.append(h["temp"][i])
    u = h["u"][t_rows].copy()
    # a truncated request keeps its frontier draw in its last slot
    for n, (i, k) in enumerate(reqs):
        u[off[n + 1] - 1] = h["u"][int(ro[i + 1]) - 1]
    return (h["target"][t_rows], h["draft"][d_rows], np.asarray(off, np.int32), h["toks"][d_rows], u,
            np.asarray(temps, np.float32))


def plan_sample(h, rows_budget, cursor):
    ro = h["row_off"]
    B = len(ro) - 1
    reqs, rows = [], 0
    while rows < rows_budget:
        i = cursor % B
        K = int(ro[i + 1] - ro[i] - 1)
        k = min(K, rows_budget - rows - 1)
        reqs.append((i, k))
        rows += k + 1
        cursor += 1
    return reqs, rows, cursor


def time_oracle(h, rows_budget, cursor):
    import oracle
    reqs, rows, cursor = plan_sample(h, rows_budget, cursor)
    args = oracle_rows(h, reqs)
    t0 = time.perf_counter()
    oracle.verify(*args)
    return rows, time.perf_counter() - t0, cursor


def cpu_baseline(rd, seconds):
    """The oracle as it stands (single-threaded C, float64) on this host, on a bounded sample."""
    import oracle
    oracle.build()
    h = _host_round(rd)
    rows_total, secs, cursor = 0, 0.0, 0
    rows_budget = 1
    while secs < seconds:
        r, s, cursor = time_oracle(h, rows_budget, cursor)
        rows_total += r
        secs += s
        per_row = s / r
        rows_budget = max(1, min(int(h["row_off"][-1]), int(0.25 * seconds / per_row)))
    return {"value": rows_total / secs, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{rows_total} verified rows of the same workload (requests in order, truncated "
                      f"to fit), {secs:.1f} s of single-thread float64 CPU time"}


# ------------------------------------------------------------------ our arm

def run_ours(args):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    dev = torch.device("cuda", local)
    from speculative_decoding_verification_43_gb300 import api

    wl = W.WORKLOADS[WORKLOAD]
    seed = 0
    sets = [W.make_round(wl, seed=seed, rnd=r + 1000 * rank, device=dev) for r in range(args.input_sets)]
    rows = sets[0].T
    logit_bytes = wl.bytes_per_round(seed)
    verifiers, compactors = [], []
    for rd in sets:
        v = api.Verifier(rd.B, rd.target.shape[1], rd.T, rd.target.dtype, K_max=8, device=dev)
        v.bind(rd.target, rd.draft, rd.row_off, rd.draft_tokens, rd.uniforms, rd.temperature)
        ci = W.make_compaction_inputs(rd, wl.prefix_len, wl.page_size)
        c = api.Compactor(rd.B, rd.T, device=dev)
        c.bind(rd.row_off, v.out.accept_len, v.out.n_emitted, v.out.out_tokens, v.out.req_status,
               ci["prefix_len"], ci["cand_kv_rows"], ci["block_table"], ci["page_size"])
        verifiers.append(v)
        compactors.append(c)
    gout = (torch.empty(1, dtype=torch.int32, device=dev), torch.empty(1, dtype=torch.float64, device=dev))
    stream = torch.cuda.current_stream(dev)

    def step(s):
        k = s % len(sets)
        v = verifiers[k]
        api.run_round(v, compactors[k], 0.5, GAMMA_COST, 0, 8, out=gout, stream=stream)

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize(dev)

    # per-launch events around the per-position kernel, on the stream it runs on, on every
    # KERNEL_SAMPLE-th timed step: an event between the per-position kernel and the round's tail
    # kernel makes the tail wait for the kernel to finish before it can start (no early launch),
    # so bracketing every step would slow the very steps being timed
    sampled = list(range(0, args.steps, KERNEL_SAMPLE))
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in sampled]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in sampled]
    for ev in ev_b + ev_e:
        ev.record(stream)  # torch creates the CUDA event on its first record
    torch.cuda.synchronize(dev)
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    t_begin.record(stream)
    for s in range(args.steps):
        v = verifiers[s % len(sets)]
        if s % KERNEL_SAMPLE == 0:
            v.time_rows_with(ev_b[s // KERNEL_SAMPLE], ev_e[s // KERNEL_SAMPLE])
        step(s)
        if s % KERNEL_SAMPLE == 0:
            v.time_rows_with(None, None)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    for v in verifiers:
        v.time_rows_with(None, None)
    ms_total = t_begin.elapsed_time(t_end)
    ms_total = max_over_ranks(ms_total, world, dev)
    ms_step = ms_total / args.steps
    rows_ms = statistics.fmean(b.elapsed_time(e) for b, e in zip(ev_b, ev_e))
    value = job_value(world, rows, args.steps, ms_total)

    # end to end through the public API, host buffers in, host results out
    e2e = run_e2e(args, sets, verifiers, compactors, gout, stream, dev, world) if args.e2e_steps > 0 else None

    if rank != 0:
        return
    peak, peak_kind = measured_peak()
    achieved = logit_bytes / (rows_ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded), no dataset or weights",
        "config": workload_config(wl, rows, logit_bytes),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": recorded_traffic(logit_bytes),
                     "kernel": kernel_label(wl, rows), "kernel_ms_avg": rows_ms,
                     "kernel_timing": f"CUDA events around the per-position kernel on every {KERNEL_SAMPLE}th "
                                      f"timed step ({len(sampled)} launches)",
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)",
                     "algorithmic_bytes_per_launch": logit_bytes},
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,  # the per-position kernel and the round's tail kernel
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(sets[0], args.cpu_seconds)
    print(json.dumps(line), flush=True)


def run_e2e(args, sets, verifiers, compactors, gout, stream, dev, world):
    """The same step through the public API with inputs in pinned host memory: each step copies
    its logits, tokens, uniforms and offsets to the device, runs the step, and copies the
    packed results back."""
    n = len(sets)
    host_in = []
    for rd in sets:
        host_in.append({k: getattr(rd, k).cpu().pin_memory() for k in
                        ("target", "draft", "row_off", "draft_tokens", "uniforms", "temperature")})
    outs = []
    for v, c in zip(verifiers, compactors):
        names = [(v.out, k) for k in ("accept_len", "n_emitted", "out_tokens", "req_status")] + \
                [(c.out, k) for k in ("out_off", "packed_tokens", "packed_pos", "kv_off", "kv_src", "kv_dst",
                                      "new_seq_len", "new_kv_len")]
        outs.append([(getattr(o, k), torch.empty_like(getattr(o, k), device="cpu").pin_memory()) for o, k in names])
    g_host = [torch.empty(1, dtype=torch.int32).pin_memory(), torch.empty(1, dtype=torch.float64).pin_memory()]
    h2d = sum(t.numel() * t.element_size() for t in host_in[0].values())
    d2h = sum(d.numel() * d.element_size() for d, _ in outs[0]) + 12

    from speculative_decoding_verification_43_gb300 import api

    def step(s):
        k = s % n
        rd = sets[k]
        for name, t in host_in[k].items():
            getattr(rd, name).copy_(t, non_blocking=True)
        api.run_round(verifiers[k], compactors[k], 0.5, GAMMA_COST, 0, 8, out=gout, stream=stream)
        for d, h in outs[k]:
            h.copy_(d, non_blocking=True)
        g_host[0].copy_(gout[0], non_blocking=True)
        g_host[1].copy_(gout[1], non_blocking=True)

    for s in range(5):
        step(s)
    torch.cuda.synchronize(dev)
    steps = args.e2e_steps
    b = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    barrier(world)
    b.record(stream)
    for s in range(steps):
        step(s)
    e.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(b.elapsed_time(e), world, dev)
    return {"value": world * sets[0].T * steps / (ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": ms / steps}


# ------------------------------------------------------------------ reference arm (the oracle)

def run_reference(args):
    world, rank, local = dist_env()
    if world > 1 and rank != 0:
        return  # rank 0 alone times the CPU oracle
    import oracle
    oracle.build()
    wl = W.WORKLOADS[WORKLOAD]
    rd = W.make_round(wl, seed=0, rnd=0, device="cpu")
    h = _host_round(rd)
    logit_bytes = wl.bytes_per_round(0)
    # size each step so that the whole run stays within about 90 s of CPU time
    r, s, cursor = time_oracle(h, 1, 0)
    per_row = s / r
    budget = 90.0 / max(1, args.steps + args.warmup)
    rows_budget = max(1, int(budget / per_row))
    for _ in range(args.warmup):
        _, _, cursor = time_oracle(h, rows_budget, cursor)
    rows_total, secs = 0, 0.0
    for _ in range(args.steps):
        r, s, cursor = time_oracle(h, rows_budget, cursor)
        rows_total += r
        secs += s
    value = rows_total / secs
    sample = (f"each step verifies {rows_budget} rows of the same workload (requests in order, truncated "
              f"to fit) with the single-thread float64 oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded), no dataset or weights",
        "config": workload_config(wl, rd.T, logit_bytes),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

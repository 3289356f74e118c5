#!/usr/bin/env python3
"""Throughput of the batched speculative-decoding verifier step on GB300.

One step = one pass of the whole hot path over one batch: one spec_verify_round call, which
enqueues the verifier's four kernels (per-chunk statistics of every row; per-request accept
decisions; pass 2 over the draft positions for alpha and the frontier's residual; per-item
finishing: draws, per-request selection, and in the CTA that completes the batch the
compaction and the gamma choice). Workload (synthetic, seeded): by default
"B=64 ragged K_i ~ U{0..7}, V=128256, bf16 Zipf logits, T=0.7"; --workload c4 or c5 selects
the larger configurations. Four input sets rotate between steps, together well above the
126 MB L2, so every step reads its logits from HBM.

Prints one JSON line:
  value       verified rows/s (sum_i (K_i+1) per step over the step time), whole job;
  roofline    the dominant kernel (spec_stats_kernel, the one pass that reads every target and
              draft logit) timed alone with CUDA events over 64 launches of its own after the
              step loop: algorithmic bytes (every logit once) over its mean duration, against
              the measured copy bandwidth; `verifier` gives the same for the four kernels;
  acceptance  mean accepted length and mean alpha of the timed inputs, and the band and
              mismatch counts of one full round checked against the float64 oracle;
  e2e         the same step through the public API from pinned host memory and back, with the
              next step's input copy and the previous step's result copy on two copy streams
              overlapping the current step's kernels;
  truncation  the cost of top-k 50 then top-p 0.9 on every request (SDCP "Session Model"):
              spec_verify calls with and without, timed whole;
  cpu_baseline the float64 oracle on this host: one thread, and all cores (OpenMP over
              requests).

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
WORKLOADS = ("c3", "c4", "c5")
GAMMA_COST = 0.05  # relative draft cost c used by the gamma controller each step
KERNEL_LAUNCHES = 64  # launches timed one by one for the dominant kernel and for the verifier
BAND = 1e-6  # a draw whose uniform lies this close to a decision boundary (oracle's side)
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "stats_kernel_{wl}_traffic.json")
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
    ap.add_argument("--workload", choices=WORKLOADS, default="c3")
    ap.add_argument("--input-sets", type=int, default=4)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--copy-streams", type=int, default=1, help="streams sharing each e2e input copy")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--truncation", type=int, default=1, help="also time top-k 50 / top-p 0.9 calls (1: yes)")
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


def recorded_traffic(wl_name):
    """DRAM bytes per launch of the statistics kernel from the committed ncu capture, if it was
    taken on this workload and on this kernel's code."""
    try:
        d = json.load(open(PROFILE_TRAFFIC.format(wl=wl_name)))
    except Exception:
        return None
    if d.get("kernel_src_sha256_16") != kernel_hash():
        return None
    return d.get("dram_bytes_per_launch")


def kernel_label(wl, rows):
    """The dominant kernel the library launches for this workload, and its grid."""
    from speculative_decoding_verification_43_gb300 import api
    plan = api.verify_plan(wl.B, wl.V, rows, wl.dtype)
    if plan is None:
        return "none"
    name, c, n = plan
    return f"{name}<{'bf16' if wl.dtype == torch.bfloat16 else 'f32'}>, {n} CTAs"


def workload_config(wl, rows, logit_bytes, sets):
    return {
        "workload": f"{wl.name}: {wl.note}",
        "B": wl.B, "V": wl.V, "input_dtype": "bf16" if wl.dtype == torch.bfloat16 else "f32",
        "rows_per_step": rows, "logit_bytes_per_step": logit_bytes,
        "step": f"spec_verify_round: spec_verify + spec_compact (P={wl.prefix_len}, page {wl.page_size}) + "
                "spec_choose_gamma in one call",
        "l2": (f"inputs larger than L2: {sets} rotating input sets of {logit_bytes / 1e6:.0f} MB of logits each "
               "(L2 126 MB)") if sets > 1 else "not applicable (host CPU)",
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


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_full_round(h, threads):
    """The oracle on every request of one round (OpenMP over requests); (result, seconds)."""
    import oracle
    t0 = time.perf_counter()
    o = oracle.verify(h["target"], h["draft"], h["row_off"], h["toks"], h["u"], h["temp"], threads=threads)
    return o, time.perf_counter() - t0


def check_counts(h, orc, gpu):
    """One round's tokens against the oracle: requests inside the band (judged on the oracle's
    margins alone), mismatches outside it, and alpha's largest relative error (rows >= 1e-6)."""
    ro = h["row_off"]
    near = mism = 0
    for i in range(len(ro) - 1):
        r0, r1 = int(ro[i]), int(ro[i + 1])
        K, d0 = r1 - r0 - 1, r0 - i
        walked = range(min(int(orc["accept_len"][i]) + 1, K))
        in_band = float(h["temp"][i]) > 0 and orc["req_status"][i] == 0 and (
            any(abs(orc["accept_margin"][d0 + j]) < BAND for j in walked) or orc["sample_margin"][i] < BAND)
        same = (orc["req_status"][i] == gpu["req_status"][i] and orc["accept_len"][i] == gpu["accept_len"][i]
                and orc["n_emitted"][i] == gpu["n_emitted"][i]
                and np.array_equal(orc["out_tokens"][r0:r1], gpu["out_tokens"][r0:r1]))
        if in_band:
            near += 1
        elif not same:
            mism += 1
    a_o = orc["alpha"]
    big = np.isfinite(a_o) & (a_o >= 1e-6)
    rel = np.abs(gpu["alpha_rows"][big].astype(np.float64) - a_o[big]) / a_o[big]
    return {"requests": len(ro) - 1, "compared": len(ro) - 1 - near, "near_boundary": near, "mismatches": mism,
            "alpha_max_rel": float(rel.max()) if rel.size else 0.0,
            "oracle_mean_alpha": float(np.nanmean(a_o)) if a_o.size else None}


def cpu_baseline(rd, seconds, gpu_out=None):
    """The oracle as it stands (C, float64) on this host, on bounded samples of the workload:
    one leg single-threaded, one on all cores (OpenMP over requests; reported as `value`). The
    all-cores leg's first call is a full round, which also checks the GPU's outputs of it."""
    import oracle
    oracle.build()
    h = _host_round(rd)
    # single thread: requests in order, truncated to fit, about half the time
    rows_1, secs_1, cursor, rows_budget = 0, 0.0, 0, 1
    while secs_1 < seconds / 2:
        r, s, cursor = time_oracle(h, rows_budget, cursor)
        rows_1 += r
        secs_1 += s
        rows_budget = max(1, min(int(h["row_off"][-1]), int(0.25 * seconds / (s / r))))
    # all cores: full rounds
    cores = host_cores()
    rows_n, secs_n, calls, used, check = 0, 0.0, 0, 1, None
    while secs_n < seconds / 2 or calls == 0:
        o, s = oracle_full_round(h, cores)
        used = o["threads_used"]
        if check is None and gpu_out is not None:
            check = check_counts(h, o, gpu_out)
        rows_n += int(h["row_off"][-1])
        secs_n += s
        calls += 1
    return {"value": rows_n / secs_n, "unit": UNIT, "cores": used, "kind": "oracle",
            "host_cores": cores,
            "sample": f"{calls} full rounds ({rows_n} verified rows) of the same workload on {used} OpenMP threads "
                      f"(requests split across them), {secs_n:.1f} s",
            "single_thread": {"value": rows_1 / secs_1, "unit": UNIT, "cores": 1,
                              "sample": f"{rows_1} verified rows (requests in order, truncated to fit), "
                                        f"{secs_1:.1f} s of one thread"}}, check


# ------------------------------------------------------------------ our arm

def time_kernels(verifiers, stream, n):
    """The verifier's kernels timed launch by launch with CUDA events on their own stream,
    outside the step loop: n launches of spec_verify with events around all four kernels, then
    n with events around the statistics kernel alone. Input sets rotate, so each launch reads
    logits that are not in L2. Returns ms lists (verifier, stats)."""
    def loop(stats_only):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for b, e in evs:  # torch creates the CUDA event on its first record
            b.record(stream)
            e.record(stream)
        torch.cuda.synchronize()
        for k in range(n):
            v = verifiers[k % len(verifiers)]
            b, e = evs[k]
            v.time_rows_with(b, None, e) if stats_only else v.time_rows_with(b, e)
            v.run(stream)
            v.time_rows_with(None, None)
        torch.cuda.synchronize()
        return [b.elapsed_time(e) for b, e in evs]
    for v in verifiers:  # warm the launch path with events attached
        v.time_rows_with(None, None)
        v.run(stream)
    return loop(False), loop(True)


def time_truncation(sets, stream, dev, n, top_k=50, top_p=0.9):
    """spec_verify with top-k then top-p on every request, against the same calls without: CUDA
    events around each whole call (the truncation kernel included), input sets rotating."""
    from speculative_decoding_verification_43_gb300 import api
    res = {}
    for label, trunc in (("plain", False), ("truncated", True)):
        vs = []
        for rd in sets:
            v = api.Verifier(rd.B, rd.target.shape[1], rd.T, rd.target.dtype, device=dev)
            kw = {}
            if trunc:
                kw = dict(top_k=torch.full((rd.B,), top_k, dtype=torch.int32, device=dev),
                          top_p=torch.full((rd.B,), top_p, dtype=torch.float32, device=dev))
            v.bind(rd.target, rd.draft, rd.row_off, rd.draft_tokens, rd.uniforms, rd.temperature, **kw)
            vs.append(v)
        for v in vs:
            v.run(stream)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize(dev)
        for k, (b, e) in enumerate(evs):
            b.record(stream)
            vs[k % len(vs)].run(stream)
            e.record(stream)
        torch.cuda.synchronize(dev)
        ms = [b.elapsed_time(e) for b, e in evs]
        res[label] = statistics.fmean(ms)
    return {"top_k": top_k, "top_p": top_p, "calls": n, "call_ms_mean": res["truncated"],
            "plain_call_ms_mean": res["plain"], "extra_us": 1e3 * (res["truncated"] - res["plain"]),
            "timing": "CUDA events around each spec_verify call (truncation kernel included)"}


def run_ours(args):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    dev = torch.device("cuda", local)
    from speculative_decoding_verification_43_gb300 import api

    wl = W.WORKLOADS[args.workload]
    seed = 0
    sets = [W.make_round(wl, seed=seed, rnd=r + 1000 * rank, device=dev) for r in range(args.input_sets)]
    rows = sets[0].T
    assert all(rd.T == rows for rd in sets)
    logit_bytes = wl.bytes_per_round(seed)
    K_max = max(int(np.max(rd.K)) for rd in sets)
    verifiers, compactors = [], []
    for rd in sets:
        v = api.Verifier(rd.B, rd.target.shape[1], rd.T, rd.target.dtype, K_max=max(K_max, 1), device=dev)
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
        api.run_round(verifiers[k], compactors[k], 0.5, GAMMA_COST, 0, 8, out=gout, stream=stream)

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize(dev)

    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    t_begin.record(stream)
    for s in range(args.steps):
        step(s)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    ms_total = t_begin.elapsed_time(t_end)
    ms_total = max_over_ranks(ms_total, world, dev)
    ms_step = ms_total / args.steps
    value = job_value(world, rows, args.steps, ms_total)

    # the statistics (dominant) kernel and the verifier, launch by launch
    ver_ms, stats_ms = time_kernels(verifiers, stream, KERNEL_LAUNCHES)
    trunc = time_truncation(sets, stream, dev, KERNEL_LAUNCHES) if args.truncation else None

    # acceptance of the timed inputs (set 0, as every step computed it)
    step(0)
    torch.cuda.synchronize(dev)
    o0 = verifiers[0].out
    gpu0 = {k: getattr(o0, k).cpu().numpy() for k in ("accept_len", "n_emitted", "out_tokens", "req_status",
                                                      "alpha_rows")}
    ok = gpu0["req_status"] == 0
    acceptance = {"mean_accept_len": float(gpu0["accept_len"][ok].mean()) if ok.any() else None,
                  "mean_alpha": float(o0.alpha_sum.item()) / max(int(o0.alpha_count.item()), 1),
                  "mean_emitted": float(gpu0["n_emitted"][ok].mean()) if ok.any() else None,
                  "round": "input set 0"}

    # end to end through the public API, host buffers in, host results out
    e2e = run_e2e(args, sets, verifiers, compactors, gout, stream, dev, world) if args.e2e_steps > 0 else None

    if rank != 0:
        return
    peak, peak_kind = measured_peak()

    def stat(ms):
        return {"mean_ms": statistics.fmean(ms), "median_ms": statistics.median(ms), "min_ms": min(ms),
                "max_ms": max(ms), "launches": len(ms)}
    st, vr = stat(stats_ms), stat(ver_ms)
    achieved = logit_bytes / (st["mean_ms"] / 1e3) / 1e9
    v_achieved = logit_bytes / (vr["mean_ms"] / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded), no dataset or weights",
        "config": workload_config(wl, rows, logit_bytes, len(sets)),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": recorded_traffic(wl.name),
                     "kernel": kernel_label(wl, rows), "kernel_ms_avg": st["mean_ms"],
                     "kernel_ms_median": st["median_ms"],
                     "kernel_timing": f"CUDA events on the launching stream around the statistics kernel alone, "
                                      f"{st['launches']} launches after the step loop (input sets rotating)",
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json), burst copy",
                     "algorithmic_bytes_per_launch": logit_bytes,
                     "algorithmic_bytes": "every target and draft logit once"},
        "verifier": {"kernels": 4, **vr, "achieved_gbs": v_achieved, "frac": v_achieved / peak,
                     "timing": "CUDA events around spec_verify's four kernels, launch by launch"},
        "acceptance": acceptance,
        "truncation": trunc,
        "e2e": e2e,
        "gpu_launches": 4 * args.steps,  # per step: statistics, decisions, pass 2, finishing
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"], check = cpu_baseline(sets[0], args.cpu_seconds, gpu0)
        acceptance.update(check or {})
    print(json.dumps(line), flush=True)


def run_e2e(args, sets, verifiers, compactors, gout, stream, dev, world):
    """The same step through the public API with inputs in pinned host memory: each step copies
    its logits, tokens, uniforms and offsets to the device, runs the step, and copies the
    packed results back. Copies run on two copy streams (host to device, device to host), so
    step s+1's inputs travel while step s computes; events order each input set's reuse."""
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
    g_host = [[torch.empty(1, dtype=torch.int32).pin_memory(), torch.empty(1, dtype=torch.float64).pin_memory()]
              for _ in range(n)]
    g_dev = [(torch.empty_like(gout[0]), torch.empty_like(gout[1])) for _ in range(n)]
    h2d = sum(t.numel() * t.element_size() for t in host_in[0].values())
    d2h = sum(d.numel() * d.element_size() for d, _ in outs[0]) + 12

    from speculative_decoding_verification_43_gb300 import api
    s_in = torch.cuda.Stream(dev)
    # the large input tensors are copied in args.copy_streams slices on streams of their own, so
    # that several copy engines share each step's host-to-device transfer
    s_sl = [torch.cuda.Stream(dev) for _ in range(max(1, args.copy_streams))]
    ev_sl = [[torch.cuda.Event() for _ in s_sl] for _ in range(n)]
    s_out = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(n)]     # set k's inputs are on the device
    ev_comp = [torch.cuda.Event() for _ in range(n)]   # set k's step has finished
    ev_out = [torch.cuda.Event() for _ in range(n)]    # set k's results are on the host
    for k in range(n):
        ev_out[k].record(s_out)

    def copy_in(s):
        k = s % n
        rd = sets[k]
        s_in.wait_event(ev_comp[k])  # the last step on set k no longer reads its inputs
        with torch.cuda.stream(s_in):
            for name, t in host_in[k].items():
                if name not in ("target", "draft"):
                    getattr(rd, name).copy_(t, non_blocking=True)
        for j, sj in enumerate(s_sl):
            sj.wait_event(ev_comp[k])
            with torch.cuda.stream(sj):
                for name in ("target", "draft"):
                    dst, src = getattr(rd, name), host_in[k][name]
                    rows = dst.shape[0]
                    r0, r1 = rows * j // len(s_sl), rows * (j + 1) // len(s_sl)
                    if r1 > r0:
                        dst[r0:r1].copy_(src[r0:r1], non_blocking=True)
            ev_sl[k][j].record(sj)
        for e in ev_sl[k]:
            s_in.wait_event(e)
        ev_in[k].record(s_in)

    def compute(s):
        k = s % n
        stream.wait_event(ev_in[k])
        stream.wait_event(ev_out[k])  # set k's previous results have been read out
        api.run_round(verifiers[k], compactors[k], 0.5, GAMMA_COST, 0, 8, out=g_dev[k], stream=stream)
        ev_comp[k].record(stream)
        s_out.wait_event(ev_comp[k])
        with torch.cuda.stream(s_out):
            for d, h in outs[k]:
                h.copy_(d, non_blocking=True)
            g_host[k][0].copy_(g_dev[k][0], non_blocking=True)
            g_host[k][1].copy_(g_dev[k][1], non_blocking=True)
        ev_out[k].record(s_out)

    def run(steps):
        copy_in(0)
        for s in range(steps):
            if s + 1 < steps:
                copy_in(s + 1)
            compute(s)
        # the end waits for the last results to reach the host
        stream.wait_event(ev_out[(steps - 1) % n])

    for k in range(n):
        ev_comp[k].record(stream)
    run(5)
    torch.cuda.synchronize(dev)
    steps = args.e2e_steps
    b = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    barrier(world)
    b.record(stream)
    s_in.wait_event(b)
    s_out.wait_event(b)
    for sj in s_sl:
        sj.wait_event(b)
    run(steps)
    e.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(b.elapsed_time(e), world, dev)
    return {"value": world * sets[0].T * steps / (ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": ms / steps, "copies_declared": True,
            "overlap": f"inputs of step s+1 copied while step s computes (logits in {len(s_sl)} slices on "
                       f"{len(s_sl)} streams); results copied back on another stream"}


# ------------------------------------------------------------------ reference arm (the oracle)

def run_reference(args):
    world, rank, local = dist_env()
    if world > 1 and rank != 0:
        return  # rank 0 alone times the CPU oracle
    import oracle
    oracle.build()
    wl = W.WORKLOADS[args.workload]
    rd = W.make_round(wl, seed=0, rnd=0, device="cpu")
    h = _host_round(rd)
    logit_bytes = wl.bytes_per_round(0)
    cores = host_cores()
    # size each step so that the whole run stays within about 90 s of CPU time
    _, s0 = oracle_full_round(h, cores)
    per_row = s0 / int(h["row_off"][-1])
    budget = 90.0 / max(1, args.steps + args.warmup)
    rows_budget = max(1, int(budget / per_row))
    used = 1

    def one(cursor):
        reqs, rows, cursor = plan_sample(h, rows_budget, cursor)
        a = oracle_rows(h, reqs)
        t0 = time.perf_counter()
        o = oracle.verify(*a, threads=cores)
        return rows, time.perf_counter() - t0, cursor, o["threads_used"]

    cursor = 0
    for _ in range(args.warmup):
        _, _, cursor, used = one(cursor)
    rows_total, secs = 0, 0.0
    for _ in range(args.steps):
        r, s, cursor, used = one(cursor)
        rows_total += r
        secs += s
    value = rows_total / secs
    sample = (f"each step verifies {rows_budget} rows of the same workload (requests in order, cycling, the "
              f"last truncated to fit) with the float64 oracle on {used} OpenMP threads (requests split "
              f"across them)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded), no dataset or weights",
        "config": workload_config(wl, rd.T, logit_bytes, 1),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle", "sample": sample,
                         "host_cores": cores},
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

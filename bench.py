"""Benchmark of the ZeRO-DP partitioned mixed-precision AdamW step on GB300.

One step = the whole hot path on one batch of synthetic gradients: the reduce-scatter
arithmetic of N simulated ranks' bf16 gradient copies (with unscale, overflow flag and
per-tile sums of squares), the global norm / clip / scaler kernel, and the fused AdamW +
bf16 cast into the gathered parameter layout.  Workload: the GPT-2-1.5B-shaped flat
buffer (psi = 1,557,611,200, N = 8, ZeRO-2), inputs resident in HBM; its 65 GB working
set is far larger than the 129 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

The same line carries the Llama-7B buffer (ZeRO-3, 51 gradient buckets) and the
1,000,003-parameter fp16 workload under `workloads`, each timed by the same code after the
previous workload's buffers are freed, and an end-to-end figure (`e2e`) through
zero_step_host with the gradient copies in pinned host memory.  --impl reference times the
CPU oracle (the build's own baseline) on bounded samples of the same workload on the host
cores.  Under torchrun (N > 1) the workload's ranks are spread over the N processes, one
GPU each, and exchange over torch.distributed (ranks.RankStep: the gradient copies window
by window, the norm's partials and overflow flag, the gathered parameters); the whole job
updates the workload's parameters once per step (strong scaling), and rank 0 prints one
JSON line with the maximum time over ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "params updated/s and achieved HBM GB/s (% of ~8 TB/s) for the fused shard step"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
ADAMW_BYTES = 30   # per parameter: g, master, m, v read (16); master, m, v, bf16 written (14)
L2_FLUSH_BELOW = 4 * 129e6   # working sets below this are timed with L2 flushed between steps
L2_FLUSH_BYTES = 512 << 20


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clocks, power and throttle reasons sampled during the timed region."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "clocks.mem,temperature.gpu")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.t_on = self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, on: bool):
        if on:
            self.t_on = time.time()
        else:
            self.t_off = time.time()

    def stop(self) -> dict:
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = [r for t, r in self.rows if self.t_on and self.t_on - 0.15 <= t <= (self.t_off or t) + 0.15]
        if not rows:
            rows = [r for _, r in self.rows]
        sm = [float(r[1]) for r in rows if len(r) > 8 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) > 8 and r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if len(r) > 8 and r[3].replace(".", "").isdigit()]
        mem = [float(r[9]) for r in rows if len(r) > 10 and r[9].replace(".", "").isdigit()]
        temp = [float(r[10]) for r in rows if len(r) > 10 and r[10].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows if len(r) > 8 for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "mem_mhz": statistics.median(mem) if mem else None,
                "temp_c_max": max(temp) if temp else None,
                "samples": len(rows), "reasons": reasons}


def cpu_oracle_baseline(steps: int = 1, psi_sample: int = 1 << 24, base=None):
    """Time the CPU oracle (as it stands, single-threaded) on a bounded sample of a
    workload (default the GPT-2 one): the same recipe at psi_sample parameters, N = 8;
    params/s."""
    import numpy as np

    import oracle
    import synth
    from synth import workloads as W

    base = W.C2 if base is None else base
    wl = base if psi_sample == base.psi else W.scaled(base, psi_sample, steps=steps)
    orc = oracle.load()
    lay = orc.partition(wl.psi, wl.n_ranks, wl.stage)
    P = lay.psi_padded
    hp = oracle.hparams(**wl.hp.__dict__)
    reps = [synth.fill_host(wl.grad_out, wl.grad_kind, wl.grad_key(1, k), 0, P, wl.psi,
                            wl.grad_sigma, wl.loss_scale) for k in range(wl.n_ranks)]
    st = [synth.fill_host(synth.OUT_F32, synth.NORMAL, wl.state_key(synth.ROLE_MASTER), 0, P,
                          wl.psi, wl.master_sigma)]
    if wl.random_moments:
        st += [synth.fill_host(synth.OUT_F32, kind, wl.state_key(role), 0, P, wl.psi, wl.mom_sigma)
               for role, kind in ((synth.ROLE_MOM, synth.NORMAL), (synth.ROLE_VAR, synth.NORMAL_SQ))]
    else:
        st += [np.zeros(P, np.float32), np.zeros(P, np.float32)]
    g = np.zeros(P, np.float32)
    out = np.zeros(P, np.uint16)
    sc = oracle.scaler(wl.loss_scale, wl.dynamic, wl.growth_interval)
    dt_ = oracle.F16 if wl.grad_dtype == "f16" else oracle.BF16
    t0 = time.perf_counter()
    for _ in range(steps):
        orc.step(lay, hp, dt_, reps, g, *st, out, sc)
    dt = time.perf_counter() - t0
    return wl.psi * steps / dt, dt, wl


def cpu_baseline_all_cores(base, psi_sample: int, seconds: float = 8.0) -> dict:
    """The oracle on every host core (oracle.parallel: fixed 2^20-element chunks on a
    pool of spawned processes, so the result does not depend on the core count), timed
    for about `seconds` on a psi_sample-parameter sample of the workload's recipe; plus
    the single-threaded oracle step on a smaller sample for comparison."""
    from oracle.parallel import ParallelOracle, host_cores
    from synth import workloads as W

    wl = base if psi_sample == base.psi else W.scaled(base, psi_sample)
    cores = host_cores()
    single_psi = min(1 << 22, base.psi)
    v1, dt1, _ = cpu_oracle_baseline(2, single_psi, base)
    single = {"value": v1, "unit": "params/s", "cores": 1,
              "sample": f"2 serial oracle steps at psi={single_psi}, {dt1:.1f} s"}
    try:
        with ParallelOracle(wl, cores) as par:
            one = par.time_steps(1)
            steps = max(2, min(200, int(seconds / max(one, 1e-3))))
            dt = par.time_steps(steps)
    except Exception as e:  # e.g. no room for the shared arrays: report the serial oracle
        return dict(single, kind="oracle", single_core=single,
                    note=f"the all-core oracle could not run here ({type(e).__name__}: {e}); "
                         "value is the serial oracle on one core")
    return {"value": wl.psi * steps / dt, "unit": "params/s", "cores": cores, "kind": "oracle",
            "sample": f"{steps} oracle steps of the {_recipe_name(base)} recipe at psi="
                      f"{wl.psi} (N={wl.n_ranks} {wl.grad_dtype} copies) on {cores} host "
                      f"processes (2^20-element chunks), {dt:.1f} s",
            "single_core": single}


def run_reference(args):
    from oracle.parallel import ParallelOracle, host_cores
    from synth import workloads as W

    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    base = _base_workload(args.workload)
    sample = min(1 << 24, base.psi)
    wl = base if sample == base.psi else W.scaled(base, sample)
    cores = host_cores()
    how = f"one oracle step on {cores} host processes (2^20-element chunks)"
    try:
        with ParallelOracle(wl, cores) as par:
            par.time_steps(args.warmup)
            total = par.time_steps(args.steps)
    except Exception as e:  # e.g. no room for the shared arrays: the serial oracle instead
        cores, total = 1, 0.0
        how = f"one serial oracle step on one core (the all-core oracle failed: {type(e).__name__})"
        for _ in range(args.warmup):
            cpu_oracle_baseline(1, sample, base)
        for _ in range(args.steps):
            total += cpu_oracle_baseline(1, sample, base)[1]
    value = sample * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "params/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": _config(base=base),
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: the {_recipe_name(base)} recipe at psi={sample} "
                                   f"(N={base.n_ranks} {base.grad_dtype} copies), {how}"},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _base_workload(name):
    from synth import workloads as W
    return {"gpt2-1.5b": W.C2, "llama-7b": W.C3, "c1": W.C1}[name]


def _recipe_name(base):
    from synth import workloads as W
    return {id(W.C2): "GPT-2-1.5B", id(W.C3): "Llama-7B", id(W.C1): "odd-size fp16"}[id(base)]


def _config(extra=None, psi=None, base=None):
    from synth import workloads as W
    base = W.C2 if base is None else base
    psi = base.psi if psi is None else psi
    if base is W.C3:
        name = ("Llama-7B-shaped flat buffer, psi=6,738,415,616, N=8 simulated ranks, ZeRO-3, "
                "gradients in 2^27-element buckets of 8 bf16 copies (51 buckets, each reduced "
                "by its own launch)")
    elif base is W.C1:
        name = ("odd-size fp16 buffer, psi=1,000,003 (last shard padded), N=4 simulated ranks, "
                "ZeRO-2, fp16 gradient copies fp16(N(0,1e-3)*1024), dynamic loss scale 1024, "
                "fp32 master ~N(0,0.02), m = v = 0")
    else:
        name = ("GPT-2-1.5B-shaped flat buffer, psi=1,557,611,200" if psi == W.C2.psi else
                f"GPT-2-1.5B recipe at a reduced psi={psi:,} (profiling case, not the headline)")
        name += ", N=8 simulated ranks, ZeRO-2"
    if base is not W.C1:
        name += ", bf16 gradient copies ~N(0,1e-4), fp32 master/m/v random-init"
    ws_bytes = (34 + 2 * base.n_ranks) * psi
    c = {"workload": name + ", AdamW lr 1e-3 betas 0.9/0.999 eps 1e-8 wd 0.01 clip 1.0",
         "psi": psi, "n_ranks": base.n_ranks, "stage": base.stage, "grad_dtype": base.grad_dtype,
         "l2": (f"inputs larger than L2 ({ws_bytes / 1e9:.1f} GB working set vs 129 MB L2); "
                "no flush needed") if ws_bytes > L2_FLUSH_BELOW else
               (f"L2 flushed before every step (a {L2_FLUSH_BYTES >> 20} MiB write, outside the "
                f"timed events): the {ws_bytes / 1e6:.0f} MB working set would otherwise stay "
                "in the 129 MB L2")}
    if base.bucket_elems:
        c["bucket_elems"] = base.bucket_elems
    if extra:
        c.update(extra)
    return c


def run_ours(args):
    import torch

    ws, rank, local = _dist()
    if ws > 1:
        return run_ranks(args)
    torch.cuda.set_device(local)
    base = _base_workload(args.workload)
    line = _measure_simulated(args, base, args.psi)
    torch.cuda.empty_cache()
    if not args.no_extra_workloads and args.psi is None and args.workload == "gpt2-1.5b":
        # the other two workloads the target names, timed by the same code on this GPU
        # (one at a time: the headline's buffers are freed first)
        line["workloads"] = {}
        for name, min_steps in (("llama-7b", 0), ("c1", 200)):
            sub = _measure_simulated(args, _base_workload(name), None, max(args.steps, min_steps))
            torch.cuda.empty_cache()
            line["workloads"][name] = {k: sub[k] for k in (
                "value", "unit", "steps", "ms_per_step", "ms_per_step_spread", "config", "hbm",
                "roofline", "kernels", "launches_per_step", "gpu_launches", "clocks", "e2e",
                "final_state")}
        line["gpu_launches_all_workloads"] = line["gpu_launches"] + sum(
            w["gpu_launches"] for w in line["workloads"].values())
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_all_cores(base, min(1 << 26, base.psi))
    print(json.dumps(line), flush=True)
    return 0


def _measure_simulated(args, base, psi=None, steps=None):
    """Time the step of one workload, all N ranks simulated on this GPU (zero_step, inputs
    resident in HBM); returns the JSON line without its cpu_baseline.  Every buffer it
    allocates is released when it returns."""
    import torch

    import synth
    import zero_partitioned_optimizer_shard_gb300 as z
    from synth import workloads as W

    steps = args.steps if steps is None else steps
    dev = torch.device("cuda", torch.cuda.current_device())
    wl = base if psi in (None, base.psi) else W.scaled(base, psi)
    gdt = z.ZERO_F16 if wl.grad_dtype == "f16" else z.ZERO_BF16
    lay = z.zero_partition(wl.psi, wl.n_ranks, wl.stage, 1, wl.bucket_elems)
    P, N = lay.psi_padded, lay.n_ranks
    Wb, nb = lay.bucket_elems, lay.n_buckets
    hp = z.hparams(**wl.hp.__dict__)
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream

    reps = [torch.empty(P, dtype=torch.int16, device=dev) for _ in range(N)]
    for k, r in enumerate(reps):
        synth.fill_dev(r.data_ptr(), wl.grad_out, wl.grad_kind, wl.grad_key(1, k), 0, P, wl.psi,
                       wl.grad_sigma, wl.loss_scale, s)
    master = torch.empty(P, dtype=torch.float32, device=dev)
    m = torch.zeros(P, dtype=torch.float32, device=dev)
    v = torch.zeros(P, dtype=torch.float32, device=dev)
    fills = [(master, synth.ROLE_MASTER, synth.NORMAL, wl.master_sigma)]
    if wl.random_moments:
        fills += [(m, synth.ROLE_MOM, synth.NORMAL, wl.mom_sigma),
                  (v, synth.ROLE_VAR, synth.NORMAL_SQ, wl.mom_sigma)]
    for t_, role, kind, sig in fills:
        synth.fill_dev(t_.data_ptr(), synth.OUT_F32, kind, wl.state_key(role), 0, P, wl.psi, sig,
                       1.0, s)
    g = torch.empty(P, dtype=torch.float32, device=dev)
    out = torch.empty(P, dtype=torch.int16, device=dev)
    partials = torch.empty(lay.n_tiles, dtype=torch.float64, device=dev)
    st = torch.empty(z.STATE_BYTES, dtype=torch.uint8, device=dev)
    z.zero_step_state_init(lay, wl.loss_scale, wl.dynamic, wl.growth_interval, st, partials, stream)
    rep_ptrs = [r.data_ptr() for r in reps]
    flush = None
    if (34 + 2 * N) * P <= L2_FLUSH_BELOW:
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    # one window per bucket: every bucket's N copies stay resident, each reduced by its own
    # launch (a single window over the whole buffer when the workload is not bucketed)
    windows = [(b * Wb, min(Wb, P - b * Wb), [p + 2 * b * Wb for p in rep_ptrs]) for b in range(nb)]

    bucket_ptrs = [p for _, _, ptrs in windows for p in ptrs]
    launches = z.zero_step_launches(lay, gdt)  # 1: the single-launch step; else nb + 2

    def step():  # the public call: zero_step over every bucket, the norm and AdamW
        z.zero_step(lay, hp, gdt, bucket_ptrs, g, partials, master, m, v, out, st, stream)

    def step_split(ev):  # the same launches one by one, with an event after each part
        for begin, count, ptrs in windows:
            z.zero_reduce_shard_unscale(lay, gdt, ptrs, begin, count, g, partials, st, stream)
        ev[1].record(stream)
        z.zero_grad_norm(lay, hp, partials, st, stream)
        ev[2].record(stream)
        z.zero_adamw_cast_gather(lay, hp, g, master, m, v, out, st, stream)
        ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(dev.index)
    clocks.start()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    torch.cuda.synchronize(dev)
    clocks.mark(True)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(steps):
        if flush is not None:
            flush.fill_(float(i))  # evicts the step's working set from L2; not timed
            evs[i][0].record(stream)
        step()
        if flush is not None:
            evs[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark(False)
    elapsed_ms = t_start.elapsed_time(t_end)
    if flush is not None:  # the flushes between steps are not part of the step
        elapsed_ms = sum(e[0].elapsed_time(e[1]) for e in evs)
    clk = clocks.stop()

    # --- per-kernel breakdown: the same launches made one by one, an event after each --
    n_split = min(steps, 20)
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_split)]
    for i in range(n_split):
        if flush is not None:
            flush.fill_(float(i))
        sev[i][0].record(stream)
        step_split(sev[i])
    torch.cuda.synchronize(dev)
    reduce_ms = [e[0].elapsed_time(e[1]) for e in sev]
    norm_ms = [e[1].elapsed_time(e[2]) for e in sev]
    adamw_ms = [e[2].elapsed_time(e[3]) for e in sev]
    stt = z.zero_step_state_read(st, stream)
    assert stt.t == args.warmup + steps + n_split and stt.skip == 0 and stt.norm == stt.norm
    assert stt.error == 0

    # --- end to end through zero_step_host: gradients from pinned host memory -----------
    e2e = None
    if nb > 1:
        e2e = {"value": None, "unit": "params/s", "h2d_bytes_per_step": N * P * 2,
               "d2h_bytes_per_step": z.STATE_BYTES,
               "note": "not measured for the bucketed buffer: its gradient copies "
                       f"({N * P * 2 / 1e9:.0f} GB) would all have to be pinned in host memory"}
    elif not args.no_e2e:
        e2e = _e2e(args, z, torch, dev, wl, hp, reps, g, partials, master, m, v, out, st, stream)

    peak, peak_kind = _peaks()
    ms = elapsed_ms / steps
    if flush is not None:
        per_step = sorted(e[0].elapsed_time(e[1]) for e in evs)
        spread = {"p10": _pct(per_step, 10), "p50": _pct(per_step, 50), "p90": _pct(per_step, 90),
                  "from": "the timed steps (an event on each side of every step)"}
    else:
        # the timed steps run back to back (no event between them, so each launch overlaps
        # the previous kernel's tail); the spread comes from the breakdown steps, whose
        # events sit between the calls
        per_step = sorted(e[0].elapsed_time(e[3]) for e in sev)
        spread = {"p10": _pct(per_step, 10), "p50": _pct(per_step, 50), "p90": _pct(per_step, 90),
                  "from": f"the {n_split} breakdown steps (separate calls, events between them)"}
    params_per_s = wl.psi * steps / (elapsed_ms / 1e3)
    bytes_26 = (26 + 2 * N) * P
    moved = _fused_moved(N, lay, True) if launches == 1 else (34 + 2 * N)  # g re-read if split
    adamw_avg = statistics.mean(adamw_ms)
    reduce_avg = statistics.mean(reduce_ms)
    ach = ADAMW_BYTES * P / (adamw_avg / 1e3) / 1e9
    red_bytes = (2 * N + 4) * P
    if launches == 1:
        fused_bytes = (30 + 2 * N) * P
        ach_f = fused_bytes / (ms / 1e3) / 1e9
        roof = {"kernel": "k_step_fused (the whole step in one cooperative launch)",
                "bound": "hbm", "achieved": ach_f, "peak": peak, "unit": "GB/s",
                "frac": ach_f / peak, "peak_kind": peak_kind + ", burst figure of a kernel "
                "timed alone", "traffic": None, "bytes_per_launch": fused_bytes,
                "avg_launch_ms": ms,
                "note": "latency-bound size: one launch per step, timed as the step"}
    else:
        roof = {"kernel": "k_adamw (fused AdamW + bf16 cast + gathered write)",
                "bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                "peak_kind": peak_kind + ", burst figure of a kernel timed alone",
                "traffic": _traffic_from_profile(P), "bytes_per_launch": ADAMW_BYTES * P,
                "avg_launch_ms": adamw_avg}
    line = {
        "metric": METRIC, "value": params_per_s, "unit": "params/s", "n_gpus": 1,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms,
        "ms_per_step_spread": spread,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": _config({"parallelism": f"1 GPU, {N} simulated ranks"}, psi=wl.psi, base=base),
        "hbm": {
            "gbs_at_26p2n_bytes": bytes_26 / (ms / 1e3) / 1e9,
            "pct_of_8tbs": 100 * bytes_26 / (ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
            "pct_of_measured_peak": 100 * bytes_26 / (ms / 1e3) / 1e9 / peak,
            "bytes_per_param_moved": moved,
            "gbs_moved": moved * P / (ms / 1e3) / 1e9,
            "note": "(26+2N) B/param is the headline roofline; an exact step must also write "
                    "and re-read the fp32 gradient (34+2N) because clipping needs the global "
                    "norm before any update; the single-launch step of small layouts keeps g "
                    "on chip (30+2N: g is written for the caller but not read back; +2 with at "
                    "most one tile per SM, where the gathered parameters are read so that the "
                    "update made ahead of the norm can be undone)",
        },
        "roofline": roof,
        "kernels": {
            "timing": f"{n_split} extra steps made of the separate calls, an event after each",
            "k_reduce": {"avg_ms": reduce_avg, "bytes_per_launch": red_bytes,
                         "gbs": red_bytes / (reduce_avg / 1e3) / 1e9} if nb == 1 else
                        {"launches_per_step": nb, "avg_ms_all_buckets": reduce_avg,
                         "bytes_all_buckets": red_bytes,
                         "gbs": red_bytes / (reduce_avg / 1e3) / 1e9},
            "k_finalize": {"avg_ms": statistics.mean(norm_ms)},
            "k_adamw": {"avg_ms": adamw_avg, "bytes_per_launch": ADAMW_BYTES * P, "gbs": ach},
        },
        "launches_per_step": launches,
        "gpu_launches": launches * steps,
        "clocks": clk,
        "e2e": e2e,
        "final_state": {"t": stt.t, "norm": stt.norm, "clip_coef": stt.clip_coef},
    }
    return line


def run_ranks(args):
    """The step with its ranks spread over the processes of a torchrun job, one GPU each:
    the workload's N ranks in contiguous groups of N/G per process
    (zero_partitioned_optimizer_shard_gb300.ranks.RankStep), the gradient reduce-scatter,
    the norm's all-gather and the parameter all-gather over torch.distributed.  The
    whole job updates the workload's psi parameters per step, so the total work is fixed
    as G grows (strong scaling).  Rank 0 prints the line; times are the maximum over
    ranks."""
    import torch
    import torch.distributed as dist

    import synth
    import zero_partitioned_optimizer_shard_gb300 as z
    from synth import workloads as W
    from zero_partitioned_optimizer_shard_gb300.ranks import RankStep, layout_for

    ws, rank, local = _dist()
    torch.cuda.set_device(local % torch.cuda.device_count())
    dist.init_process_group(args.dist_backend)
    dev = torch.device("cuda", torch.cuda.current_device())
    base = _base_workload(args.workload)
    wl = base if args.psi in (None, base.psi) else W.scaled(base, args.psi)
    if wl.n_ranks % ws:
        raise SystemExit(f"{wl.n_ranks} ranks cannot be spread evenly over {ws} processes")
    # the gradient exchange goes in 2^24-element windows of every process's range (the next
    # windows' exchanges overlapping this window's reduce, constant-size receive buffers)
    lay = layout_for(wl.psi, wl.n_ranks, wl.stage, wl.bucket_elems)
    P, N = lay.psi_padded, lay.n_ranks
    gdt = z.ZERO_F16 if wl.grad_dtype == "f16" else z.ZERO_BF16
    rs = RankStep(lay, z.hparams(**wl.hp.__dict__), gdt, wl.loss_scale, wl.dynamic,
                  wl.growth_interval, dev, exchange_elems=1 << 24)
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream
    fills = [(rs.master, synth.ROLE_MASTER, synth.NORMAL, wl.master_sigma)]
    if wl.random_moments:
        fills += [(rs.m, synth.ROLE_MOM, synth.NORMAL, wl.mom_sigma),
                  (rs.v, synth.ROLE_VAR, synth.NORMAL_SQ, wl.mom_sigma)]
    for t_, role, kind, sig in fills:
        synth.fill_dev(t_.data_ptr(), synth.OUT_F32, kind, wl.state_key(role), rs.origin,
                       rs.local_len, wl.psi, sig, 1.0, s)
    copies = [torch.empty(P, dtype=torch.int16, device=dev) for _ in range(rs.rank_count)]
    for j, c in enumerate(copies):
        synth.fill_dev(c.data_ptr(), wl.grad_out, wl.grad_kind, wl.grad_key(1, rs.rank_begin + j),
                       0, P, wl.psi, wl.grad_sigma, wl.loss_scale, s)
    for _ in range(args.warmup):
        rs.step(copies)
    torch.cuda.synchronize(dev)
    dist.barrier()
    clocks = ClockSampler(dev.index)
    clocks.start()
    torch.cuda.synchronize(dev)
    clocks.mark(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        rs.step(copies)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark(False)
    clk = clocks.stop()
    elapsed = torch.tensor([e0.elapsed_time(e1)], dtype=torch.float64, device=dev)
    dist.all_reduce(elapsed, op=dist.ReduceOp.MAX)
    elapsed_ms = float(elapsed.item())

    # per-part breakdown: more steps with an event after each part (max over ranks)
    names = ["gradients", "norm inputs", "norm", "adamw", "parameters"]
    n_split = min(args.steps, 10)
    parts = {n: [] for n in names}
    for _ in range(n_split):
        evs = {"start": torch.cuda.Event(enable_timing=True)}
        evs["start"].record(stream)

        def mark(name):
            evs[name] = torch.cuda.Event(enable_timing=True)
            evs[name].record(stream)
        rs.step(copies, mark)
        torch.cuda.synchronize(dev)
        prev = "start"
        for n in names:
            parts[n].append(evs[prev].elapsed_time(evs[n]))
            prev = n
    avg = torch.tensor([statistics.mean(parts[n]) for n in names], dtype=torch.float64, device=dev)
    dist.all_reduce(avg, op=dist.ReduceOp.MAX)
    avg = dict(zip(names, avg.tolist()))
    stt = z.zero_step_state_read(rs.st)
    assert stt.error == 0 and stt.skip == 0 and stt.t == args.warmup + args.steps + n_split

    # end to end: every step copies this process's gradient copies in from pinned host
    # memory and reads the step state back
    e2e = None
    if not args.no_e2e:
        hcopies = [torch.empty(P, dtype=torch.int16, pin_memory=True) for _ in copies]
        for h, c in zip(hcopies, copies):
            h.copy_(c)
        hstate = torch.empty(z.STATE_BYTES, dtype=torch.uint8, pin_memory=True)
        n_e2e = max(1, args.e2e_steps)
        dist.barrier()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            for h, c in zip(hcopies, copies):
                c.copy_(h, non_blocking=True)
            rs.step(copies)
            hstate.copy_(rs.st, non_blocking=True)
            torch.cuda.synchronize(dev)
        dt = torch.tensor([time.perf_counter() - t0], dtype=torch.float64, device=dev)
        dist.all_reduce(dt, op=dist.ReduceOp.MAX)
        e2e = {"value": wl.psi * n_e2e / float(dt.item()), "unit": "params/s",
               "h2d_bytes_per_step": ws * len(copies) * P * 2,
               "d2h_bytes_per_step": ws * z.STATE_BYTES, "steps": n_e2e,
               "ms_per_step": float(dt.item()) / n_e2e * 1e3,
               "path": "every process: its gradient copies from pinned host memory, RankStep "
                       "(gradient windows exchanged while the previous ones are reduced, norm "
                       "exchange, norm, local AdamW, parameter all-gather), step state read back"}
    peak, peak_kind = _peaks()
    ms = elapsed_ms / args.steps
    L = rs.local_len
    ach = ADAMW_BYTES * L / (avg["adamw"] / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": wl.psi * args.steps / (elapsed_ms / 1e3), "unit": "params/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": _config({"parallelism": f"{ws} GPUs x {rs.rank_count} of the {N} ZeRO ranks "
                                          f"each ({args.dist_backend}: the 16-bit gradient "
                                          "copies exchanged window by window, all-gather of tile "
                                          "partials and parameters, max of the overflow flag)",
                           "exchange_window_elems": 1 << 24},
                          psi=wl.psi, base=base),
        "roofline": {"kernel": "k_adamw on this process's ranks (zero_adamw_cast_gather_local)",
                     "bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
                     "frac": ach / peak, "peak_kind": peak_kind, "traffic": None,
                     "bytes_per_launch": ADAMW_BYTES * L, "avg_launch_ms": avg["adamw"]},
        "parts_ms": avg,
        "launches_per_step": len(rs.windows()) + 2,
        "gpu_launches": (len(rs.windows()) + 2) * args.steps,
        "clocks": clk, "e2e": e2e,
        "final_state": {"t": stt.t, "norm": stt.norm, "clip_coef": stt.clip_coef},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    dist.barrier()
    dist.destroy_process_group()
    return 0


def _pct(sorted_vals, q):  # nearest-rank percentile
    return sorted_vals[min(len(sorted_vals) - 1, max(0, round(q / 100 * len(sorted_vals)) - 1))]


def _fused_moved(N: int, lay, g_written: bool) -> int:
    """Bytes per parameter the single-launch step moves: the copies, master/m/v both ways
    and the gathered parameters (26 + 2N), g when written (+4), and with at most one tile
    per SM (the staged shape) the gathered parameters as found (+2)."""
    import torch
    staged = lay.n_tiles <= torch.cuda.get_device_properties(0).multi_processor_count
    return 26 + 2 * N + (4 if g_written else 0) + (2 if staged else 0)


def kernel_code_hash(paths) -> str:
    """sha256 of C++/CUDA sources with their comments and whitespace runs removed: it
    changes when the code changes, not when a comment is edited."""
    import hashlib
    import re
    h = hashlib.sha256()
    for path in paths:
        with open(path) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()


def _traffic_from_profile(psi_padded):
    """DRAM bytes per k_adamw launch over psi_padded parameters from the committed ncu
    captures: a line slope * psi + intercept through three sizes (the intercept is the
    fixed amount of the launch's last writes still in L2 when it ends), or None when the
    kernel's code has changed since those counters were taken."""
    path = os.path.join(ROOT, "profiles", "k_adamw_traffic.json")
    csrc = os.path.join(ROOT, "zero_partitioned_optimizer_shard_gb300", "csrc")
    try:
        with open(path) as f:
            rec = json.load(f)
        sha = kernel_code_hash([os.path.join(csrc, n) for n in ("adamw.cu", "adamw_elem.cuh")])
        if not sha.startswith(rec["source_sha256_prefix"]):
            return None
        return round(rec["slope_bytes_per_param"] * psi_padded + rec["intercept_bytes"])
    except Exception:
        return None


def _e2e(args, z, torch, dev, wl, hp, reps, g, partials, master, m, v, out, st, stream):
    P, N = reps[0].numel(), len(reps)
    need = N * P * 2
    try:
        avail = int([l for l in open("/proc/meminfo") if l.startswith("MemAvailable")][0].split()[1]) * 1024
    except Exception:
        avail = 0
    if avail < 2 * need:
        return {"value": None, "unit": "params/s", "h2d_bytes_per_step": need,
                "d2h_bytes_per_step": z.STATE_BYTES, "note": f"skipped: {avail/1e9:.0f} GB host RAM free"}
    W = 1 << 24  # 2^24-element buckets: 256 MB of copies per bucket keeps the pipeline short
    lay = z.zero_partition(wl.psi, wl.n_ranks, wl.stage, 1, W)
    hreps = [torch.empty(P, dtype=torch.int16, pin_memory=True) for _ in range(N)]
    for h, r in zip(hreps, reps):
        h.copy_(r)
    staging = torch.empty(2 * N * W, dtype=torch.int16, device=dev)
    gdt = z.ZERO_F16 if wl.grad_dtype == "f16" else z.ZERO_BF16
    hstate = torch.empty(z.STATE_BYTES, dtype=torch.uint8, pin_memory=True)
    cs = torch.cuda.Stream(dev)
    z.zero_step_host(lay, hp, gdt, hreps, staging, staging.numel() * 2, g, partials,
                     master, m, v, out, st, hstate, stream, cs)
    torch.cuda.synchronize(dev)
    # at least --e2e-steps, and enough steps for ~50 ms of host-clock timing on small buffers
    t0 = time.perf_counter()
    z.zero_step_host(lay, hp, gdt, hreps, staging, staging.numel() * 2, g, partials,
                     master, m, v, out, st, hstate, stream, cs)
    stream.synchronize()
    one = time.perf_counter() - t0
    steps = max(1, args.e2e_steps, min(1000, int(0.05 / max(one, 1e-6))))
    t0 = time.perf_counter()
    for _ in range(steps):
        z.zero_step_host(lay, hp, gdt, hreps, staging, staging.numel() * 2, g, partials,
                         master, m, v, out, st, hstate, stream, cs)
        stream.synchronize()  # the step's result (norm, flag, scale) is on the host
    dt = time.perf_counter() - t0
    return {"value": wl.psi * steps / dt, "unit": "params/s", "h2d_bytes_per_step": need,
            "d2h_bytes_per_step": z.STATE_BYTES, "steps": steps, "ms_per_step": dt / steps * 1e3,
            "path": ("zero_step_host: N pinned host gradient copies read in place over the "
                     "CPU-GPU link by the single launch (reduce, norm and AdamW in one kernel); "
                     "step state copied back to pinned host memory"
                     if z.zero_step_launches(lay, gdt) == 1 else
                     "zero_step_host: N pinned host gradient copies -> 2 x 16M-element staging "
                     "ring (H2D on a copy stream, overlapped with the bucket reduces) -> norm -> "
                     "AdamW; step state copied back to pinned host memory")}


def run_sweep(args):
    """Bandwidth sweep (one JSON line per point): psi = 2^k and 2^k+1, N in {2,4,8,16,64},
    bf16 gradients ~N(0,1e-3).  Points whose N gradient copies do not fit beside the
    state run bucketed: 2^27-element windows, each read from one bucket buffer per rank
    (every window's copies are re-read from HBM; the buffers are far larger than L2)."""
    import torch

    import synth
    import zero_partitioned_optimizer_shard_gb300 as z
    from synth import workloads as W

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)  # a side stream: CUDA graphs cannot capture the default one
    torch.cuda.set_stream(stream)    # and graph.replay() launches on the current stream
    s_ = stream.cuda_stream
    ks = [int(k) for k in args.sweep_k.split(",")]
    ns = [int(n) for n in args.sweep_n.split(",")]
    free_total = torch.cuda.mem_get_info(dev)[1]
    for k in ks:
        for plus in (0, 1):
            for N in ns:
                for stage in ([1, 2, 3] if (k == ks[0] and plus == 0) else [2]):
                    psi = (1 << k) + plus
                    wl = W.sweep_point(psi, N, stage)
                    lay0 = z.zero_partition(psi, N, stage)
                    P = lay0.psi_padded
                    state_bytes = 18 * P + 8 * lay0.n_tiles
                    bucketed = N * P * 2 + state_bytes > 0.8 * free_total
                    W_ = 1 << 27 if bucketed else 0
                    lay = z.zero_partition(psi, N, stage, 1, W_)
                    rep_len = lay.bucket_elems
                    reps = [torch.empty(rep_len, dtype=torch.int16, device=dev) for _ in range(N)]
                    for kk, r in enumerate(reps):
                        synth.fill_dev(r.data_ptr(), wl.grad_out, wl.grad_kind, wl.grad_key(1, kk), 0,
                                       rep_len, psi, wl.grad_sigma, 1.0, s_)
                    bufs = {n: torch.empty(P, dtype=torch.float32, device=dev)
                            for n in ("g", "master", "m", "v")}
                    for t_, role, kind, sig in ((bufs["master"], synth.ROLE_MASTER, synth.NORMAL, 0.02),
                                                (bufs["m"], synth.ROLE_MOM, synth.NORMAL, 1e-4),
                                                (bufs["v"], synth.ROLE_VAR, synth.NORMAL_SQ, 1e-4)):
                        synth.fill_dev(t_.data_ptr(), synth.OUT_F32, kind, wl.state_key(role), 0, P,
                                       psi, sig, 1.0, s_)
                    out = torch.empty(P, dtype=torch.int16, device=dev)
                    partials = torch.empty(lay.n_tiles, dtype=torch.float64, device=dev)
                    st = torch.empty(z.STATE_BYTES, dtype=torch.uint8, device=dev)
                    z.zero_step_state_init(lay, 1.0, False, 1000, st, partials, stream)
                    ptrs = [reps[kk].data_ptr() for b in range(lay.n_buckets) for kk in range(N)]
                    hp = z.hparams()
                    # N = 2 with resident copies: re-read the copies in AdamW (26 + 4N = 34
                    # bytes per parameter) instead of writing and re-reading g (34 + 2N = 38)
                    reread = N == 2 and not bucketed and not args.sweep_materialise
                    g_arg = None if reread else bufs["g"]
                    moved = 26 + 4 * N if reread else 34 + 2 * N
                    launches = z.zero_step_launches(lay, z.ZERO_BF16)
                    if launches == 1:  # one launch, g kept on chip (written when given)
                        moved = _fused_moved(N, lay, not reread)

                    def step():
                        z.zero_step(lay, hp, z.ZERO_BF16, ptrs, g_arg, partials, bufs["master"],
                                    bufs["m"], bufs["v"], out, st, stream)

                    for _ in range(3):
                        step()
                    torch.cuda.synchronize(dev)
                    steps = max(3, min(200, int(2e9 / ((34 + 2 * N) * P)) + 1))
                    run = step
                    graph = None
                    if args.graph:  # replay the step's launches from a CUDA graph
                        graph = torch.cuda.CUDAGraph()
                        with torch.cuda.graph(graph, stream=stream):
                            step()
                        run = graph.replay
                        for _ in range(3):
                            run()
                        torch.cuda.synchronize(dev)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    for _ in range(steps):
                        run()
                    e1.record(stream)
                    torch.cuda.synchronize(dev)
                    ms = e0.elapsed_time(e1) / steps
                    print(json.dumps({
                        "sweep": True, "psi": psi, "n_ranks": N, "stage": stage,
                        "mode": "bucketed 2^27" if bucketed else "resident", "steps": steps,
                        "schedule": ("single launch, g not written" if reread else
                                     "single launch, g written") if launches == 1 else
                                    ("re-read copies" if reread else "materialise g"),
                        "launches_per_step": launches,
                        "launch": "cuda graph replay" if args.graph else "direct",
                        "ms_per_step": ms, "params_per_s": psi / (ms / 1e3),
                        "gbs_at_26p2n": (26 + 2 * N) * P / (ms / 1e3) / 1e9,
                        "bytes_moved_per_param": moved,
                        "gbs_moved": moved * P / (ms / 1e3) / 1e9,
                        "l2": "L2-resident regime" if moved * P < 129e6 else "HBM"}), flush=True)
                    del reps, bufs, out, partials, st, graph
                    torch.cuda.empty_cache()
    return 0


def run_overlap(args):
    """Gradient buckets arriving from a synthetic backward pass, reduced as they arrive.

    The Llama-7B-shaped buffer (psi = 6,738,415,616, N = 8, ZeRO-3) with its gradients in
    2^27-element buckets through a two-slot ring of constant-size buffers: a producer
    stream writes bucket b+1's N gradient copies (the seeded generator stands in for the
    backward pass) while the compute stream reduces bucket b; then the norm and AdamW.
    Reported: the overlapped step, the producer alone, the consumer alone (reduces of
    already-produced buckets + norm + AdamW), and the overlap efficiency
    hidden fraction of the reduces ((producer + consumer - overlapped) / reduces alone;
    AdamW cannot overlap: it needs every bucket's gradient first)."""
    import torch

    import synth
    import zero_partitioned_optimizer_shard_gb300 as z
    from synth import workloads as W

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = W.C3
    lay = z.zero_partition(wl.psi, wl.n_ranks, wl.stage, 1, wl.bucket_elems)
    P, N, Wb, nb = lay.psi_padded, lay.n_ranks, lay.bucket_elems, lay.n_buckets
    # the reduce runs on a high-priority stream; the producer (the synthetic backward)
    # leaves room on every SM (4 of the generator's blocks per SM) so the two can co-reside
    comp = torch.cuda.Stream(dev, priority=-1)
    prod = torch.cuda.Stream(dev)
    PRODUCER_BLOCKS_PER_SM = args.producer_blocks
    ring = [[torch.empty(Wb, dtype=torch.int16, device=dev) for _ in range(N)] for _ in range(2)]
    bufs = {n: torch.empty(P, dtype=torch.float32, device=dev) for n in ("g", "master", "m", "v")}
    for t_, role, kind, sig in ((bufs["master"], synth.ROLE_MASTER, synth.NORMAL, wl.master_sigma),
                                (bufs["m"], synth.ROLE_MOM, synth.NORMAL, wl.mom_sigma),
                                (bufs["v"], synth.ROLE_VAR, synth.NORMAL_SQ, wl.mom_sigma)):
        synth.fill_dev(t_.data_ptr(), synth.OUT_F32, kind, wl.state_key(role), 0, P, wl.psi, sig,
                       1.0, comp.cuda_stream)
    out = torch.empty(P, dtype=torch.int16, device=dev)
    partials = torch.empty(lay.n_tiles, dtype=torch.float64, device=dev)
    st = torch.empty(z.STATE_BYTES, dtype=torch.uint8, device=dev)
    z.zero_step_state_init(lay, 1.0, False, 1000, st, partials, comp)
    hp = z.hparams(**wl.hp.__dict__)
    filled = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def produce(step, b, slot, stream):
        begin, count = b * Wb, min(Wb, P - b * Wb)
        for k in range(N):
            synth.fill_dev(ring[slot][k].data_ptr(), wl.grad_out, wl.grad_kind, wl.grad_key(step, k),
                           begin, count, wl.psi, wl.grad_sigma, 1.0, stream.cuda_stream,
                           PRODUCER_BLOCKS_PER_SM)
        return begin, count

    def reduce(b, slot):
        begin, count = b * Wb, min(Wb, P - b * Wb)
        z.zero_reduce_shard_unscale(lay, z.ZERO_BF16, [r.data_ptr() for r in ring[slot]], begin, count,
                                    bufs["g"], partials, st, comp)

    def tail():
        z.zero_grad_norm(lay, hp, partials, st, comp)
        z.zero_adamw_cast_gather(lay, hp, bufs["g"], bufs["master"], bufs["m"], bufs["v"], out, st, comp)

    def overlapped(step):
        prod.wait_stream(comp)
        for b in range(nb):
            slot = b & 1
            if b >= 2:
                prod.wait_event(consumed[slot])
            produce(step, b, slot, prod)
            filled[slot].record(prod)
            comp.wait_event(filled[slot])
            reduce(b, slot)
            consumed[slot].record(comp)
        tail()

    def timed(fn, reps):
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        for r in range(reps):
            fn(r)
        e1.record(comp)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / reps

    reps = max(1, args.steps // 10)
    for w in range(args.warmup):
        overlapped(1 + w)
    t_over = timed(lambda r: overlapped(100 + r), reps)
    t_prod = timed(lambda r: [produce(200 + r, b, b & 1, comp) for b in range(nb)], reps)

    def consumer_only(r):  # the ring already holds data; reduce every bucket from it
        for b in range(nb):
            reduce(b, b & 1)
        tail()
    t_cons = timed(consumer_only, reps)

    def reduces_only(r):  # the part that can overlap: AdamW needs every bucket first
        for b in range(nb):
            reduce(b, b & 1)
        z.zero_grad_norm(lay, hp, partials, st, comp)
    t_red = timed(reduces_only, reps)
    line = {"overlap": True, "workload": wl.name, "buckets": nb, "bucket_elems": Wb,
            "ring_bytes": 2 * N * Wb * 2, "steps": reps,
            "ms_overlapped_step": t_over, "ms_producer_alone": t_prod, "ms_consumer_alone": t_cons,
            "ms_serial_sum": t_prod + t_cons,
            "ms_reduces_alone": t_red, "producer_blocks_per_sm": PRODUCER_BLOCKS_PER_SM,
            "hidden_fraction_of_reduces": (t_prod + t_cons - t_over) / t_red,
            "params_per_s_overlapped": wl.psi / (t_over / 1e3)}
    print(json.dumps(line), flush=True)
    return 0


def _link_bandwidth(torch, dev, nbytes=1 << 31):
    """Copy-engine bandwidth of the CPU-GPU link, measured here: pinned host -> HBM,
    HBM -> pinned host, and both at once on two streams (GB/s each way)."""
    h = [torch.empty(nbytes, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    d = [torch.empty(nbytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    s = [torch.cuda.Stream(dev) for _ in range(2)]
    e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]

    def one(dst, src, stream):
        with torch.cuda.stream(stream):
            dst.copy_(src, non_blocking=True)

    best = {"h2d": 0.0, "d2h": 0.0, "both_each": 0.0}
    for _ in range(3):
        torch.cuda.synchronize(dev)
        e[0].record(s[0]); one(d[0], h[0], s[0]); e[1].record(s[0])
        torch.cuda.synchronize(dev)
        best["h2d"] = max(best["h2d"], nbytes / e[0].elapsed_time(e[1]) / 1e6)
        e[0].record(s[0]); one(h[1], d[1], s[0]); e[1].record(s[0])
        torch.cuda.synchronize(dev)
        best["d2h"] = max(best["d2h"], nbytes / e[0].elapsed_time(e[1]) / 1e6)
        e[0].record(s[0])
        s[1].wait_event(e[0])
        one(d[0], h[0], s[0])
        one(h[1], d[1], s[1])
        e[1].record(s[0]); e[2].record(s[1])
        torch.cuda.synchronize(dev)
        ms = max(e[0].elapsed_time(e[1]), e[0].elapsed_time(e[2]))
        best["both_each"] = max(best["both_each"], nbytes / ms / 1e6)
    return best


def run_offload(args):
    """The GPT-2-1.5B step with the optimizer state offloaded to host memory.

    master, m and v (18.7 GB) live in page-locked Grace memory; the N gradient copies,
    g and the gathered parameters stay in HBM.  Per step: the reduce and the norm on the
    device, then zero_adamw_cast_gather_host_state, which reads and writes the state in
    place over NVLink-C2C (12 B per parameter each way).  Reported against the link's
    copy bandwidth measured in the same run."""
    import torch

    import synth
    import zero_partitioned_optimizer_shard_gb300 as z
    from synth import workloads as W

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    link = _link_bandwidth(torch, dev)
    wl = W.C2 if args.psi in (None, W.C2.psi) else W.scaled(W.C2, args.psi)
    lay = z.zero_partition(wl.psi, wl.n_ranks, wl.stage)
    P, N = lay.psi_padded, lay.n_ranks
    hp = z.hparams(**wl.hp.__dict__)
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream
    reps = [torch.empty(P, dtype=torch.int16, device=dev) for _ in range(N)]
    for k, r in enumerate(reps):
        synth.fill_dev(r.data_ptr(), wl.grad_out, wl.grad_kind, wl.grad_key(1, k), 0, P, wl.psi,
                       wl.grad_sigma, 1.0, s)
    g = torch.empty(P, dtype=torch.float32, device=dev)
    host = {}
    for name, role, kind, sig in (("master", synth.ROLE_MASTER, synth.NORMAL, wl.master_sigma),
                                  ("m", synth.ROLE_MOM, synth.NORMAL, wl.mom_sigma),
                                  ("v", synth.ROLE_VAR, synth.NORMAL_SQ, wl.mom_sigma)):
        synth.fill_dev(g.data_ptr(), synth.OUT_F32, kind, wl.state_key(role), 0, P, wl.psi, sig, 1.0, s)
        host[name] = torch.empty(P, dtype=torch.float32, pin_memory=True)
        host[name].copy_(g)
    out = torch.empty(P, dtype=torch.int16, device=dev)
    partials = torch.empty(lay.n_tiles, dtype=torch.float64, device=dev)
    st = torch.empty(z.STATE_BYTES, dtype=torch.uint8, device=dev)
    z.zero_step_state_init(lay, 1.0, False, 1000, st, partials, stream)
    ptrs = [r.data_ptr() for r in reps]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps + 1)]

    def step(e=None):
        z.zero_reduce_shard_unscale(lay, z.ZERO_BF16, ptrs, 0, P, g, partials, st, stream)
        z.zero_grad_norm(lay, hp, partials, st, stream)
        if e:
            e[1].record(stream)
        z.zero_adamw_cast_gather_host_state(lay, hp, g, host["master"], host["m"], host["v"], out,
                                            st, stream)
        if e:
            e[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(0)
    clocks.start()
    clocks.mark(True)
    ev[0][2].record(stream)
    for i in range(args.steps):
        step(ev[i + 1])
    torch.cuda.synchronize(dev)
    clocks.mark(False)
    clk = clocks.stop()
    total = ev[0][2].elapsed_time(ev[args.steps][2])
    adamw = [ev[i + 1][1].elapsed_time(ev[i + 1][2]) for i in range(args.steps)]
    stt = z.zero_step_state_read(st, stream)
    assert stt.t == args.warmup + args.steps and stt.skip == 0 and stt.error == 0
    a_ms = statistics.mean(adamw)
    link_gbs_each = 12 * P / (a_ms / 1e3) / 1e9
    line = {"offload": True, "workload": wl.name, "psi": wl.psi, "n_ranks": N,
            "state_in_host_memory_gb": 12 * P / 1e9, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total / args.steps, "params_per_s": wl.psi / (total / args.steps / 1e3),
            "ms_adamw_host_state": a_ms,
            "link_gbs_each_way": link_gbs_each,
            "link_copy_peak_gbs": link,
            "frac_of_copy_both_ways": link_gbs_each / link["both_each"],
            "clocks": clk}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="bandwidth sweep over psi and N (one JSON line per point)")
    ap.add_argument("--sweep-k", default="20,24,27,29,30,31")
    ap.add_argument("--sweep-materialise", action="store_true",
                    help="sweep: write and re-read g at N = 2 too (default: re-read the copies)")
    ap.add_argument("--graph", action="store_true", help="sweep: replay each step from a CUDA graph")
    ap.add_argument("--producer-blocks", type=int, default=2,
                    help="overlap: generator blocks per SM for the synthetic backward")
    ap.add_argument("--overlap", action="store_true",
                    help="bucket arrival overlapped with a synthetic backward producer "
                         "(Llama-7B buffer, 2^27-element buckets)")
    ap.add_argument("--offload", action="store_true",
                    help="optimizer state (master/m/v) in pinned host memory, updated over "
                         "the CPU-GPU link")
    ap.add_argument("--sweep-n", default="2,4,8,16,64")
    ap.add_argument("--workload", default="gpt2-1.5b", choices=["gpt2-1.5b", "llama-7b", "c1"],
                    help="gpt2-1.5b: psi=1,557,611,200, N=8, ZeRO-2 (the headline); llama-7b: "
                         "psi=6,738,415,616, N=8, ZeRO-3, 51 gradient buckets of 2^27 elements; "
                         "c1: psi=1,000,003, N=4, fp16 copies, dynamic loss scale (latency-bound, "
                         "L2 flushed before every step)")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="time only the headline workload (no llama-7b / c1 sub-lines)")
    ap.add_argument("--dist-backend", default="nccl", choices=["nccl", "gloo"],
                    help="under torchrun: the exchange's backend (gloo stages through host "
                         "memory; for checking the path where only one GPU is present)")
    ap.add_argument("--psi", type=int, default=None,
                    help="profiling only: the same recipe at another size (default: the "
                         "GPT-2-1.5B buffer)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.impl == "reference":
        return run_reference(args)
    import fcntl

    import __graft_entry__
    os.makedirs(os.path.join(ROOT, "_build"), exist_ok=True)
    with open(os.path.join(ROOT, "_build", ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)  # ranks of one node build once, in turn
        __graft_entry__.build()
        fcntl.flock(lock, fcntl.LOCK_UN)
    if args.sweep:
        return run_sweep(args)
    if args.overlap:
        return run_overlap(args)
    if args.offload:
        return run_offload(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

#!/usr/bin/env python
"""Benchmark of the verify step of MTP speculative decoding on GB300.

Headline workload (greedy k=1): hidden 2560, bf16 LM head of 151,936 rows, draft head over the
first 64,000 rows, 2 verify rows, batch 1. One STEP is one verify cycle -- the verify LM-head
GEMV over the k+1 rows plus acceptance, one launch (the greedy acceptance runs in the GEMV's
last block) -- on device-resident inputs (drafts produced by the draft head before the timed
region). Printed as one JSON line (rank 0):

  value        verify cycles/s over all ranks (replicas: every rank runs the same workload)
  roofline     the step's kernel: algorithmic bytes per launch / its average launch duration
               over the timed region (K launches back to back, the region's only kernel),
               against the measured HBM copy bandwidth; `isolated` beside it: the verify alone,
               3,000 launches each between CUDA events (no programmatic overlap), with the SM
               clock sampled over that loop
  step_two_kernels  the same step as two launches (verify, then the acceptance kernel)
  full_cycle   k draft-head steps + verify + acceptance: cycles/s and emitted tokens/s
  sweep        k = 1..7 at temperature 0, and at temperature 1 on the sampled workload's recipe
               (Philox seeds 0..99, EOS injected in 5% of cycles), 512 distinct cycles a point
  commit       snapshot commit and replay of the 64K-context state
  c3_cycle     the adaptive-rollback workload's verify cycle (k ~ U{1..7}: verify k+1 rows,
               acceptance, commit of the 64K-context state) timed end to end
  e2e          the same verify cycle through SpecVerifyEngine with host buffers (pinned H2D of the
               step's hidden rows and drafts, D2H of the 64-byte result) inside the timed region
  cpu_baseline the float64 oracle on the host cores, on a bounded sample

``--impl reference`` times the float64 oracle instead (the only other implementation of this
method here), on the same workload, metric and unit.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synth import configs, gen  # noqa: E402

METRIC = "verify cycles/s & emitted tok/s at k=1..7; LM-head HBM GB/s vs 8 TB/s"
# sources of the verify kernel: an ncu traffic figure holds only for the source it was taken on
GEMV_TC_SOURCES = ("gemv_tc.cu", "gemv_epilogue.cuh", "tcgen05.cuh", "common.cuh", "params.cuh")


def source_digest(names):
    """First 16 hex digits of the SHA-256 of the named kernel sources, concatenated."""
    import hashlib
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "mtp_speculative_decoding_spec_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(summary, section, sources):
    """DRAM bytes (read + written) of one launch from an ncu summary under profiles/: the
    ``- DRAM read:`` and ``- DRAM write:`` lines (Mbyte) of the first section whose heading
    contains ``section``, used only when the summary's ``source sha256:`` line names the
    current kernel sources. Returns (bytes or None, note)."""
    path = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(path):
        return None, "no ncu summary"
    text = open(path).read()
    digest = source_digest(sources)
    if f"source sha256: {digest}" not in text:
        return None, "kernel source changed since the ncu capture"
    part = text.split(section, 1)
    if len(part) < 2:
        return None, "section not in the ncu summary"
    vals = {}
    for line in part[1].splitlines():
        for key in ("DRAM read", "DRAM write"):
            if line.startswith(f"- {key}:") and key not in vals:
                x, unit = line.split(":", 1)[1].split()[:2]
                vals[key] = float(x) * {"Mbyte": 1e6, "Kbyte": 1e3, "Gbyte": 1e9,
                                        "byte": 1.0}[unit]
        if len(vals) == 2:
            break
    if len(vals) < 2:
        return None, "DRAM lines missing"
    return int(round(vals["DRAM read"] + vals["DRAM write"])), f"ncu, source {digest}"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--clocks-dir", default=None,
                    help="directory for the raw nvidia-smi clock samples (default: temp dir)")
    ap.add_argument("--profile", action="store_true",
                    help="few launches, no sweep/baseline: for ncu launch lists")
    return ap.parse_args()


def rank_reduce(x, op, device):
    """All-reduce one float over the ranks ("max" or "sum"); the identity on a single rank.
    The bench's only collective: timing and unit counts, never the data path."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def whole_job_value(units_per_rank, elapsed_max_s, world):
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return world * units_per_rank / elapsed_max_s


def rank_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def workload_config(cfg, extra=None):
    c = {"workload": f"{cfg.name}: d={cfg.d}, V={cfg.V} {cfg.wdtype} LM head, draft rows "
                     f"{cfg.Vd}, k={cfg.k}, {cfg.k + 1} verify rows, batch {cfg.batch}",
         "hidden": cfg.d, "vocab": cfg.V, "draft_rows": cfg.Vd, "k": cfg.k,
         "verify_rows": cfg.k + 1, "batch": cfg.batch, "temperature": cfg.temps[0],
         "l2": "inputs larger than L2 (778 MB of weights streamed per step); no flush"}
    if extra:
        c.update(extra)
    return c


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), d.get("bf16_tflops"), "measured"
    return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, csv_dir=None, tag=""):
        import tempfile
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(csv_dir or tempfile.gettempdir(),
                                 f"clocks{tag}_rank{gpu_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:  # no nvidia-smi: the line carries no clock record
            self.proc = None
            if getattr(self, "f", None) is not None:
                self.f.close()
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            lines = f.readlines()
        for line in lines:
            w = [x.strip() for x in line.split(",")]
            if len(w) < 9:
                continue
            try:
                sm.append(float(w[1]))
                smax.append(float(w[2]))
            except ValueError:
                continue
            for n, v in zip(names, w[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------- GPU arm
def build_inputs(cfg, W, n_pool, k, T, rng_seed):
    """Pool of cycle inputs: verify rows [n, k+1, d] and draft rows [n, k, d] (bf16 bits)."""
    H = np.empty((n_pool, k + 1, cfg.d), dtype=np.uint16)
    Hd = np.empty((n_pool, max(k, 1), cfg.d), dtype=np.uint16)
    for c in range(n_pool):
        inp = gen.cycle_inputs(cfg, W, c, seed=rng_seed, k=k)
        H[c] = inp["H"]
        if k:
            Hd[c, :k] = inp["Hd"]
    return H, Hd


def run_ours(args, rank, local_rank, world):
    import torch

    import mtp_speculative_decoding_spec_gb300 as spec
    from mtp_speculative_decoding_spec_gb300 import build as _build
    from mtp_speculative_decoding_spec_gb300.engine import SpecVerifyEngine

    _build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def max_over_ranks(x):
        return rank_reduce(x, "max", dev)

    def sum_over_ranks(x):
        return rank_reduce(x, "sum", dev)

    cfg = configs.get(1)
    W = gen.lm_weights(cfg)
    Wd = torch.from_numpy(W.view(np.int16)).to(dev)
    hbm_peak, tf_peak, peak_src = measured_peaks()
    n_pool = 16 if args.profile else 512
    k = cfg.k
    Hp, Hdp = build_inputs(cfg, W, n_pool, k, cfg.temps[0], rng_seed=100 + rank)
    Hp_d = torch.from_numpy(Hp.view(np.int16)).to(dev)
    Hdp_d = torch.from_numpy(Hdp.view(np.int16)).to(dev)

    eng = SpecVerifyEngine(Wd, spec.SPEC_BF16, cfg.V, cfg.d, cfg.Vd, 1, k + 1, k, cfg.eos_id,
                           device=dev, want_q_logits=False, fuse_greedy=True)
    eng.set_requests(temps=[0.0], seeds=[0], pos=[0], k=[k])
    # drafts of every pool entry, produced by the draft head on the GPU before timing
    drafts_pool = torch.zeros((n_pool, 1, k), dtype=torch.int32, device=dev)
    for c in range(n_pool):
        for i in range(1, k + 1):
            eng.draft_step(i, Hdp_d[c, i - 1:i])
        drafts_pool[c].copy_(eng.drafts[:, :k])
    torch.cuda.synchronize()

    def step(c):  # greedy verify + acceptance, fused into the LM-head kernel's last block
        spec.spec_verify_accept_greedy(Wd, spec.SPEC_BF16, cfg.V, cfg.d, Hp_d[c], 1, k + 1,
                                       eng.temps, eng.logits, eng.stats, k, eng.k,
                                       drafts_pool[c], cfg.eos_id, eng.out, eng.counters, eng.ws)

    def step_two_kernels(c):  # the same step as two launches: verify, then acceptance
        eng.verify(Hp_d[c])
        spec.spec_accept(1, k, eng.k, drafts_pool[c], eng.logits, eng.stats, cfg.V, k + 1,
                         None, None, cfg.Vd, cfg.Vd, eng.temps, cfg.eos_id, eng.seeds, eng.pos,
                         eng.out, eng.counters, eng.ws)

    K, Wm = args.steps, args.warmup
    stream = torch.cuda.current_stream()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank, args.clocks_dir)
    barrier()
    torch.cuda.synchronize()
    with clocks:
        # the warm-up steps run after the clock sampler has started (it idles the GPU for a
        # moment), right before the timed ones
        for c in range(Wm):
            step(c % n_pool)
        torch.cuda.synchronize()
        barrier()
        t_start.record(stream)
        for c in range(K):
            step(c % n_pool)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    elapsed = t_start.elapsed_time(t_end) / 1e3
    err = int(eng.ws[4:8].cpu().numpy().view(np.uint32)[0])
    cnt = eng.counters.cpu().numpy().view(spec.COUNTERS_DTYPE)[0]
    elapsed_max = max_over_ranks(elapsed)
    value = whole_job_value(K, elapsed_max, world)
    algo_bytes = cfg.V * cfg.d * 2 + (k + 1) * cfg.d * 2 + (k + 1) * 16
    roof = verify_launch_roofline(eng, Hp_d, n_pool, algo_bytes, hbm_peak, peak_src, local_rank,
                                  args.clocks_dir, 8 if args.profile else 3000)
    # The timed region holds K launches of the one kernel of the step, back to back: its
    # average launch duration is the region's time / K. The loop of launches each alone between
    # events (no programmatic overlap) is kept beside it.
    step_s = elapsed_max / K
    iso = {key: roof.pop(key) for key in ("achieved", "frac", "mean_launch_us",
                                          "median_launch_us", "launches_timed", "sm_mhz",
                                          "clock_samples")}
    iso["timing"] = "each launch alone between CUDA events, after 100 warm-up launches"
    roof.update({"kernel": "gemv_tc_kernel (verify, 2 rows; greedy acceptance in its last block)",
                 "achieved": round(algo_bytes / step_s / 1e9, 1),
                 "frac": round(algo_bytes / step_s / 1e9 / hbm_peak, 4),
                 "mean_launch_us": round(step_s * 1e6, 2), "launches_timed": K,
                 "timing": "the timed region: K launches of the step's only kernel, back to back",
                 "isolated": iso})
    roof["step_frac"] = roof["frac"]

    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "verify cycles/s",
        "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": round(elapsed_max / K * 1e3, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(cfg, {"parallelism": f"replicas x{world}",
                                        "step": "verify GEMV (2 rows) + greedy acceptance, "
                                                "fused into the GEMV's last block"}),
        "roofline": roof,
        "acceptance": round(float(cnt["accepted"]) / max(1.0, float(cnt["drafted"])), 4),
        "gpu_launches": K,
        "workspace_error": err,
    }
    # the same step as two launches (verify, then the acceptance kernel), timed the same way,
    # after the same warm-up (its acceptance kernel's first launch loads its code)
    for c in range(Wm):
        step_two_kernels(c % n_pool)
    torch.cuda.synchronize()
    t_start.record(stream)
    for c in range(K):
        step_two_kernels(c % n_pool)
    t_end.record(stream)
    torch.cuda.synchronize()
    e2k = max_over_ranks(t_start.elapsed_time(t_end) / 1e3)
    res["step_two_kernels"] = {"value": round(whole_job_value(K, e2k, world), 2),
                               "unit": "verify cycles/s", "ms_per_step": round(e2k / K * 1e3, 5)}
    cs = clocks.summary()
    res["clocks"] = cs

    if args.profile:
        profile_extras(dev, W, Wd)
    if not args.profile:
        # secondary figures: at least 500 cycles whatever --steps is (each reports its count)
        n_sec = min(max(K, 500), 2000)
        res["full_cycle"] = full_cycle(eng, cfg, Hp_d, Hdp_d, n_pool, k, n_sec, dev)
        res["e2e"] = e2e(eng, cfg, Hp, drafts_pool, n_pool, k, n_sec, dev, world,
                         max_over_ranks)
        if not args.no_sweep:
            res["sweep"] = sweep(dev, W, Wd, hbm_peak)
            step_us = elapsed_max / K * 1e6
            draft_us = max(1.0, 1e6 / res["full_cycle"]["cycles_s"] - step_us)
            res["adaptive"] = adaptive_bench(dev, W, Wd, step_us, draft_us)
            res["commit"] = commit_bench(dev, hbm_peak)
            res["c3_cycle"] = c3_cycle(dev, W, Wd, hbm_peak)
            res["q4"] = q4_bench(dev, W, hbm_peak)
            res["batched"] = batched_bench(dev, W, Wd, hbm_peak, tf_peak)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.profile:
        res["cpu_baseline"] = cpu_baseline(cfg, W, args.cpu_seconds)
    if world > 1:
        res["value_check"] = sum_over_ranks(K / elapsed)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def verify_launch_roofline(eng, Hp_d, n_pool, algo_bytes, hbm_peak, peak_src, gpu, clocks_dir,
                           n):
    """The verify kernel alone: n launches, each bracketed by CUDA events on the launch stream
    (events between kernels stop the programmatic overlap, so each launch runs by itself),
    after 100 warm-up launches, with the SM clock sampled over the loop (the `isolated` figure
    beside the timed region's own)."""
    import torch
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    with ClockSampler(gpu, clocks_dir, tag="roofline") as ck:
        for c in range(100):
            eng.verify(Hp_d[c % n_pool])
        for c in range(n):
            ev[c][0].record(stream)
            eng.verify(Hp_d[c % n_pool])
            ev[c][1].record(stream)
        torch.cuda.synchronize()
    us = [a.elapsed_time(b) * 1e3 for a, b in ev]
    mean_s = statistics.mean(us) / 1e6
    achieved = algo_bytes / mean_s / 1e9
    traffic, note = profiled_traffic("gemv_tc_kernel_verify_V151936_d2560.md", "## 2-row verify",
                                     GEMV_TC_SOURCES)
    cs = ck.summary()
    return {"bound": "hbm", "kernel": "gemv_tc_kernel (verify, 2 rows)",
            "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4), "peak_source": peak_src,
            "algorithmic_bytes_per_launch": algo_bytes,
            "mean_launch_us": round(mean_s * 1e6, 2),
            "median_launch_us": round(statistics.median(us), 2),
            "launches_timed": n, "traffic": traffic, "traffic_source": note,
            "sm_mhz": None if cs is None else cs["sm_mhz"],
            "clock_samples": None if cs is None else cs["samples"]}


def profile_extras(dev, W, Wd):
    """Launches for ncu captures after the greedy section: 5 sampled k=7 cycles (7 draft
    steps, an 8-row verify, acceptance with residual/bonus draws), 3 snapshot commits and 3
    replay commits of the 64K-context state, 5 batched 256-row verifies on the tensor
    cores (each followed by a 32-request acceptance), then the 4-bit head's section with 20
    steps (20 warm-up cycles, 20 verify + acceptance steps, 20 cycles)."""
    import torch

    import mtp_speculative_decoding_spec_gb300 as spec
    from mtp_speculative_decoding_spec_gb300.engine import SpecVerifyEngine
    cfg = configs.get(2)
    k = cfg.k
    Hp, Hdp = build_inputs(cfg, W, 5, k, 1.0, rng_seed=5)
    Hp_d = torch.from_numpy(Hp.view(np.int16)).to(dev)
    Hdp_d = torch.from_numpy(Hdp.view(np.int16)).to(dev)
    eng = SpecVerifyEngine(Wd, spec.SPEC_BF16, cfg.V, cfg.d, cfg.Vd, 1, k + 1, k, cfg.eos_id,
                           device=dev, want_q_logits=True)
    eng.set_requests(temps=[1.0], seeds=[3], pos=[0], k=[k])
    for c in range(5):
        eng.cycle(Hp_d[c], Hdp_d[c, :, None, :], k)
    torch.cuda.synchronize()
    hbm_peak, tf_peak, _ = measured_peaks()
    commit_bench(dev, hbm_peak, reps=3, warm=0)
    batched_bench(dev, W, Wd, hbm_peak, tf_peak, reps=2, with_commit=False)
    q4_bench(dev, W, hbm_peak, K=20)


def full_cycle(eng, cfg, Hp_d, Hdp_d, n_pool, k, K, dev):
    import torch
    for c in range(10):
        eng.cycle(Hp_d[c % n_pool], Hdp_d[c % n_pool, :, None, :], k)
    eng.counters.zero_()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for c in range(K):
        eng.cycle(Hp_d[c % n_pool], Hdp_d[c % n_pool, :, None, :], k)
    b.record()
    torch.cuda.synchronize()
    s = a.elapsed_time(b) / 1e3
    import mtp_speculative_decoding_spec_gb300 as spec
    cnt = eng.counters.cpu().numpy().view(spec.COUNTERS_DTYPE)[0]
    return {"cycles_s": round(K / s, 2), "emitted_tok_s": round(float(cnt["emitted"]) / s, 1),
            "tokens_per_cycle": round(float(cnt["emitted"]) / K, 4), "steps": K,
            "step": f"{k} draft-head step(s) + verify + acceptance"}


def e2e(eng, cfg, Hp, drafts_pool, n_pool, k, K, dev, world, max_over_ranks):
    """The headline step end to end through the C ABI from pinned host memory: each step moves
    its verify rows and drafts host -> device (one spec_copy_from_host of the cycle's packed
    inputs), runs the verify with the greedy acceptance fused into it, which writes its result
    straight into pinned host memory (spec_host_alias). Both transfers stay inside the chain of kernels,
    so the next kernel still starts in the previous one's tail (a cudaMemcpyAsync between them
    would end that overlap)."""
    import torch

    import mtp_speculative_decoding_spec_gb300 as spec
    hb = Hp[0].nbytes                                  # verify rows of a cycle
    db = drafts_pool[0].numel() * 4                    # its drafts (int32)
    xb = (hb + db + 15) // 16 * 16                     # packed and padded to 16 bytes
    X_np = np.zeros((n_pool, xb), dtype=np.uint8)
    X_np[:, :hb] = Hp.reshape(n_pool, -1).view(np.uint8)
    X_np[:, hb:hb + db] = drafts_pool.reshape(n_pool, -1).cpu().numpy().view(np.uint8)
    X_host = torch.from_numpy(X_np).pin_memory()
    out_host = torch.zeros((max(K, 10), spec.ACCEPT_OUT_BYTES), dtype=torch.uint8).pin_memory()
    out_alias = [spec.spec_host_alias(out_host[j]) for j in range(out_host.shape[0])]
    X_dev = torch.empty(xb, dtype=torch.uint8, device=dev)
    H_dev = X_dev[:hb].view(torch.int16).view(Hp.shape[1:])
    D_dev = X_dev[hb:hb + db].view(torch.int32).view(drafts_pool.shape[1:])

    def one(c, j):
        spec.spec_copy_from_host(X_dev, X_host[c], xb)
        spec.spec_verify_accept_greedy(eng.W, eng.wdt, cfg.V, cfg.d, H_dev, 1, k + 1, eng.temps,
                                       eng.logits, eng.stats, k, eng.k, D_dev, cfg.eos_id,
                                       out_alias[j], eng.counters, eng.ws)

    for c in range(10):
        one(c % n_pool, c)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for c in range(K):
        one(c % n_pool, c)
    torch.cuda.synchronize()
    s = max_over_ranks(time.perf_counter() - t0)
    return {"value": round(whole_job_value(K, s, world), 2), "unit": "verify cycles/s",
            "h2d_bytes_per_step": int(hb + db), "d2h_bytes_per_step": spec.ACCEPT_OUT_BYTES,
            "steps": K, "api": "spec_copy_from_host + spec_verify_accept_greedy (result into "
                               "pinned host memory)"}


def recipe_inputs(cfg, W, n_pool, k, T, rng_seed):
    """Pool of cycle inputs on the recipe of the workload ``cfg``: verify rows [n, k+1, d] and
    draft rows [n, k, d] (bf16 bits). At T > 0 the EOS id is injected at a random proposal
    position in cfg.eos_inject of the cycles (the verify row that checks that proposal, and the
    draft row derived from it, are planted on EOS). Also returns how many cycles carry EOS."""
    H = np.empty((n_pool, k + 1, cfg.d), dtype=np.uint16)
    Hd = np.empty((n_pool, max(k, 1), cfg.d), dtype=np.uint16)
    n_eos = 0
    for c in range(n_pool):
        e = gen.eos_injection(cfg, c, k, seed=rng_seed) if T > 0 else 0
        n_eos += e > 0
        inp = gen.cycle_inputs(cfg, W, c, seed=rng_seed, k=k, eos_at=e)
        H[c] = inp["H"]
        if k:
            Hd[c, :k] = inp["Hd"]
    return H, Hd, n_eos


def acceptance_rates(cnt, k):
    """accepted / drafted, and accepted / ratio tests: every draft tested is accepted or ends
    the chain, and a chain that did not reach depth k ended at a failed test unless it ended on
    an accepted EOS (cycles that ended on EOS are counted as having no failed test)."""
    acc, drafted = float(cnt["accepted"]), float(cnt["drafted"])
    fails = float(cnt["cycles"]) - float(cnt["depth"][k]) - float(cnt["eos"])
    return (round(acc / max(1.0, drafted), 4), round(acc / max(1.0, acc + max(0.0, fails)), 4))


def sweep(dev, W, Wd, hbm_peak):
    """k = 1..7 at temperature 0 (greedy) and at temperature 1 on the sampled workload's recipe
    (ratio rule with the draft head's q rows, Philox seeds 0..99 cycling over the cycles, EOS
    injected in 5% of the cycles); exact-match acceptance, and acceptance against the top-k 20 /
    top-p 0.95 filtered target (argmax drafts), at temperature 1 for k = 1, 3, 7. Each point
    runs 512 distinct cycles three times: with events around each verify and acceptance launch
    (their durations: lmhead_frac, accept_us), verify + acceptance back to back on the cycles'
    drafts (verify_cycles_s, verify_accept_frac) and whole cycles with their k draft steps
    (full_cycles_s, emitted_tok_s)."""
    import torch

    import mtp_speculative_decoding_spec_gb300 as spec
    from mtp_speculative_decoding_spec_gb300.engine import SpecVerifyEngine
    out = {}
    base = configs.get(2)
    n_pool = K = 512
    points = [(T, k, "ratio") for T in (0.0, 1.0) for k in range(1, 8)]
    points += [(1.0, k, mode) for mode in ("exact", "filtered") for k in (1, 3, 7)]
    seeds_pool = torch.arange(100, dtype=torch.int64, device=dev)
    pos_pool = torch.arange(n_pool, dtype=torch.int64, device=dev) * 16
    for T, k, mode in points:
        cfg = configs.Config(**{**base.__dict__, "k": k, "temps": (T,)})
        Hp, Hdp, n_eos = recipe_inputs(cfg, W, n_pool, k, T, rng_seed=7 * k + int(T))
        Hp_d = torch.from_numpy(Hp.view(np.int16)).to(dev)
        Hdp_d = torch.from_numpy(Hdp.view(np.int16)).to(dev)
        eng = SpecVerifyEngine(Wd, spec.SPEC_BF16, cfg.V, cfg.d, cfg.Vd, 1, k + 1, k,
                               cfg.eos_id, device=dev, want_q_logits=True,
                               acceptance=mode, fuse_greedy=True)
        eng.set_requests(temps=[T], seeds=[0], pos=[0], k=[k], top_k=[20], top_p=[0.95])
        # each cycle's drafts and draft rows (q), kept so that verify + acceptance can also be
        # timed on their own
        q_pool = torch.empty((n_pool, k, cfg.Vd), dtype=torch.float32, device=dev)
        qs_pool = torch.zeros((n_pool, k * spec.ROWSTATS_BYTES), dtype=torch.uint8, device=dev)
        d_pool = torch.zeros((n_pool, 1, k), dtype=torch.int32, device=dev)

        def use(c):
            cc = c % n_pool
            eng.seeds = seeds_pool[c % 100:c % 100 + 1]  # this cycle's Philox seed and position
            eng.pos = pos_pool[cc:cc + 1]
            eng.q, eng.qs, eng.drafts = q_pool[cc], qs_pool[cc], d_pool[cc]
            return cc

        def drafts(c):
            cc = use(c)
            for i in range(1, k + 1):
                eng.draft_step(i, Hdp_d[cc, i - 1:i])
            return cc

        for c in range(n_pool):
            drafts(c)
        for c in range(5):
            eng.verify(Hp_d[use(c)])
            eng.accept()
        torch.cuda.synchronize()
        # pass 1: verify and acceptance launches bracketed by events; each chunk of cycles is
        # queued behind a short device-side wait so that the host's call overhead is not timed
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for c0 in range(0, K, 32):
            torch.cuda._sleep(20_000_000)
            for c in range(c0, min(K, c0 + 32)):
                cc = use(c)
                ev[c][0].record()
                eng.verify(Hp_d[cc])
                ev[c][1].record()
                eng.accept()
                ev[c][2].record()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # pass 2: verify + acceptance back to back (the verify cycle, overlapped as in use; one
        # fused launch at T = 0)
        a.record()
        for c in range(K):
            eng.verify_accept(Hp_d[use(c)])
        b.record()
        torch.cuda.synchronize()
        va_s = a.elapsed_time(b) / 1e3
        eng.counters.zero_()
        # pass 3: full cycles (k draft steps + verify + acceptance)
        a.record()
        for c in range(K):
            cc = drafts(c)
            eng.verify_accept(Hp_d[cc])
        b.record()
        torch.cuda.synchronize()
        s = a.elapsed_time(b) / 1e3
        gemv_s = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) / 1e3
        cnt = eng.counters.cpu().numpy().view(spec.COUNTERS_DTYPE)[0]
        lm_bytes = (cfg.V * cfg.d * 2 + (k + 1) * cfg.d * 2 + (k + 1) * 16 +
                    (k + 1) * cfg.V * 4 * (T > 0))
        # verify + acceptance: the LM head's bytes plus, at T > 0, one logit row and one draft
        # row read by the acceptance's draw
        va_bytes = lm_bytes + (cfg.V + cfg.Vd) * 4 * (T > 0)
        gbs = lm_bytes / gemv_s / 1e9
        accept_us = statistics.mean(e[1].elapsed_time(e[2]) for e in ev) * 1e3
        per_drafted, per_test = acceptance_rates(cnt, k)
        out[f"T{T:g}_k{k}" + ("" if mode == "ratio" else f"_{mode}")] = {
            "verify_cycles_s": round(K / va_s, 1),
            "verify_accept_frac": round(va_bytes / (va_s / K) / 1e9 / hbm_peak, 4),
            "full_cycles_s": round(K / s, 1),
            "emitted_tok_s": round(float(cnt["emitted"]) / s, 1),
            "tokens_per_cycle": round(float(cnt["emitted"]) / K, 3),
            "acceptance": per_drafted, "acceptance_per_test": per_test,
            "eos_cycles": int(n_eos), "cycles": K,
            "lmhead_gbs": round(gbs, 1), "lmhead_frac": round(gbs / hbm_peak, 4),
            "accept_us": round(accept_us, 2)}
        del eng, Hp_d, Hdp_d, q_pool, qs_pool, d_pool
    return out


def adaptive_bench(dev, W, Wd, step_us, draft_us, K=512):
    """Adaptive verify width on the k-sweep's greedy workload: the width of every cycle is
    chosen on the device (spec_adapt_width) from the per-depth acceptance and the request's
    cycle-cost fit (cycles timed on the device; a prior table from this run's measured verify
    step and draft step until the fit is usable). One request, two schedules:
    host-scheduled widths (the headline: cycle n runs exactly the width chosen after cycle
    n - 2, which the width update writes into pinned host memory; the host reads it once that
    cycle has completed; acceptance and width update run in the verify kernel's last block),
    and the width graph (each cycle a graph launch whose select kernel
    picks the body of the chosen width, the cycle's inputs first copied into the graph's input
    buffers). Compared with every fixed width on the same inputs."""
    import torch

    import mtp_speculative_decoding_spec_gb300 as spec
    from mtp_speculative_decoding_spec_gb300.engine import SpecVerifyEngine
    k_max, n_pool = 7, 256
    cfg = configs.Config(**{**configs.get(2).__dict__, "k": k_max, "temps": (0.0,)})
    Hp, Hdp = build_inputs(cfg, W, n_pool, k_max, 0.0, rng_seed=7 * k_max)
    Hp_d = torch.from_numpy(Hp.view(np.int16)).to(dev)
    Hdp_d = torch.from_numpy(Hdp.view(np.int16)).to(dev)
    cost = [(step_us + k * draft_us) / step_us for k in range(k_max + 1)]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def run(lag):
        eng = SpecVerifyEngine(Wd, spec.SPEC_BF16, cfg.V, cfg.d, cfg.Vd, 1, k_max + 1, k_max,
                               cfg.eos_id, device=dev, adaptive_cost=cost, alpha=0.1,
                               width_lag=lag, fuse_greedy=True)
        eng.set_requests(temps=[0.0], seeds=[1], pos=[0], k=[1])
        for c in range(20):
            eng.cycle(Hp_d[c % n_pool], Hdp_d[c % n_pool, :, None, :], k_max)
        torch.cuda.synchronize()
        eng.counters.zero_()
        a.record()
        for c in range(K):
            eng.cycle(Hp_d[c % n_pool], Hdp_d[c % n_pool, :, None, :], k_max)
        b.record()
        torch.cuda.synchronize()
        s = a.elapsed_time(b) / 1e3
        cnt = eng.counters.cpu().numpy().view(spec.COUNTERS_DTYPE)[0]
        st = eng.width_state.cpu().numpy().view(spec.WIDTH_STATE_DTYPE)[0]
        out = {"full_cycles_s": round(K / s, 1),
               "emitted_tok_s": round(float(cnt["emitted"]) / s, 1),
               "tokens_per_cycle": round(float(cnt["emitted"]) / K, 3),
               "mean_width": round(float(cnt["drafted"]) / K, 3),
               "final_width": int(st["k"]),
               "rates": [round(float(st["rate"][d]), 3) if (int(st["seen"]) >> d) & 1 else None
                         for d in range(1, k_max + 1)],
               "fitted_cost_ratio": round(float(st["rate"][0]), 4),
               "fit_usable": bool(float(st["rate"][0]) > 0)}
        eng.close()
        del eng
        return out

    res = run(True)
    res["mode"] = "host-scheduled widths, one cycle late"
    res["prior_cost"] = [round(x, 3) for x in cost]
    res["workload"] = "k = 7 greedy sweep inputs (256 distinct cycles), k_max = 7"
    g = run(False)
    res["width_graph"] = {key: g[key] for key in ("full_cycles_s", "emitted_tok_s",
                                                  "tokens_per_cycle", "mean_width")}
    # every fixed width on the same inputs (the first k + 1 verify rows and k draft rows)
    fixed = {}
    for k in range(1, k_max + 1):
        eng = SpecVerifyEngine(Wd, spec.SPEC_BF16, cfg.V, cfg.d, cfg.Vd, 1, k + 1, k,
                               cfg.eos_id, device=dev, fuse_greedy=True)
        eng.set_requests(temps=[0.0], seeds=[1], pos=[0], k=[k])
        for c in range(5):
            eng.cycle(Hp_d[c, :k + 1], Hdp_d[c, :k, None, :], k)
        torch.cuda.synchronize()
        eng.counters.zero_()
        a.record()
        for c in range(K):
            eng.cycle(Hp_d[c % n_pool, :k + 1], Hdp_d[c % n_pool, :k, None, :], k)
        b.record()
        torch.cuda.synchronize()
        s = a.elapsed_time(b) / 1e3
        cnt = eng.counters.cpu().numpy().view(spec.COUNTERS_DTYPE)[0]
        fixed[f"k{k}"] = round(float(cnt["emitted"]) / s, 1)
        del eng
    res["fixed_emitted_tok_s"] = fixed
    best = max(fixed.values())
    res["vs_best_fixed"] = round(res["emitted_tok_s"] / best, 4)
    res["width_graph"]["vs_best_fixed"] = round(res["width_graph"]["emitted_tok_s"] / best, 4)
    return res


def c3_cycle(dev, W, Wd, hbm_peak, K=400):
    """The adaptive-rollback workload's verify cycle, timed end to end: per cycle k ~ U{1..7}
    (the workload's own draws), the verify LM head over its k+1 rows, greedy acceptance and the
    snapshot commit of the 64K-context state (one full-attention KV layer of 4 x 256 bf16 at
    65,536 positions, 36 recurrent layers of [16,128,128] fp32 and [3,8192] conv rows) driven
    on the device by the acceptance. Drafts come from the draft head before the timed region
    (a second timing adds the k draft steps: the full cycle). P starts at 63,488 and grows by
    the kept rows."""
    import torch

    import mtp_speculative_decoding_spec_gb300 as spec
    cfg = configs.get(3)
    n_pool, ns = 256, 9
    L, Hh, dk, dv = cfg.rec_layers, cfg.rec_heads, cfg.rec_dk, cfg.rec_dv
    ks, Hs, Hds = [], [], []
    for c in range(n_pool):
        inp = gen.cycle_inputs(cfg, W, c, seed=33)
        ks.append(inp["k"])
        H = np.zeros((8, cfg.d), dtype=np.uint16)
        H[:inp["k"] + 1] = inp["H"]
        Hd = np.zeros((7, cfg.d), dtype=np.uint16)
        Hd[:inp["k"]] = inp["Hd"]
        Hs.append(H)
        Hds.append(Hd)
    Hp_d = torch.from_numpy(np.stack(Hs).view(np.int16)).to(dev)
    Hdp_d = torch.from_numpy(np.stack(Hds).view(np.int16)).to(dev)
    k_pool = torch.tensor(ks, dtype=torch.int32, device=dev)
    st = BatchedState(cfg, 1, dev)
    ws = torch.zeros(spec.spec_workspace_bytes(cfg.V, 1), dtype=torch.uint8, device=dev)
    stats = torch.zeros(8 * spec.ROWSTATS_BYTES, dtype=torch.uint8, device=dev)
    qs = torch.zeros(7 * spec.ROWSTATS_BYTES, dtype=torch.uint8, device=dev)
    temps = torch.zeros(1, dtype=torch.float32, device=dev)
    seeds = torch.zeros(1, dtype=torch.int64, device=dev)
    pos = torch.zeros(1, dtype=torch.int64, device=dev)
    drafts_pool = torch.zeros((n_pool, 7), dtype=torch.int32, device=dev)
    out = torch.zeros(spec.ACCEPT_OUT_BYTES, dtype=torch.uint8, device=dev)
    cnt = torch.zeros(spec.COUNTERS_BYTES, dtype=torch.uint8, device=dev)

    def drafts_of(c):
        for i in range(1, ks[c] + 1):
            spec.spec_draft_argmax(Wd, spec.SPEC_BF16, cfg.Vd, cfg.d, Hdp_d[c, i - 1:i], 1, temps,
                                   seeds, pos, i - 1, drafts_pool[c, i - 1:], 7, None, cfg.Vd,
                                   qs[(i - 1) * spec.ROWSTATS_BYTES:], None, ws)

    def verify_cycle(c, mode=spec.SPEC_COMMIT_SNAPSHOT):
        k = ks[c]
        spec.spec_lmhead_verify(Wd, spec.SPEC_BF16, cfg.V, cfg.d, Hp_d[c], 1, k + 1, temps, None,
                                stats, ws)
        spec.spec_accept(1, 7, k_pool[c:c + 1], drafts_pool[c:c + 1], None, stats, cfg.V, k + 1,
                         None, None, cfg.Vd, cfg.Vd, temps, cfg.eos_id, seeds, pos, out, cnt, ws)
        spec.spec_commit_rollback(1, st.desc, out, k_pool[c:c + 1], mode)

    for c in range(n_pool):
        drafts_of(c)
    res = {}
    snap, index = spec.SPEC_COMMIT_SNAPSHOT, spec.SPEC_COMMIT_INDEX
    for name, with_drafts, mode in (("verify_cycle", False, snap), ("full_cycle", True, snap),
                                    ("verify_cycle_index", False, index)):
        st.kv_len.fill_(cfg.context)
        for c in range(5):
            verify_cycle(c, mode)
        st.kv_len.fill_(cfg.context)
        cnt.zero_()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for c in range(K):
            if with_drafts:
                drafts_of(c % n_pool)
            verify_cycle(c % n_pool, mode)
        b.record()
        torch.cuda.synchronize()
        s_ = a.elapsed_time(b) / 1e3
        cn = cnt.cpu().numpy().view(spec.COUNTERS_DTYPE)[0]
        rows = sum(ks[c % n_pool] + 1 for c in range(K))
        emitted = float(cn["emitted"])
        commit_bytes = 2 * 4 * (st.rec_elems + st.conv_elems) if mode == snap else 0
        zero_fill = (rows - emitted) * 2 * cfg.kv_layers * cfg.kv_row_bytes
        cyc_bytes = (K * (cfg.V * cfg.d * 2 + commit_bytes) + rows * (cfg.d * 2 + 16) +
                     zero_fill) / K
        res[name] = {"cycles_s": round(K / s_, 1), "emitted_tok_s": round(emitted / s_, 1),
                     "tokens_per_cycle": round(emitted / K, 3), "mean_k": round(rows / K - 1, 3)}
        if not with_drafts:
            res[name].update({"algorithmic_bytes_per_cycle": int(cyc_bytes),
                              "hbm_gbs": round(cyc_bytes * K / s_ / 1e9, 1),
                              "hbm_frac": round(cyc_bytes * K / s_ / 1e9 / hbm_peak, 4)})
    res["final_len"] = int(st.kv_len.cpu()[0])
    res["workload"] = ("k ~ U{1..7}, verify k+1 rows + greedy acceptance + snapshot commit of the "
                       "64K-context state, P from 63,488; verify_cycle_index: the same with the "
                       "index commit (the live state a slot, no state bytes moved)")
    del st
    return res


def q4_bench(dev, W, hbm_peak, K=2000):
    """The headline step (greedy, k = 1: verify 2 rows + acceptance) over the same LM head
    quantised to 4-bit affine codes in groups of 32 (SPEC_Q4A32, 1,600 bytes per row): verify
    launches bracketed by events in one step of ten (their mean is the kernel's duration alone),
    the steps back to back, and full cycles with the draft head over the same quantised rows."""
    import torch

    import mtp_speculative_decoding_spec_gb300 as spec
    from mtp_speculative_decoding_spec_gb300.engine import SpecVerifyEngine
    cfg = configs.get(1)
    Wq = gen.q4_weights(cfg)
    Wq_d = torch.from_numpy(Wq).to(dev)
    n_pool, k = 64, 1
    Hp, Hdp = build_inputs(cfg, W, n_pool, k, 0.0, rng_seed=300)
    Hp_d = torch.from_numpy(Hp.view(np.int16)).to(dev)
    Hdp_d = torch.from_numpy(Hdp.view(np.int16)).to(dev)
    eng = SpecVerifyEngine(Wq_d, spec.SPEC_Q4A32, cfg.V, cfg.d, cfg.Vd, 1, k + 1, k, cfg.eos_id,
                           device=dev, want_q_logits=False)
    eng.set_requests(temps=[0.0], seeds=[0], pos=[0], k=[k])
    for c in range(20):
        eng.cycle(Hp_d[c % n_pool], Hdp_d[c % n_pool, :, None, :], k)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K // 10)]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for c in range(K):
        if c % 10 == 0:
            ev[c // 10][0].record()
        eng.verify(Hp_d[c % n_pool])
        if c % 10 == 0:
            ev[c // 10][1].record()
        eng.accept()
    b.record()
    torch.cuda.synchronize()
    step_s = a.elapsed_time(b) / 1e3
    launch_s = statistics.mean(x.elapsed_time(y) for x, y in ev) / 1e3
    eng.counters.zero_()
    a.record()
    for c in range(K):
        eng.cycle(Hp_d[c % n_pool], Hdp_d[c % n_pool, :, None, :], k)
    b.record()
    torch.cuda.synchronize()
    cyc_s = a.elapsed_time(b) / 1e3
    cnt = eng.counters.cpu().numpy().view(spec.COUNTERS_DTYPE)[0]
    err = int(eng.ws[4:8].cpu().numpy().view(np.uint32)[0])
    algo = cfg.V * (5 * cfg.d // 8) + (k + 1) * cfg.d * 2 + (k + 1) * 16
    gbs = algo / launch_s / 1e9
    return {"kernel": "gemv_q4_kernel (verify, 2 rows)", "verify_cycles_s": round(K / step_s, 1),
            "mean_launch_us": round(launch_s * 1e6, 2), "algorithmic_bytes_per_launch": algo,
            "lmhead_gbs": round(gbs, 1), "lmhead_frac": round(gbs / hbm_peak, 4),
            "full_cycles_s": round(K / cyc_s, 1),
            "emitted_tok_s": round(float(cnt["emitted"]) / cyc_s, 1),
            "acceptance": round(float(cnt["accepted"]) / max(1.0, float(cnt["drafted"])), 4),
            "workspace_error": err,
            "workload": "greedy k = 1 step over the 4-bit affine head (group 32), "
                        "inputs larger than L2"}


def commit_bench(dev, hbm_peak, reps=64, warm=8):
    """Snapshot commit and replay of the 64K-context state (36 x [16,128,128] + conv rows), one
    request. The working set of one commit (75 MB) fits in the 129 MB L2, so the timed commits
    rotate over sources and destinations: four state descriptors, each with a live state of its
    own and its slot array shifted by one slot, and (snapshot) m cycling over 1..8. A commit's
    bytes were last touched at least four commits (302 MB) earlier. The launches are queued
    behind a device-side wait and timed back to back, each between events."""
    import torch

    import mtp_speculative_decoding_spec_gb300 as spec
    cfg = configs.get(3)
    ns, n_live = 9, 4
    L, H, dk, dv = cfg.rec_layers, cfg.rec_heads, cfg.rec_dk, cfg.rec_dv
    rec_elems, conv_elems = L * H * dk * dv, L * cfg.conv_rows * cfg.conv_width
    kvb = cfg.kv_layers * 2 * cfg.kv_capacity * cfg.kv_row_bytes
    kv = torch.zeros(kvb, dtype=torch.uint8, device=dev)
    kv_len = torch.tensor([cfg.context], dtype=torch.int64, device=dev)
    lives = [torch.zeros(rec_elems, device=dev) for _ in range(n_live)]
    clives = [torch.zeros(conv_elems, device=dev) for _ in range(n_live)]
    slots = torch.randn((ns + n_live - 1) * rec_elems, device=dev)
    cslots = torch.randn((ns + n_live - 1) * conv_elems, device=dev)
    a = torch.rand((ns - 1) * L * H, device=dev)
    b = torch.randn((ns - 1) * L * H * dk, device=dev)
    c = torch.randn((ns - 1) * L * H * dv, device=dev)
    x = torch.randn((ns - 1) * L * cfg.conv_width, device=dev)
    descs = []
    live_slot = torch.zeros(n_live, dtype=torch.int32, device=dev)  # index mode
    for j in range(n_live):
        d = spec.spec_state_desc()
        d.kv, d.kv_request_stride, d.kv_layers = kv.data_ptr(), kvb, cfg.kv_layers
        d.kv_capacity, d.kv_row_bytes = cfg.kv_capacity, cfg.kv_row_bytes
        d.kv_len = kv_len.data_ptr()
        d.rec_layers, d.rec_heads, d.rec_dk, d.rec_dv = L, H, dk, dv
        d.rec_live, d.rec_slots = lives[j].data_ptr(), slots.data_ptr() + 4 * j * rec_elems
        d.conv_rows, d.conv_width = cfg.conv_rows, cfg.conv_width
        d.conv_live = clives[j].data_ptr()
        d.conv_slots, d.n_slots = cslots.data_ptr() + 4 * j * conv_elems, ns
        d.step_a, d.step_b, d.step_c, d.conv_in = (a.data_ptr(), b.data_ptr(), c.data_ptr(),
                                                   x.data_ptr())
        d.live_slot = live_slot[j:].data_ptr()
        descs.append(d)
    accs = []
    for m in range(1, 9):  # n_emit = m: slot m is copied, KV rows [P+m, P+8) are cleared
        acc = np.zeros(1, dtype=spec.ACCEPT_OUT_DTYPE)
        acc["n_emit"] = m
        accs.append(torch.from_numpy(acc.view(np.uint8)).to(dev))
    k_d = torch.tensor([7], dtype=torch.int32, device=dev)
    state_bytes = 2 * 4 * (rec_elems + conv_elems)
    out = {}
    for mode, name in ((spec.SPEC_COMMIT_SNAPSHOT, "snapshot"), (spec.SPEC_COMMIT_REPLAY, "replay"),
                       (spec.SPEC_COMMIT_INDEX, "index")):
        def launch(i):
            m_idx = (i // n_live) % 8 if mode != spec.SPEC_COMMIT_REPLAY else 3
            spec.spec_commit_rollback(1, descs[i % n_live], accs[m_idx], k_d, mode)
            return m_idx + 1
        kv_len.fill_(cfg.context)  # each commit keeps at most 8 rows: P stays below capacity
        for i in range(warm):
            launch(i)
        torch.cuda.synchronize()
        ts, kept = [], []
        # a device-side wait lets the host queue every timed launch before the first one runs,
        # so the events time back-to-back kernels, not the host's call overhead
        torch.cuda._sleep(5_000_000)
        for i in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            kept.append(launch(warm + i))
            e1.record()
            ts.append((e0, e1))
        torch.cuda.synchronize()
        t = statistics.mean(a_.elapsed_time(b_) for a_, b_ in ts) / 1e3
        # KV rows cleared: [P+m, P+k+1) of both planes of every KV layer
        kv_bytes = statistics.mean(8 - m for m in kept) * cfg.kv_row_bytes * 2 * cfg.kv_layers
        moved = (state_bytes if mode != spec.SPEC_COMMIT_INDEX else 0) + kv_bytes
        out[name] = {"us": round(t * 1e6, 2), "bytes": int(moved),
                     "gbs": round(moved / t / 1e9, 1), "frac": round(moved / t / 1e9 / hbm_peak, 4)}
    out["method"] = ("one request, 64 launches back to back between events; sources and "
                     "destinations rotated over 302 MB so no commit hits L2 from an earlier one; "
                     "index: the live state a slot, only the index and the KV rows move")
    return out


def batched_bench(dev, W, Wd, hbm_peak, tf_peak, reps=20, with_commit=True):
    """32 requests x 8 rows: tensor-core LM head (256 rows), acceptance for 32 requests (half
    greedy, half T = 1 with one-hot q), and the 32 requests' snapshot commit at 16K context."""
    import torch

    import mtp_speculative_decoding_spec_gb300 as spec
    cfg = configs.get(4)
    B, R = cfg.batch, cfg.rows_per_request
    rng = np.random.default_rng(4)
    H, _, targets = gen.planted_rows(cfg, W, B * R, rng)
    H_d = torch.from_numpy(H.view(np.int16)).to(dev)
    ws = torch.zeros(spec.spec_workspace_bytes(cfg.V, B), dtype=torch.uint8, device=dev)
    logits = torch.empty((B * R, cfg.V), dtype=torch.float32, device=dev)
    stats = torch.zeros(B * R * spec.ROWSTATS_BYTES, dtype=torch.uint8, device=dev)
    temps = torch.tensor(cfg.temps, dtype=torch.float32, device=dev)
    ks = rng.integers(1, 8, B).astype(np.int32)
    drafts = np.zeros((B, 7), dtype=np.int32)
    for b in range(B):
        drafts[b, :ks[b]] = targets[b * R:b * R + ks[b]]
    k_d = torch.from_numpy(ks).to(dev)
    dr_d = torch.from_numpy(drafts).to(dev)
    seeds = torch.arange(B, dtype=torch.int64, device=dev)
    pos = torch.full((B,), cfg.context, dtype=torch.int64, device=dev)
    out = torch.zeros(B * spec.ACCEPT_OUT_BYTES, dtype=torch.uint8, device=dev)
    cnt = torch.zeros(B * spec.COUNTERS_BYTES, dtype=torch.uint8, device=dev)

    def verify():
        spec.spec_lmhead_verify(Wd, spec.SPEC_BF16, cfg.V, cfg.d, H_d, B, R, temps, logits, stats,
                                ws)

    def accept():
        spec.spec_accept(B, 7, k_d, dr_d, logits, stats, cfg.V, R, None, None, cfg.Vd, cfg.Vd,
                         temps, cfg.eos_id, seeds, pos, out, cnt, ws)

    st = None
    if with_commit:
        st = BatchedState(cfg, B, dev)

    def commit():
        st.kv_len.fill_(cfg.context)
        spec.spec_commit_rollback(B, st.desc, out, k_d, spec.SPEC_COMMIT_SNAPSHOT)

    for _ in range(3):
        verify()
        accept()
        if st:
            commit()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(reps)]
    for i in range(reps):
        ev[i][0].record()
        verify()
        ev[i][1].record()
        accept()
        ev[i][2].record()
        if st:
            commit()
        ev[i][3].record()
    torch.cuda.synchronize()
    tv = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) / 1e3
    ta = statistics.mean(e[1].elapsed_time(e[2]) for e in ev) / 1e3
    tc = statistics.mean(e[2].elapsed_time(e[3]) for e in ev) / 1e3
    o = out.cpu().numpy().view(spec.ACCEPT_OUT_DTYPE)
    flops = 2.0 * B * R * cfg.d * cfg.V
    gemm_bytes = cfg.V * cfg.d * 2 + B * R * cfg.d * 2 + (B // 2) * R * cfg.V * 4
    res = {"workload": "32 requests x 8 rows, d=2560, V=151936 bf16, half T=0 / half T=1, "
                       "16K context state",
           "verify_us": round(tv * 1e6, 2), "tflops": round(flops / tv / 1e12, 1),
           "tensor_frac": round(flops / tv / 1e12 / tf_peak, 4),
           "hbm_gbs": round(gemm_bytes / tv / 1e9, 1),
           "hbm_frac": round(gemm_bytes / tv / 1e9 / hbm_peak, 4),
           "accept_us": round(ta * 1e6, 2),
           "emitted_tokens_per_cycle": int(o["n_emit"].sum()),
           "verify_cycles_s": round(1.0 / (tv + ta), 1),
           "tokens_s_verify_accept": round(float(o["n_emit"].sum()) / (tv + ta), 1),
           "workspace_error": int(ws[4:8].cpu().numpy().view(np.uint32)[0])}
    if st:
        moved = B * (2 * 4 * (st.rec_elems + st.conv_elems))
        res.update({"commit_us": round(tc * 1e6, 2), "commit_bytes": moved,
                    "commit_gbs": round(moved / tc / 1e9, 1),
                    "commit_frac": round(moved / tc / 1e9 / hbm_peak, 4),
                    "full_cycles_s": round(1.0 / (tv + ta + tc), 1)})
        del st
    return res


class BatchedState:
    """Device state of B requests at the batched workload's sizes (KV, recurrent, conv, 9
    snapshot slots) for the commit timing; contents are random, the commit copies them."""

    def __init__(self, cfg, B, dev):
        import torch

        import mtp_speculative_decoding_spec_gb300 as spec
        ns = 9
        L, H, dk, dv = cfg.rec_layers, cfg.rec_heads, cfg.rec_dk, cfg.rec_dv
        self.rec_elems = L * H * dk * dv
        self.conv_elems = L * cfg.conv_rows * cfg.conv_width
        kvb = cfg.kv_layers * 2 * cfg.kv_capacity * cfg.kv_row_bytes
        self.kv = torch.zeros(B * kvb, dtype=torch.uint8, device=dev)
        self.kv_len = torch.full((B,), cfg.context, dtype=torch.int64, device=dev)
        self.live = torch.zeros(B * self.rec_elems, device=dev)
        self.slots = torch.randn(B * ns * self.rec_elems, device=dev)
        self.clive = torch.zeros(B * self.conv_elems, device=dev)
        self.cslots = torch.randn(B * ns * self.conv_elems, device=dev)
        d = spec.spec_state_desc()
        d.kv, d.kv_request_stride, d.kv_layers = self.kv.data_ptr(), kvb, cfg.kv_layers
        d.kv_capacity, d.kv_row_bytes = cfg.kv_capacity, cfg.kv_row_bytes
        d.kv_len = self.kv_len.data_ptr()
        d.rec_layers, d.rec_heads, d.rec_dk, d.rec_dv = L, H, dk, dv
        d.rec_live, d.rec_slots = self.live.data_ptr(), self.slots.data_ptr()
        d.conv_rows, d.conv_width = cfg.conv_rows, cfg.conv_width
        d.conv_live, d.conv_slots, d.n_slots = self.clive.data_ptr(), self.cslots.data_ptr(), ns
        self.live_slot = torch.zeros(B, dtype=torch.int32, device=dev)  # index mode
        d.live_slot = self.live_slot.data_ptr()
        self.desc = d


def cpu_baseline(cfg, W, seconds):
    """The float64 oracle as it stands: verify cycles on the host cores until `seconds`."""
    from oracle import accept as o_accept
    from oracle import lmhead as o_lm
    n, t0 = 0, time.perf_counter()
    while n < 2 or time.perf_counter() - t0 < seconds:
        inp = gen.cycle_inputs(cfg, W, n, seed=999, k=cfg.k)
        z = o_lm.logits(W, inp["H"])
        y = o_lm.logits(W, inp["Hd"], rows=cfg.Vd)
        d, _ = o_accept.draft_chain_tokens(y, 0.0, None, 0)
        o_accept.accept_request(z, None, d, cfg.k, 0.0, cfg.eos_id, None, 0)
        n += 1
    s = time.perf_counter() - t0
    return {"value": round(n / s, 4), "unit": "verify cycles/s", "kind": "oracle",
            "cores": len(os.sched_getaffinity(0)),
            "sample": f"{n} full cycles (draft-head logits over {cfg.Vd} rows, verify logits "
                      f"over {cfg.V} rows x {cfg.k + 1}, greedy acceptance) in float64 numpy",
            "seconds": round(s, 2)}


# ------------------------------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    if rank != 0:
        return
    from oracle import accept as o_accept
    from oracle import lmhead as o_lm
    cfg = configs.get(1)
    W = gen.lm_weights(cfg)
    K, Wm = args.steps, args.warmup

    def one_step(c, rows):
        inp = gen.cycle_inputs(cfg, W, c, seed=999, k=cfg.k)
        z = o_lm.logits(W[:rows], inp["H"])
        o_accept.accept_request(z, None, [0] * cfg.k, cfg.k, 0.0, cfg.eos_id, None, 0)

    t0 = time.perf_counter()
    one_step(0, 2048)
    probe = time.perf_counter() - t0
    budget = 90.0
    rows = int(max(256, min(cfg.V, 2048 * budget / max(1, K + Wm) / max(probe, 1e-6))))
    for c in range(Wm):
        one_step(c, rows)
    t0 = time.perf_counter()
    for c in range(K):
        one_step(c, rows)
    s = time.perf_counter() - t0
    per_cycle = s / K * cfg.V / rows
    value = 1.0 / per_cycle
    sample = (f"each step: float64 oracle verify cycle over {rows} of {cfg.V} LM-head rows "
              f"(2 verify rows) + greedy acceptance; time scaled by {cfg.V}/{rows}")
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 4),
           "unit": "verify cycles/s", "n_gpus": world, "steps": K, "warmup": Wm,
           "ms_per_step": round(per_cycle * 1e3, 3), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": workload_config(cfg, {"parallelism": "host cores"}),
           "cpu_baseline": {"value": round(value, 4), "unit": "verify cycles/s",
                            "kind": "oracle", "cores": len(os.sched_getaffinity(0)),
                            "sample": sample},
           "e2e": {"value": round(value, 4), "unit": "verify cycles/s",
                   "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    args = parse()
    rank, local_rank, world = rank_info()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, local_rank, world)


if __name__ == "__main__":
    main()

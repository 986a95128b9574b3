"""Benchmark of linear_logp on GB300: tokens/s of forward + backward at the
Qwen3-8B output-layer shape, with the tensor-core roofline fraction.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl rlk|reference]
                [--workload qwen3_8b|qwen3_30b_tp2|tiny] [--quick]
python bench.py --case fwd|dz|dh|dw|fwd8|dz8 [--tokens T] [--vocab V]
python bench.py --record-traffic NCU_CSV --traffic-command CMD

A step is one pass of the whole path over one synthetic batch: the fused
forward (tile GEMM + online statistics + fixed-tree merge; for the sharded
workload one call per vocab shard plus rlk_lse_merge) and the backward (dz
recompute, dH, dW; sharded: per shard plus the fixed-order dH sum), the
backward launched as its three stages so that a CUDA event between the calls
times each GEMM inside the step. N > 1 runs one independent batch per rank
(weak scaling; no collective on the data path, only a barrier and a max of
the elapsed times). Rank 0 prints one JSON line; at N = 1 it also carries the
small-batch and tiny legs (run first), the end-to-end leg from host buffers,
the forward-only, saved-logits, saved-probabilities and FP8 legs, the two-shard
Qwen3-30B step, one rank's calls of that split, and the CPU oracle baseline.

--impl reference times the fp64 CPU oracle on the host cores instead (each
step a bounded sample of the same workload, extrapolated per token).
--case times one stage alone (per-kernel timings, small ncu captures).
--record-traffic writes the per-launch DRAM bytes of an ncu capture of the
step to profiles/traffic_qwen3_8b.json together with the library sources' hash.
"""
from __future__ import annotations

import argparse
import datetime
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

import workloads  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024


# DRAM traffic per launch of each tile kernel, from one ncu capture of the full-size step
# (`--record-traffic` writes it; bench reads it back only while the library's sources
# still hash to the value recorded with it).
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_qwen3_8b.json")
STAGE_OF_MODE = {0: "fwd", 1: "dz", 2: "dH", 3: "dW"}


def record_traffic(csv_path: str, command: str, out_path: str = TRAFFIC_FILE):
    """Parse an ncu --csv log of dram__bytes_read.sum / dram__bytes_write.sum over tile-kernel
    launches and write the per-launch averages with the current sources hash."""
    import csv
    import re
    from deterministic_token_logprob_gb300 import build as libbuild
    acc = {}
    with open(csv_path, newline="") as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for row in csv.DictReader(lines):
        m = re.search(r"gemm_kernel<\(?(?:int\))?(\d+)>", row.get("Kernel Name", ""))
        metric = row.get("Metric Name", "")
        if not m or int(m.group(1)) not in STAGE_OF_MODE or not metric.startswith("dram__bytes_"):
            continue
        scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}.get(row.get("Metric Unit", "byte"))
        if scale is None:
            raise ValueError(f"unknown unit {row.get('Metric Unit')}")
        val = float(row["Metric Value"].replace(",", "")) * scale
        e = acc.setdefault(STAGE_OF_MODE[int(m.group(1))], {"ids": set(), "read": 0.0, "write": 0.0})
        e["ids"].add(row["ID"])
        e["read" if "read" in metric else "write"] += val
    kernels = {}
    for stage, e in acc.items():
        n = len(e["ids"])
        kernels[stage] = {"launches": n, "dram_bytes_read_per_launch": e["read"] / n,
                          "dram_bytes_write_per_launch": e["write"] / n,
                          "traffic_bytes_per_launch": (e["read"] + e["write"]) / n}
    rec = {"workload": "qwen3_8b fwd+bwd T=8192 H=4096 V=151936 V_true=151669",
           "metrics": "dram__bytes_read.sum + dram__bytes_write.sum (ncu, 1 pass per launch)",
           "command": command, "library_sources_sha256": libbuild.sources_sha256(),
           "kernels": kernels}
    with open(out_path, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    return rec


def traffic_per_launch(stage: str):
    """(bytes, note): the recorded DRAM traffic of one launch of `stage`'s kernel on the
    Qwen3-8B workload, or (None, why) when there is no record for the current sources."""
    from deterministic_token_logprob_gb300 import build as libbuild
    if not os.path.exists(TRAFFIC_FILE):
        return None, "no traffic record"
    with open(TRAFFIC_FILE) as f:
        rec = json.load(f)
    if rec.get("library_sources_sha256") != libbuild.sources_sha256():
        return None, "traffic record predates the current library sources"
    k = rec.get("kernels", {}).get(stage)
    if not k:
        return None, f"no {stage} launch in the traffic record"
    return k["traffic_bytes_per_launch"], f"ncu capture: {rec.get('command')}"


def print_line(line: dict):
    """Print the JSON line as the last thing on stdout: C-level stdio output buffered by
    libraries (a communication library's version banner, say) is flushed first."""
    try:
        import ctypes
        ctypes.CDLL(None).fflush(None)
    except (OSError, AttributeError):
        pass
    sys.stdout.flush()
    print(json.dumps(line), flush=True)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock, power and throttle reasons. Only samples
    whose timestamps fall between mark_start() and mark_end() (the timed region) are kept."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_id: str, interval_ms: int = 50):
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None
        try:
            fd, self.path = tempfile.mkstemp(prefix="rlk_clocks_", suffix=".csv")
            self.out = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(interval_ms), "-i", gpu_id], stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def wait_running(self, timeout_s: float = 5.0):
        """Return once the first sample has been written (or after timeout_s)."""
        t_end = time.time() + timeout_s
        while self.proc is not None and time.time() < t_end:
            if os.path.getsize(self.path) > 0:
                return
            time.sleep(0.02)

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        samples = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    samples.append((ts, float(parts[2]), float(parts[3]),
                                    [n for n, v in zip(self.REASONS, parts[6:10])
                                     if v.lower().startswith("active")]))
                except ValueError:
                    continue
        os.unlink(self.path)
        inside = [x for x in samples if self.t0 is not None and self.t1 is not None
                  and self.t0 <= x[0] <= self.t1]
        use = inside or samples
        if not use:
            return None
        return {"sm_mhz": statistics.median(x[1] for x in use), "sm_max_mhz": max(x[2] for x in use),
                "samples": len(use), "samples_in_timed_region": bool(inside),
                "reasons": sorted({r for x in use for r in x[3]})}


# ----------------------------------------------------------------------------- oracle timing


def oracle_sample_rate(w: workloads.Workload, d: dict, n_tok: int = 0, n_vrows: int = 1024,
                       seed: int = 0):
    """Oracle (fp64, all host cores) fwd+bwd throughput on a bounded sample.

    n_tok sampled tokens (default 8 per host thread, the oracle's own block of tokens per
    thread) go through the oracle's forward and dH. dW is linear in the tokens with
    non-zero g, so it is evaluated with g restricted to the sampled tokens for n_vrows
    sampled vocab rows; its per-row time is scaled to all V rows, and its fixed cost
    (widening h once per call) is charged per token (n_tok / T of it), as in a full step.
    Returns (tokens/s, cores, sample text).
    """
    import oracle
    oracle.build()
    cores = oracle.default_threads()
    n_tok = min(w.T, n_tok or 8 * cores)
    rows = workloads.sample_rows(w.T, n_tok, seed=seed, stream=11)
    vrows = workloads.sample_rows(w.V, n_vrows, seed=seed, stream=12)
    g_sub = np.zeros(w.T, np.float64)
    g_sub[rows] = d["g"][rows]
    t0 = time.perf_counter()
    _, lse_rows = oracle.forward(d["h"], d["W"], d["y"], w.V_true, rows=rows)
    t1 = time.perf_counter()
    oracle.backward_dh(d["h"], d["W"], d["y"], d["g"].astype(np.float64), w.V_true, rows=rows)
    t2 = time.perf_counter()
    lse_full = np.zeros(w.T)
    lse_full[rows] = lse_rows
    oracle.backward_dw(d["h"], d["W"], d["y"], g_sub, lse_full, w.V_true,
                       vrows=np.zeros(0, np.int64))
    t3 = time.perf_counter()
    oracle.backward_dw(d["h"], d["W"], d["y"], g_sub, lse_full, w.V_true, vrows=vrows)
    t4 = time.perf_counter()
    fixed = t3 - t2
    per_row = max(0.0, (t4 - t3) - fixed) / len(vrows)
    per_step = (t1 - t0) + (t2 - t1) + per_row * w.V + fixed * len(rows) / w.T
    sample = (f"{len(rows)} of {w.T} tokens: oracle forward + dH over all {w.V_true} columns; "
              f"dW for {len(vrows)} of {w.V} vocab rows (per-row time x {w.V}), "
              f"its fixed per-call cost charged {len(rows)}/{w.T}")
    return len(rows) / per_step, cores, sample


def run_reference(args, w: workloads.Workload, rank: int, world: int):
    """--impl reference: the fp64 oracle on the host cores, same metric and workload."""
    if rank != 0:
        return
    d = workloads.make_inputs(w)
    import oracle
    oracle.build()
    # a bounded sample per step (about 10 s): 8 tokens per host thread, the block of tokens
    # the oracle's forward and dH widen each W row for, as in the GPU arm's cpu_baseline
    n_tok = min(w.T, 8 * oracle.default_threads())
    for i in range(args.warmup):
        oracle_sample_rate(w, d, n_tok=min(n_tok, 4), n_vrows=64, seed=100 + i)
    rates = []
    t0 = time.perf_counter()
    for i in range(args.steps):
        r, cores, sample = oracle_sample_rate(w, d, n_tok=n_tok, n_vrows=256, seed=i)
        rates.append(r)
    wall = time.perf_counter() - t0
    value = float(statistics.median(rates))
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "impl": "reference",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * w.T / value, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w, world),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "wall_s": wall}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU path

METRIC = "linear_logp tokens/s fwd & fwd+bwd at Qwen3-8B shape; % of GB300 BF16 TC roofline"


def config_dict(w: workloads.Workload, world: int):
    return {"workload": f"{w.name} fwd+bwd T={w.T} H={w.H} V={w.V} V_true={w.V_true}"
                        + (f" shards={len(w.shards)}" if w.shards else ""),
            "tokens_per_rank": w.T, "H": w.H, "V": w.V, "V_true": w.V_true,
            "global_tokens": w.T * world, "parallelism": f"replicas{world}",
            "l2_policy": "inputs larger than L2 (W alone exceeds 129 MB); no flush"}


class Path:
    """Device buffers and the C-ABI calls of one step."""

    def __init__(self, rlk, torch, w: workloads.Workload, d: dict, device, with_dW: bool = True):
        self.rlk, self.torch, self.w = rlk, torch, w
        bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)  # noqa: E731
        self.h = bf(d["h"])
        self.W = bf(d["W"]) if "W" in d else None
        self.y = torch.from_numpy(d["y"]).to(device)
        self.g = torch.from_numpy(d["g"]).to(device)
        T, H, V = w.T, w.H, w.V
        f32 = torch.float32
        self.logp = torch.empty(T, dtype=f32, device=device)
        self.lse = torch.empty(T, dtype=f32, device=device)
        self.dW = torch.empty((V, H), dtype=f32, device=device) if with_dW else None
        shards = w.shards or ((0, V),)
        self.shards = shards
        self.fws = torch.empty(max(rlk.fwd_workspace_bytes(T, H, n) for _, n in shards),
                               dtype=torch.uint8, device=device)
        self.bws = torch.empty(max(rlk.bwd_workspace_bytes(T, H, n) for _, n in shards),
                               dtype=torch.uint8, device=device)
        if w.shards:
            self.parts = torch.empty((len(shards), T, 3), dtype=f32, device=device)
            self.dH_parts = torch.empty((len(shards), T, H), dtype=f32, device=device)
            self.dH = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        else:
            self.dH = torch.empty((T, H), dtype=torch.bfloat16, device=device)

    def launches_per_step(self):
        n = len(self.shards)
        return (2 * n + 1 + 3 * n + 1) if self.w.shards else 5

    def staged_calls(self):
        """The step as a list of (stage, call): the forward, then the backward as its three
        stages (rlk_linear_logp_bwd_stages: the launches of one rlk_linear_logp_bwd call, one
        call each), so that each stage can be timed inside the step."""
        rlk, w = self.rlk, self.w
        DZ, DH, DW = rlk.RLK_BWD_DZ, rlk.RLK_BWD_DH, rlk.RLK_BWD_DW
        if not w.shards:
            def bwd(stage):
                return lambda: rlk.linear_logp_bwd(self.h, self.W, self.y, self.lse, self.g, w.V_true,
                                                   out=(self.dH, self.dW), workspace=self.bws,
                                                   stages=stage)
            return [("fwd", self.forward), ("dz", bwd(DZ)), ("dH", bwd(DH)), ("dW", bwd(DW))]
        calls = []
        for i, (a, n) in enumerate(self.shards):
            calls.append(("fwd", lambda a=a, n=n, i=i: rlk.linear_logp_fwd(
                self.h, self.W[a:a + n], self.y, w.V_true, vocab_start=a, partial=True,
                out=(self.parts[i],), workspace=self.fws)))
        calls.append(("merge", lambda: rlk.lse_merge(self.parts, out=(self.logp, self.lse))))
        for i, (a, n) in enumerate(self.shards):
            for name, stage in (("dz", DZ), ("dH", DH), ("dW", DW)):
                calls.append((name, lambda a=a, n=n, i=i, stage=stage: rlk.linear_logp_bwd(
                    self.h, self.W[a:a + n], self.y, self.lse, self.g, w.V_true, vocab_start=a,
                    dH_fp32_partial=True, out=(self.dH_parts[i], self.dW[a:a + n]),
                    workspace=self.bws, stages=stage)))
        calls.append(("sum", lambda: rlk.shard_sum_bf16(self.dH_parts, out=self.dH)))
        return calls

    def forward(self):
        rlk, w = self.rlk, self.w
        if not w.shards:
            rlk.linear_logp_fwd(self.h, self.W, self.y, w.V_true, out=(self.logp, self.lse),
                                workspace=self.fws)
        else:
            for i, (a, n) in enumerate(self.shards):
                rlk.linear_logp_fwd(self.h, self.W[a:a + n], self.y, w.V_true, vocab_start=a,
                                    partial=True, out=(self.parts[i],), workspace=self.fws)
            rlk.lse_merge(self.parts, out=(self.logp, self.lse))

    def backward(self):
        rlk, w = self.rlk, self.w
        if not w.shards:
            rlk.linear_logp_bwd(self.h, self.W, self.y, self.lse, self.g, w.V_true,
                                out=(self.dH, self.dW), workspace=self.bws)
        else:
            for i, (a, n) in enumerate(self.shards):
                rlk.linear_logp_bwd(self.h, self.W[a:a + n], self.y, self.lse, self.g, w.V_true,
                                    vocab_start=a, dH_fp32_partial=True,
                                    out=(self.dH_parts[i], self.dW[a:a + n]), workspace=self.bws)
            rlk.shard_sum_bf16(self.dH_parts, out=self.dH)


def rank_workload(w: workloads.Workload, rank: int) -> workloads.Workload:
    """Rank `rank`'s batch: its own seeded h, y, g (seed = rank); W (model state) is shared."""
    return workloads.Workload(w.name, T=w.T, H=w.H, V=w.V, V_true=w.V_true, seed=rank,
                              backward=w.backward, g_kind=w.g_kind, shards=w.shards)


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest x over all ranks (the job's elapsed time is its slowest rank's)."""
    if world <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, steps: int, max_total_ms: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world * steps / (max_total_ms / 1e3)


def gpu_uuid(torch, device):
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        return str(device.index or 0)


def run_gpu(args, w: workloads.Workload, rank: int, world: int, local_rank: int):
    import torch

    import deterministic_token_logprob_gb300 as rlk
    from deterministic_token_logprob_gb300 import build as libbuild
    if rank == 0 or world == 1:
        libbuild.build()
    if world > 1:
        torch.distributed.barrier()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    peaks, peaks_src = load_peaks()

    # model weight shared by all ranks (seed 0); each rank its own batch
    W_bits = workloads.make_W(w.V, w.H, seed=0)
    wr = rank_workload(w, rank)
    d = workloads.make_inputs(wr, with_W=False)
    d["W"] = W_bits
    path = Path(rlk, torch, wr, d, device)
    stream = torch.cuda.current_stream(device)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    first_legs = {}
    if rank == 0 and world == 1 and not args.quick:
        # the short, HBM-bound and launch-bound legs first, before any power-capped loop has
        # heated the GPU, each with its own clock record
        if w.name == "qwen3_8b":
            first_legs["small_T_forward"] = small_t_leg(rlk, torch, path, device, peaks,
                                                        gpu_uuid(torch, device))
        first_legs["tiny"] = tiny_leg(rlk, torch, device, args, gpu_uuid(torch, device))

    calls = path.staged_calls()
    for _ in range(args.warmup):
        for _, fn in calls:
            fn()
    torch.cuda.synchronize(device)

    K = args.steps
    sampler = ClockSampler(gpu_uuid(torch, device)) if rank == 0 else None
    if sampler:
        sampler.wait_running()
    barrier()
    torch.cuda.synchronize(device)
    if sampler:
        sampler.mark_start()
    res = timed_steps(torch, stream, calls, K)
    if sampler:
        sampler.mark_end()
    barrier()
    clocks = sampler.stop() if sampler else None
    total_ms = max_over_ranks(res["total_ms"], world, device)
    ms_per_step = total_ms / K
    tokens_per_s = job_tokens_per_s(w.T, world, K, total_ms)

    flops_gemm = 2.0 * w.T * w.H * w.V_true   # one GEMM-equivalent: each of fwd, dz, dH, dW
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    step_flops = 3.0 * flops_gemm
    roofline_ms = step_flops / (peak * 1e12) * 1e3
    per_kernel = per_kernel_roofline(res["stage_ms"], flops_gemm, peak, peak_sus)
    dominant = max(per_kernel, key=lambda k: per_kernel[k]["ms"])
    dk = per_kernel[dominant]
    traffic, traffic_note = (traffic_per_launch(dominant) if w.name == "qwen3_8b"
                             else (None, "traffic is recorded for the qwen3_8b workload only"))
    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(w, world),
        "gpu_launches": K * path.launches_per_step(),
        # the dominant (slowest) GEMM kernel of the step, timed with CUDA events around its call
        # inside the back-to-back, power-capped loop: its denominator is the sustained bf16
        # figure; the burst fraction is kept beside it
        "roofline": {"bound": "tensor", "kernel": STAGE_LABEL[dominant],
                     "achieved": dk["tflops"], "peak": peak_sus, "unit": "TFLOP/s",
                     "frac": dk["frac_of_sustained"], "traffic": traffic,
                     "traffic_source": traffic_note,
                     "peak_source": f"{peaks_src} bf16 sustained (kernel timed inside the step loop)",
                     "frac_of_burst": dk["frac_of_burst"],
                     "algorithmic_flops_per_launch": flops_gemm, "avg_launch_ms": dk["ms"],
                     "per_kernel": per_kernel},
        "step_roofline": {"flops_counted": step_flops, "roofline_ms": roofline_ms,
                          "frac_of_burst": roofline_ms / ms_per_step,
                          "frac_of_sustained": (step_flops / (peak_sus * 1e12) * 1e3) / ms_per_step,
                          "stage_ms": res["stage_ms"],
                          "step_ms_median": statistics.median(res["step_ms"]),
                          "step_ms_best": min(res["step_ms"]),
                          "note": "step = forward call + the backward's three stages (one call each)"},
        "clocks": clocks,
    }
    line.update(first_legs)

    if not args.quick:
        # the end-to-end step first, right after the device-timed loop, so that both run in
        # the same thermal and power state (every rank: its own batch); the other legs follow
        line["e2e"] = e2e(rlk, torch, path, wr, d, device, args,
                          gpu_uuid(torch, device) if rank == 0 else None, world)
    if rank == 0 and world == 1 and not args.quick:
        if w.name == "qwen3_8b":  # legs defined on the Qwen3-8B weight
            line["fwd_only"] = fwd_only(rlk, torch, W_bits, path, device, args, peak)
            line["saved_logits"] = saved_logits_leg(rlk, torch, path, wr, device, args, peak, peak_sus)
            line["saved_probs_bf16"] = saved_probs_leg(rlk, torch, path, wr, device, args, peak)
            line["fp8_e4m3"] = fp8_leg(rlk, torch, path, wr, device, args, peak)
            del path, calls
            torch.cuda.empty_cache()
            line["qwen3_30b_tp2"] = sharded_leg(rlk, torch, device, args, peak, peak_sus,
                                                gpu_uuid(torch, device))
            line["qwen3_30b_tp2_rank_calls"] = tp2_rank_calls_leg(rlk, torch, device, args, peak)
        rate, cores, sample = oracle_sample_rate(wr, d)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print_line(line)


STAGE_LABEL = {"fwd": "forward tile GEMM + online statistics (call incl. leaf tree)",
               "dz": "dz: logits recompute + softmax gradient (MODE_DZ)",
               "dH": "dH = dz W (MODE_DH)", "dW": "dW = dz^T h (MODE_DW)"}


def timed_steps(torch, stream, calls, K):
    """K back-to-back steps of `calls` ([(stage, fn)]) with a CUDA event on `stream` before
    every call and after the last: total ms, per-step ms and mean ms per step of each stage
    (a stage's calls summed within a step)."""
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(K)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(K):
        for j, (_, fn) in enumerate(calls):
            evs[i][j].record(stream)
            fn()
        evs[i][-1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    stage_ms = {}
    for i in range(K):
        for j, (name, _) in enumerate(calls):
            stage_ms[name] = stage_ms.get(name, 0.0) + evs[i][j].elapsed_time(evs[i][j + 1]) / K
    return {"total_ms": t_start.elapsed_time(t_end),
            "step_ms": [e[0].elapsed_time(e[-1]) for e in evs], "stage_ms": stage_ms}


def per_kernel_roofline(stage_ms, flops_gemm, peak, peak_sus):
    """Achieved TFLOP/s of each GEMM stage (one GEMM-equivalent, 2 T H V_true FLOP, per call)
    against the measured sustained and burst bf16 peaks."""
    out = {}
    for k in ("fwd", "dz", "dH", "dW"):
        if k in stage_ms:
            tf = flops_gemm / (stage_ms[k] / 1e3) / 1e12
            out[k] = {"ms": stage_ms[k], "tflops": tf, "frac_of_sustained": tf / peak_sus,
                      "frac_of_burst": tf / peak}
    return out


def sharded_leg(rlk, torch, device, args, peak, peak_sus, gpu_id):
    """The Qwen3-30B-A3B-shaped step with two vocab shards emulated on this GPU (T = 16384,
    H = 2048; shards [0, 77824) and [77824, 151936)): per shard the forward statistics, then
    rlk_lse_merge; per shard dz, the fp32 dH partial and its dW rows, then rlk_shard_sum_bf16."""
    w = workloads.QWEN3_30B_TP2
    d = workloads.make_inputs(w)
    path = Path(rlk, torch, w, d, device)
    calls = path.staged_calls()
    for _ in range(max(3, args.warmup)):
        for _, fn in calls:
            fn()
    torch.cuda.synchronize(device)
    sampler = ClockSampler(gpu_id) if gpu_id else None
    if sampler:
        sampler.wait_running()
        sampler.mark_start()
    res = timed_steps(torch, torch.cuda.current_stream(device), calls, args.steps)
    if sampler:
        sampler.mark_end()
    clocks = sampler.stop() if sampler else None
    ms = res["total_ms"] / args.steps
    flops_gemm = 2.0 * w.T * w.H * w.V_true
    step_flops = 3.0 * flops_gemm
    out = {"workload": config_dict(w, 1)["workload"], "tokens_per_s": w.T / (ms / 1e3),
           "ms_per_step": ms, "steps": args.steps,
           "frac_of_burst": step_flops / (peak * 1e12) / (ms / 1e3),
           "frac_of_sustained": step_flops / (peak_sus * 1e12) / (ms / 1e3),
           "gpu_launches_per_step": path.launches_per_step(),
           "per_kernel": per_kernel_roofline(res["stage_ms"], flops_gemm, peak, peak_sus),
           "stage_ms": res["stage_ms"], "clocks": clocks,
           "shards": [list(x) for x in w.shards]}
    del path
    torch.cuda.empty_cache()
    return out


def tp2_rank_calls_leg(rlk, torch, device, args, peak):
    """One rank's share of a two-way vocab split at the Qwen3-30B-A3B output layer (H = 2048,
    shard [0, 77824) of V = 151936, V_true = 151669), for 796, 1820 and 6827 tokens per call:
    the forward (the shard's statistics, then rlk_lse_merge with the other shard's) and the
    forward + backward (plus dz, the fp32 dH partial and the shard's dW rows), each timed as
    back-to-back calls with CUDA events. The exchange between ranks is not included."""
    H, V, Vt = 2048, 151936, 151669
    (a0, n0), (a1, n1) = rlk.shard_bounds(V, Vt, 2)
    W = torch.from_numpy(workloads.make_W(n0, H, 3).view(np.int16)).view(torch.bfloat16).to(device)
    out = {"shard": [a0, n0], "H": H, "V": V, "V_true": Vt}
    for T in (796, 1820, 6827):
        h = torch.from_numpy(workloads.make_h(T, H, T).view(np.int16)).view(torch.bfloat16).to(device)
        y = torch.from_numpy(workloads.make_y(T, Vt, T)).to(device)
        g = torch.from_numpy(np.random.default_rng(T).standard_normal(T).astype(np.float32)).to(device)
        parts = torch.empty((2, T, 3), dtype=torch.float32, device=device)
        parts[1, :, 0], parts[1, :, 1], parts[1, :, 2] = 5.0, 1000.0, float("-inf")  # other shard
        logp = torch.empty(T, dtype=torch.float32, device=device)
        lse = torch.empty(T, dtype=torch.float32, device=device)
        dHp = torch.empty((T, H), dtype=torch.float32, device=device)
        dW = torch.empty((n0, H), dtype=torch.float32, device=device)
        fws = torch.empty(rlk.fwd_workspace_bytes(T, H, n0), dtype=torch.uint8, device=device)
        bws = torch.empty(rlk.bwd_workspace_bytes(T, H, n0), dtype=torch.uint8, device=device)

        def fwd():
            rlk.linear_logp_fwd(h, W, y, Vt, vocab_start=a0, partial=True, out=(parts[0],),
                                workspace=fws)
            rlk.lse_merge(parts, out=(logp, lse))

        def fwd_bwd():
            fwd()
            rlk.linear_logp_bwd(h, W, y, lse, g, Vt, vocab_start=a0, dH_fp32_partial=True,
                                out=(dHp, dW), workspace=bws)

        K = max(args.steps, 10)
        f_ms, fb_ms = _time_calls(torch, device, fwd, K), _time_calls(torch, device, fwd_bwd, K)
        flops = 2.0 * T * H * min(n0, Vt - a0)
        # memory of one forward + backward call pair whose every buffer (workspaces, statistics,
        # dH partial, dW rows) the binding allocates, with the inputs already resident
        torch.cuda.synchronize(device)
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats(device)
        m_alloc, m_res = torch.cuda.memory_allocated(device), torch.cuda.memory_reserved(device)
        p0 = rlk.linear_logp_fwd(h, W, y, Vt, vocab_start=a0, partial=True)
        lp, ls = rlk.lse_merge(torch.stack([p0, parts[1]]))
        dh_m, dw_m = rlk.linear_logp_bwd(h, W, y, ls, g, Vt, vocab_start=a0, dH_fp32_partial=True)
        torch.cuda.synchronize(device)
        mem = {"peak_allocated_delta_MB": (torch.cuda.max_memory_allocated(device) - m_alloc) / 2**20,
               "peak_reserved_delta_MB": (torch.cuda.max_memory_reserved(device) - m_res) / 2**20}
        del p0, lp, ls, dh_m, dw_m
        out[str(T)] = {"fwd_ms": f_ms, "fwd_bwd_ms": fb_ms, "memory": mem,
                       "fwd_tflops": flops / (f_ms / 1e3) / 1e12,
                       "fwd_bwd_tflops": 3 * flops / (fb_ms / 1e3) / 1e12,
                       "fwd_frac_of_burst": flops / (f_ms / 1e3) / 1e12 / peak}
    out["note"] = ("per-rank single-operator times; the backward's recompute GEMM is not "
                   "counted in fwd_bwd_tflops (3 GEMM-equivalents credited, 4 run); memory = peak "
                   "delta of one fwd + bwd call pair with every buffer allocated by the binding "
                   "(dz workspace, fp32 dH partial, fp32 dW rows of the shard), inputs excluded")
    return out


def tiny_leg(rlk, torch, device, args, gpu_id):
    """The tiny workload (T = 64, H = 256, V = V_true = 4096) fwd+bwd: launch-bound."""
    w = workloads.TINY
    d = workloads.make_inputs(w)
    path = Path(rlk, torch, w, d, device)
    K = max(50, args.steps)
    for _ in range(max(3, args.warmup)):
        path.forward()
        path.backward()
    torch.cuda.synchronize(device)
    sampler = ClockSampler(gpu_id) if gpu_id else None
    if sampler:
        sampler.wait_running()
        sampler.mark_start()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(K):
        path.forward()
        path.backward()
    b.record()
    torch.cuda.synchronize(device)
    if sampler:
        sampler.mark_end()
    clocks = sampler.stop() if sampler else None
    ms = a.elapsed_time(b) / K
    # the same step captured once in a CUDA graph and replayed: what remains is the kernels'
    # own latency (prologue, one short tile pass, tail) without the host's launch overhead
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            path.forward()
            path.backward()
    torch.cuda.current_stream(device).wait_stream(side)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize(device)
    a.record()
    for _ in range(K):
        graph.replay()
    b.record()
    torch.cuda.synchronize(device)
    gms = a.elapsed_time(b) / K
    del graph
    return {"workload": config_dict(w, 1)["workload"], "tokens_per_s": w.T / (ms / 1e3),
            "us_per_step": ms * 1e3, "steps": K, "gpu_launches_per_step": path.launches_per_step(),
            "graph_replay": {"us_per_step": gms * 1e3, "tokens_per_s": w.T / (gms / 1e3)},
            "bound": "launch latency (5 kernels of a few microseconds each)", "clocks": clocks}


def saved_logits_leg(rlk, torch, path, w, device, args, peak, peak_sus):
    """The same fwd+bwd step through the saved-logits pair (forward stores fp32 z,
    backward forms dz from it instead of recomputing the logits GEMM)."""
    z = rlk.saved_logits_buffer(w.T, w.V, device)

    def step():
        rlk.linear_logp_fwd_save(path.h, path.W, path.y, w.V_true, z_saved=z,
                                 out=(path.logp, path.lse), workspace=path.fws)
        rlk.linear_logp_bwd_saved(path.h, path.W, path.y, path.lse, path.g, z, w.V_true,
                                  out=(path.dH, path.dW), workspace=path.bws)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(device)
    K = args.steps
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(K):
        step()
    b.record()
    torch.cuda.synchronize(device)
    ms = a.elapsed_time(b) / K
    # the parts: the forward that also stores z, and dz formed from z alone (an HBM-bound
    # pass: fp32 z of the columns below V_true read, bf16 dz of all padded columns written)
    fwd_ms = _time_calls(torch, device, lambda: rlk.linear_logp_fwd_save(
        path.h, path.W, path.y, w.V_true, z_saved=z, out=(path.logp, path.lse), workspace=path.fws), K)
    dz_ms = _time_calls(torch, device, lambda: rlk.linear_logp_bwd_saved(
        path.h, path.W, path.y, path.lse, path.g, z, w.V_true, want_dH=False, want_dW=False,
        out=(None, None), workspace=path.bws), K)
    dz_bytes = w.T * w.V_true * 4 + w.T * (-(-w.V // 256) * 256) * 2
    hbm = _peaks_hbm()
    del z
    step_flops = 3.0 * 2.0 * w.T * w.H * w.V_true
    return {"tokens_per_s": w.T / (ms / 1e3), "ms_per_step": ms,
            "frac_of_burst": step_flops / (peak * 1e12) / (ms / 1e3),
            "frac_of_sustained": step_flops / (peak_sus * 1e12) / (ms / 1e3),
            "saved_logits_bytes": rlk.saved_logits_bytes(w.T, w.V), "steps": K,
            "gpu_launches_per_step": 5,
            "forward_with_save_ms": fwd_ms,
            "dz_from_logits": {"ms": dz_ms, "algorithmic_bytes": dz_bytes,
                               "GBps": dz_bytes / (dz_ms / 1e3) / 1e9,
                               "frac_of_hbm": dz_bytes / (dz_ms / 1e3) / 1e9 / hbm}}


def _peaks_hbm():
    peaks, _ = load_peaks()
    return float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))


def small_t_leg(rlk, torch, path, device, peaks, gpu_id=None):
    """Forward latency at small T (the batch-invariance workload's batch sizes) on the
    Qwen3-8B weight: these calls stream W once and are HBM-bound; reported as achieved
    GB/s of algorithmic bytes (W + h read, statistics written) against measured HBM.
    Runs before the power-capped legs, with its own clock record."""
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    W = path.W
    V, H = W.shape
    Vt = path.w.V_true
    out = {}
    sampler = ClockSampler(gpu_id) if gpu_id else None
    if sampler:
        sampler.wait_running()
        sampler.mark_start()
    for T in (1, 7, 128, 1000):
        h = torch.from_numpy(workloads.make_h(T, H, 9).view(np.int16)).view(torch.bfloat16).to(device)
        y = torch.from_numpy(workloads.make_y(T, Vt, 9)).to(device)
        logp = torch.empty(T, dtype=torch.float32, device=device)
        lse = torch.empty(T, dtype=torch.float32, device=device)
        ws = torch.empty(rlk.fwd_workspace_bytes(T, H, V), dtype=torch.uint8, device=device)
        for _ in range(5):
            rlk.linear_logp_fwd(h, W, y, Vt, out=(logp, lse), workspace=ws)
        # five repeats of 20 back-to-back calls, the median repeat reported: right after the
        # heavy legs the power controller is still settling, which moved single repeats by ~10 %
        n, reps = 20, []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(device)
            a.record()
            for _ in range(n):
                rlk.linear_logp_fwd(h, W, y, Vt, out=(logp, lse), workspace=ws)
            b.record()
            torch.cuda.synchronize(device)
            reps.append(a.elapsed_time(b) / n)
        ms = statistics.median(reps)
        nbytes = V * H * 2 + T * H * 2 + 3 * 4 * T * -(-V // 1024)
        gbs = nbytes / (ms / 1e3) / 1e9
        out[str(T)] = {"us_per_call": ms * 1e3, "us_per_call_best": min(reps) * 1e3,
                       "algorithmic_GBps": gbs, "frac_of_hbm": gbs / hbm}
    if sampler:
        sampler.mark_end()
    out["clocks"] = sampler.stop() if sampler else None
    out["note"] = ("W and L2 are not flushed between calls; W (1.24 GB) exceeds L2 on its own; "
                   "median of 5 repeats of 20 calls; run first, before the power-capped legs")
    return out


def saved_probs_leg(rlk, torch, path, w, device, args, peak):
    """The fwd+bwd step through the saved bf16-probabilities pair."""
    pbuf = torch.empty(rlk.saved_probs_bytes(w.T, w.V), dtype=torch.uint8, device=device)

    def step():
        rlk.linear_logp_fwd_save_probs(path.h, path.W, path.y, w.V_true, p_saved=pbuf,
                                       out=(path.logp, path.lse), workspace=path.fws)
        rlk.linear_logp_bwd_saved_probs(path.h, path.W, path.y, path.lse, path.g, pbuf, w.V_true,
                                        out=(path.dH, path.dW), workspace=path.bws)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(device)
    K = args.steps
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(K):
        step()
    b.record()
    torch.cuda.synchronize(device)
    ms = a.elapsed_time(b) / K
    # the parts: the forward that also stores the probabilities, and dz formed from them
    # alone (HBM-bound: bf16 e(z - m) of the columns below V_true and the fp32 chunk maxima
    # read, bf16 dz of all padded columns written)
    fwd_ms = _time_calls(torch, device, lambda: rlk.linear_logp_fwd_save_probs(
        path.h, path.W, path.y, w.V_true, p_saved=pbuf, out=(path.logp, path.lse),
        workspace=path.fws), K)
    dz_ms = _time_calls(torch, device, lambda: rlk.linear_logp_bwd_saved_probs(
        path.h, path.W, path.y, path.lse, path.g, pbuf, w.V_true, want_dH=False, want_dW=False,
        out=(None, None), workspace=path.bws), K)
    Vd = -(-w.V // 256) * 256
    dz_bytes = w.T * w.V_true * 2 + w.T * (Vd // 64) * 4 + w.T * Vd * 2
    hbm = _peaks_hbm()
    del pbuf
    step_flops = 3.0 * 2.0 * w.T * w.H * w.V_true
    return {"tokens_per_s": w.T / (ms / 1e3), "ms_per_step": ms,
            "frac_of_burst": step_flops / (peak * 1e12) / (ms / 1e3),
            "saved_probs_bytes": rlk.saved_probs_bytes(w.T, w.V), "steps": K,
            "forward_with_save_ms": fwd_ms,
            "dz_from_probs": {"ms": dz_ms, "algorithmic_bytes": dz_bytes,
                              "GBps": dz_bytes / (dz_ms / 1e3) / 1e9,
                              "frac_of_hbm": dz_bytes / (dz_ms / 1e3) / 1e9 / hbm}}


def _time_calls(torch, device, fn, K, warmup=3):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(K):
        fn()
    b.record()
    torch.cuda.synchronize(device)
    return a.elapsed_time(b) / K


def fp8_leg(rlk, torch, path, w, device, args, peak_bf16):
    """The FP8 (E4M3, per-row power-of-two scales) LM head on the Qwen3-8B weight:
    forward-only at T = 4096 with the weight codes resident (inference-style) and with
    the weight re-quantized every call (training-style); the straight-through fwd+bwd
    step at T = 8192 (quantize W and h, FP8 forward, FP8 dz recompute, bf16 dH / dW).
    The FP8 GEMM rate is reported against 2x the measured bf16 burst (the nominal
    dense fp8 : bf16 tensor ratio, 4.5 : 2.25 PFLOP/s)."""
    peak8 = 2.0 * peak_bf16
    K = max(args.steps, 10)
    W = path.W
    V, H = W.shape
    Vt = w.V_true
    Wq = torch.empty((V, H), dtype=torch.uint8, device=device)
    Ws = torch.empty(V, dtype=torch.float32, device=device)
    out = {"format": "OCP E4M3, one power-of-two scale per row", "peak_tflops_fp8": peak8,
           "peak_source": "2 x measured bf16 burst (nominal dense fp8:bf16 ratio)"}

    wf = workloads.QWEN3_8B_FWD
    h4 = torch.from_numpy(workloads.make_h(wf.T, H, 0).view(np.int16)).view(torch.bfloat16).to(device)
    y4 = torch.from_numpy(workloads.make_y(wf.T, Vt, 0)).to(device)
    hq4 = torch.empty((wf.T, H), dtype=torch.uint8, device=device)
    hs4 = torch.empty(wf.T, dtype=torch.float32, device=device)
    lp4 = torch.empty(wf.T, dtype=torch.float32, device=device)
    ls4 = torch.empty(wf.T, dtype=torch.float32, device=device)
    ws4 = torch.empty(rlk.fwd_workspace_bytes(wf.T, H, V), dtype=torch.uint8, device=device)
    rlk.quantize_rows_e4m3(W, out=(Wq, Ws))

    def fwd_resident():
        rlk.quantize_rows_e4m3(h4, out=(hq4, hs4))
        rlk.linear_logp_fwd_fp8(hq4, hs4, Wq, Ws, y4, Vt, out=(lp4, ls4), workspace=ws4)

    def fwd_gemm_only():
        rlk.linear_logp_fwd_fp8(hq4, hs4, Wq, Ws, y4, Vt, out=(lp4, ls4), workspace=ws4)

    def fwd_requant():
        rlk.quantize_rows_e4m3(W, out=(Wq, Ws))
        fwd_resident()

    def quant_W():
        rlk.quantize_rows_e4m3(W, out=(Wq, Ws))

    flops4 = 2.0 * wf.T * H * Vt
    ms_g = _time_calls(torch, device, fwd_gemm_only, K)
    ms_r = _time_calls(torch, device, fwd_resident, K)
    ms_q = _time_calls(torch, device, fwd_requant, K)
    ms_w = _time_calls(torch, device, quant_W, K)
    qbytes = V * H * 3 + V * 4     # read bf16 W, write codes and scales
    out["forward_T4096"] = {
        "workload": f"{wf.name} T={wf.T} H={H} V={V} V_true={Vt}",
        "gemm_call_ms": ms_g, "gemm_tflops": flops4 / (ms_g / 1e3) / 1e12,
        "gemm_frac_of_fp8_peak": flops4 / (ms_g / 1e3) / 1e12 / peak8,
        "tokens_per_s_W_resident": wf.T / (ms_r / 1e3), "ms_W_resident": ms_r,
        "tokens_per_s_W_requantized": wf.T / (ms_q / 1e3), "ms_W_requantized": ms_q}
    out["quantize_W"] = {"ms": ms_w, "GBps": qbytes / (ms_w / 1e3) / 1e9}
    del hq4, hs4, lp4, ls4, ws4

    hq = torch.empty((w.T, H), dtype=torch.uint8, device=device)
    hs = torch.empty(w.T, dtype=torch.float32, device=device)

    def step():
        rlk.quantize_rows_e4m3(W, out=(Wq, Ws))
        rlk.quantize_rows_e4m3(path.h, out=(hq, hs))
        rlk.linear_logp_fwd_fp8(hq, hs, Wq, Ws, path.y, Vt, out=(path.logp, path.lse),
                                workspace=path.fws)
        rlk.linear_logp_bwd_fp8(path.h, W, hq, hs, Wq, Ws, path.y, path.lse, path.g, Vt,
                                out=(path.dH, path.dW), workspace=path.bws)

    ms = _time_calls(torch, device, step, args.steps)
    step_flops = 3.0 * 2.0 * w.T * H * Vt
    out["ste_fwd_bwd_T8192"] = {
        "tokens_per_s": w.T / (ms / 1e3), "ms_per_step": ms,
        "frac_of_bf16_burst": step_flops / (peak_bf16 * 1e12) / (ms / 1e3),
        "gpu_launches_per_step": 7, "steps": args.steps,
        "note": "per step: quantize W and h, FP8 forward (2 kernels), FP8 dz + bf16 dH + bf16 dW"}
    del Wq, Ws, hq, hs
    return out


def fwd_only(rlk, torch, W_bits, path, device, args, peak):
    """Forward-only tokens/s on the Qwen3-8B forward workload (T=4096), same W."""
    w = workloads.QWEN3_8B_FWD
    h = torch.from_numpy(workloads.make_h(w.T, w.H, 0).view(np.int16)).view(torch.bfloat16).to(device)
    y = torch.from_numpy(workloads.make_y(w.T, w.V_true, 0)).to(device)
    logp = torch.empty(w.T, dtype=torch.float32, device=device)
    lse = torch.empty(w.T, dtype=torch.float32, device=device)
    ws = torch.empty(rlk.fwd_workspace_bytes(w.T, w.H, w.V), dtype=torch.uint8, device=device)
    W = path.W
    for _ in range(max(3, args.warmup)):
        rlk.linear_logp_fwd(h, W, y, w.V_true, out=(logp, lse), workspace=ws)
    K = max(args.steps, 10)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    a.record()
    for _ in range(K):
        rlk.linear_logp_fwd(h, W, y, w.V_true, out=(logp, lse), workspace=ws)
    b.record()
    torch.cuda.synchronize(device)
    ms = a.elapsed_time(b) / K
    tf = 2.0 * w.T * w.H * w.V_true / (ms / 1e3) / 1e12
    return {"workload": f"{w.name} T={w.T} H={w.H} V={w.V} V_true={w.V_true}",
            "tokens_per_s": w.T / (ms / 1e3), "ms_per_call": ms, "tflops": tf,
            "frac_of_burst": tf / peak, "steps": K}


def e2e(rlk, torch, path, w, d, device, args, gpu_id=None, world=1):
    """Same step through the public API from pinned host buffers: every step copies
    its inputs (h, y, g) host -> device, runs the C-ABI calls and copies its result
    (logp) device -> host, all inside the timed region. The weight W is model state
    and stays resident, as in a training step. Like a training input pipeline, the
    copies of step k+1's inputs run on a second stream into a second set of device
    buffers while step k computes (double buffering, ordered by events). With several
    ranks, each runs its own batch between two barriers, and the job's throughput is
    every rank's tokens over the slowest rank's time."""
    h_host = torch.from_numpy(d["h"].view(np.int16)).view(torch.bfloat16).pin_memory()
    y_host = torch.from_numpy(d["y"]).pin_memory()
    g_host = torch.from_numpy(d["g"]).pin_memory()
    logp_host = torch.empty(w.T, dtype=torch.float32).pin_memory()
    h2d = h_host.numel() * 2 + y_host.numel() * 8 + g_host.numel() * 4
    d2h = logp_host.numel() * 4
    sets = [(path.h, path.y, path.g),
            (torch.empty_like(path.h), torch.empty_like(path.y), torch.empty_like(path.g))]
    compute = torch.cuda.current_stream(device)
    copy = torch.cuda.Stream(device)
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]

    def load(i):  # H2D of one step's inputs into set i, after the compute that last read it
        with torch.cuda.stream(copy):
            copy.wait_event(done[i])
            for dst, src in zip(sets[i], (h_host, y_host, g_host)):
                dst.copy_(src, non_blocking=True)
            ready[i].record(copy)

    def run(K):
        for i in range(2):
            done[i].record(compute)
        load(0)
        for k in range(K):
            i = k % 2
            if k + 1 < K:
                load(1 - i)                       # prefetch the next step's inputs
            compute.wait_event(ready[i])
            path.h, path.y, path.g = sets[i]
            path.forward()
            path.backward()
            logp_host.copy_(path.logp, non_blocking=True)   # D2H of the step's result
            done[i].record(compute)
        compute.wait_stream(copy)

    run(max(3, args.warmup))
    torch.cuda.synchronize(device)
    K = args.steps
    sampler = ClockSampler(gpu_id) if gpu_id else None
    if sampler:
        sampler.wait_running()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    if sampler:
        sampler.mark_start()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(compute)
    run(K)
    b.record(compute)
    torch.cuda.synchronize(device)
    if sampler:
        sampler.mark_end()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    path.h, path.y, path.g = sets[0]
    ms = max_over_ranks(a.elapsed_time(b), world, device) / K
    out = {"value": w.T * world / (ms / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d * world, "d2h_bytes_per_step": d2h * world, "ms_per_step": ms,
           "pipeline": "inputs of step k+1 copied on a second stream while step k computes",
           "d2h": ("logp only; dH and dW stay on the device, where the model's backward and the "
                   "optimizer consume them"),
           "clocks": clocks}
    if world > 1:
        out["h2d_bytes_per_step_per_rank"] = h2d
        out["d2h_bytes_per_step_per_rank"] = d2h
    return out


def run_vocab_parallel(args, w: workloads.Workload, rank: int, world: int, local_rank: int):
    """--parallel vocab: the ranks hold one contiguous shard of W each (shard_bounds(V, V_true, S),
    S = the number of ranks) and the same batch; a step is the forward and backward across the
    group (deterministic_token_logprob_gb300.vocab_parallel: all-gather of the shard statistics
    and rlk_lse_merge; fp32 dH partials summed in rank order by all-to-all, rlk_shard_sum_bf16
    and all-gather; dW rows local). The total work is fixed, so this is strong scaling."""
    import torch

    import deterministic_token_logprob_gb300 as rlk
    from deterministic_token_logprob_gb300 import build as libbuild
    from deterministic_token_logprob_gb300 import vocab_parallel as vp
    if rank == 0:
        libbuild.build()
    torch.distributed.barrier()
    device = torch.device("cuda", local_rank)
    peaks, peaks_src = load_peaks()
    start, n = vp.shard_of_rank(w.V, w.V_true)
    d = workloads.make_inputs(w, with_W=False)   # the same batch on every rank (seed 0)
    W_bits = workloads.make_W(w.V, w.H, seed=0)[start:start + n]
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)  # noqa: E731
    h, W = bf(d["h"]), bf(W_bits)
    y, g = torch.from_numpy(d["y"]).to(device), torch.from_numpy(d["g"]).to(device)
    fws = torch.empty(rlk.fwd_workspace_bytes(w.T, w.H, n), dtype=torch.uint8, device=device)
    bws = torch.empty(rlk.bwd_workspace_bytes(w.T, w.H, n), dtype=torch.uint8, device=device)

    def step():
        _, lse = vp.linear_logp_fwd_tp(h, W, y, w.V_true, w.V, workspace=fws)
        vp.linear_logp_bwd_tp(h, W, y, lse, g, w.V_true, w.V, workspace=bws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    K = args.steps
    sampler = ClockSampler(gpu_uuid(torch, device)) if rank == 0 else None
    if sampler:
        sampler.wait_running()
    torch.distributed.barrier()
    torch.cuda.synchronize(device)
    if sampler:
        sampler.mark_start()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(K):
        step()
    b.record()
    torch.cuda.synchronize(device)
    if sampler:
        sampler.mark_end()
    torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    total_ms = max_over_ranks(a.elapsed_time(b), world, device)
    ms = total_ms / K
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    step_flops = 3.0 * 2.0 * w.T * w.H * w.V_true
    line = {"metric": METRIC, "value": w.T / (ms / 1e3), "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(config_dict(w, world), parallelism=f"vocab{world}",
                           global_tokens=w.T, shard_of_rank_0=list(rlk.shard_bounds(w.V, w.V_true, world)[0])),
            "gpu_launches": K * 7,  # per rank and step: forward 2 + merge 1, backward 3 + sum 1
            "step_roofline": {"flops_counted": step_flops,
                              "frac_of_burst": step_flops / (peak * world * 1e12) / (ms / 1e3),
                              "peak_source": f"{peaks_src} bf16 burst x {world} GPUs"},
            "clocks": clocks}
    if rank == 0:
        print_line(line)


def run_case(args):
    """One stage of the path at the Qwen3-8B H and V with --tokens tokens, timed per call
    with CUDA events (for per-kernel timing and small-case ncu captures)."""
    import torch

    import deterministic_token_logprob_gb300 as rlk
    from deterministic_token_logprob_gb300 import build as libbuild
    libbuild.build()
    base = workloads.QWEN3_8B
    V = args.vocab or base.V
    V_true = V - (base.V - base.V_true) if V > base.V - base.V_true else V
    w = workloads.Workload(f"case_{args.case}", T=args.tokens, H=base.H, V=V, V_true=V_true,
                           g_kind="grpo")
    d = workloads.make_inputs(w)
    dev = torch.device("cuda", 0)
    path = Path(rlk, torch, w, d, dev, with_dW=args.case == "dw")
    path.forward()
    if args.case == "fwd":
        call = path.forward
    elif args.case in ("fwd8", "dz8"):
        hq, hs = rlk.quantize_rows_e4m3(path.h)
        Wq, Ws = rlk.quantize_rows_e4m3(path.W)
        if args.case == "fwd8":
            def call():
                rlk.linear_logp_fwd_fp8(hq, hs, Wq, Ws, path.y, w.V_true, out=(path.logp, path.lse),
                                        workspace=path.fws)
        else:
            def call():
                rlk.linear_logp_bwd_fp8(path.h, path.W, hq, hs, Wq, Ws, path.y, path.lse, path.g,
                                        w.V_true, out=(None, None), want_dH=False, want_dW=False,
                                        workspace=path.bws)
    else:
        want_dH, want_dW = args.case == "dh", args.case == "dw"

        def call():
            rlk.linear_logp_bwd(path.h, path.W, path.y, path.lse, path.g, w.V_true,
                                out=(path.dH if want_dH else None, path.dW if want_dW else None),
                                want_dH=want_dH, want_dW=want_dW, workspace=path.bws)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    ms = []
    for _ in range(args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        torch.cuda.synchronize(dev)
        ms.append(a.elapsed_time(b))
    flops = 2.0 * w.T * w.H * w.V_true * (1 if args.case in ("fwd", "dz", "fwd8", "dz8") else 2)
    print(json.dumps({"case": args.case, "T": w.T, "H": w.H, "V": w.V, "V_true": w.V_true,
                      "ms": ms, "tflops_best": flops / (min(ms) / 1e3) / 1e12,
                      "kernels_per_call": {"fwd": 2, "dz": 1, "dh": 2, "dw": 2, "fwd8": 2,
                                           "dz8": 1}[args.case]}),
          flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["rlk", "reference"], default="rlk")
    ap.add_argument("--workload", choices=["qwen3_8b", "qwen3_30b_tp2", "tiny"], default="qwen3_8b")
    ap.add_argument("--quick", action="store_true", help="skip the forward-only, e2e and CPU legs")
    ap.add_argument("--parallel", choices=["replicas", "vocab"], default="replicas",
                    help="replicas: one independent batch per rank (default); vocab: one batch, "
                         "W split into one vocab shard per rank (1, 2, 4 or 8 ranks)")
    ap.add_argument("--case", choices=["fwd", "dz", "dh", "dw", "fwd8", "dz8"], default=None,
                    help="time one stage only (dz alone; dh / dw each after its dz)")
    ap.add_argument("--tokens", type=int, default=1024, help="tokens for --case")
    ap.add_argument("--vocab", type=int, default=0,
                    help="vocab rows for --case (default 151936; V_true = V - 267)")
    ap.add_argument("--record-traffic", metavar="NCU_CSV", default=None,
                    help="write the per-launch DRAM traffic of an ncu --csv capture of the "
                         "qwen3_8b step to profiles/traffic_qwen3_8b.json and exit")
    ap.add_argument("--traffic-command", default="", help="the command that made NCU_CSV")
    args = ap.parse_args()
    if args.record_traffic:
        print(json.dumps(record_traffic(args.record_traffic, args.traffic_command), indent=1))
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.case:
        run_case(args)
        return
    w = workloads.CONFIGS[args.workload]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    vocab = args.parallel == "vocab"
    if vocab and world not in (1, 2, 4, 8):
        ap.error("--parallel vocab needs 1, 2, 4 or 8 ranks")
    if world > 1 or vocab:
        import torch
        torch.cuda.set_device(local_rank)
        if world > 1:
            torch.distributed.init_process_group("nccl")
        else:   # a one-rank group, so that the exchange runs its collectives
            torch.distributed.init_process_group(
                "nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1)
    try:
        if vocab:
            run_vocab_parallel(args, w, rank, world, local_rank)
        else:
            run_gpu(args, w, rank, world, local_rank)
    finally:
        if world > 1 or vocab:
            import torch
            torch.distributed.destroy_process_group()


def _free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


if __name__ == "__main__":
    main()

"""Benchmark: row-wise online softmax on GB300, one JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one softmax over the whole workload matrix (every kernel the path launches for it).
The default headline workload is the largest of the problem statement that fits one GPU: bf16
attention-score-shaped rows, 4 x 32 heads x 4096 queries = 524,288 rows over 4096 keys, scores
z / sqrt(128) with z ~ N(0, 1) (seed 4), keys after the query set to -inf in the matrix, every
entry read.  By default (one GPU) the line also carries, under "configs", the other workloads
of 4096 x 4096 and larger, each timed over the same K steps: fp32 4096 x 4096 (the shape
measured on "5.2 CUDA Online Softmax 实现优化" §2.4; AUTO, the one-read shared-memory and the
two-pass kernels), bf16 16384 x 32768 logits with per-row LSE, fp32 32 x 4,194,304 long rows,
and the causal workload through softmax_rows_causal (masked keys not read).  Inputs are
synthetic (synth/) and already resident in HBM when timing starts.

Metric: effective HBM GB/s with minimum bytes = read x once + write y once (2 M N s), plus
rows/s and the fraction of the HBM roofline.  L2: steps rotate over enough input/output buffer
sets that every step's operands are evicted from L2 (126 MB) before they are used again; each
batch of steps is one CUDA graph replay, timed with CUDA events on the launching stream.

Multi-GPU (torchrun): rows are independent, so each rank processes its own shard (its own
rows of the same seeded matrix) with no data-path collective: weak scaling, max time over ranks.

--impl reference times the fp64 CPU oracle (oracle/) on the host cores, on a bounded sample of
the same workload per step.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "softmax effective HBM GB/s (read+write once) and % of GB300 HBM peak, rows/s"
DEFAULT_WORKLOAD = "bf16_causal_4x32x4096x4096"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES_NOMINAL = 126 * 2 ** 20
# The pages' best number on this workload: V3 register-cached one-pass, A100 80GB SXM4, fp32,
# M = N = 4096, about 1672 GB/s ("5.2 CUDA Online Softmax 实现优化" §6.3).  Another machine.
PAGE_GBS = {"fp32_4096x4096": 1672.0}


# ----------------------------------------------------------------------------------------------
# helpers shared with the tests (no GPU needed)
# ----------------------------------------------------------------------------------------------

def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard_row0(rank: int, rows_per_rank: int) -> int:
    """First global row of a rank's shard: rank r owns rows [r * M, (r + 1) * M)."""
    return rank * rows_per_rank


def reduce_max(value: float, world: int) -> float:
    """Max of a float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    backend = dist.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def measured_hbm_peak() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def code_only(text: str) -> str:
    """C++ / CUDA source without its comments (string and character literals kept), blank lines
    and runs of white space (one space between tokens): what a change of comments or layout
    leaves unchanged."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(" ".join(line.split()) for line in "".join(out).splitlines() if line.strip())


def kernel_source_hash(files=None) -> str:
    """Hash of the code (comments excluded) of the named files of row_wise_online_gb300/csrc (all
    of them when files is None)."""
    csrc = os.path.join(ROOT, "row_wise_online_gb300", "csrc")
    paths = sorted(glob.glob(os.path.join(csrc, "*"))) if files is None else [os.path.join(csrc, f) for f in sorted(files)]
    h = hashlib.sha256()
    for p in paths:
        with open(p, encoding="utf-8") as fh:
            h.update(os.path.basename(p).encode())
            h.update(code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str) -> float | None:
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current sources
    (the summary names the source files its kernel is built from, and their hash)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}__{workload}.md")
    try:
        text = open(path, encoding="utf-8").read()
    except OSError:
        return None
    src = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    files = re.search(r"source_files:\s*(.+)", text)
    tb = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not src or not tb:
        return None
    try:
        current = kernel_source_hash(files.group(1).split() if files else None)
    except OSError:
        return None
    return float(tb.group(1)) if src.group(1) == current else None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.proc = None
        self.out = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm = [float(r[1]) for r in rows]
        smax = max(float(r[2]) for r in rows)
        power = [float(r[3]) for r in rows]
        loaded = [s for s, p in zip(sm, power) if p >= 0.6 * max(power)] or sm
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power)}


# ----------------------------------------------------------------------------------------------
# the CUDA arm
# ----------------------------------------------------------------------------------------------

def _pinned_workload(w: synth.Workload, row0: int):
    import torch

    tdt = torch.float32 if w.dtype == synth.F32 else torch.int16
    host = torch.empty((w.M, w.N), dtype=tdt).pin_memory()
    synth.fill(w, host.data_ptr(), row0, w.M)
    if w.dtype == synth.BF16:
        host = host.view(torch.bfloat16)
    return host


def _graph_time(run_step, nsteps: int, stream, graph_batch: int):
    """Capture `graph_batch` steps in a CUDA graph, replay to cover exactly nsteps; return ms."""
    import torch

    full, rest = divmod(nsteps, graph_batch)
    graphs = []
    for count in ((graph_batch,) if full else ()) + ((rest,) if rest else ()):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(count):
                run_step(i)
        graphs.append((g, count))
    return graphs, full, rest


# The configurations timed by default, in the order they run.  The first is the headline: the
# largest workload of the problem statement (bf16 attention-score-shaped rows, 524,288 x 4096,
# causal -inf written into the matrix, every entry read).  The others are the remaining
# workloads of 4096 x 4096 and larger, with the variants the statement asks to measure.
#   (label, workload, mode, forced variant or None, state outputs)
SUITE = (
    ("bf16_causal_4x32x4096x4096", "bf16_causal_4x32x4096x4096", "softmax", None, ""),
    ("fp32_4096x4096", "fp32_4096x4096", "softmax", None, ""),
    ("fp32_4096x4096/oneread_smem", "fp32_4096x4096", "softmax", "smem", ""),
    ("fp32_4096x4096/twopass", "fp32_4096x4096", "softmax", "twopass", ""),
    ("bf16_logits_16384x32768+lse", "bf16_logits_16384x32768", "softmax", None, "lse"),
    ("fp32_longrow_32x4194304", "fp32_longrow_32x4194304", "softmax", None, ""),
    ("bf16_causal_4x32x4096x4096/causal_skip", "bf16_causal_4x32x4096x4096", "causal", None, ""),
)

VARIANT_ARG = {"auto": 0, "reg": 1, "smem": 2, "twopass": 3, "splitrow": 4, "splitrow_stream": 5}


class _Run:
    """One workload's buffers on this rank's device, and the step that softmaxes it."""

    def __init__(self, w: synth.Workload, row0: int, dev, stream, mode: str, state: str, host_x=None):
        import torch

        import row_wise_online_gb300 as rwo

        self.w, self.mode, self.stream, self.rwo = w, mode, stream, rwo
        if host_x is None:
            host_x = _pinned_workload(w, row0)
        self.host_x = host_x
        set_bytes = 2 * w.M * w.N * w.elem_bytes
        # rotate over enough buffer sets that a step's operands were evicted from L2 since last use
        self.nbuf = 1 if set_bytes >= 4 * L2_BYTES_NOMINAL else max(2, -(-4 * L2_BYTES_NOMINAL // set_bytes))
        self.set_bytes = set_bytes
        self.xs = [host_x.to(dev) for _ in range(self.nbuf)]
        self.ys = [torch.empty_like(self.xs[0]) for _ in range(self.nbuf)]
        self.lse = torch.empty(w.M, dtype=torch.float32, device=dev) if "lse" in state else None
        if mode == "ce":  # synthetic labels, uniform over the classes
            self.labels = torch.from_numpy(np.random.default_rng(5).integers(0, w.N, w.M)).to(dev)
            self.loss = torch.empty(w.M, dtype=torch.float32, device=dev)
        self.variant = rwo.VARIANT_AUTO

    def step(self, i: int) -> None:
        rwo, w, k = self.rwo, self.w, i % self.nbuf
        if self.mode == "causal":  # masked keys are not read: the causal rule replaces the -inf entries
            rwo.softmax_rows_causal(self.xs[k], w.causal_q, 0, self.ys[k], lse_out=self.lse, stream=self.stream)
        elif self.mode == "log":
            rwo.log_softmax_rows(self.xs[k], self.ys[k], lse_out=self.lse, stream=self.stream)
        elif self.mode == "ce":
            rwo.cross_entropy_rows(self.xs[k], self.labels, self.loss, stream=self.stream)
        else:
            rwo.softmax_rows_ex(self.xs[k], self.ys[k], lse_out=self.lse, variant=self.variant, stream=self.stream)

    def bytes_per_step(self) -> int:
        """The metric's bytes: read x once + write y once (x + labels + losses for cross entropy)."""
        w = self.w
        if self.mode == "ce":
            return w.M * w.N * w.elem_bytes + 12 * w.M
        return w.min_bytes

    def algorithmic_bytes(self, row0: int) -> int:
        """Bytes the launch must move: the metric's bytes, or for the causal skip the live prefix of
        every row (whole 16-byte vectors) plus all of y; state outputs add 4 bytes per row each."""
        w = self.w
        b = self.bytes_per_step()
        if self.mode == "causal":
            vec = 16 // w.elem_bytes
            r = np.arange(row0, row0 + w.M, dtype=np.int64)
            live = np.clip(r % w.causal_q + 1, 0, w.N)
            b = int(((live + vec - 1) // vec).sum()) * 16 + w.M * w.N * w.elem_bytes
        if self.lse is not None:
            b += 4 * w.M
        return b

    def release(self) -> None:
        self.xs = self.ys = None


def _time_steps(run: _Run, nsteps: int, warm: int, world: int, dev) -> tuple[float, dict]:
    """Time exactly nsteps steps of `run` between CUDA events on its stream; returns (ms, spread).

    Warm-up steps run eagerly; the steps are then captured in CUDA graphs of up to 256 steps (a
    multiple of the buffer rotation).  After the barrier and synchronisation that open the timed
    region, one untimed replay is issued right before the first event, so the GPU is busy and at
    its working clock when the first timed step starts (no idle gap, no launch latency inside).
    """
    import torch

    stream = run.stream
    with torch.cuda.stream(stream):
        for i in range(warm):
            run.step(i)
    graph_batch = max(run.nbuf, min(nsteps, 256) // run.nbuf * run.nbuf)
    graphs, full, rest = _graph_time(run.step, nsteps, stream, graph_batch)
    with torch.cuda.stream(stream):
        graphs[0][0].replay()  # page the graph in
    stream.synchronize()
    batches = [graphs[0]] * full + ([graphs[-1]] if rest else [])
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(batches) + 1)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        graphs[0][0].replay()  # untimed, immediately before the timed region
        evs[0].record(stream)
        for i, (g, _) in enumerate(batches):
            g.replay()
            evs[i + 1].record(stream)
    stream.synchronize()
    torch.cuda.synchronize(dev)
    barrier(world)
    ms = evs[0].elapsed_time(evs[-1])
    per_step = sorted(evs[i].elapsed_time(evs[i + 1]) / n for i, (_, n) in enumerate(batches))
    spread = {"median": round(per_step[len(per_step) // 2] * 1e3, 3), "best": round(per_step[0] * 1e3, 3),
              "replays": len(per_step), "steps_per_replay": batches[0][1]}
    status = run.rwo.get_status(stream)
    if status != run.rwo.OK:
        raise run.rwo.SoftmaxError(status, "kernel status after timing")
    return ms, spread


def _kernel_name(rwo, used: int, w: synth.Workload, mode: str) -> str:
    """The kernel a step of this workload launches (as the library's variant choice makes it)."""
    row_bytes = w.N * w.elem_bytes
    if mode == "causal":
        return "k_causal_warp" if row_bytes <= 16384 else "k_twopass"
    if used == rwo.VARIANT_ONEREAD_REG:
        return "k_oneread_reg"
    if used == rwo.VARIANT_ONEREAD_SMEM:
        if row_bytes > (64 << 10):
            return "k_splitrow_onchip"  # a thread-block cluster per row, segments held on chip
        return "k_oneread_warp" if row_bytes <= 8192 and mode == "softmax" else "k_oneread_tma"
    if used == rwo.VARIANT_SPLITROW:
        return "k_splitrow_onchip"
    if used == rwo.VARIANT_SPLITROW_STREAM:
        return "k_splitrow"
    if used == rwo.VARIANT_TWOPASS and row_bytes > (64 << 10) and mode != "ce":
        return "k_clusterrow"
    return "k_twopass"


def measure_config(label: str, w: synth.Workload, mode: str, forced: str | None, state: str, args, world: int,
                   rank: int, dev, stream, peak: float, host_x=None) -> tuple[dict, "_Run"]:
    """Time one configuration over exactly --steps steps; returns its record and the run."""
    import row_wise_online_gb300 as rwo

    row0 = shard_row0(rank, w.M)
    run = _Run(w, row0, dev, stream, mode, state, host_x=host_x)
    run.variant = VARIANT_ARG[forced] if forced else rwo.VARIANT_AUTO
    try:
        run.step(0)
    except rwo.SoftmaxError as e:
        run.release()
        return {"label": label, "workload": w.name, "unsupported": str(e)}, run
    used = rwo.last_variant()
    ms_local, spread = _time_steps(run, args.steps, args.warmup, world, dev)
    ms = reduce_max(ms_local, world)
    per_step_ms = ms / args.steps
    bytes_step = run.bytes_per_step()
    gbs = world * bytes_step * args.steps / (ms * 1e-3) / 1e9
    kernel = _kernel_name(rwo, used, w, mode)
    profile_key = kernel + ("-log" if mode == "log" else "-ce" if mode == "ce" else "")
    alg = run.algorithmic_bytes(row0)
    achieved = alg / (per_step_ms * 1e-3) / 1e9
    variant_name = rwo.VARIANT_NAMES[used] + {"causal": "+causal_skip", "log": "+log_softmax",
                                              "ce": "+cross_entropy"}.get(mode, "")
    rec = {
        "label": label, "workload": w.name, "M": w.M, "N": w.N,
        "dtype": "f32" if w.dtype == synth.F32 else "bf16",
        "variant": variant_name + ("" if not forced else " (forced)"),
        "kernel": kernel,
        "state_outputs": state or None,
        "gbs": round(gbs, 1),
        "us_per_step": round(per_step_ms * 1e3, 3),
        "step_us": spread,
        "rows_per_s": round(world * w.M * args.steps / (ms * 1e-3), 1),
        "pct_of_8tbs": round(100 * gbs / world / NOMINAL_HBM_GBS, 2),
        "frac": round(achieved / peak, 4),
        "achieved_gbs": round(achieved, 1),
        "algorithmic_bytes_per_launch": alg,
        "traffic": profiled_traffic(profile_key, w.name),
        "l2": (f"{run.nbuf} rotating x/y buffer sets ({run.nbuf * run.set_bytes >> 20} MiB > L2)" if run.nbuf > 1
               else "inputs larger than L2"),
        "steps": args.steps,
    }
    return rec, run


def bench_ours(args) -> dict | None:
    import torch

    import row_wise_online_gb300 as rwo
    from row_wise_online_gb300 import _build

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    if rank == 0 or not _build.up_to_date():
        _build.build()
    barrier(world)
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.Stream(device=dev)
    peak, peak_kind = measured_hbm_peak()

    w = synth.WORKLOADS[args.workload]
    if args.rows:
        w = w.with_rows(args.rows)
    mode = {"causal": "causal", "log": "log", "ce": "ce"}.get(args.variant, "softmax")
    if mode == "causal" and not w.causal_q:
        raise SystemExit("--variant causal needs a workload with a causal mask")
    forced = args.variant if args.variant in VARIANT_ARG and args.variant != "auto" else None
    state = "lse" if args.workload == "bf16_logits_16384x32768" and mode == "softmax" else ""

    # nvidia-smi samples over every timed region of this run (started before the first warm-up)
    sampler = ClockSampler(dev.index)
    rec, run = measure_config(args.workload, w, mode, forced, state, args, world, rank, dev, stream, peak)
    if "unsupported" in rec:
        sampler.stop()
        raise SystemExit(f"{args.workload}: {rec['unsupported']}")

    # End to end through the public host-buffer call: H2D of x, kernels, D2H of y, every step.
    e2e = None
    if not args.no_e2e and mode == "softmax":
        host_x = run.host_x
        run.release()
        torch.cuda.empty_cache()
        y_host = torch.empty_like(host_x).pin_memory()
        for _ in range(2):
            rwo.softmax_rows_host(host_x, y_host)
        k = max(3, min(args.steps, 20))
        barrier(world)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(k):
            rwo.softmax_rows_host(host_x, y_host)
        torch.cuda.synchronize(dev)
        t = reduce_max(time.perf_counter() - t0, world)
        e2e = {"value": round(world * w.min_bytes * k / t / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": w.M * w.N * w.elem_bytes, "d2h_bytes_per_step": w.M * w.N * w.elem_bytes,
               "steps": k, "ms_per_step": round(t * 1e3 / k, 4), "call": "softmax_rows_host (pinned host buffers)"}
        del y_host
    run.release()
    del run
    torch.cuda.empty_cache()

    # The other configurations, each over exactly --steps steps (one GPU; --quick skips them).
    configs = []
    if world == 1 and not args.quick and args.workload == DEFAULT_WORKLOAD and not args.rows and args.variant == "auto":
        for label, wname, cmode, cforced, cstate in SUITE[1:]:
            cw = synth.WORKLOADS[wname]
            crec, crun = measure_config(label, cw, cmode, cforced, cstate, args, world, rank, dev, stream, peak)
            crun.release()
            del crun
            torch.cuda.empty_cache()
            configs.append(crec)
    clk = sampler.stop()

    if rank != 0:
        return None
    result = {
        "metric": METRIC,
        "value": round(rec["gbs"], 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(rec["us_per_step"] / 1e3, 6),
        "step_us": rec["step_us"],  # this rank's median and best µs per step over single graph replays
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": round(rec["gbs"] / world / PAGE_GBS[w.name], 3) if w.name in PAGE_GBS else None,
        "vs_baseline_ref": ("pages' V3 register one-pass kernel, ~1672 GB/s on A100 80GB SXM4 "
                            "(another machine: context, not the target)") if w.name in PAGE_GBS else None,
        "dtype": rec["dtype"],
        "data": "synthetic",
        "config": {"workload": w.name if not args.rows else f"{w.name}[rows={w.M}]", "M": w.M, "N": w.N,
                   "rows_total": w.M * world, "variant": rec["variant"], "state_outputs": rec["state_outputs"],
                   "parallelism": f"rows sharded over {world} GPU(s)", "l2": rec["l2"],
                   "timing": ("CUDA graph replays between CUDA events on the launching stream, an untimed "
                              "replay issued right before the first event")},
        "rows_per_s": rec["rows_per_s"],
        "pct_of_8tbs": rec["pct_of_8tbs"],
        "pct_of_measured_peak": round(100 * rec["gbs"] / world / peak, 2),
        "roofline": {"bound": "hbm", "achieved": rec["achieved_gbs"], "peak": peak, "unit": "GB/s",
                     "frac": rec["frac"], "traffic": rec["traffic"],
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s", "kernel": rec["kernel"],
                     "algorithmic_bytes_per_launch": rec["algorithmic_bytes_per_launch"]},
        "gpu_launches": args.steps,
        "e2e": e2e,
        "clocks": clk,
        "configs": configs,
    }
    if configs:
        result["gpu_launches_all_configs"] = args.steps * (1 + sum(1 for c in configs if "gbs" in c))
    if world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w)
    return result

# ----------------------------------------------------------------------------------------------
# the oracle (CPU) arms
# ----------------------------------------------------------------------------------------------

def _oracle_rate(w: synth.Workload, threads: int, target_s: float):
    """Whole passes of the fp64 oracle over (up to) the full matrix for about `target_s` seconds
    on `threads` host threads: (GB/s on the read-once + write-once basis, passes, rows, seconds)."""
    import oracle

    probe = synth.generate(w, row0=0, nrows=min(w.M, 4 * threads))
    t0 = time.perf_counter()
    oracle.softmax_rows(probe, nthreads=threads)
    per_row = (time.perf_counter() - t0) / probe.shape[0]
    nrows = int(max(threads, min(w.M, target_s / max(per_row, 1e-9))))
    x = synth.generate(w, row0=0, nrows=nrows)
    reps, t = 0, 0.0
    t0 = time.perf_counter()
    while reps < 200 and (reps == 0 or t < target_s):
        oracle.softmax_rows(x, nthreads=threads)
        reps += 1
        t = time.perf_counter() - t0
    return 2 * nrows * w.N * w.elem_bytes * reps / t / 1e9, reps, nrows, t


def cpu_baseline(w: synth.Workload, target_s: float = 1.5) -> dict:
    """The fp64 oracle as it stands, on the host cores, on a bounded sample of the workload:
    as many whole passes over (up to) the full matrix as fit in about `target_s` seconds.  For
    the two fp32 workloads of 64 x 1024 and 4096 x 4096 also on one thread."""
    import oracle

    threads = oracle.default_threads()
    gbs, reps, nrows, t = _oracle_rate(w, threads, target_s)
    out = {"value": round(gbs, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
           "sample": f"{reps} pass(es) over rows 0..{nrows - 1} of {w.name} ({nrows} x {w.N}), fp64 three-pass, "
                     f"{t:.2f} s wall on {threads} threads (~{t * threads:.0f} CPU-s)",
           "rows_per_s": round(nrows * reps / t, 1)}
    if w.name in ("fp32_64x1024", "fp32_4096x4096"):
        gbs1, reps1, nrows1, t1 = _oracle_rate(w, 1, target_s / 2)
        out["single_thread"] = {"value": round(gbs1, 3), "unit": "GB/s", "cores": 1,
                                "sample": f"{reps1} pass(es) over rows 0..{nrows1 - 1}, {t1:.2f} s wall"}
    return out


def bench_reference(args) -> dict | None:
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import oracle

    w = synth.WORKLOADS[args.workload]
    threads = oracle.default_threads()
    probe = synth.generate(w, row0=0, nrows=min(w.M, 2 * threads))
    t0 = time.perf_counter()
    oracle.softmax_rows(probe, nthreads=threads)
    per_row = (time.perf_counter() - t0) / probe.shape[0]
    budget_s = 120.0  # the whole run, warm-up included
    rows = int(max(1, min(w.M, budget_s / max(1, args.steps + args.warmup) / max(per_row, 1e-9))))
    x = synth.generate(w, row0=0, nrows=rows)
    for _ in range(args.warmup):
        oracle.softmax_rows(x, nthreads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.softmax_rows(x, nthreads=threads)
    t = time.perf_counter() - t0
    gbs = 2 * rows * w.N * w.elem_bytes * args.steps / t / 1e9
    sample = f"rows 0..{rows - 1} of {w.name} ({rows} x {w.N}) per step, fp64 three-pass oracle"
    return {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3 / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "M": w.M, "N": w.N, "rows_per_step": rows},
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


ATTN_WORKLOADS = {
    # name: (BH, S, d, causal) -- 4 x 32 heads of 4096 queries over 4096 keys, head dimension 128
    # (and 4 x 64 heads of head dimension 64: the same bytes of q, k and v)
    "attn_bf16_4x32x4096x128_causal": (128, 4096, 128, True),
    "attn_bf16_4x32x4096x128": (128, 4096, 128, False),
    "attn_bf16_4x64x4096x64_causal": (256, 4096, 64, True),
    "attn_bf16_4x64x4096x64": (256, 4096, 64, False),
}


def attention_flops(BH: int, S: int, d: int, causal: bool) -> int:
    """2 S x S x d products (Q K^T and P V), 2 flops per multiply-add; causal: keys j <= i only."""
    pairs = S * (S + 1) // 2 if causal else S * S
    return 4 * BH * pairs * d


def measured_tensor_peak() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def bench_attention(args) -> dict | None:
    """attention_forward on the attention workload: TFLOP/s of the two products."""
    import torch

    import row_wise_online_gb300 as rwo
    from row_wise_online_gb300 import _build

    rank, world, local = dist_env()
    torch.cuda.set_device(local if torch.cuda.device_count() > 1 else 0)
    if rank == 0 or not _build.up_to_date():
        _build.build()
    barrier(world)
    dev = torch.device("cuda", torch.cuda.current_device())
    BH, S, d, causal = ATTN_WORKLOADS[args.workload]
    gen = torch.Generator(device=dev)
    gen.manual_seed(7 + rank)
    q, k, v = (torch.randn((BH, S, d), device=dev, generator=gen).to(torch.bfloat16) for _ in range(3))
    o = torch.empty_like(q)
    lse = torch.empty((BH, S), device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(i):
        rwo.attention_forward(q, k, v, o, lse, causal=causal, stream=stream)

    sampler = ClockSampler(dev.index)  # nvidia-smi samples from before the warm-up to the end
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    stream.synchronize()
    graphs, full, rest = _graph_time(step, args.steps, stream, max(1, min(args.steps, 64)))
    with torch.cuda.stream(stream):
        graphs[0][0].replay()
    stream.synchronize()
    barrier(world)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        graphs[0][0].replay()  # untimed, immediately before the timed region
        ev0.record(stream)
        for _ in range(full):
            graphs[0][0].replay()
        if rest:
            graphs[-1][0].replay()
        ev1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = sampler.stop()
    status = rwo.get_status(stream)
    if status != rwo.OK:
        raise rwo.SoftmaxError(status, "kernel status after timing")
    ms = reduce_max(ev0.elapsed_time(ev1), world)
    if rank != 0:
        return None
    flops = attention_flops(BH, S, d, causal)
    tflops = world * flops * args.steps / (ms * 1e-3) / 1e12
    peak, kind = measured_tensor_peak()
    per_launch = ms / args.steps
    return {
        "metric": "attention forward TFLOP/s (Q K^T and P V, 2 flops per multiply-add)",
        "value": round(tflops, 1), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(per_launch, 6), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "BH": BH, "S": S, "d": d, "causal": causal,
                   "parallelism": f"heads sharded over {world} GPU(s)",
                   "l2": "q, k, v 384 MiB (larger than L2)",
                   "timing": "CUDA graph replays between CUDA events on the launching stream"},
        "roofline": {"bound": "tensor", "achieved": round(tflops / world, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(tflops / world / peak, 4),
                     "traffic": profiled_traffic("k_attention_fwd", args.workload),
                     "peak_source": f"{kind} (MEASURED_PEAKS.json bf16_tflops, burst)", "kernel": "k_attention_fwd"},
        "gpu_launches": args.steps,
        "clocks": clk,
    }


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS) + sorted(ATTN_WORKLOADS))
    ap.add_argument("--variant", default="auto",
                    choices=["auto", "reg", "smem", "twopass", "splitrow", "splitrow_stream", "causal", "log", "ce"],
                    help="causal: softmax_rows_causal on a causal workload (masked keys not read); "
                         "log: log_softmax_rows; ce: cross_entropy_rows with uniform synthetic labels")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--rows", type=int, default=0, help="use only the first ROWS rows (profiling small cases)")
    ap.add_argument("--quick", action="store_true", help="skip the other-variant measurements")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.workload in ATTN_WORKLOADS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the attention forward has no CPU reference arm "
                              "(the fp64 oracle checks sampled rows in the tests)"}), flush=True)
            return 0
        res = bench_attention(args)
    else:
        res = bench_reference(args) if args.impl == "reference" else bench_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)
    rank, world, _ = dist_env()
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

"""Benchmark of the coalesced varlen attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 1..9] [--mode step|fwd] [--seed S] [--bf16-partials]
                    [--no-e2e] [--no-cpu-baseline] [--per-config 2,3,4 | --per-config none]

One step = one pass of the whole path over one batch: the forward over whole
sequences and shard tiles in one launch, the exact LSE merge of the tiles, the
backward preprocess, the backward, and the dQ conversion.  The default
workload is the training-step batch (a 720p 81-frame video of 75,600 tokens
split into a 2 x 2 tile grid, two 480p 81-frame videos of 32,760 tokens, four
4,096-token and 32 1,024-token images; 40 heads, head dim 128, bf16).

The metric is attention TFLOP/s: algorithmic FLOPs (forward 4 * sum(Lq * Lk)
* d * H; forward + backward 3.5x that) over device time, timed with CUDA
events over exactly K steps after W warm-up steps.  Every input tensor is
larger than L2 (129 MB), so no L2 flush is needed between steps.

With torchrun (N > 1) every rank runs an independent replica of the same
workload on its own GPU (the path has no cross-GPU exchange); the time is the
maximum over ranks and the value is the work of all ranks over that time.

--impl reference times the float64 CPU oracle (the correctness reference) on a
bounded sample of the same workload, on rank 0 only.

Besides the metric the JSON line carries: the per-kernel launch times of the
timed region (the library's event hook), the dominant kernel's roofline
(algorithmic FLOPs or bytes per launch over its mean launch time, against the
measured peak, with the DRAM bytes of the last ncu capture of the same kernel
source), the oracle's CPU throughput on a bounded sample, an end-to-end leg
(pinned host inputs in and all results out inside the timed region) with its
own clock record, the number of library launches, and the SM clock, power,
temperature and throttle reasons sampled while each timed region ran.
--bf16-partials keeps the partial rows of key-split sequences in bf16.

`per_config` adds, for the image-only mix (2), the mixed Wan batch (3) and the
131,072-token shard mode (4), the forward (with its merge) and the fwd+bwd
step timed on their own batches: CUDA events over K steps after 3 warm-up
steps (K chosen so each timed region lasts about half a second, at least 5
steps), each with its own clock record and its fraction of the burst and
sustained bf16 peaks, against the target of 60% (forward) and 45% (fwd+bwd)
of the dense bf16 peak.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "varlen attn TFLOP/s (fwd; fwd+bwd) on mixed image-video batch, % of BF16 peak"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")
CSRC = os.path.join(ROOT, "mixed_length_dit_gb300", "csrc")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- helpers
def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_hash(name: str) -> str:
    with open(os.path.join(CSRC, name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def algorithmic_bytes(wl, kernel: str, bf16_partials: bool = False) -> float:
    """Algorithmic DRAM bytes of one step's launches of `kernel` (every input
    read once, every output written once):
      fwd_tc   q, k, v read; bf16 O and float32 LSE of whole sequences and of
               sequences split only by queries and heads written; the partial
               O (float32, or bf16) and LSE of every key chunk of a key-split
               sequence written;
      bwd_tc   q, k, v, dO (bf16) and LSE, D (float32) read; dK, dV written;
               the float32 dQ accumulator read and written once;
      lse_merge  merge_bytes."""
    h, d = wl.num_heads, wl.head_dim
    t = wl.total_tokens
    if kernel == "lse_merge":
        return merge_bytes(wl, bf16_partials)
    if kernel == "bwd_tc":
        return t * h * (4 * d * 2 + 2 * 4 + 2 * d * 2 + 2 * d * 4)
    if kernel == "fwd_tc":
        part = (2 if bf16_partials else 4) * d + 4
        total = 3.0 * t * h * d * 2
        for s, n in enumerate(wl.seqlens):
            n_kv = wl.splits.get(s, (1, 1))[1]
            total += n * h * (n_kv * part if n_kv > 1 else 2 * d + 4)
        return total
    raise KeyError(kernel)


def recorded_traffic(kernel: str, wl, bf16_partials: bool = False):
    """DRAM bytes per step of `kernel` on workload wl, scaled from a capture:
    profiles/traffic.txt records, per kernel, the DRAM bytes of one launch on
    a small workload (dram__bytes_read.sum + dram__bytes_write.sum) and that
    launch's algorithmic bytes; the ratio of the two times wl's algorithmic
    bytes is the estimate.  None when no record exists for the current kernel
    source (src hash)."""
    try:
        with open(TRAFFIC_FILE) as f:
            lines = f.read().splitlines()
    except OSError:
        return None
    src = {"fwd_tc": "fwd_tc.cu", "bwd_tc": "bwd_tc.cu", "lse_merge": "merge.cu"}.get(kernel)
    if src is None:
        return None
    h = source_hash(src)
    for line in lines:
        if line.startswith("#") or not line.strip():
            continue
        f = dict(x.split("=", 1) for x in line.split())
        if f.get("kernel") == kernel and f.get("src") == h and "algorithmic_bytes" in f:
            ratio = float(f["bytes_per_launch"]) / float(f["algorithmic_bytes"])
            return {"bytes": ratio * algorithmic_bytes(wl, kernel, bf16_partials), "ratio": round(ratio, 4),
                    "captured_on": f.get("workload")}
    return None


def workload_desc(wl) -> str:
    counts = {}
    for n in wl.seqlens:
        counts[n] = counts.get(n, 0) + 1
    parts = []
    for n, c in sorted(counts.items(), key=lambda x: -x[0]):
        parts.append(f"{c}x{n}")
    split = ", ".join(f"seq {s} ({wl.seqlens[s]} tokens) as {'x'.join(str(c) for c in sp)} tiles"
                      for s, sp in wl.splits.items())
    return (f"{wl.name}: " + " + ".join(parts) + f" tokens; H={wl.num_heads}, d={wl.head_dim}"
            + (f"; {split}" if split else ""))


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "temperature.gpu,clocks.mem")

    def __init__(self, gpu_index: str):
        fd, self.path = tempfile.mkstemp(prefix="zl_clocks_", suffix=".csv")
        self.proc = None
        self.fh = os.fdopen(fd, "w")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", gpu_index], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        """Ends sampling and removes the sample file; None if nvidia-smi could
        not be started."""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.fh.close()
        lines = []
        if self.proc is not None:
            with open(self.path) as f:
                lines = f.readlines()
        os.unlink(self.path)
        return parse_clock_samples(lines) if self.proc is not None else None


def parse_clock_samples(lines):
    """Summary of `nvidia-smi --query-gpu=<ClockSampler.FIELDS>` CSV lines:
    median SM clock, the highest max clock, the throttle reasons seen active
    in any sample, median power and memory clock, peak temperature."""
    rows = []
    for line in lines:
        parts = [x.strip() for x in line.split(",")]
        if len(parts) >= 9:
            rows.append(parts)
    if not rows:
        return None

    def column(i):
        return [float(r[i]) for r in rows if len(r) > i and r[i].replace(".", "").isdigit()]

    sm, mx, pw, tc, mem = column(1), column(2), column(3), column(9), column(10)
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
            "reasons": reasons, "samples": len(rows),
            "power_w": round(statistics.median(pw), 1) if pw else None,
            "temp_c": max(tc) if tc else None, "mem_mhz": statistics.median(mem) if mem else None}


def gpu_index_for_smi(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local_rank < len(ids) and ids[local_rank].isdigit():
            return ids[local_rank]
    return str(local_rank)


def reduce_max_ms(ms_local: float, world: int, device) -> float:
    """Slowest rank's time: the job is done when its last replica is."""
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, steps: int, flops_step: float, ms_max: float) -> float:
    """Whole-job throughput: the work of every replica over the slowest time."""
    return world * steps * flops_step / (ms_max * 1e-3) / 1e12


def fwd_flops(wl) -> float:
    return 4.0 * wl.head_dim * wl.num_heads * wl.pair_count()


def merge_bytes(wl, bf16_partials: bool = False) -> float:
    """Algorithmic bytes the merge moves per step: every sequence split over
    keys (n_kv > 1; splits are (n_q, n_kv[, n_h])) reads its n_kv partial rows
    (float32, or bf16 with bf16_partials) and float32 LSEs and writes its bf16
    O rows and LSEs."""
    h, d = wl.num_heads, wl.head_dim
    part = (2 if bf16_partials else 4) * d + 4
    total = 0.0
    for s, sp in wl.splits.items():
        n_kv = sp[1]
        if n_kv > 1:
            total += wl.seqlens[s] * h * (n_kv * part + (2 * d + 4))
    return total


def e2e_timeline(steps):
    """Where the end-to-end leg's time goes, from per-step event times (ms
    from the start of the timed region): [h2d start, h2d end, compute start,
    compute end, then the start and end of each device-to-host copy group]
    per step (the output O leaves after the forward, the gradients after the
    backward).  Reports the mean copy and compute durations, the compute
    stream's idle time between steps (what the copies failed to hide) and the
    share of copy time that ran while a compute interval was open."""
    if not steps:
        return None
    comp = [(s[2], s[3]) for s in steps]
    outs = [[(s[i], s[i + 1]) for i in range(4, len(s) - 1, 2)] for s in steps]
    copies = [(s[0], s[1]) for s in steps] + [c for o in outs for c in o]

    def overlap(a, b):
        return max(0.0, min(a[1], b[1]) - max(a[0], b[0]))

    copy_ms = sum(b - a for a, b in copies)
    hidden = sum(overlap(c, k) for c in copies for k in comp)
    idle = [comp[i + 1][0] - comp[i][1] for i in range(len(comp) - 1)]
    n = len(steps)
    return {"h2d_ms": round(sum(s[1] - s[0] for s in steps) / n, 2),
            "d2h_ms": round(sum(b - a for o in outs for a, b in o) / n, 2),
            "compute_ms": round(sum(b - a for a, b in comp) / n, 2),
            "compute_idle_ms_between_steps": round(sum(idle) / max(1, len(idle)), 2),
            "first_compute_start_ms": round(comp[0][0], 2),
            "last_d2h_after_compute_ms": round(steps[-1][-1] - steps[-1][3], 2),
            "copy_time_overlapped": round(hidden / copy_ms, 4) if copy_ms > 0 else None}


# ----------------------------------------------------------------- CPU oracle
def oracle_sample(wl, inp, target_tokens: int, n_heads: int):
    """The first `n_heads` heads of the sequence of the workload nearest
    `target_tokens` long, copied to float64 host arrays, and their algorithmic
    fwd+bwd FLOPs."""
    lens = wl.seqlens
    s = min(range(len(lens)), key=lambda i: (abs(lens[i] - target_tokens), i))
    cu = wl.cu_seqlens()
    a, b = cu[s], cu[s + 1]
    n_heads = min(n_heads, wl.num_heads)
    arrs = [inp[n][a:b, :n_heads].to("cpu", torch.float64).numpy() for n in ("q", "k", "v", "do")]
    L = b - a
    return arrs, L, n_heads, n_heads * 3.5 * 4.0 * L * L * wl.head_dim


def time_oracle(arrs, L):
    import oracle
    q, k, v, do = arrs
    cu = [0, L]
    t0 = time.perf_counter()
    oracle.varlen_attn_fwd(q, k, v, cu, cu)
    oracle.varlen_attn_bwd(q, k, v, do, cu, cu)
    return time.perf_counter() - t0


def cpu_threads() -> int:
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


# ----------------------------------------------------------------- per configuration
TARGET_FRAC = {"fwd": 0.60, "step": 0.45}


def time_config(zl, n: int, dev, seed: int, peaks, target_s: float = 0.5, warmup: int = 3):
    """Forward (with its merge) and fwd+bwd step of workload n, each timed by
    itself: `warmup` untimed calls (timed as a group to size the run), then K
    calls bracketed by CUDA events on the launching stream, with the clocks
    sampled meanwhile.  Returns one dict per mode."""
    wl = synth.config(n)
    inp = synth.make_inputs(wl, seed=seed, device=dev)
    cu = wl.cu_seqlens()
    tiles = wl.tiles() or None
    H, D, T = wl.num_heads, wl.head_dim, wl.total_tokens
    o = torch.empty_like(inp["q"])
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    fws = zl.alloc_workspace(zl.fwd_workspace_bytes(cu, cu, H, D, tiles), dev)
    dq, dk, dv = (torch.empty_like(inp["q"]) for _ in range(3))
    bws = zl.alloc_workspace(zl.bwd_workspace_bytes(cu, cu, H, D), dev)
    burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    out = {"workload": workload_desc(wl)}
    for mode in ("fwd", "step"):
        def run():
            zl.varlen_attn_fwd(inp["q"], inp["k"], inp["v"], cu, cu, tiles=tiles, out=o, lse=lse, workspace=fws)
            if mode == "step":
                zl.varlen_attn_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], cu, cu, tiles=tiles,
                                   dq=dq, dk=dk, dv=dv, workspace=bws)
        w0 = torch.cuda.Event(enable_timing=True)
        w1 = torch.cuda.Event(enable_timing=True)
        w0.record()
        for _ in range(warmup):
            run()
        w1.record()
        torch.cuda.synchronize()
        zl.sync_check()
        est_ms = w0.elapsed_time(w1) / warmup
        steps = max(5, int(np.ceil(target_s * 1e3 / max(est_ms, 1e-3))))
        sampler = ClockSampler(gpu_index_for_smi(dev.index or 0))
        time.sleep(0.3)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            run()
        e1.record()
        torch.cuda.synchronize()
        clocks = sampler.stop()
        zl.sync_check()
        ms = e0.elapsed_time(e1) / steps
        flops = fwd_flops(wl) * (3.5 if mode == "step" else 1.0)
        tf = flops / (ms * 1e-3) / 1e12
        out[mode] = {"tflops": round(tf, 1), "ms": round(ms, 4), "steps": steps, "flops": flops,
                     "frac_burst": round(tf / burst, 4), "frac_sustained": round(tf / sustained, 4),
                     "target_frac_burst": TARGET_FRAC[mode], "meets_target": bool(tf / burst >= TARGET_FRAC[mode]),
                     "clocks": clocks}
    del inp, o, lse, fws, dq, dk, dv, bws
    torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=5)
    ap.add_argument("--seed", type=int, default=0, help="input seed (rank r draws with seed + r)")
    ap.add_argument("--mode", choices=["step", "fwd"], default="step")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bf16-partials", action="store_true",
                    help="keep the partial O rows of key-split sequences in bf16")
    ap.add_argument("--oracle-tokens", type=int, default=4096,
                    help="length of the sequence whose heads the CPU oracle times")
    ap.add_argument("--oracle-heads", type=int, default=16,
                    help="number of heads of that sequence the CPU oracle times")
    ap.add_argument("--per-config", default="2,3,4",
                    help="workloads whose forward and fwd+bwd step are also timed by themselves "
                         "(comma-separated; 'none' to skip)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    wl = synth.config(args.workload)
    peaks, peak_kind = load_peaks()

    if args.impl == "reference":
        if rank != 0:
            return 0
        return run_reference(args, wl, world)

    import torch.distributed as dist
    import mixed_length_dit_gb300 as zl

    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", local_rank)
    inp = synth.make_inputs(wl, seed=args.seed + rank, device=dev)
    cu = wl.cu_seqlens()
    tiles = wl.tiles() or None
    H, D, T = wl.num_heads, wl.head_dim, wl.total_tokens
    o = torch.empty_like(inp["q"])
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    fws = zl.alloc_workspace(zl.fwd_workspace_bytes(cu, cu, H, D, tiles), dev)
    dq, dk, dv = (torch.empty_like(inp["q"]) for _ in range(3))
    bws = zl.alloc_workspace(zl.bwd_workspace_bytes(cu, cu, H, D), dev)
    step_bwd = args.mode == "step"

    def step(q, k, v, do):
        zl.varlen_attn_fwd(q, k, v, cu, cu, tiles=tiles, out=o, lse=lse, workspace=fws,
                           bf16_partials=args.bf16_partials)
        if step_bwd:
            zl.varlen_attn_bwd(q, k, v, o, lse, do, cu, cu, tiles=tiles, dq=dq, dk=dk, dv=dv, workspace=bws)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step(inp["q"], inp["k"], inp["v"], inp["do"])
    zl.sync_check()

    sampler = ClockSampler(gpu_index_for_smi(local_rank))
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    n_launch0 = zl.launch_count()
    zl.profile_begin()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step(inp["q"], inp["k"], inp["v"], inp["do"])
    e1.record()
    torch.cuda.synchronize()
    barrier()
    prof = zl.profile_end()
    clocks = sampler.stop()
    launches = zl.launch_count() - n_launch0
    zl.sync_check()
    ms_total = reduce_max_ms(e0.elapsed_time(e1), world, dev)
    flops_fwd = fwd_flops(wl)
    flops_step = flops_fwd * (3.5 if step_bwd else 1.0)
    value = job_tflops(world, args.steps, flops_step, ms_total)

    # ---------------- per-kernel roofline of the dominant kernel
    dom = max(prof.items(), key=lambda kv: kv[1][1])[0] if prof else None
    roof = None
    sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    if dom is not None:
        n_l, tot = prof[dom]
        avg_ms = tot / n_l
        rec = recorded_traffic(dom, wl, args.bf16_partials)
        # per launch, scaled from the small-case capture's ratio to its algorithmic bytes
        traffic = round(rec["bytes"] * args.steps / n_l) if rec else None
        traffic_note = (f"ncu DRAM bytes of one launch on {rec['captured_on']} = {rec['ratio']} x its "
                        f"algorithmic bytes, times this launch's algorithmic bytes") if rec else None
        if dom in ("fwd_tc", "bwd_tc"):
            per_launch = (flops_fwd if dom == "fwd_tc" else 2.5 * flops_fwd) * args.steps / n_l
            ach = per_launch / (avg_ms * 1e-3) / 1e12
            roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": sustained, "unit": "TFLOP/s",
                    "frac": round(ach / sustained, 4), "traffic": traffic, "traffic_note": traffic_note,
                    "kernel": dom, "peak_kind": f"bf16 sustained ({peak_kind})",
                    "flops_per_launch": per_launch, "avg_launch_ms": round(avg_ms, 4)}
        elif dom == "lse_merge":
            hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
            per_launch = merge_bytes(wl, args.bf16_partials) * args.steps / max(1, n_l)
            ach = per_launch / (avg_ms * 1e-3) / 1e9
            roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                    "frac": round(ach / hbm, 4), "traffic": traffic, "traffic_note": traffic_note,
                    "kernel": dom}
    kernels = {k: {"launches": v[0], "avg_ms": round(v[1] / v[0], 4),
                   "share": round(v[1] / sum(x[1] for x in prof.values()), 4)} for k, v in prof.items()}
    fwd_ms = sum(prof[k][1] for k in ("fwd_tc", "lse_merge") if k in prof) / args.steps
    bwd_ms = sum(prof[k][1] for k in ("bwd_preprocess", "bwd_tc", "dq_convert") if k in prof) / args.steps
    phases = {"fwd_tflops": round(flops_fwd / (fwd_ms * 1e-3) / 1e12, 1) if fwd_ms else None}
    if step_bwd and bwd_ms:
        phases["bwd_tflops"] = round(2.5 * flops_fwd / (bwd_ms * 1e-3) / 1e12, 1)
    if "lse_merge" in prof and wl.splits:
        n_l, tot = prof["lse_merge"]
        per_launch = merge_bytes(wl, args.bf16_partials) * args.steps / n_l
        gbs = per_launch / (tot / n_l * 1e-3) / 1e9
        hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        phases["merge"] = {"gbs": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4),
                           "bytes_per_launch": per_launch, "avg_launch_ms": round(tot / n_l, 4)}

    # ---------------- forward and fwd+bwd per configuration, each timed by itself
    per_config = None
    if args.per_config.strip().lower() not in ("", "none"):
        per_config = {}
        for n in (int(x) for x in args.per_config.split(",")):
            per_config[str(n)] = time_config(zl, n, dev, args.seed + rank, peaks)

    # ---------------- CPU oracle baseline (rank 0, single GPU)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        arrs, L, nh_s, fl = oracle_sample(wl, inp, args.oracle_tokens, args.oracle_heads)
        secs = time_oracle(arrs, L)
        cpu = {"value": round(fl / secs / 1e12, 5), "unit": "TFLOP/s", "cores": cpu_threads(),
               "kind": "oracle",
               "sample": f"float64 numpy oracle, fwd+bwd of {nh_s} heads of one {L}-token sequence of the "
                         f"workload ({fl / 1e12:.3f} TFLOP algorithmic) in {secs:.1f} s"}

    # ---------------- end to end through the public API with host buffers
    # (the last leg: it pins 2 x 7.8 GB of host memory)
    # Every step copies its four inputs in from pinned host memory and its
    # four results (O, dQ, dK, dV) back out, all inside the timed region.  The
    # copies of neighbouring steps overlap the compute of the current one
    # (inputs and outputs double-buffered on the device, one stream each for
    # host-to-device and device-to-host copies); within a step the forward
    # starts once q, k and v are in (dO follows) and O leaves while the
    # backward runs.
    e2e = None
    if not args.no_e2e:
        k_e2e = max(2, args.steps)
        names_in = ("q", "k", "v", "do")
        names_out = ("o", "dq", "dk", "dv") if step_bwd else ("o",)
        host_in = {n: inp[n].to("cpu").pin_memory() for n in names_in}
        host_out = {n: torch.empty(inp["q"].shape, dtype=inp["q"].dtype).pin_memory() for n in names_out}
        dev_in = [{n: torch.empty_like(inp[n]) for n in names_in} for _ in range(2)]
        dev_out = [{n: torch.empty_like(inp["q"]) for n in names_out} for _ in range(2)]
        lse2 = [torch.empty_like(lse) for _ in range(2)]
        comp = torch.cuda.current_stream()
        h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
        ev = {key: [torch.cuda.Event() for _ in range(2)] for key in ("qkv", "h2d", "fwd", "comp", "d2h")}
        for key in ev:
            for e in ev[key]:
                e.record(comp)

        def timed_event(stream, marks):
            if marks is not None:
                e = torch.cuda.Event(enable_timing=True)
                e.record(stream)
                marks.append(e)

        def e2e_step(i, marks=None):
            # marks (timed region only): h2d start/end, compute start/end, the
            # O copy's start/end and the gradients' copy start/end of this
            # step, each recorded on its own stream
            sl = i % 2
            din, dout = dev_in[sl], dev_out[sl]
            with torch.cuda.stream(h2d):
                h2d.wait_event(ev["comp"][sl])            # step i-2 no longer reads this slot
                timed_event(h2d, marks)
                for n in ("q", "k", "v"):
                    din[n].copy_(host_in[n], non_blocking=True)
                ev["qkv"][sl].record(h2d)                 # the forward's inputs are in
                din["do"].copy_(host_in["do"], non_blocking=True)
                ev["h2d"][sl].record(h2d)
                timed_event(h2d, marks)
            comp.wait_event(ev["qkv"][sl])
            comp.wait_event(ev["d2h"][sl])                # step i-2's results have left this slot
            timed_event(comp, marks)
            zl.varlen_attn_fwd(din["q"], din["k"], din["v"], cu, cu, tiles=tiles, out=dout["o"],
                               lse=lse2[sl], workspace=fws, bf16_partials=args.bf16_partials)
            ev["fwd"][sl].record(comp)
            if step_bwd:
                comp.wait_event(ev["h2d"][sl])            # dO is in
                zl.varlen_attn_bwd(din["q"], din["k"], din["v"], dout["o"], lse2[sl], din["do"], cu, cu,
                                   tiles=tiles, dq=dout["dq"], dk=dout["dk"], dv=dout["dv"], workspace=bws)
            ev["comp"][sl].record(comp)
            timed_event(comp, marks)
            with torch.cuda.stream(d2h):
                d2h.wait_event(ev["fwd"][sl])             # O leaves while the backward runs
                timed_event(d2h, marks)
                host_out["o"].copy_(dout["o"], non_blocking=True)
                timed_event(d2h, marks)
                d2h.wait_event(ev["comp"][sl])
                timed_event(d2h, marks)
                for n in names_out[1:]:
                    host_out[n].copy_(dout[n], non_blocking=True)
                ev["d2h"][sl].record(d2h)
                timed_event(d2h, marks)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        e2e_sampler = ClockSampler(gpu_index_for_smi(local_rank))
        f0.record(comp)
        h2d.wait_event(f0)
        marks = []
        for i in range(k_e2e):
            e2e_step(i, marks)
        comp.wait_stream(d2h)
        f1.record(comp)
        torch.cuda.synchronize()
        e2e_clocks = e2e_sampler.stop()
        barrier()
        ems = reduce_max_ms(f0.elapsed_time(f1), world, dev)
        timeline = e2e_timeline([[f0.elapsed_time(e) for e in marks[8 * i:8 * i + 8]] for i in range(k_e2e)])
        bi = sum(t.numel() * t.element_size() for t in host_in.values())
        bo = sum(t.numel() * t.element_size() for t in host_out.values())
        e2e = {"value": round(job_tflops(world, k_e2e, flops_step, ems), 1),
               "unit": "TFLOP/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": k_e2e,
               "ms_per_step": round(ems / k_e2e, 3),
               "note": ("copies of neighbouring steps overlap compute (2 copy streams, double-buffered device "
                        "tensors); the forward starts once q, k, v are in, O leaves during the backward"),
               "timeline": timeline, "clocks": e2e_clocks}
        del dev_in, dev_out, host_in, host_out, lse2

    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return 0
    bf16_peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_total / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: q, k, v, dO ~ N(0,1) drawn in float32 from a seeded generator, rounded to bf16",
        "config": {"workload": workload_desc(wl), "mode": "fwd+bwd step" if step_bwd else "fwd only",
                   "total_tokens": wl.total_tokens, "sequences": len(wl.seqlens),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "no flush: every input tensor (>= %.2f GB) is larger than the 129 MB L2"
                         % (wl.total_tokens * H * D * 2 / 1e9),
                   "flops_per_step": flops_step,
                   "partials": "bf16" if args.bf16_partials else "float32"},
        "pct_of_peak": round(100 * value / world / bf16_peak, 2),
        "peak_tflops": bf16_peak,
        "phases": phases,
        "kernels": kernels,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "per_config": per_config,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args, wl, world):
    """The float64 CPU oracle, as it stands, on a bounded sample of the same
    workload: each step is the fwd+bwd of one head of one sequence."""
    g = torch.Generator().manual_seed(args.seed)
    target = 4096
    lens = wl.seqlens
    s = min(range(len(lens)), key=lambda i: (abs(lens[i] - target), i))
    L = lens[s]
    arrs = [torch.randn((L, 1, wl.head_dim), generator=g).to(torch.bfloat16).double().numpy() for _ in range(4)]
    fl = 3.5 * 4.0 * L * L * wl.head_dim
    for _ in range(args.warmup):
        time_oracle(arrs, L)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        time_oracle(arrs, L)
    secs = time.perf_counter() - t0
    value = args.steps * fl / secs / 1e12
    sample = (f"float64 numpy oracle, fwd+bwd of one head of one {L}-token sequence of the workload "
              f"({fl / 1e9:.1f} GFLOP algorithmic) per step")
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 5),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * secs / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic: N(0,1) rounded to bf16, upcast to float64",
        "config": {"workload": workload_desc(wl), "mode": "fwd+bwd step (sampled)"},
        "cpu_baseline": {"value": round(value, 5), "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 5), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())

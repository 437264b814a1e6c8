"""Replica aggregation of bench.py across ranks, on CPU with gloo (world size
2): the job time is the slowest rank's, the value counts every rank's work,
and the reference arm runs on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.reduce_max_ms(100.0 + 50.0 * rank, world, torch.device("cpu"))
    out[rank] = (ms, bench.job_tflops(world, 10, 1e15, ms))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_value():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 150.0
    # 2 replicas x 10 steps x 1 PFLOP in 150 ms
    assert abs(res[0][1] - 2 * 10 * 1e15 / 0.150 / 1e12) < 1e-6


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_prints_the_contract_line():
    """A single-process reference arm prints one JSON line with the keys the
    benchmark contract asks for (oracle on the host cores, no GPU needed)."""
    import json
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "1", "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_merge_bytes_count_key_split_sequences_only():
    """The merge reads n_kv float32 partials (O row + LSE) per row and head and
    writes the bf16 row and its LSE, for sequences split over keys only:
    tiles of query or head splits write their rows directly."""
    import synth
    wl = synth.config(8)                      # splits (1,1,4), (2,2,2), (2,1,5)
    h, d = wl.num_heads, wl.head_dim
    row = 2 * (4 * d + 4) + (2 * d + 4)
    assert bench.merge_bytes(wl) == wl.seqlens[1] * h * row
    wl5 = synth.config(5)                     # one sequence as 2 x 2 tiles
    assert bench.merge_bytes(wl5) == wl5.seqlens[0] * wl5.num_heads * row
    assert bench.merge_bytes(synth.config(2)) == 0


def test_workload_descriptions_cover_every_workload():
    """Every workload bench.py can time describes itself (splits of two or
    three chunk counts) and prices its merge without error."""
    import synth
    for n in range(1, 10):
        wl = synth.config(n)
        desc = bench.workload_desc(wl)
        assert wl.name in desc
        for s, sp in wl.splits.items():
            assert f"as {'x'.join(str(c) for c in sp)} tiles" in desc
        assert bench.merge_bytes(wl) >= 0


def test_clock_samples_summary():
    """The clock record: median SM clock, every throttle reason seen active
    in any sample (a hw or thermal slowdown rejects a run), medians of power
    and memory clock, peak temperature."""
    lines = [
        "0, 1980, 2070, 1360.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active, 55, 3996\n",
        "0, 1965, 2070, 1371.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active, 58, 3996\n",
        "0, 2010, 2070, 1300.0, 0x0000000000000008, Active, Not Active, Not Active, Not Active, 57, 3996\n",
        "garbage line\n",
    ]
    c = bench.parse_clock_samples(lines)
    assert c["sm_mhz"] == 1980 and c["sm_max_mhz"] == 2070 and c["samples"] == 3
    assert c["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert c["power_w"] == 1360.5 and c["temp_c"] == 58 and c["mem_mhz"] == 3996
    assert bench.parse_clock_samples([]) is None
    # the older nine-column form still parses
    c9 = bench.parse_clock_samples(["0, 1900, 2070, 1200, 0x0, Not Active, Not Active, Not Active, Not Active\n"])
    assert c9["reasons"] == [] and c9["temp_c"] is None


def test_traffic_record_follows_the_kernel_source(tmp_path, monkeypatch):
    """roofline.traffic is scaled from the record whose source hash matches
    the kernel source (its DRAM bytes over its algorithmic bytes, times the
    bench workload's algorithmic bytes); a record taken on another version of
    the source reads None."""
    import synth
    h = bench.source_hash("bwd_tc.cu")
    f = tmp_path / "traffic.txt"
    f.write_text("# comment\n"
                 f"kernel=bwd_tc workload=small src={h} bytes_per_launch=300 algorithmic_bytes=200\n"
                 "kernel=fwd_tc workload=small src=0000000000000000 bytes_per_launch=456 algorithmic_bytes=400\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    wl = synth.config(5)
    rec = bench.recorded_traffic("bwd_tc", wl)
    assert rec["ratio"] == 1.5 and rec["captured_on"] == "small"
    assert rec["bytes"] == 1.5 * bench.algorithmic_bytes(wl, "bwd_tc")
    assert bench.recorded_traffic("fwd_tc", wl) is None
    assert bench.recorded_traffic("nonsense", wl) is None


def test_algorithmic_bytes_of_the_training_step():
    """The training-step batch's algorithmic bytes per step, from the sizes:
    T = 190,272 tokens, H = 40, d = 128; the 75,600-token video split 2 x 2."""
    import synth
    wl = synth.config(5)
    thd = 190272 * 40 * 128
    assert bench.algorithmic_bytes(wl, "bwd_tc") == thd * 2 * 4 + 190272 * 40 * 8 + thd * 2 * 2 + thd * 8
    whole = (190272 - 75600) * 40 * (2 * 128 + 4)
    parts = 2 * 75600 * 40 * (4 * 128 + 4)
    assert bench.algorithmic_bytes(wl, "fwd_tc") == 3 * thd * 2 + whole + parts
    assert bench.algorithmic_bytes(wl, "lse_merge") == bench.merge_bytes(wl)


def test_clock_sampler_cleans_up_without_nvidia_smi(monkeypatch):
    """Where nvidia-smi cannot start, the sampler reports None and leaves no
    sample file behind."""
    def no_smi(*a, **k):
        raise OSError("no nvidia-smi")
    monkeypatch.setattr(bench.subprocess, "Popen", no_smi)
    s = bench.ClockSampler("0")
    path = s.path
    assert os.path.exists(path)
    assert s.stop() is None
    assert not os.path.exists(path)


def test_e2e_timeline_summary():
    """Two steps: input copies of 10 ms, compute of 100 ms; the second
    step's input copy runs during the first compute, its compute starts 5 ms
    after the first one ends.  Each step's output leaves in two groups: O
    (4 ms, during the compute) and the gradients (6 ms, after it); the last
    step's gradients leave after all compute."""
    steps = [[0, 10, 10, 110, 50, 54, 110, 116],
             [20, 30, 115, 215, 155, 159, 215, 221]]
    t = bench.e2e_timeline(steps)
    assert t["h2d_ms"] == 10 and t["d2h_ms"] == 10 and t["compute_ms"] == 100
    assert t["compute_idle_ms_between_steps"] == 5
    assert t["first_compute_start_ms"] == 10 and t["last_d2h_after_compute_ms"] == 6
    # hidden: step 2's h2d (20..30) overlaps compute 1 (10 ms); both O copies
    # overlap their compute (8 ms); step 1's gradients (110..116) overlap
    # compute 2 for 1 ms
    assert t["copy_time_overlapped"] == round((10 + 8 + 1) / 40, 4)
    assert bench.e2e_timeline([]) is None

"""Per-bucket attention price table on one GPU.

The Zellige paper's Hardware Profiler (arXiv 2608.01150v1, §IV-B) measures,
once per training setup, the execution time of every sequence bucket under
every parallelism configuration, and the planner then treats a rank's load as
the sum of the prices of the sequences placed on it (the additive model its
§V-B evaluates).  This module is the single-GPU, whole-sequence slice of that
profiler for the attention hot path:

* ``catalog()``: the buckets the paper's workloads span (§V-A: 256p-1080p
  images, 480p-1080p videos of several durations), as latent token counts;
* ``measure_prices()``: the price P_b of one whole sequence of each bucket,
  measured with this library's kernels while the GPU is full (many copies of
  the bucket packed into one coalesced call, time divided by the copies), so
  a price is the sequence's marginal cost inside a busy launch;
* ``predict_ms()``: the additive estimate of a packed batch, sum of prices;
* ``predict_lpt_ms()``: the same prices replayed through the launch's own
  schedule: every work item, in the order the library runs them, goes to the
  SM that comes free first (longest first, as the kernels' work stealing
  does), so a batch of few large items shows its tail.

The measurement uses CUDA events around the library's calls; no arithmetic
happens here.

    python -m mixed_length_dit_gb300.profiler --heads 12 --mode fwd+bwd --out prices.json
"""
from __future__ import annotations

import argparse
import json
import math
import statistics
from dataclasses import dataclass

FPS = 16  # frame rate of the paper's token examples (15 s 1080p -> 241 frames)

# Pixel sizes of the resolutions named in the paper's workloads (§V-A).
_RES = {"256p": (256, 256), "480p": (480, 832), "720p": (720, 1280), "1080p": (1080, 1920)}


def _tokens_video(frames: int, h: int, w: int) -> int:
    return ((frames - 1) // 4 + 1) * math.ceil(h / 16) * math.ceil(w / 16)


def _tokens_image(h: int, w: int) -> int:
    return math.ceil(h / 16) * math.ceil(w / 16)


@dataclass(frozen=True)
class Bucket:
    name: str
    tokens: int
    kind: str  # "image" or "video"


def catalog(durations=(2, 5, 10, 15)):
    """Image buckets 256p-1080p and video buckets 480p-1080p x durations (s),
    smallest first."""
    out = [Bucket(f"img_{r}", _tokens_image(*_RES[r]), "image") for r in ("256p", "480p", "720p", "1080p")]
    for r in ("480p", "720p", "1080p"):
        for sec in durations:
            frames = sec * FPS + 1
            out.append(Bucket(f"vid_{r}_{sec}s", _tokens_video(frames, *_RES[r]), "video"))
    return sorted(out, key=lambda b: b.tokens)


def predict_ms(seqlens, prices: dict, buckets) -> float:
    """Additive estimate of one coalesced call over `seqlens`: the sum of the
    prices of the buckets the sequences fall in (a sequence takes the price of
    the bucket with the nearest token count, scaled by (L / L_bucket)^2, the
    quadratic growth of attention work)."""
    by_tokens = sorted((b.tokens, prices[b.name]) for b in buckets if b.name in prices)
    if not by_tokens:
        raise ValueError("no priced bucket")
    total = 0.0
    for L in seqlens:
        if L <= 0:
            continue
        t, p = min(by_tokens, key=lambda tp: (abs(tp[0] - L), tp[0]))
        total += p * (L / t) ** 2
    return total


def _price(L, by_tokens):
    t, p = min(by_tokens, key=lambda tp: (abs(tp[0] - L), tp[0]))
    return p * (L / t) ** 2


def device_sms(device=None) -> int:
    """SM count of the CUDA device (the current one by default)."""
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("no CUDA device: pass the SM count explicitly")
    d = torch.cuda.current_device() if device is None else device
    return int(torch.cuda.get_device_properties(d).multi_processor_count)


def predict_lpt_ms(seqlens, prices: dict, buckets, num_heads: int, head_dim: int = 128, sms=None,
                   fwd_prices=None, mode: str = "fwd+bwd", tiles=None, fwd_share: float = 0.25) -> float:
    """Makespan estimate of one coalesced call (forward then backward launch
    for mode "fwd+bwd", the forward alone for "fwd").

    A sequence's price is its GPU time while the GPU is full, i.e. its SM time
    over the GPU's SM count (`sms`, by default queried from the current
    device); that SM time is spread over the sequence's work items (from the
    library's own schedule queries, with the tile table `tiles` when some
    sequences are split) in proportion to their query x key work, and the
    items of each launch are dealt in schedule order to the SM that comes free
    first.  With mode "fwd+bwd", `prices` are fwd+bwd prices and the forward
    launch takes each sequence's forward price from `fwd_prices` (measured
    with mode "fwd"), the backward launch the rest; without `fwd_prices` the
    forward takes the fixed share `fwd_share`.  With mode "fwd", `prices` are
    forward prices.  For a batch with many items per SM this equals
    predict_ms; with few, it adds the tail."""
    import heapq

    from . import attention as _attn
    if sms is None:
        sms = device_sms()
    by_tokens = sorted((b.tokens, prices[b.name]) for b in buckets if b.name in prices)
    if not by_tokens:
        raise ValueError("no priced bucket")
    by_tokens_f = None
    if fwd_prices is not None and mode == "fwd+bwd":
        by_tokens_f = sorted((b.tokens, fwd_prices[b.name]) for b in buckets if b.name in fwd_prices)
        if not by_tokens_f:
            raise ValueError("no bucket with a forward price")
    cu = [0]
    for L in seqlens:
        cu.append(cu[-1] + max(0, int(L)))
    price = [_price(L, by_tokens) if L > 0 else 0.0 for L in seqlens]
    if mode == "fwd":
        price_f = price
    elif by_tokens_f is not None:
        price_f = [min(_price(L, by_tokens_f), p) if L > 0 else 0.0 for L, p in zip(seqlens, price)]
    else:
        price_f = [fwd_share * p for p in price]
    price_b = [p - f for p, f in zip(price, price_f)]

    def makespan(items, seq_price):
        # work of every item of a sequence, to split the sequence's SM time
        work = [0.0] * len(seqlens)
        for s, w in items:
            work[s] += w
        free = [0.0] * sms
        for s, w in items:
            t = heapq.heappop(free)
            heapq.heappush(free, t + seq_price[s] * sms * (w / work[s]))
        return max(free)

    fwd = [(it[1], float(it[5]) * it[7]) for it in _attn.fwd_schedule(cu, cu, num_heads, head_dim, tiles)]
    if mode == "fwd":
        return makespan(fwd, price_f)
    bwd = [(it[1], float(it[4]) * it[5]) for it in _attn.bwd_schedule(cu, cu, num_heads, head_dim, tiles)]
    return makespan(fwd, price_f) + makespan(bwd, price_b)


def _time_call(fn, reps: int, warmup: int = 2) -> float:
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.median(times)


def time_batch(seqlens, num_heads: int, head_dim: int = 128, mode: str = "fwd+bwd", reps: int = 3,
               seed: int = 0, tiles=None) -> float:
    """Median device time in ms of one coalesced call (forward, or forward +
    backward) over a packed batch of sequences, split by the tile table
    `tiles` where given."""
    import torch
    from . import attention as zl
    g = torch.Generator(device="cuda").manual_seed(seed)
    t = int(sum(seqlens))
    shape = (t, num_heads, head_dim)
    q, k, v, do = (torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16) for _ in range(4))
    cu = [0]
    for n in seqlens:
        cu.append(cu[-1] + int(n))
    o = torch.empty_like(q)
    lse = torch.empty((num_heads, t), dtype=torch.float32, device="cuda")
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    fws = zl.alloc_workspace(zl.fwd_workspace_bytes(cu, cu, num_heads, head_dim, tiles), "cuda")
    bws = zl.alloc_workspace(zl.bwd_workspace_bytes(cu, cu, num_heads, head_dim), "cuda")

    def call():
        zl.varlen_attn_fwd(q, k, v, cu, cu, tiles=tiles, out=o, lse=lse, workspace=fws)
        if mode == "fwd+bwd":
            zl.varlen_attn_bwd(q, k, v, o, lse, do, cu, cu, tiles=tiles, dq=dq, dk=dk, dv=dv, workspace=bws)

    ms = _time_call(call, reps)
    zl.sync_check()
    return ms


def measure_prices(buckets, num_heads: int = 12, head_dim: int = 128, mode: str = "fwd+bwd",
                   fill_tokens: int = 400_000, reps: int = 3) -> dict:
    """Price (ms) of one whole sequence of each bucket inside a full launch:
    ceil(fill_tokens / tokens) copies packed into one call, time / copies."""
    prices = {}
    for b in buckets:
        n = max(1, math.ceil(fill_tokens / b.tokens))
        prices[b.name] = time_batch([b.tokens] * n, num_heads, head_dim, mode, reps) / n
    return prices


def validate_batch(seqlens, num_heads: int, head_dim: int = 128, tiles=None, fill_tokens: int = 100_000,
                   reps: int = 3) -> dict:
    """Measures the batch's fwd+bwd time and compares it with both estimates,
    the additive one (predict_ms) and the schedule replay (predict_lpt_ms),
    from prices measured on this GPU for exactly the batch's sequence
    lengths (fwd+bwd and forward-only prices, so the replay splits each
    sequence's time between the two launches by measurement).  Returns the
    measured and predicted times (ms) and the relative errors."""
    lens = sorted({int(L) for L in seqlens if L > 0})
    bks = [Bucket(f"len_{L}", L, "batch") for L in lens]
    prices = measure_prices(bks, num_heads, head_dim, "fwd+bwd", fill_tokens, reps)
    fwd_prices = measure_prices(bks, num_heads, head_dim, "fwd", fill_tokens, reps)
    measured = time_batch(seqlens, num_heads, head_dim, "fwd+bwd", reps, tiles=tiles)
    additive = predict_ms(seqlens, prices, bks)
    lpt = predict_lpt_ms(seqlens, prices, bks, num_heads, head_dim, fwd_prices=fwd_prices, tiles=tiles)
    return {"measured_ms": measured, "additive_ms": additive, "lpt_ms": lpt,
            "additive_err": (additive - measured) / measured, "lpt_err": (lpt - measured) / measured,
            "prices_ms": {b.tokens: prices[b.name] for b in bks},
            "fwd_prices_ms": {b.tokens: fwd_prices[b.name] for b in bks}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--heads", type=int, default=12)
    ap.add_argument("--head-dim", type=int, default=128)
    ap.add_argument("--mode", choices=["fwd", "fwd+bwd"], default="fwd+bwd")
    ap.add_argument("--max-tokens", type=int, default=200_000, help="skip buckets longer than this")
    ap.add_argument("--out", default=None)
    ap.add_argument("--validate", default=None,
                    help="comma-separated workload numbers of the repository's synthetic batches (synth.config): "
                         "print measured fwd+bwd time against the additive and schedule-replay estimates")
    args = ap.parse_args()
    if args.validate:
        import synth
        rows = {}
        for n in (int(x) for x in args.validate.split(",")):
            wl = synth.config(n)
            r = validate_batch(wl.seqlens, wl.num_heads, wl.head_dim, tiles=wl.tiles() or None)
            rows[wl.name] = {k: (round(v, 4) if isinstance(v, float) else v) for k, v in r.items()
                             if not k.endswith("prices_ms")}
            print(json.dumps({wl.name: rows[wl.name]}), flush=True)
        if args.out:
            with open(args.out, "w") as f:
                f.write(json.dumps(rows, indent=1) + "\n")
        return
    bks = [b for b in catalog() if b.tokens <= args.max_tokens]
    prices = measure_prices(bks, args.heads, args.head_dim, args.mode)
    flops = {b.name: (3.5 if args.mode == "fwd+bwd" else 1.0) * 4.0 * b.tokens ** 2 * args.head_dim * args.heads
             for b in bks}
    table = {b.name: {"tokens": b.tokens, "kind": b.kind, "ms": round(prices[b.name], 4),
                      "tflops": round(flops[b.name] / (prices[b.name] * 1e-3) / 1e12, 1)} for b in bks}
    text = json.dumps({"heads": args.heads, "head_dim": args.head_dim, "mode": args.mode, "buckets": table},
                      indent=1)
    if args.out:
        with open(args.out, "w") as f:
            f.write(text + "\n")
    print(text)


if __name__ == "__main__":
    main()

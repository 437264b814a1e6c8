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


def predict_lpt_ms(seqlens, prices: dict, buckets, num_heads: int, head_dim: int = 128, sms: int = 152,
                   fwd_share: float = 0.25, mode: str = "fwd+bwd") -> float:
    """Makespan estimate of one coalesced call (forward then backward launch
    for mode "fwd+bwd", the forward alone for "fwd").

    A sequence's price is its GPU time while the GPU is full, i.e. its SM time
    over `sms`; that SM time is spread over the sequence's work items (from
    the library's own schedule queries) in proportion to their query x key
    work, and the items of each launch are dealt in schedule order to the SM
    that comes free first.  With mode "fwd+bwd" the price is split between
    the two launches by `fwd_share` (the forward's share of the training
    step's kernel time, ~0.25 measured); with "fwd" it is all forward.  For a
    batch with many items per SM this equals predict_ms; with few, it adds
    the tail."""
    import heapq

    from . import attention as _attn
    by_tokens = sorted((b.tokens, prices[b.name]) for b in buckets if b.name in prices)
    if not by_tokens:
        raise ValueError("no priced bucket")
    cu = [0]
    for L in seqlens:
        cu.append(cu[-1] + max(0, int(L)))
    price = [_price(L, by_tokens) if L > 0 else 0.0 for L in seqlens]

    def makespan(items, share):
        # work of every item of a sequence, to split the sequence's SM time
        work = [0.0] * len(seqlens)
        for s, w in items:
            work[s] += w
        free = [0.0] * sms
        for s, w in items:
            t = heapq.heappop(free)
            heapq.heappush(free, t + share * price[s] * sms * (w / work[s]))
        return max(free)

    fwd = [(it[1], float(it[5]) * it[7]) for it in _attn.fwd_schedule(cu, cu, num_heads, head_dim)]
    if mode == "fwd":
        return makespan(fwd, 1.0)
    bwd = [(it[1], float(it[4]) * it[5]) for it in _attn.bwd_schedule(cu, cu, num_heads, head_dim)]
    return makespan(fwd, fwd_share) + makespan(bwd, 1.0 - fwd_share)


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
               seed: int = 0) -> float:
    """Median device time in ms of one coalesced call (forward, or forward +
    backward) over a packed batch of whole sequences."""
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
    bws = zl.alloc_workspace(zl.bwd_workspace_bytes(cu, cu, num_heads, head_dim), "cuda")

    def call():
        zl.varlen_attn_fwd(q, k, v, cu, cu, out=o, lse=lse)
        if mode == "fwd+bwd":
            zl.varlen_attn_bwd(q, k, v, o, lse, do, cu, cu, dq=dq, dk=dk, dv=dv, workspace=bws)

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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--heads", type=int, default=12)
    ap.add_argument("--head-dim", type=int, default=128)
    ap.add_argument("--mode", choices=["fwd", "fwd+bwd"], default="fwd+bwd")
    ap.add_argument("--max-tokens", type=int, default=200_000, help="skip buckets longer than this")
    ap.add_argument("--out", default=None)
    args = ap.parse_args()
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

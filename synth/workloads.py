"""Seeded synthetic workloads shaped like the mixed image-video DiT batches.

This module only describes inputs: sequence lengths, head counts, how a long
sequence is cut into (query-chunk x KV-chunk) tiles, and seeded random tensors.
It holds none of the attention arithmetic, so both the CUDA path and the oracle
can take their inputs from it.

Token counts follow the Wan-style latent geometry used by the Zellige paper
("Moldable Sequence Placement for Mixed Image-Video DiT Training", §I and the
Fig. 1 caption): a VAE that compresses time 4x (4k+1 frames -> k+1 latent
frames) and space 8x, then 1x2x2 patches, so a frame of H x W pixels becomes
ceil(H/16) * ceil(W/16) tokens.  The paper's own examples pin this reading:
a 15 s 1080p video at 16 fps (241 frames) is 61 * 68 * 120 = 497,760 tokens
(§I), and a 10 s 1080p video against a 256p image is a 1,307x token ratio
(Fig. 1).  Images use the same 16-pixel token stride (Flux-like 2x2 patches).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

# Pixel sizes of the resolutions named in the paper's workloads (§V-A).
RESOLUTIONS = {
    "256p": (256, 256),
    "480p": (480, 832),
    "720p": (720, 1280),
    "1080p": (1080, 1920),
}


def video_tokens(frames: int, height: int, width: int) -> int:
    """Latent tokens of a video: 4x temporal / 8x spatial VAE, 1x2x2 patch."""
    if frames < 1 or (frames - 1) % 4 != 0:
        raise ValueError("frame count must be 4k+1")
    t = (frames - 1) // 4 + 1
    return t * math.ceil(height / 16) * math.ceil(width / 16)


def image_tokens(height: int, width: int) -> int:
    """Latent tokens of an image with the same 16-pixel token stride."""
    return math.ceil(height / 16) * math.ceil(width / 16)


@dataclass
class Workload:
    name: str
    seqlens: list          # packed order == listed order
    num_heads: int
    head_dim: int
    splits: dict = field(default_factory=dict)  # seq index -> (n_q, n_kv) or (n_q, n_kv, n_h) chunks
    dtype: str = "bf16"

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seqlens))

    def cu_seqlens(self):
        cu = [0]
        for n in self.seqlens:
            cu.append(cu[-1] + int(n))
        return cu

    def tiles(self):
        """Tile table of the split sequences (see chunk_bounds)."""
        out = []
        for s, sp in sorted(self.splits.items()):
            nq, nk = sp[0], sp[1]
            nh = sp[2] if len(sp) > 2 else 1
            out.extend(grid_tiles(s, self.seqlens[s], self.seqlens[s], nq, nk, nh, self.num_heads))
        return out

    def pair_count(self) -> int:
        """Number of (query, key) pairs attended: sum of L^2 over sequences.
        A tile grid covers its sequence exactly once, so splits do not change it."""
        return int(sum(int(n) * int(n) for n in self.seqlens))


def chunk_bounds(length: int, n: int):
    """Contiguous chunks of ceil(length/n) tokens, the last one shorter.
    Returns a list of (start, len)."""
    step = -(-length // n)
    out = []
    for i in range(n):
        a = min(length, i * step)
        b = min(length, (i + 1) * step)
        out.append((a, b - a))
    return out


def grid_tiles(seq: int, q_len: int, k_len: int, n_q: int, n_kv: int, n_h: int = 1, num_heads: int = 0):
    """The full (head-chunk x query-chunk x KV-chunk) grid of one split
    sequence, the (q, h, k) parallelism configuration of the Zellige paper
    (§IV-A), as tuples (seq, q_start, q_len, k_start, k_len, q_chunk,
    kv_chunk, n_kv_chunks, h_start, h_len, h_chunk).  With n_h = 1 the head
    range is left as (0, 0, 0), meaning all heads; with n_h > 1 the num_heads
    heads are cut into chunk_bounds(num_heads, n_h)."""
    qb = chunk_bounds(q_len, n_q)
    kb = chunk_bounds(k_len, n_kv)
    if n_h == 1:
        hb = [(0, 0)]
    else:
        if num_heads < n_h:
            raise ValueError("head split needs num_heads >= n_h")
        hb = chunk_bounds(num_heads, n_h)
        if any(hl == 0 for _, hl in hb):
            raise ValueError(f"{num_heads} heads do not make {n_h} non-empty chunks")
    return [(seq, qa, ql, ka, kl, i, j, n_kv, ha, hl, c)
            for c, (ha, hl) in enumerate(hb)
            for i, (qa, ql) in enumerate(qb)
            for j, (ka, kl) in enumerate(kb)]


def config(n: int) -> Workload:
    """The batches used for parity and measurement (1-based numbering).

    1  tiny correctness batch: lengths 37, 64, 100, 256; 2 heads, d = 64
    2  image-only mix: 16 x 256, 8 x 1024, 4 x 4096 tokens; 24 heads, d = 128
    3  Wan mix: one 480p 81-frame video, two 480p 33-frame videos,
       24 images of 1024 and 8 of 4096 tokens; 40 heads, d = 128
    4  shard mode: one 131,072-token sequence as a 4 x 4 tile grid in the same
       launch as 64 images of 1024 tokens; 40 heads, d = 128
    5  training step: one 720p 81-frame video as a 2 x 2 tile grid, two 480p
       81-frame videos, 4 images of 4096 and 32 of 1024 tokens; 40 heads
    6  profiling case: one 480p 81-frame video (32,760 tokens), 24 heads
    7  the Fig. 2 batch of the Zellige paper: three 720p 10-second videos
       (147,600 tokens, each as a 2 x 2 tile grid) and 228 720p images
       (3,600 tokens); 12 heads, d = 128 (Wan2.1-1.3B)
    8  (q, h, k) configurations (§IV-A): one 720p 81-frame video as (1, 4, 1)
       (Ulysses degree 4: 10 heads per shard), a 480p 81-frame video as
       (2, 2, 2), another as (2, 5, 1), and 24 images of 1024 tokens whole;
       40 heads, d = 128
    9  profiling case of the shard path and the merge: workload 6's video
       as a 2 x 2 tile grid (float32 partials 0.8 GB, above L2)

    `splits` maps a sequence to (n_q, n_kv) or (n_q, n_kv, n_h) chunk counts.
    """
    v480_81 = video_tokens(81, *RESOLUTIONS["480p"])     # 32,760
    v480_33 = video_tokens(33, *RESOLUTIONS["480p"])     # 14,040
    v720_81 = video_tokens(81, *RESOLUTIONS["720p"])     # 75,600
    img256 = image_tokens(*RESOLUTIONS["256p"])          # 256
    img512 = image_tokens(512, 512)                      # 1,024
    img1024 = image_tokens(1024, 1024)                   # 4,096
    if n == 1:
        return Workload("tiny", [37, 64, 100, 256], 2, 64)
    if n == 2:
        return Workload("image_mix", [img256] * 16 + [img512] * 8 + [img1024] * 4, 24, 128)
    if n == 3:
        return Workload("wan_mix",
                        [v480_81] + [v480_33] * 2 + [img512] * 24 + [img1024] * 8, 40, 128)
    if n == 4:
        return Workload("shard_131k", [131072] + [img512] * 64, 40, 128, splits={0: (4, 4)})
    if n == 5:
        return Workload("train_step",
                        [v720_81] + [v480_81] * 2 + [img1024] * 4 + [img512] * 32, 40, 128,
                        splits={0: (2, 2)})
    if n == 6:
        # profiling case: one long video alone, fewer heads (inputs ~200 MB)
        return Workload("video_32k_h24", [v480_81], 24, 128)
    if n == 7:
        # the paper's Fig. 2 batch: three 720p 10-second videos (161 frames at
        # 16 fps) and 228 720p images, with Wan2.1-1.3B's 12 heads of 128;
        # each video runs as a 2 x 2 tile grid beside the whole images
        v720_161 = video_tokens(161, *RESOLUTIONS["720p"])   # 147,600
        img720 = image_tokens(*RESOLUTIONS["720p"])          # 3,600
        return Workload("fig2_mix", [v720_161] * 3 + [img720] * 228, 12, 128,
                        splits={0: (2, 2), 1: (2, 2), 2: (2, 2)})
    if n == 8:
        return Workload("qhk_mix", [v720_81, v480_81, v480_81] + [img512] * 24, 40, 128,
                        splits={0: (1, 1, 4), 1: (2, 2, 2), 2: (2, 1, 5)})
    if n == 9:
        return Workload("video_32k_h24_split", [v480_81], 24, 128, splits={0: (2, 2)})
    raise ValueError(f"no workload {n}")


def make_inputs(wl: Workload, seed: int = 0, device="cpu", dtype=None, with_grad_out=True):
    """q, k, v (and dO) ~ N(0,1), drawn in float32 from one seeded generator in
    that order, then cast to the workload dtype (bf16 rounds to nearest even).
    Shapes [T, H, d].  Returns a dict of tensors on `device`."""
    if dtype is None:
        dtype = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    shape = (wl.total_tokens, wl.num_heads, wl.head_dim)
    out = {}
    names = ["q", "k", "v"] + (["do"] if with_grad_out else [])
    for name in names:
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        out[name] = x.to(dtype)
    return out

"""Randomised parity on the GPU: many small seeded batches, each compared
element by element with the float64 oracle, forward and backward.

Each draw packs 1-9 sequences whose lengths mix exact multiples of the
128-row block (full tiles, which the forward writes with TMA stores) with
ragged ones (a partial last tile, stored row by row), over 1-5 heads of
dimension 64 or 128, and splits some sequences into a (query x head x key)
tile grid (the (q, h, k) configurations of the Zellige paper,
arXiv 2608.01150v1, §IV-A; key-split tiles are merged exactly, §II-B).  The
forward output must be within 2e-2 (max-abs) and the LSE within 1e-3 of the
oracle; each gradient within 2e-2 relative L2 (the backward runs the
sequence whole, whatever its tiles).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import mixed_length_dit_gb300 as zl
from _helpers import TOL_GRAD_REL_L2, TOL_LSE, TOL_O_BF16, f64, rel_l2

pytestmark = pytest.mark.gpu

N_DRAWS = 64


def _draw(rng):
    n_seq = int(rng.integers(1, 10))
    lens = []
    for _ in range(n_seq):
        kind = rng.integers(0, 3)
        if kind == 0:
            lens.append(int(128 * rng.integers(1, 5)))          # whole 128-row tiles
        elif kind == 1:
            lens.append(int(rng.integers(1, 130)))              # up to one partial tile
        else:
            lens.append(int(rng.integers(130, 700)))            # several tiles and a ragged tail
    heads = int(rng.integers(1, 6))
    hd = int(rng.choice([64, 128]))
    tiles = []
    for s, L in enumerate(lens):
        if L >= 4 and rng.random() < 0.35:
            n_q = _nonempty(L, int(rng.integers(1, 4)))
            n_kv = _nonempty(L, int(rng.integers(1, 4)))
            n_h = _nonempty(heads, int(rng.integers(1, heads + 1))) if rng.random() < 0.5 else 1
            if n_q * n_kv * n_h > 1:
                tiles += synth.grid_tiles(s, L, L, n_q, n_kv, n_h, heads)
    return lens, heads, hd, tiles


def _nonempty(length, n):
    """The largest chunk count <= n whose contiguous ceil(length / n) chunks
    are all non-empty (the tile table takes no empty chunk)."""
    while n > 1 and any(c == 0 for _, c in synth.chunk_bounds(length, n)):
        n -= 1
    return n


@pytest.mark.parametrize("draw", range(N_DRAWS))
def test_random_batch_matches_the_oracle(draw):
    rng = np.random.default_rng(1000 + draw)
    lens, heads, hd, tiles = _draw(rng)
    wl = synth.Workload("random", lens, heads, hd)
    inp = synth.make_inputs(wl, seed=draw, device="cuda")
    cu = wl.cu_seqlens()
    o, lse = zl.varlen_attn_fwd(inp["q"], inp["k"], inp["v"], cu, cu, tiles=tiles or None)
    dq, dk, dv = zl.varlen_attn_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], cu, cu, tiles=tiles or None)
    zl.sync_check()
    q, k, v, do = (f64(inp[n]) for n in ("q", "k", "v", "do"))
    o_ref, lse_ref = oracle.varlen_attn_fwd(q, k, v, cu, cu)
    what = (lens, heads, hd, len(tiles))
    assert np.abs(f64(o) - o_ref).max() <= TOL_O_BF16, what
    assert np.abs(f64(lse) - lse_ref).max() <= TOL_LSE, what
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), oracle.varlen_attn_bwd(q, k, v, do, cu, cu)):
        assert torch.isfinite(got).all(), (name, what)
        assert rel_l2(f64(got), ref) <= TOL_GRAD_REL_L2, (name, what, rel_l2(f64(got), ref))


def test_draws_cover_the_cases():
    """The seeded draws include full tiles, partial tiles, both head
    dimensions, key-split and head-split tile grids."""
    seen = {"full": False, "partial": False, 64: False, 128: False, "kv_split": False, "h_split": False}
    for draw in range(N_DRAWS):
        lens, heads, hd, tiles = _draw(np.random.default_rng(1000 + draw))
        seen["full"] |= any(L % 128 == 0 for L in lens)
        seen["partial"] |= any(L % 128 != 0 for L in lens)
        seen[hd] = True
        seen["kv_split"] |= any(t[7] > 1 for t in tiles)
        seen["h_split"] |= any(t[9] > 0 for t in tiles)
    assert all(seen.values()), seen

"""Backward parity on the GPU against the float64 oracle's analytic gradient
of O = softmax(Q K^T * scale) V (exact backward, as the Zellige paper trains
with, arXiv 2608.01150v1 §V-A).  The GPU backward consumes the GPU forward's
own O and LSE; the oracle recomputes everything in float64 from q, k, v, dO.
Tolerance: relative L2 error 2e-2 per gradient.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import mixed_length_dit_gb300 as zl
from _helpers import TOL_GRAD_REL_L2, f64, rel_l2, sample_rows

pytestmark = pytest.mark.gpu


def _fwd_bwd(q, k, v, do, cu_q, cu_k, tiles=None):
    o, lse = zl.varlen_attn_fwd(q, k, v, cu_q, cu_k, tiles=tiles)
    dq, dk, dv = zl.varlen_attn_bwd(q, k, v, o, lse, do, cu_q, cu_k, tiles=tiles)
    zl.sync_check()
    return dq, dk, dv


def _full_grad_check(q, k, v, do, cu_q, cu_k, grads, heads=None):
    ref = oracle.varlen_attn_bwd(f64(q), f64(k), f64(v), f64(do), cu_q, cu_k, heads=heads)
    hs = slice(None) if heads is None else list(heads)
    errs = []
    for name, got, r in zip(("dq", "dk", "dv"), grads, ref):
        e = rel_l2(f64(got)[:, hs], r[:, hs])
        errs.append(e)
        assert e <= TOL_GRAD_REL_L2, (name, e)
    return errs


@pytest.mark.parametrize("hd", [64, 128])
def test_tiny(hd):
    wl = synth.Workload("tiny", [37, 64, 100, 256], 2, hd)
    inp = synth.make_inputs(wl, seed=0, device="cuda")
    cu = wl.cu_seqlens()
    grads = _fwd_bwd(inp["q"], inp["k"], inp["v"], inp["do"], cu, cu)
    _full_grad_check(inp["q"], inp["k"], inp["v"], inp["do"], cu, cu, grads)


def test_ragged_edges():
    lens = [1, 2, 127, 128, 129, 0, 255, 257, 3]
    wl = synth.Workload("edges", lens, 3, 128)
    inp = synth.make_inputs(wl, seed=4, device="cuda")
    cu = wl.cu_seqlens()
    grads = _fwd_bwd(inp["q"], inp["k"], inp["v"], inp["do"], cu, cu)
    _full_grad_check(inp["q"], inp["k"], inp["v"], inp["do"], cu, cu, grads)


def test_cross_lengths_and_keys_without_queries():
    """Sequence 1 has keys but no queries: its dK/dV are zero."""
    cu_q = [0, 70, 70, 400]
    cu_k = [0, 200, 330, 500]
    g = torch.Generator(device="cuda").manual_seed(3)
    mk = lambda n: torch.randn((n, 2, 128), generator=g, device="cuda").to(torch.bfloat16)
    q, k, v, do = mk(400), mk(500), mk(500), mk(400)
    grads = _fwd_bwd(q, k, v, do, cu_q, cu_k)
    _full_grad_check(q, k, v, do, cu_q, cu_k, grads)
    assert torch.all(grads[1][200:330] == 0) and torch.all(grads[2][200:330] == 0)


@pytest.mark.parametrize("n_q,n_kv,n_h", [(3, 2, 1), (2, 2, 2), (1, 1, 2)])
def test_tiles_equal_whole(n_q, n_kv, n_h):
    """The backward of a split sequence sums its tiles' contributions, which is
    the backward of the whole sequence, for query, key and head splits
    (the (q, h, k) configurations of the Zellige paper, §IV-A)."""
    wl = synth.Workload("split", [700, 90, 300], 2, 128)
    inp = synth.make_inputs(wl, seed=8, device="cuda")
    cu = wl.cu_seqlens()
    tiles = synth.grid_tiles(0, 700, 700, n_q, n_kv, n_h, 2)
    g_t = _fwd_bwd(inp["q"], inp["k"], inp["v"], inp["do"], cu, cu, tiles)
    g_w = _fwd_bwd(inp["q"], inp["k"], inp["v"], inp["do"], cu, cu, None)
    for a, b in zip(g_t, g_w):
        assert (a.float() - b.float()).abs().max().item() <= 2e-2
    _full_grad_check(inp["q"], inp["k"], inp["v"], inp["do"], cu, cu, g_t)


def test_image_mix_heads():
    """Image-only mix (28 sequences, 24 heads): all sequences, two heads."""
    wl = synth.config(2)
    inp = synth.make_inputs(wl, seed=0, device="cuda")
    cu = wl.cu_seqlens()
    grads = _fwd_bwd(inp["q"], inp["k"], inp["v"], inp["do"], cu, cu)
    _full_grad_check(inp["q"], inp["k"], inp["v"], inp["do"], cu, cu, grads, heads=[0, 23])


def test_train_step_sampled():
    """Training-step batch (75,600-token video as 2 x 2 tiles, two 32,760-token
    videos, 36 images; 40 heads): dQ rows and dK/dV rows sampled per sequence
    kind on one head each; every row value is exact, so sampling loses nothing."""
    wl = synth.config(5)
    inp = synth.make_inputs(wl, seed=0, device="cuda")
    cu = wl.cu_seqlens()
    dq, dk, dv = _fwd_bwd(inp["q"], inp["k"], inp["v"], inp["do"], cu, cu, wl.tiles())
    rng = np.random.default_rng(1)
    checks = [(0, 7), (1, 0), (3, 39), (7, 21)]       # (sequence, head)
    for s, h in checks:
        L = wl.seqlens[s]
        a, b = cu[s], cu[s + 1]
        rows = sample_rows(L, synth.chunk_bounds(L, wl.splits.get(s, (1, 1))[0]), 256, rng)
        qs, ks, vs, dos = (f64(inp[n][a:b]) for n in ("q", "k", "v", "do"))
        cu1 = [0, L]
        dq_ref = oracle.dq_rows(qs, ks, vs, dos, cu1, cu1, 0, h, rows)
        dk_ref, dv_ref = oracle.dkdv_rows(qs, ks, vs, dos, cu1, cu1, 0, h, rows)
        for name, got, ref in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
            e = rel_l2(f64(got[a:b][rows, h]), ref)
            assert e <= TOL_GRAD_REL_L2, (s, h, name, e)


def test_dk_dv_isolation_bitwise():
    """Changing one sequence leaves the other sequences' dK and dV bit-identical
    (they are written once per key block, without atomics)."""
    wl = synth.Workload("iso", [300, 64, 1000, 129], 2, 128)
    inp = synth.make_inputs(wl, seed=2, device="cuda")
    cu = wl.cu_seqlens()
    g1 = _fwd_bwd(inp["q"], inp["k"], inp["v"], inp["do"], cu, cu)
    inp2 = {n: t.clone() for n, t in inp.items()}
    a, b = cu[2], cu[3]
    inp2["k"][a:b] += 0.5
    inp2["do"][a:b] *= 2
    g2 = _fwd_bwd(inp2["q"], inp2["k"], inp2["v"], inp2["do"], cu, cu)
    for s in (0, 1, 3):
        x, y = cu[s], cu[s + 1]
        assert torch.equal(g1[1][x:y], g2[1][x:y])
        assert torch.equal(g1[2][x:y], g2[2][x:y])


def test_concurrent_launches_on_two_streams():
    """Two backward launches in flight at once on different streams each do
    every one of their own work items exactly once: dK and dV (written once
    per key block) are bit-identical to the launches run one after the other,
    dQ (summed by additions in L2, whose order varies) agrees to rounding."""
    wa = synth.config(2)
    wb = synth.Workload("two_streams_b", [9000, 3000, 500, 1024], 8, 128)

    def prep(wl, seed):
        inp = synth.make_inputs(wl, seed=seed, device="cuda")
        cu = wl.cu_seqlens()
        o, lse = zl.varlen_attn_fwd(inp["q"], inp["k"], inp["v"], cu, cu)
        ws = zl.alloc_workspace(zl.bwd_workspace_bytes(cu, cu, wl.num_heads, wl.head_dim), "cuda")
        grads = tuple(torch.empty_like(inp[n]) for n in ("q", "k", "v"))
        return inp, cu, o, lse, ws, grads

    a, b = prep(wa, 5), prep(wb, 6)

    def launch(x, stream):
        inp, cu, o, lse, ws, (dq, dk, dv) = x
        zl.varlen_attn_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], cu, cu, dq=dq, dk=dk, dv=dv,
                           workspace=ws, stream=stream)

    launch(a, None)
    launch(b, None)
    torch.cuda.synchronize()
    ref = [tuple(g.clone() for g in x[5]) for x in (a, b)]
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        for x in (a, b):
            for g in x[5]:
                g.zero_()
        torch.cuda.synchronize()
        launch(a, s1)
        launch(b, s2)
        torch.cuda.synchronize()
        for x, r in zip((a, b), ref):
            dq, dk, dv = x[5]
            assert torch.equal(dk, r[1]) and torch.equal(dv, r[2])
            assert (dq.float() - r[0].float()).abs().max().item() <= 1e-2 * r[0].float().abs().max().item()
    zl.sync_check()

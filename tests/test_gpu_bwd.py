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
        qs, ks, vs, dos = (f64(inp[n][a:b, h:h + 1]) for n in ("q", "k", "v", "do"))   # one head
        cu1 = [0, L]
        dq_ref = oracle.dq_rows(qs, ks, vs, dos, cu1, cu1, 0, 0, rows)
        dk_ref, dv_ref = oracle.dkdv_rows(qs, ks, vs, dos, cu1, cu1, 0, 0, rows)
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


def _sampled_grad_check(wl, inp, cu, grads, checks, n_random=256, seed=1):
    dq, dk, dv = grads
    rng = np.random.default_rng(seed)
    for s, h in checks:
        L = wl.seqlens[s]
        a, b = cu[s], cu[s + 1]
        rows = sample_rows(L, synth.chunk_bounds(L, wl.splits.get(s, (1, 1))[0]), n_random, rng)
        qs, ks, vs, dos = (f64(inp[n][a:b, h:h + 1]) for n in ("q", "k", "v", "do"))   # one head
        cu1 = [0, L]
        dq_ref = oracle.dq_rows(qs, ks, vs, dos, cu1, cu1, 0, 0, rows)
        dk_ref, dv_ref = oracle.dkdv_rows(qs, ks, vs, dos, cu1, cu1, 0, 0, rows)
        for name, got, ref in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
            e = rel_l2(f64(got[a:b][rows, h]), ref)
            assert e <= TOL_GRAD_REL_L2, (s, h, name, e)


def test_wan_mix_sampled():
    """Wan mix (32,760- and 14,040-token videos, 1,024- and 4,096-token images,
    40 heads): dQ, dK and dV rows sampled on one head per sequence kind."""
    wl = synth.config(3)
    inp = synth.make_inputs(wl, seed=0, device="cuda")
    cu = wl.cu_seqlens()
    grads = _fwd_bwd(inp["q"], inp["k"], inp["v"], inp["do"], cu, cu)
    _sampled_grad_check(wl, inp, cu, grads, [(0, 5), (1, 39), (3, 12), (30, 27)])


def test_shard_mode_131k_dense():
    """131,072-token sequence (run as 4 x 4 tiles in the forward) beside 64
    images, dense dO: dQ rows of the long sequence sampled on two heads, every
    gradient of two images on one head each, and on every head of the long
    sequence the identity sum_j dV_j = sum_i dO_i (rows of P sum to one)."""
    wl = synth.config(4)
    inp = synth.make_inputs(wl, seed=0, device="cuda")
    cu = wl.cu_seqlens()
    dq, dk, dv = _fwd_bwd(inp["q"], inp["k"], inp["v"], inp["do"], cu, cu, wl.tiles())
    L = wl.seqlens[0]
    rng = np.random.default_rng(2)
    rows = sample_rows(L, synth.chunk_bounds(L, 4), 256, rng)
    for h in (0, 33):
        qs, ks, vs, dos = (f64(inp[n][:L, h:h + 1]) for n in ("q", "k", "v", "do"))   # one head
        ref = oracle.dq_rows(qs, ks, vs, dos, [0, L], [0, L], 0, 0, rows)
        e = rel_l2(f64(dq[rows, h]), ref)
        assert e <= TOL_GRAD_REL_L2, (h, e)
    _sampled_grad_check(wl, inp, cu, (dq, dk, dv), [(1, 7), (64, 39)], n_random=1024)
    # bf16 rounding of P and of dV (2^-9 relative per entry, random in sign)
    # leaves the identity's relative error near 1e-5
    sv = dv[:L].double().sum(dim=0)
    so = inp["do"][:L].double().sum(dim=0)
    e = ((sv - so).norm() / so.norm()).item()
    assert e <= 1e-3, e


def test_shard_mode_131k_one_query_row():
    """The same batch with dO zero except one query row of the long sequence on
    three heads: dK and dV of all 131,072 keys of those heads come from that
    row's softmax alone and are checked exactly, as is dQ of the row; every
    other dQ row, and every gradient of the other heads and sequences, is
    zero."""
    wl = synth.config(4)
    inp = synth.make_inputs(wl, seed=1, device="cuda")
    cu = wl.cu_seqlens()
    L = wl.seqlens[0]
    picks = {0: 0, 17: 65535, 39: 131071}            # head -> query row
    do = torch.zeros_like(inp["do"])
    for h, r in picks.items():
        do[r, h] = inp["do"][r, h]
    dq, dk, dv = _fwd_bwd(inp["q"], inp["k"], inp["v"], do, cu, cu, wl.tiles())
    for h, r in picks.items():
        qs, ks, vs = (f64(inp[n][:L, h:h + 1]) for n in ("q", "k", "v"))            # one head
        dq_r, dk_ref, dv_ref = oracle.grads_one_query_row(qs, ks, vs, f64(do[r, h]), [0, L], [0, L], 0, 0, r)
        for name, got, ref in (("dq", dq[r, h], dq_r), ("dk", dk[:L, h], dk_ref), ("dv", dv[:L, h], dv_ref)):
            e = rel_l2(f64(got), ref)
            assert e <= TOL_GRAD_REL_L2, (h, name, e)
        others = torch.ones(dq.shape[0], dtype=torch.bool, device="cuda")
        others[r] = False
        assert torch.count_nonzero(dq[others, h]).item() == 0
    quiet = [h for h in range(wl.num_heads) if h not in picks]
    for g in (dq, dk, dv):
        assert torch.count_nonzero(g[:, quiet]).item() == 0
        assert torch.count_nonzero(g[L:]).item() == 0


def test_fig2_mix_dense():
    """The Fig. 2 batch (three 147,600-token videos, run as 2 x 2 tiles in the
    forward, beside 228 images of 3,600 tokens; 12 heads), dense dO: dQ rows of
    one video sampled on two heads, every gradient of two images on one head
    each, and for each video on every head sum_j dV_j = sum_i dO_i."""
    wl = synth.config(7)
    inp = synth.make_inputs(wl, seed=0, device="cuda")
    cu = wl.cu_seqlens()
    dq, dk, dv = _fwd_bwd(inp["q"], inp["k"], inp["v"], inp["do"], cu, cu, wl.tiles())
    L = wl.seqlens[1]
    a = cu[1]
    rng = np.random.default_rng(3)
    rows = sample_rows(L, synth.chunk_bounds(L, 2), 256, rng)
    for h in (0, 11):
        qs, ks, vs, dos = (f64(inp[n][a:a + L, h:h + 1]) for n in ("q", "k", "v", "do"))
        ref = oracle.dq_rows(qs, ks, vs, dos, [0, L], [0, L], 0, 0, rows)
        e = rel_l2(f64(dq[a:a + L][rows, h]), ref)
        assert e <= TOL_GRAD_REL_L2, (h, e)
    _sampled_grad_check(wl, inp, cu, (dq, dk, dv), [(3, 4), (230, 9)], n_random=1024)
    for s in range(3):
        x, y = cu[s], cu[s + 1]
        sv = dv[x:y].double().sum(dim=0)
        so = inp["do"][x:y].double().sum(dim=0)
        e = ((sv - so).norm() / so.norm()).item()
        assert e <= 1e-3, (s, e)


def test_more_sequences_than_one_launch_holds():
    """1,400 short sequences (more than two launches' 640-segment tables): the
    forward and the backward each run as three launches, whose work items
    are numbered per launch and stolen within their own grid; every output
    and gradient element against the oracle."""
    rng = np.random.default_rng(6)
    lens = [int(x) for x in rng.integers(1, 150, size=1400)]
    wl = synth.Workload("many", lens, 2, 64)
    inp = synth.make_inputs(wl, seed=6, device="cuda")
    cu = wl.cu_seqlens()
    n0 = zl.launch_count()
    o, lse = zl.varlen_attn_fwd(inp["q"], inp["k"], inp["v"], cu, cu)
    zl.sync_check()
    assert zl.launch_count() - n0 == 3
    o_ref, l_ref = oracle.varlen_attn_fwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), cu, cu)
    assert np.abs(f64(o) - o_ref).max() <= 2e-2
    assert np.abs(f64(lse) - l_ref).max() <= 1e-3
    grads = zl.varlen_attn_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], cu, cu)
    zl.sync_check()
    _full_grad_check(inp["q"], inp["k"], inp["v"], inp["do"], cu, cu, grads)

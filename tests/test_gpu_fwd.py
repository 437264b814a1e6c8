"""Forward parity on the GPU: the CUDA path through the C ABI against the
float64 oracle on the same seeded inputs.

The operation is the coalesced block-diagonal attention of Zellige
(arXiv 2608.01150v1) §IV-D, with shards of split sequences computed as
(query-chunk x KV-chunk) tiles and merged exactly (§II-B, Table II).
Tolerances: bf16 O max-abs 2e-2 and LSE 1e-3 against float64; float32 mode
1e-4.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import mixed_length_dit_gb300 as zl
from _helpers import TOL_FP32, TOL_GRAD_REL_L2, TOL_LSE, TOL_O_BF16, f64, rel_l2, sample_rows

pytestmark = pytest.mark.gpu


def _run(inp, wl, tiles=None, cu_q=None, cu_k=None):
    cu = wl.cu_seqlens()
    o, lse = zl.varlen_attn_fwd(inp["q"], inp["k"], inp["v"], cu_q or cu, cu_k or cu, tiles=tiles)
    zl.sync_check()
    return o, lse


def _full_check(q, k, v, cu_q, cu_k, o, lse, tol_o, tol_lse):
    o_ref, lse_ref = oracle.varlen_attn_fwd(f64(q), f64(k), f64(v), cu_q, cu_k)
    err_o = np.abs(f64(o) - o_ref).max()
    mask = np.isfinite(lse_ref)
    err_l = np.abs(f64(lse)[mask] - lse_ref[mask]).max() if mask.any() else 0.0
    assert err_o <= tol_o, f"O max-abs {err_o}"
    assert err_l <= tol_lse, f"LSE max-abs {err_l}"
    return err_o, err_l


@pytest.mark.parametrize("split", [False, True])
def test_tiny_bf16(split):
    wl = synth.config(1)
    inp = synth.make_inputs(wl, seed=0, device="cuda", with_grad_out=False)
    tiles = None
    if split:
        tiles = synth.grid_tiles(3, 256, 256, 2, 2) + synth.grid_tiles(2, 100, 100, 3, 2)
    o, lse = _run(inp, wl, tiles)
    cu = wl.cu_seqlens()
    _full_check(inp["q"], inp["k"], inp["v"], cu, cu, o, lse, TOL_O_BF16, TOL_LSE)


@pytest.mark.parametrize("split", [False, True])
def test_tiny_fp32(split):
    wl = synth.config(1)
    inp = synth.make_inputs(wl, seed=0, device="cuda", dtype=torch.float32, with_grad_out=False)
    tiles = synth.grid_tiles(3, 256, 256, 2, 2) if split else None
    o, lse = _run(inp, wl, tiles)
    assert o.dtype == torch.float32
    cu = wl.cu_seqlens()
    _full_check(inp["q"], inp["k"], inp["v"], cu, cu, o, lse, TOL_FP32, TOL_FP32)


@pytest.mark.parametrize("split", [False, True])
def test_tiny_fp32_head_dim_128(split):
    """The float32 path at head_dim 128, whose kernel splits each query row's
    dot products over two threads: the tiny batch's lengths at d = 128, whole
    and with the 256-token sequence as a 2 x 2 tile grid."""
    wl = synth.Workload("tiny128", [37, 64, 100, 256], 2, 128)
    inp = synth.make_inputs(wl, seed=3, device="cuda", dtype=torch.float32, with_grad_out=False)
    tiles = synth.grid_tiles(3, 256, 256, 2, 2) if split else None
    o, lse = _run(inp, wl, tiles)
    assert o.dtype == torch.float32
    cu = wl.cu_seqlens()
    _full_check(inp["q"], inp["k"], inp["v"], cu, cu, o, lse, TOL_FP32, TOL_FP32)


@pytest.mark.parametrize("hd", [64, 128])
def test_ragged_edges(hd):
    """Lengths around the 128-row block: 1, 2, 127, 128, 129, 255, 257, an
    empty sequence, and a short tail."""
    lens = [1, 2, 127, 128, 129, 0, 255, 257, 3]
    wl = synth.Workload("edges", lens, 3, hd)
    inp = synth.make_inputs(wl, seed=5, device="cuda", with_grad_out=False)
    o, lse = _run(inp, wl)
    cu = wl.cu_seqlens()
    _full_check(inp["q"], inp["k"], inp["v"], cu, cu, o, lse, TOL_O_BF16, TOL_LSE)



@pytest.mark.parametrize("case", ["block", "inner", "growing"])
@pytest.mark.parametrize("split", [False, True])
def test_running_max_jumps(case, split):
    """Keys whose scores jump after the first key block, so that the running
    maximum of nearly every query row grows by more than the lazy-rescale
    threshold (2^8) in the middle of the sequence, which N(0, 1) inputs never
    do: a whole 128-key block scaled by 6 (its first 32 columns already
    exceed the threshold), only keys 40-99 of a block scaled by 6 (the
    exponentials of the block's first 32 columns start on the old maximum
    and must be redone), and every block scaled by 1.5^j (repeated
    rescales, the last one in the partial block).  Forward O and LSE against
    the oracle, whole and as a 2 x 2 tile grid, then the backward's
    gradients from that O and LSE."""
    L = 1000
    wl = synth.Workload("jumps", [L, 300], 2, 128)
    inp = synth.make_inputs(wl, seed=11, device="cuda")
    k = inp["k"].float()
    if case == "block":
        k[384:512] *= 6
    elif case == "inner":
        k[384 + 40:384 + 100] *= 6
    else:
        for j in range(8):
            k[128 * j:128 * (j + 1)] *= 1.5 ** j
    inp["k"] = k.to(torch.bfloat16)
    tiles = synth.grid_tiles(0, L, L, 2, 2) if split else None
    cu = wl.cu_seqlens()
    o, lse = _run(inp, wl, tiles)
    _full_check(inp["q"], inp["k"], inp["v"], cu, cu, o, lse, TOL_O_BF16, TOL_LSE)
    dq, dk, dv = zl.varlen_attn_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], cu, cu, tiles=tiles)
    zl.sync_check()
    refs = oracle.varlen_attn_bwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["do"]), cu, cu)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        assert rel_l2(f64(got), ref) <= TOL_GRAD_REL_L2, (name, rel_l2(f64(got), ref))


def test_binding_refuses_tensors_that_disagree_with_the_batch():
    """The C ABI receives pointers only, so the binding refuses, before any
    launch, tensors whose rows, heads, head dimension, dtype or device
    disagree with the batch (a shorter tensor would be read or written past
    its end)."""
    wl = synth.Workload("chk", [100, 60], 2, 64)
    inp = synth.make_inputs(wl, seed=0, device="cuda")
    cu = wl.cu_seqlens()
    q, k, v, do = inp["q"], inp["k"], inp["v"], inp["do"]
    n0 = zl.launch_count()
    bad_inputs = [
        (q[:150], k, v),                          # fewer rows than cu_seqlens_q ends at
        (q, torch.cat([k, k[:8]]), v),            # more key rows than cu_seqlens_k ends at
        (q, k[:, :1].contiguous(), v),            # another head count
        (q, k, v[..., :32].contiguous()),         # another head dimension
        (q, k, v.float()),                        # another dtype
    ]
    for qq, kk, vv in bad_inputs:
        with pytest.raises(ValueError):
            zl.varlen_attn_fwd(qq, kk, vv, cu, cu)
    with pytest.raises(ValueError):
        zl.varlen_attn_fwd(q, k, v, cu, cu, out=torch.empty_like(q[:10]))
    with pytest.raises(ValueError):
        zl.varlen_attn_fwd(q, k, v, cu, cu, lse=torch.empty((2, 10), device="cuda"))
    assert zl.launch_count() == n0
    o, lse = zl.varlen_attn_fwd(q, k, v, cu, cu)
    zl.sync_check()
    n1 = zl.launch_count()
    for args, kw in [((q, k, v, o, lse, do[:, :1].contiguous()), {}),
                     ((q, k, v, o, lse.t().contiguous(), do), {}),
                     ((q, k, v, o[:100], lse, do), {}),
                     ((q, k, v, o, lse, do), {"dk": torch.empty_like(k[:100])}),
                     ((q, k, v, o, lse, do), {"dq": torch.empty_like(q).float()})]:
        with pytest.raises(ValueError):
            zl.varlen_attn_bwd(*args, cu, cu, **kw)
    part = torch.zeros((2, 16, 2, 64), device="cuda")
    with pytest.raises(ValueError):
        zl.lse_merge(part, torch.zeros((2, 16, 2), device="cuda"))        # [P, R, H] instead of [P, H, R]
    with pytest.raises(ValueError):
        zl.lse_merge(part, torch.zeros((2, 2, 16), device="cuda"), rows=17)
    assert zl.launch_count() == n1

def test_different_query_and_key_lengths():
    cu_q = [0, 5, 200, 330]
    cu_k = [0, 130, 140, 600]
    g = torch.Generator(device="cuda").manual_seed(9)
    q = torch.randn((330, 2, 128), generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn((600, 2, 128), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((600, 2, 128), generator=g, device="cuda").to(torch.bfloat16)
    o, lse = zl.varlen_attn_fwd(q, k, v, cu_q, cu_k)
    zl.sync_check()
    _full_check(q, k, v, cu_q, cu_k, o, lse, TOL_O_BF16, TOL_LSE)
    # the same batch with sequence 2 split into a 2 x 3 grid of tiles
    tiles = synth.grid_tiles(2, 130, 460, 2, 3)
    o2, lse2 = zl.varlen_attn_fwd(q, k, v, cu_q, cu_k, tiles=tiles)
    zl.sync_check()
    _full_check(q, k, v, cu_q, cu_k, o2, lse2, TOL_O_BF16, TOL_LSE)


def test_image_mix_full():
    """Image-only mix: 16 x 256 + 8 x 1024 + 4 x 4096 tokens, 24 heads, d = 128,
    every row and head against the oracle."""
    wl = synth.config(2)
    inp = synth.make_inputs(wl, seed=0, device="cuda", with_grad_out=False)
    o, lse = _run(inp, wl)
    cu = wl.cu_seqlens()
    _full_check(inp["q"], inp["k"], inp["v"], cu, cu, o, lse, TOL_O_BF16, TOL_LSE)


def _sampled_check(wl, inp, o, lse, seed=0, n_random=2048, max_heads_long=4):
    """Row-sampled parity: rows are independent, so the oracle's value for a
    sampled row is exactly the full call's value for it."""
    rng = np.random.default_rng(seed)
    cu = wl.cu_seqlens()
    splits = wl.splits
    worst_o = worst_l = 0.0
    for s, L in enumerate(wl.seqlens):
        if L == 0:
            continue
        nq = splits.get(s, (1, 1))[0]
        rows = sample_rows(L, synth.chunk_bounds(L, nq), n_random, rng)
        heads = list(range(wl.num_heads))
        if L > 32768:
            heads = sorted(set([0, wl.num_heads - 1] + list(rng.choice(wl.num_heads, max_heads_long - 2,
                                                                        replace=False))))
        a, b = cu[s], cu[s + 1]
        cu1 = [0, L]
        idx = torch.as_tensor(rows, device=o.device)
        long_seq = L > 32768
        if not long_seq:                     # every head is checked: one bulk copy
            q_all, k_all, v_all = (f64(inp[n][a:b]) for n in ("q", "k", "v"))
        for h in heads:
            if long_seq:                     # a few heads of a long sequence: copy only those
                qs, ks, vs = (f64(inp[n][a:b, h:h + 1]) for n in ("q", "k", "v"))
                hh = 0
            else:
                qs, ks, vs, hh = q_all, k_all, v_all, h
            o_ref, l_ref = oracle.attention_rows(qs, ks, vs, cu1, cu1, 0, hh, rows)
            worst_o = max(worst_o, float(np.abs(f64(o[a:b, h][idx]) - o_ref).max()))
            worst_l = max(worst_l, float(np.abs(f64(lse[h, a:b][idx]) - l_ref).max()))
    assert worst_o <= TOL_O_BF16, worst_o
    assert worst_l <= TOL_LSE, worst_l
    return worst_o, worst_l


def test_wan_mix_sampled():
    wl = synth.config(3)
    inp = synth.make_inputs(wl, seed=0, device="cuda", with_grad_out=False)
    o, lse = _run(inp, wl)
    _sampled_check(wl, inp, o, lse, n_random=1024)


def test_shard_mode_131k():
    """One 131,072-token sequence as 4 x 4 tiles beside 64 images of 1024
    tokens in one launch, then the merge: equals the same batch run whole, and
    the oracle on sampled rows."""
    wl = synth.config(4)
    inp = synth.make_inputs(wl, seed=0, device="cuda", with_grad_out=False)
    o, lse = _run(inp, wl, wl.tiles())
    _sampled_check(wl, inp, o, lse, n_random=512, max_heads_long=3)
    o_whole, lse_whole = _run(inp, wl, None)
    assert (o - o_whole).abs().max().item() <= TOL_O_BF16
    assert (lse - lse_whole).abs().max().item() <= TOL_LSE
    # images are not split: identical work items, identical bits
    a = wl.seqlens[0]
    assert torch.equal(o[a:], o_whole[a:])


def test_train_step_mix_sampled():
    wl = synth.config(5)
    inp = synth.make_inputs(wl, seed=0, device="cuda", with_grad_out=False)
    o, lse = _run(inp, wl, wl.tiles())
    _sampled_check(wl, inp, o, lse, n_random=512, max_heads_long=3)


def test_fig2_mix_sampled():
    """The paper's Fig. 2 batch (three 147,600-token videos as 2 x 2 tiles and
    228 images of 3,600 tokens, 12 heads) through the same engine."""
    wl = synth.config(7)
    inp = synth.make_inputs(wl, seed=0, device="cuda", with_grad_out=False)
    o, lse = _run(inp, wl, wl.tiles())
    _sampled_check(wl, inp, o, lse, n_random=256, max_heads_long=3)


HEAD_SPLIT_CASES = [
    # (seq, n_q, n_kv, n_h) on the tiny batch (lengths 37, 64, 100, 256; 2 heads)
    [(3, 1, 1, 2)],
    [(3, 2, 2, 2), (2, 1, 1, 2)],
    [(3, 1, 3, 2), (0, 2, 1, 2), (1, 1, 2, 1)],
]


def _head_tiles(cases, lens, nh):
    return [t for s, nq, nk, nhc in cases for t in synth.grid_tiles(s, lens[s], lens[s], nq, nk, nhc, nh)]


@pytest.mark.parametrize("case", range(len(HEAD_SPLIT_CASES)))
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_head_sharded_tiles_tiny(case, dtype):
    """(q, h, k) configurations of the Zellige paper (§IV-A, Table II) as tile
    tables: query, head and key splits, alone and composed, against the oracle."""
    wl = synth.config(1)
    inp = synth.make_inputs(wl, seed=4, device="cuda", dtype=dtype, with_grad_out=False)
    tiles = _head_tiles(HEAD_SPLIT_CASES[case], wl.seqlens, wl.num_heads)
    o, lse = _run(inp, wl, tiles)
    cu = wl.cu_seqlens()
    tol_o, tol_l = (TOL_O_BF16, TOL_LSE) if dtype == torch.bfloat16 else (TOL_FP32, TOL_FP32)
    _full_check(inp["q"], inp["k"], inp["v"], cu, cu, o, lse, tol_o, tol_l)
    if dtype == torch.bfloat16:
        o2, l2 = zl.varlen_attn_fwd(inp["q"], inp["k"], inp["v"], cu, cu, tiles=tiles, fused_merge=True)
        zl.sync_check()
        _full_check(inp["q"], inp["k"], inp["v"], cu, cu, o2, l2, tol_o, tol_l)


def test_query_and_head_splits_are_bitwise_whole():
    """A sequence cut only along queries and heads, (q, h, 1), computes every
    row over all of its keys in the same order as the whole sequence: no
    partials, no merge launch, and bit-identical output."""
    wl = synth.Workload("qh", [3000, 517, 1024], 8, 128)
    inp = synth.make_inputs(wl, seed=5, device="cuda", with_grad_out=False)
    cu = wl.cu_seqlens()
    tiles = synth.grid_tiles(0, 3000, 3000, 3, 1, 4, 8) + synth.grid_tiles(1, 517, 517, 1, 1, 3, 8)
    assert zl.fwd_workspace_bytes(cu, cu, 8, 128, tiles) == 0
    o_whole, l_whole = _run(inp, wl, None)
    n0 = zl.launch_count()
    o, lse = _run(inp, wl, tiles)
    assert zl.launch_count() - n0 == 1
    assert torch.equal(o, o_whole) and torch.equal(lse, l_whole)


def test_qhk_mix_sampled():
    """A training-size batch with a Ulysses-style (1, 4, 1) 720p video, a
    composed (2, 2, 2) and a (2, 5, 1) 480p video beside whole images."""
    wl = synth.config(8)
    inp = synth.make_inputs(wl, seed=0, device="cuda", with_grad_out=False)
    o, lse = _run(inp, wl, wl.tiles())
    _sampled_check(wl, inp, o, lse, n_random=512, max_heads_long=3)
    o_whole, lse_whole = _run(inp, wl, None)
    cu = wl.cu_seqlens()
    for s in (0, 2, 3):           # key axis not split: identical bits
        a, b = cu[s], cu[s + 1]
        assert torch.equal(o[a:b], o_whole[a:b]) and torch.equal(lse[:, a:b], lse_whole[:, a:b])
    assert (o - o_whole).abs().max().item() <= TOL_O_BF16


def test_sequence_isolation_bitwise():
    """§IV-D keeps sequences separate: changing one sequence's q/k/v leaves
    every other sequence's output bit-identical; outputs stay in input order."""
    wl = synth.Workload("iso", [300, 64, 1000, 129], 4, 128)
    inp = synth.make_inputs(wl, seed=2, device="cuda", with_grad_out=False)
    o1, l1 = _run(inp, wl)
    cu = wl.cu_seqlens()
    inp2 = {k2: t.clone() for k2, t in inp.items()}
    a, b = cu[2], cu[3]
    inp2["k"][a:b] += 1.0
    inp2["v"][a:b] *= -1
    o2, l2 = _run(inp2, wl)
    for s in (0, 1, 3):
        x, y = cu[s], cu[s + 1]
        assert torch.equal(o1[x:y], o2[x:y])
        assert torch.equal(l1[:, x:y], l2[:, x:y])
    assert not torch.equal(o1[a:b], o2[a:b])


@pytest.mark.parametrize("hd,out_dtype", [(64, torch.float32), (128, torch.bfloat16),
                                          (128, torch.float32)])
def test_lse_merge_standalone(hd, out_dtype):
    g = torch.Generator(device="cuda").manual_seed(11)
    P, R, H = 3, 777, 5
    o_part = torch.randn((P, R, H, hd), generator=g, device="cuda")
    lse_part = 4 * torch.randn((P, H, R), generator=g, device="cuda")
    lse_part[1, :, 10:20] = float("-inf")        # an empty partial
    lse_part[:, 2, 30:33] = float("-inf")        # rows with nothing at all
    o, lse = zl.lse_merge(o_part, lse_part, out_dtype=out_dtype)
    zl.sync_check()
    o_ref, l_ref = oracle.lse_merge(f64(o_part), f64(lse_part))
    tol = TOL_O_BF16 if out_dtype == torch.bfloat16 else 1e-5
    assert np.abs(f64(o) - o_ref).max() <= tol
    fin = np.isfinite(l_ref)
    assert np.abs(f64(lse)[fin] - l_ref[fin]).max() <= 1e-5
    assert np.all(np.isneginf(f64(lse)[~fin]))
    assert np.all(f64(o)[30:33, 2] == 0)


def test_launch_counter_and_no_errors():
    wl = synth.config(1)
    inp = synth.make_inputs(wl, seed=0, device="cuda", with_grad_out=False)
    cu = wl.cu_seqlens()
    tiles = synth.grid_tiles(3, 256, 256, 2, 2)
    n0 = zl.launch_count()
    _run(inp, wl, tiles)
    assert zl.launch_count() - n0 == 2     # one attention launch + one merge
    n0 = zl.launch_count()
    zl.varlen_attn_fwd(inp["q"], inp["k"], inp["v"], cu, cu, tiles=tiles, fused_merge=True)
    zl.sync_check()
    assert zl.launch_count() - n0 == 1     # the merge happens inside the attention launch


@pytest.mark.parametrize("n,hd", [(1, 64), (4, 128)])
def test_fused_merge_matches_separate_merge(n, hd):
    """The in-launch (last-arriving tile) merge gives the same result as the
    merge kernel: the same float32 partials combined by the same identity."""
    if n == 1:
        wl = synth.Workload("tiny", [37, 64, 100, 256], 2, hd)
        tiles = synth.grid_tiles(3, 256, 256, 2, 2) + synth.grid_tiles(2, 100, 100, 3, 2)
    else:
        wl = synth.Workload("split", [20000, 1024, 5000], 4, hd)
        tiles = synth.grid_tiles(0, 20000, 20000, 3, 4) + synth.grid_tiles(2, 5000, 5000, 1, 3)
    inp = synth.make_inputs(wl, seed=3, device="cuda", with_grad_out=False)
    cu = wl.cu_seqlens()
    o1, l1 = zl.varlen_attn_fwd(inp["q"], inp["k"], inp["v"], cu, cu, tiles=tiles)
    o2, l2 = zl.varlen_attn_fwd(inp["q"], inp["k"], inp["v"], cu, cu, tiles=tiles, fused_merge=True)
    zl.sync_check()
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-5
    _full_check(inp["q"], inp["k"], inp["v"], cu, cu, o2, l2, TOL_O_BF16, TOL_LSE) if n == 1 else None


def test_concurrent_launches_on_two_streams_bitwise():
    """Two forward launches in flight at once on different streams: their CTAs
    share the SMs, and each launch takes work only from its own queue, so
    both give bit-identical results to the same launches run one after the
    other (every work item done exactly once)."""
    wa = synth.config(2)                                     # 28 sequences, 2,688 items
    wb = synth.Workload("two_streams_b", [20000, 3000, 500, 1024, 1024], 8, 128, splits={0: (2, 2)})

    def prep(wl, seed):
        inp = synth.make_inputs(wl, seed=seed, device="cuda", with_grad_out=False)
        cu = wl.cu_seqlens()
        tiles = wl.tiles() or None
        ws = zl.alloc_workspace(zl.fwd_workspace_bytes(cu, cu, wl.num_heads, wl.head_dim, tiles), "cuda")
        o = torch.empty_like(inp["q"])
        lse = torch.empty((wl.num_heads, wl.total_tokens), device="cuda")
        return inp, cu, tiles, ws, o, lse

    a, b = prep(wa, 3), prep(wb, 4)

    def launch(x, stream):
        inp, cu, tiles, ws, o, lse = x
        zl.varlen_attn_fwd(inp["q"], inp["k"], inp["v"], cu, cu, tiles=tiles, out=o, lse=lse,
                           workspace=ws, stream=stream)

    launch(a, None)
    launch(b, None)
    torch.cuda.synchronize()
    ref = [(x[4].clone(), x[5].clone()) for x in (a, b)]
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        for x in (a, b):
            x[4].zero_()
            x[5].zero_()
        torch.cuda.synchronize()
        launch(a, s1)
        launch(b, s2)
        torch.cuda.synchronize()
        for x, (o_ref, l_ref) in zip((a, b), ref):
            assert torch.equal(x[4], o_ref)
            assert torch.equal(x[5], l_ref)
    zl.sync_check()


@pytest.mark.parametrize("n,hd,fused", [(1, 64, False), (1, 128, True), (4, 128, False), (4, 128, True)])
def test_bf16_partials(n, hd, fused):
    """Partial O rows kept in bf16 (ZL_FWD_BF16_PARTIALS): each partial is
    rounded once before the merge, so O stays within the bf16 tolerance of the
    oracle and of the float32-partial result; partial LSEs stay float32, so
    LSE is bit-identical to the float32-partial run."""
    if n == 1:
        wl = synth.Workload("tiny", [37, 64, 100, 256], 2, hd)
        tiles = synth.grid_tiles(3, 256, 256, 2, 2) + synth.grid_tiles(2, 100, 100, 3, 2)
    else:
        wl = synth.Workload("split", [20000, 1024, 5000], 4, hd)
        tiles = synth.grid_tiles(0, 20000, 20000, 3, 4) + synth.grid_tiles(2, 5000, 5000, 1, 3)
    inp = synth.make_inputs(wl, seed=7, device="cuda", with_grad_out=False)
    cu = wl.cu_seqlens()
    o32, l32 = zl.varlen_attn_fwd(inp["q"], inp["k"], inp["v"], cu, cu, tiles=tiles, fused_merge=fused)
    o16, l16 = zl.varlen_attn_fwd(inp["q"], inp["k"], inp["v"], cu, cu, tiles=tiles, fused_merge=fused,
                                  bf16_partials=True)
    zl.sync_check()
    assert torch.equal(l16, l32)
    assert (o16.float() - o32.float()).abs().max().item() <= TOL_O_BF16
    # sequences that are not split over keys never touch a partial
    assert torch.equal(o16[cu[1]:cu[2]], o32[cu[1]:cu[2]])
    if n == 1:
        _full_check(inp["q"], inp["k"], inp["v"], cu, cu, o16, l16, TOL_O_BF16, TOL_LSE)
    else:
        wl_t = synth.Workload("split", wl.seqlens, wl.num_heads, hd, splits={0: (3, 4), 2: (1, 3)})
        _sampled_check(wl_t, inp, o16, l16, n_random=256, max_heads_long=4)


def test_shard_mode_131k_bf16_partials():
    """The 131,072-token sequence as 4 x 4 tiles beside 64 images, partials in
    bf16: the oracle on sampled rows."""
    wl = synth.config(4)
    inp = synth.make_inputs(wl, seed=0, device="cuda", with_grad_out=False)
    cu = wl.cu_seqlens()
    o, lse = zl.varlen_attn_fwd(inp["q"], inp["k"], inp["v"], cu, cu, tiles=wl.tiles(), bf16_partials=True)
    zl.sync_check()
    _sampled_check(wl, inp, o, lse, n_random=512, max_heads_long=3)


@pytest.mark.parametrize("hd,out_dtype,P", [(64, torch.float32, 3), (128, torch.bfloat16, 4)])
def test_lse_merge_standalone_bf16_partials(hd, out_dtype, P):
    """zl_lse_merge_ex on bf16 partials (3 parts: the any-count path; 4: the
    unrolled one): the oracle's merge of the same bf16 values (widened
    exactly), to float32 rounding."""
    g = torch.Generator(device="cuda").manual_seed(12)
    R, H = 513, 3
    o_part = torch.randn((P, R, H, hd), generator=g, device="cuda").to(torch.bfloat16)
    lse_part = 4 * torch.randn((P, H, R), generator=g, device="cuda")
    lse_part[2, :, 5:9] = float("-inf")
    o, lse = zl.lse_merge(o_part, lse_part, out_dtype=out_dtype)
    zl.sync_check()
    o_ref, l_ref = oracle.lse_merge(f64(o_part), f64(lse_part))
    tol = TOL_O_BF16 if out_dtype == torch.bfloat16 else 1e-5
    assert np.abs(f64(o) - o_ref).max() <= tol
    assert np.abs(f64(lse) - l_ref).max() <= 1e-5

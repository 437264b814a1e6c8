"""Pins for the float64 oracle: facts fixed by the mathematics of softmax
attention and by the Zellige paper's description of the coalesced engine
(arXiv 2608.01150v1, §IV-D: block-diagonal, sequences kept separate, outputs in
input order; §II-B: exact attention from block-wise K/V partials).

None of these retypes the oracle's own formula: each compares it with a closed
form, an invariant, a brute-force loop in plain Python, or a library routine.
The mutation test at the end plants one plausible mistake at a time in the
oracle's steps and checks that at least one pin fails.
"""
import math
import os
import random

import numpy as np
import pytest
import scipy.special

import oracle
import oracle.attn_f64 as of
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=0):
    return np.random.default_rng(seed)


def _packed(seqlens, nh, d, seed=0, dv=None):
    r = _rng(seed)
    t = sum(seqlens)
    q = r.standard_normal((t, nh, d))
    k = r.standard_normal((t, nh, d))
    v = r.standard_normal((t, nh, dv or d))
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int64)
    return q, k, v, cu


# ----------------------------------------------------------------------------
# Pins (each a plain function so the mutation test can rerun them).
# ----------------------------------------------------------------------------

def pin_length_one():
    """A sequence of one token attends only to itself: O = v, LSE = q.k*scale."""
    q, k, v, cu = _packed([1, 5, 1], 3, 8, seed=1)
    scale = 0.37
    o, lse = oracle.varlen_attn_fwd(q, k, v, cu, cu, scale)
    for t in (0, 6):
        for h in range(3):
            assert np.allclose(o[t, h], v[t, h], rtol=0, atol=1e-14)
            assert abs(lse[h, t] - scale * float(q[t, h] @ k[t, h])) < 1e-13


def pin_constant_keys():
    """All keys equal: uniform weights, O = mean of V rows, LSE = q.k*scale + ln L,
    and dQ = 0 (the scores do not depend on which key)."""
    L, d = 9, 6
    r = _rng(2)
    q = r.standard_normal((L, 1, d))
    krow = r.standard_normal(d)
    k = np.tile(krow, (L, 1))[:, None, :]
    v = r.standard_normal((L, 1, d))
    do = r.standard_normal((L, 1, d))
    cu = np.array([0, L])
    scale = 1 / math.sqrt(d)
    o, lse = oracle.varlen_attn_fwd(q, k, v, cu, cu, scale)
    assert np.allclose(o[:, 0], v[:, 0].mean(axis=0)[None], atol=1e-14)
    assert np.allclose(lse[0], scale * (q[:, 0] @ krow) + math.log(L), atol=1e-13)
    dq, dk, dv = oracle.varlen_attn_bwd(q, k, v, do, cu, cu, scale)
    assert np.abs(dq).max() < 1e-13
    # dV_j = sum_i P_ij dO_i = mean of dO rows for every j
    assert np.allclose(dv[:, 0], np.tile(do[:, 0].sum(axis=0) / L, (L, 1)), atol=1e-13)


def pin_identical_values():
    """All value rows equal: O is that row whatever the weights, and the
    gradients through the scores vanish: dS = 0, so dQ = dK = 0."""
    L, d = 7, 5
    r = _rng(3)
    q = r.standard_normal((L, 2, d))
    k = r.standard_normal((L, 2, d))
    vrow = r.standard_normal((2, d))
    v = np.tile(vrow[None], (L, 1, 1))
    do = r.standard_normal((L, 2, d))
    cu = np.array([0, L])
    o, _ = oracle.varlen_attn_fwd(q, k, v, cu, cu)
    assert np.allclose(o, np.tile(vrow[None], (L, 1, 1)), atol=1e-14)
    dq, dk, _ = oracle.varlen_attn_bwd(q, k, v, do, cu, cu)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13


def pin_two_keys_closed_form():
    """L = 2: O = sigma(delta) v1 + (1 - sigma(delta)) v2 with
    delta = (q.k1 - q.k2) * scale, LSE = log(e^a + e^b)."""
    r = _rng(4)
    d = 4
    q = r.standard_normal((2, 1, d))
    k = r.standard_normal((2, 1, d))
    v = r.standard_normal((2, 1, d))
    cu = np.array([0, 2])
    scale = 0.8
    o, lse = oracle.varlen_attn_fwd(q, k, v, cu, cu, scale)
    for i in range(2):
        a = scale * float(q[i, 0] @ k[0, 0])
        b = scale * float(q[i, 0] @ k[1, 0])
        sig = 1.0 / (1.0 + math.exp(-(a - b)))
        assert np.allclose(o[i, 0], sig * v[0, 0] + (1 - sig) * v[1, 0], atol=1e-14)
        assert abs(lse[0, i] - math.log(math.exp(a) + math.exp(b))) < 1e-13


def _brute_force(q, k, v, cu_q, cu_k, scale):
    """Scalar loops with math.exp, explicit normalisation, no max shift."""
    tq, nh, d = q.shape
    dv = v.shape[2]
    o = [[[0.0] * dv for _ in range(nh)] for _ in range(tq)]
    lse = [[float("-inf")] * tq for _ in range(nh)]
    for s in range(len(cu_q) - 1):
        for h in range(nh):
            for i in range(int(cu_q[s]), int(cu_q[s + 1])):
                w = []
                for j in range(int(cu_k[s]), int(cu_k[s + 1])):
                    dot = 0.0
                    for c in range(d):
                        dot += float(q[i, h, c]) * float(k[j, h, c])
                    w.append((j, math.exp(dot * scale)))
                z = sum(x for _, x in w)
                if not w:
                    continue
                lse[h][i] = math.log(z)
                for c in range(dv):
                    o[i][h][c] = sum(x * float(v[j, h, c]) for j, x in w) / z
    return np.array(o), np.array(lse)


def pin_brute_force_tiny():
    """Oracle == scalar brute force on tiny packed batches, including different
    query and key lengths per sequence and an empty sequence."""
    for seed, lq, lk, nh, d in [(5, [3, 1, 4], [3, 1, 4], 2, 4),
                                (6, [2, 0, 5], [4, 0, 3], 1, 3),
                                (7, [6], [6], 3, 2)]:
        r = _rng(seed)
        q = r.standard_normal((sum(lq), nh, d))
        k = r.standard_normal((sum(lk), nh, d))
        v = r.standard_normal((sum(lk), nh, d + 1))
        cu_q = np.concatenate([[0], np.cumsum(lq)])
        cu_k = np.concatenate([[0], np.cumsum(lk)])
        scale = 0.61
        o, lse = oracle.varlen_attn_fwd(q, k, v, cu_q, cu_k, scale)
        ob, lb = _brute_force(q, k, v, cu_q, cu_k, scale)
        assert np.allclose(o, ob, atol=1e-13, rtol=0)
        assert np.allclose(lse, lb, atol=1e-13, rtol=0)


def pin_scipy_softmax():
    """Each output row is scipy's softmax of the scaled scores times V, and
    LSE is scipy's logsumexp."""
    q, k, v, cu = _packed([50, 17], 2, 16, seed=8)
    scale = 0.25
    o, lse = oracle.varlen_attn_fwd(q, k, v, cu, cu, scale)
    for s in range(2):
        a, b = cu[s], cu[s + 1]
        for h in range(2):
            logits = scale * np.einsum("id,jd->ij", q[a:b, h], k[a:b, h])
            p = scipy.special.softmax(logits, axis=1)
            assert np.allclose(o[a:b, h], p @ v[a:b, h], atol=1e-13)
            assert np.allclose(lse[h, a:b], scipy.special.logsumexp(logits, axis=1), atol=1e-13)


def pin_merge_equals_unsplit():
    """Merging the (partial O, LSE) pairs of every tile of a full
    (query-chunk x KV-chunk) grid reproduces unsplit attention (fp64, 1e-12)."""
    for L, nq, nk in [(37, 2, 2), (100, 3, 1), (100, 1, 3), (64, 4, 4), (257, 2, 3)]:
        q, k, v, cu = _packed([L], 2, 8, seed=L + nq)
        o_ref, lse_ref = oracle.varlen_attn_fwd(q, k, v, cu, cu)
        tiles = synth.grid_tiles(0, L, L, nq, nk)
        o = np.zeros_like(o_ref)
        lse = np.zeros_like(lse_ref)
        for i, (qa, ql) in enumerate(synth.chunk_bounds(L, nq)):
            parts = [oracle.tile_partial(q, k, v, cu, cu, t) for t in tiles if t[5] == i]
            om, lm = oracle.lse_merge(np.stack([p[0] for p in parts]),
                                      np.stack([p[1] for p in parts]))
            o[qa:qa + ql] = om
            lse[:, qa:qa + ql] = lm
        assert np.abs(o - o_ref).max() < 1e-12
        assert np.abs(lse - lse_ref).max() < 1e-12


def pin_head_sharded_configurations():
    """Every composed configuration (q, h, k) of the Zellige paper (§IV-A,
    Table II: query split, head split, key split) reproduces unsplit attention
    of the split sequences, whole sequences beside them untouched (fp64)."""
    lens = [37, 100, 64]
    for cfg in [(1, 2, 1), (2, 2, 2), (1, 3, 2), (3, 1, 1), (1, 1, 3), (2, 3, 1), (1, 5, 1)]:
        nq, nk, nh = cfg[0], cfg[2], cfg[1]
        q, k, v, cu = _packed(lens, 5, 8, seed=11 + nq + 3 * nh + 7 * nk)
        o_ref, lse_ref = oracle.varlen_attn_fwd(q, k, v, cu, cu)
        tiles = (synth.grid_tiles(0, 37, 37, nq, nk, nh, 5) +
                 synth.grid_tiles(1, 100, 100, nq, nk, nh, 5))
        covered = sorted((t[0], h) for t in tiles if t[5] == 0 and t[6] == 0
                         for h in oracle.tile_heads(t, 5))
        assert covered == [(s, h) for s in (0, 1) for h in range(5)]
        o, lse = oracle.tiled_attn_fwd(q, k, v, cu, cu, tiles)
        assert np.abs(o - o_ref).max() < 1e-12, cfg
        assert np.abs(lse - lse_ref).max() < 1e-12, cfg
    # a zero-length head range means every head
    assert oracle.tile_heads((0, 0, 1, 0, 1, 0, 0, 1, 0, 0, 0), 3) == [0, 1, 2]
    assert oracle.tile_heads((0, 0, 1, 0, 1, 0, 0, 1), 3) == [0, 1, 2]


def pin_merge_empty_parts():
    """An empty partial (LSE = -inf) contributes nothing; all-empty stays empty."""
    r = _rng(9)
    o1 = r.standard_normal((3, 2, 4))
    l1 = r.standard_normal((2, 3))
    o_parts = np.stack([o1, np.zeros_like(o1)])
    l_parts = np.stack([l1, np.full_like(l1, -np.inf)])
    o, lse = oracle.lse_merge(o_parts, l_parts)
    assert np.allclose(o, o1, atol=1e-15) and np.allclose(lse, l1, atol=1e-15)
    o, lse = oracle.lse_merge(np.zeros((2, 3, 2, 4)), np.full((2, 2, 3), -np.inf))
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    # two equal halves: lse grows by ln 2, O is their common value
    o, lse = oracle.lse_merge(np.stack([o1, o1]), np.stack([l1, l1]))
    assert np.allclose(o, o1, atol=1e-14) and np.allclose(lse, l1 + math.log(2), atol=1e-14)


def pin_finite_differences():
    """Central differences of the scalar loss sum(dO * O) match the analytic
    gradients on tiny inputs."""
    for seed, lens, d in [(10, [5, 3], 4), (11, [8], 8), (12, [2, 6], 3)]:
        q, k, v, cu = _packed(lens, 2, d, seed=seed)
        do = _rng(seed + 100).standard_normal(q.shape)
        scale = 1.3 / math.sqrt(d)

        def loss(qq, kk, vv):
            o, _ = oracle.varlen_attn_fwd(qq, kk, vv, cu, cu, scale)
            return float((o * do).sum())

        dq, dk, dv = oracle.varlen_attn_bwd(q, k, v, do, cu, cu, scale)
        eps = 1e-6
        for which, x, g in ((0, q, dq), (1, k, dk), (2, v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(*x.shape):
                xp = x.copy()
                xm = x.copy()
                xp[idx] += eps
                xm[idx] -= eps
                args_p = [q, k, v]
                args_m = [q, k, v]
                args_p[which] = xp
                args_m[which] = xm
                num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            rel = np.linalg.norm(num - g) / max(np.linalg.norm(g), 1e-30)
            assert rel < 1e-7, (which, rel)


def pin_gradient_sums():
    """Softmax is shift-invariant, so dK sums to zero over the keys of each
    sequence and head; rows of P sum to one, so dV sums to the sum of dO."""
    q, k, v, cu = _packed([13, 40, 7], 3, 8, seed=13)
    do = _rng(14).standard_normal(q.shape)
    dq, dk, dv = oracle.varlen_attn_bwd(q, k, v, do, cu, cu)
    for s in range(3):
        a, b = cu[s], cu[s + 1]
        assert np.abs(dk[a:b].sum(axis=0)).max() < 1e-12
        assert np.allclose(dv[a:b].sum(axis=0), do[a:b].sum(axis=0), atol=1e-12)


def pin_sequence_isolation_and_order():
    """§IV-D: sequences are kept separate and outputs come back in input order.
    Perturbing one sequence leaves the others bit-identical, and permuting the
    packing order permutes the outputs."""
    lens = [11, 30, 5]
    q, k, v, cu = _packed(lens, 2, 8, seed=15)
    o, lse = oracle.varlen_attn_fwd(q, k, v, cu, cu)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    a, b = cu[1], cu[2]
    k2[a:b] += 3.0
    v2[a:b] *= -2.0
    q2[a:b] += 1.0
    o2, lse2 = oracle.varlen_attn_fwd(q2, k2, v2, cu, cu)
    for s in (0, 2):
        sa, sb = cu[s], cu[s + 1]
        assert np.array_equal(o[sa:sb], o2[sa:sb])
        assert np.array_equal(lse[:, sa:sb], lse2[:, sa:sb])
    assert not np.allclose(o[a:b], o2[a:b])
    perm = [2, 0, 1]
    idx = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in perm])
    cu_p = np.concatenate([[0], np.cumsum([lens[s] for s in perm])])
    op, lp = oracle.varlen_attn_fwd(q[idx], k[idx], v[idx], cu_p, cu_p)
    assert np.allclose(op, o[idx], atol=1e-15)
    assert np.allclose(lp, lse[:, idx], atol=1e-15)


def pin_row_helpers():
    """Row-sampled helpers return exactly the rows of the full call."""
    q, k, v, cu = _packed([20, 2500], 2, 8, seed=16)
    do = _rng(17).standard_normal(q.shape)
    o, lse = oracle.varlen_attn_fwd(q, k, v, cu, cu)
    dq, _, _ = oracle.varlen_attn_bwd(q, k, v, do, cu, cu)
    rows = [0, 1, 1023, 1024, 2047, 2048, 2499]
    orow, lrow = oracle.attention_rows(q, k, v, cu, cu, 1, 1, rows)
    assert np.allclose(orow, o[20 + np.array(rows), 1], atol=1e-14)
    assert np.allclose(lrow, lse[1, 20 + np.array(rows)], atol=1e-13)
    dqr = oracle.dq_rows(q, k, v, do, cu, cu, 1, 0, rows)
    assert np.allclose(dqr, dq[20 + np.array(rows), 0], atol=1e-13)
    _, dk, dv = oracle.varlen_attn_bwd(q, k, v, do, cu, cu)
    dkr, dvr = oracle.dkdv_rows(q, k, v, do, cu, cu, 1, 1, rows)
    assert np.allclose(dkr, dk[20 + np.array(rows), 1], atol=1e-12)
    assert np.allclose(dvr, dv[20 + np.array(rows), 1], atol=1e-12)


def pin_one_query_row():
    """With dO zero except at one query row, the full backward (itself pinned
    by finite differences) gives exactly the one-row gradients: dK and dV of
    every key of that sequence and head, dQ of that row, and zero dQ on every
    other row."""
    q, k, v, cu = _packed([9, 300, 17], 3, 8, seed=18)
    do_full = _rng(19).standard_normal(q.shape)
    for s, h, r in ((1, 2, 0), (1, 0, 173), (2, 1, 16), (0, 1, 4)):
        a, b = cu[s], cu[s + 1]
        do = np.zeros_like(do_full)
        do[a + r, h] = do_full[a + r, h]
        dq, dk, dv = oracle.varlen_attn_bwd(q, k, v, do, cu, cu)
        dq_r, dk_s, dv_s = oracle.grads_one_query_row(q, k, v, do[a + r, h], cu, cu, s, h, r)
        assert np.allclose(dq[a + r, h], dq_r, atol=1e-13)
        assert np.allclose(dk[a:b, h], dk_s, atol=1e-13)
        assert np.allclose(dv[a:b, h], dv_s, atol=1e-13)
        mask = np.ones(q.shape[0], dtype=bool)
        mask[a + r] = False
        assert np.all(dq[mask, h] == 0) and np.all(dq[:, [x for x in range(3) if x != h]] == 0)


def pin_default_scale():
    """Without an explicit scale every oracle entry divides the scores by
    sqrt(d): the printed numbers 1/2 at d = 4, 1/8 at d = 64 (the tiny batch's
    stated 1/sqrt(64)); a length-1 sequence's LSE is then q.k / 8, summed by a
    plain loop; and each entry called with no scale returns exactly what it
    returns with scale 1/8 passed explicitly."""
    assert of.default_scale(4) == 0.5
    assert of.default_scale(64) == 0.125
    assert of.default_scale(16) == 0.25
    assert abs(of.default_scale(128) * of.default_scale(128) * 128 - 1.0) < 1e-15
    q, k, v, cu = _packed([1, 3, 2], 2, 64, seed=12)
    do = _rng(13).standard_normal(q.shape)
    o, lse = oracle.varlen_attn_fwd(q, k, v, cu, cu)
    for h in range(2):
        dot = 0.0
        for i in range(64):
            dot += float(q[0, h, i]) * float(k[0, h, i])
        assert abs(lse[h, 0] - dot / 8.0) < 1e-12
    o8, lse8 = oracle.varlen_attn_fwd(q, k, v, cu, cu, 0.125)
    assert np.array_equal(o, o8) and np.array_equal(lse, lse8)
    g = oracle.varlen_attn_bwd(q, k, v, do, cu, cu)
    g8 = oracle.varlen_attn_bwd(q, k, v, do, cu, cu, 0.125)
    assert all(np.array_equal(a, b) for a, b in zip(g, g8))
    tiles = [(1, 0, 3, 0, 2, 0, 0, 2), (1, 0, 3, 2, 1, 0, 1, 2)]
    for a, b in zip(oracle.tiled_attn_fwd(q, k, v, cu, cu, tiles),
                    oracle.tiled_attn_fwd(q, k, v, cu, cu, tiles, 0.125)):
        assert np.array_equal(a, b)
    for a, b in zip(oracle.tile_partial(q, k, v, cu, cu, tiles[0]),
                    oracle.tile_partial(q, k, v, cu, cu, tiles[0], 0.125)):
        assert np.array_equal(a, b)
    for a, b in zip(oracle.attention_rows(q, k, v, cu, cu, 1, 0, [0, 2]),
                    oracle.attention_rows(q, k, v, cu, cu, 1, 0, [0, 2], 0.125)):
        assert np.array_equal(a, b)
    assert np.array_equal(oracle.dq_rows(q, k, v, do, cu, cu, 2, 1, [1]),
                          oracle.dq_rows(q, k, v, do, cu, cu, 2, 1, [1], 0.125))
    for a, b in zip(oracle.dkdv_rows(q, k, v, do, cu, cu, 1, 1, [0, 2]),
                    oracle.dkdv_rows(q, k, v, do, cu, cu, 1, 1, [0, 2], 0.125)):
        assert np.array_equal(a, b)
    for a, b in zip(oracle.grads_one_query_row(q, k, v, do[1, 0], cu, cu, 1, 0, 0),
                    oracle.grads_one_query_row(q, k, v, do[1, 0], cu, cu, 1, 0, 0, 0.125)):
        assert np.array_equal(a, b)


PINS = [pin_length_one, pin_constant_keys, pin_identical_values,
        pin_two_keys_closed_form, pin_brute_force_tiny, pin_scipy_softmax,
        pin_merge_equals_unsplit, pin_head_sharded_configurations, pin_merge_empty_parts,
        pin_finite_differences,
        pin_gradient_sums, pin_sequence_isolation_and_order, pin_row_helpers, pin_one_query_row,
        pin_default_scale]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ----------------------------------------------------------------------------
# Golden values printed by the paper: the latent-token formula of the workloads.
# ----------------------------------------------------------------------------

def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kind, *kv = line.split()
            rows.append((kind, {a: int(b) for a, b in (x.split("=") for x in kv)}))
    return rows


def test_golden_wan_token_counts():
    rows = _read_golden("wan_token_counts.txt")
    assert rows, "fixture is empty"
    for kind, f in rows:
        if kind == "video":
            assert synth.video_tokens(f["frames"], f["height"], f["width"]) == f["tokens"]
        elif kind == "ratio":
            r = (synth.video_tokens(f["video_frames"], f["video_height"], f["video_width"]) /
                 synth.image_tokens(f["image_height"], f["image_width"]))
            assert round(r) == f["rounded"]
        else:
            raise AssertionError(kind)


def test_workload_shapes():
    """Token totals of the batches (their descriptions list the per-video
    latent sizes, e.g. 21 x 30 x 52 = 32,760 for a 480p 81-frame video)."""
    assert synth.video_tokens(81, 480, 832) == 21 * 30 * 52
    assert synth.video_tokens(33, 480, 832) == 9 * 30 * 52
    assert synth.video_tokens(81, 720, 1280) == 21 * 45 * 80
    totals = {1: 457, 2: 28672, 3: 118184, 4: 196608, 5: 190272}
    for n, t in totals.items():
        assert synth.config(n).total_tokens == t
    # Fig. 2 of the paper: three 720p 10 s videos (41 x 45 x 80) and 228 720p images (45 x 80)
    wl7 = synth.config(7)
    assert wl7.seqlens[:3] == [41 * 45 * 80] * 3 and wl7.seqlens[3:] == [45 * 80] * 228
    assert wl7.num_heads == 12 and len(wl7.tiles()) == 12
    assert len(synth.config(4).tiles()) == 16
    assert len(synth.config(5).tiles()) == 4
    wl8 = synth.config(8)
    assert wl8.total_tokens == 75600 + 2 * 32760 + 24 * 1024
    assert len(wl8.tiles()) == 4 + 8 + 10
    wl9 = synth.config(9)
    assert wl9.seqlens == synth.config(6).seqlens and len(wl9.tiles()) == 4
    for n in (4, 5, 7, 8, 9):
        wl = synth.config(n)
        for s in wl.splits:
            ts = [t for t in wl.tiles() if t[0] == s]
            covered = sum(t[2] * t[4] * (t[9] or wl.num_heads) for t in ts)
            assert covered == wl.seqlens[s] ** 2 * wl.num_heads


def test_inputs_seeded():
    wl = synth.config(1)
    a = synth.make_inputs(wl, seed=3)
    b = synth.make_inputs(wl, seed=3)
    c = synth.make_inputs(wl, seed=4)
    for key in a:
        assert a[key].shape == (457, 2, 64)
        assert bool((a[key] == b[key]).all())
        assert not bool((a[key] == c[key]).all())


# ----------------------------------------------------------------------------
# Planted mistakes: each must be caught by at least one pin.
# ----------------------------------------------------------------------------

def _mut_no_scale(q_rows, k, scale):
    return q_rows @ k.T


def _mut_inverse_scale(q_rows, k, scale):
    return (q_rows @ k.T) / scale


def _mut_scores_use_first_dims(q_rows, k, scale):
    return (q_rows[:, :-1] @ k[:, :-1].T) * scale


def _mut_lse_drop_max(s):
    m = s.max(axis=1)
    return np.log(np.exp(s - m[:, None]).sum(axis=1))


def _mut_lse_log2(s):
    m = s.max(axis=1)
    return m + np.log2(np.exp(s - m[:, None]).sum(axis=1))


def _mut_prob_unnormalised(s, lse):
    return np.exp(s)


def _mut_prob_column_norm(s, lse):
    e = np.exp(s - s.max())
    return e / e.sum(axis=0, keepdims=True)


def _mut_merge_max_only(o_parts, lse_parts):
    j = lse_parts.argmax(axis=0)
    lse = lse_parts.max(axis=0)
    o = np.take_along_axis(o_parts, j.T[None, :, :, None], axis=0)[0]
    return o, lse


def _mut_merge_unweighted(o_parts, lse_parts):
    o, lse = _REAL["lse_merge"](o_parts, lse_parts)
    return o_parts.mean(axis=0), lse


def _mut_grad_scores_no_d(p, dp, dsum):
    return p * dp


def _mut_grad_scores_sign(p, dp, dsum):
    return p * (dsum[:, None] - dp)


def _mut_grad_q_no_scale(ds, k, scale):
    return ds @ k


def _mut_grad_k_no_transpose(ds, q_rows, scale):
    # uses dS itself instead of dS^T where shapes allow; otherwise zero
    if ds.shape[0] == ds.shape[1]:
        return scale * (ds @ q_rows)
    return np.zeros((ds.shape[1], q_rows.shape[1]))


def _mut_grad_v_wrong_side(p, do_rows):
    if p.shape[0] == p.shape[1]:
        return p @ do_rows
    return np.zeros((p.shape[1], do_rows.shape[1]))


def _mut_tile_heads_from_zero(tile, num_heads):
    # drops the head offset: every head chunk reads heads 0 .. h_len-1
    if len(tile) > 9 and int(tile[9]) > 0:
        return list(range(int(tile[9])))
    return list(range(num_heads))


def _mut_one_row_no_d(q, k, v, do_row, cu_q, cu_k, seq, head, row, scale=None):
    # the one-row gradients with the D = dO . O term of dS dropped
    d = q.shape[2]
    scale = of.default_scale(d) if scale is None else scale
    qa = int(cu_q[seq])
    ka, kb = int(cu_k[seq]), int(cu_k[seq + 1])
    qr = q[qa + row:qa + row + 1, head]
    dor = np.asarray(do_row, dtype=np.float64)[None, :]
    kk, vv = k[ka:kb, head], v[ka:kb, head]
    _, lse_r = of.attention_f64(qr, kk, vv, scale)
    p = of.probabilities(of.scores(qr, kk, scale), lse_r)
    ds = p * (dor @ vv.T)
    return scale * (ds @ kk)[0], scale * (ds.T @ qr), p.T @ dor


def _mut_default_scale_inverse_d(head_dim):
    return 1.0 / head_dim


def _mut_default_scale_sqrt(head_dim):
    return math.sqrt(head_dim)


_REAL = {name: getattr(of, name) for name in
         ("scores", "row_logsumexp", "probabilities", "lse_merge", "grad_scores",
          "grad_q", "grad_k", "grad_v", "tile_heads", "grads_one_query_row")}

MUTATIONS = [
    ("scores", _mut_no_scale), ("scores", _mut_inverse_scale),
    ("scores", _mut_scores_use_first_dims),
    ("row_logsumexp", _mut_lse_drop_max), ("row_logsumexp", _mut_lse_log2),
    ("probabilities", _mut_prob_unnormalised), ("probabilities", _mut_prob_column_norm),
    ("lse_merge", _mut_merge_max_only), ("lse_merge", _mut_merge_unweighted),
    ("grad_scores", _mut_grad_scores_no_d), ("grad_scores", _mut_grad_scores_sign),
    ("grad_q", _mut_grad_q_no_scale), ("grad_k", _mut_grad_k_no_transpose),
    ("grad_v", _mut_grad_v_wrong_side), ("tile_heads", _mut_tile_heads_from_zero),
    ("grads_one_query_row", _mut_one_row_no_d),
    ("default_scale", _mut_default_scale_inverse_d), ("default_scale", _mut_default_scale_sqrt),
]


@pytest.mark.parametrize("target,mutant", MUTATIONS,
                         ids=[f"{t}:{m.__name__}" for t, m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, target, mutant):
    monkeypatch.setattr(of, target, mutant)
    monkeypatch.setattr(oracle, target, mutant, raising=False)
    caught = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except (AssertionError, ValueError, FloatingPointError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {mutant.__name__} in {target}"


def test_pins_pass_unmutated():
    random.seed(0)
    for pin in PINS:
        pin()

"""Float64 CPU oracle for coalesced varlen attention.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
and the benchmark's CPU-baseline leg may import or run anything in this
package.  The CUDA library never calls it and it never calls the CUDA library;
the two share no code.

What it computes (Zellige, "Moldable Sequence Placement for Mixed Image-Video
DiT Training", arXiv 2608.01150v1):

* §II-A: a DiT block runs dense self-attention over all L^2 token pairs of a
  sequence.  Bidirectional, no mask.
* §IV-D, Coalesced Attention Engine: the whole sequences of a rank are packed
  into one block-diagonal attention call that keeps the sequences separate
  (no attention across sequences) and returns outputs in input order.
* §II-B / Table II (ring attention, all-gather): a split sequence is computed
  block-wise from K/V chunks and the per-block results are accumulated into
  exact attention.  The pages print no merge formula; the exact combination of
  (partial O, log-sum-exp) pairs is the plain identity of the softmax:
  lse = log sum_j exp(lse_j),  O = sum_j exp(lse_j - lse) O_j.
* §IV-A / Table II: a split sequence takes a configuration (q, h, k) that cuts
  its queries (all-gather), its heads (Ulysses) and its keys (ring).  Heads are
  independent, and a query chunk with all of its keys is final; only the key
  axis needs the merge above.
* Backward: the analytic gradient of softmax(Q K^T * scale) V.  The pages do not
  print it (they train with exact backward, §V-A); it is plain calculus.

Every step is the definition written out in float64: scores, a row-wise
log-sum-exp over the FULL key row (not an online softmax), probabilities, and
two matrix products.  Rows are processed in blocks of at most ROW_BLOCK query
rows only to bound memory; each block sees all of its keys, so blocking does not
change the result.

Readings taken where the pages are silent: scale = 1/sqrt(d) unless given;
LSE is the natural log of sum(exp(scaled score)); an empty key set gives
O = 0 and LSE = -inf.

Layouts (all float64 numpy arrays):
  q            [Tq, H, d]     packed query tokens
  k, v         [Tk, H, d]     packed key/value tokens
  cu_q, cu_k   [B+1] int      prefix sums of per-sequence lengths, cu[0] = 0
  o            [Tq, H, d]
  lse          [H, Tq]        head-major
  tile         (seq, q_start, q_len, k_start, k_len, q_chunk, kv_chunk,
               n_kv_chunks[, h_start, h_len, h_chunk])  offsets relative to
               the sequence's own query / key ranges; heads absolute, a
               missing or zero-length head range meaning all heads
"""
from __future__ import annotations

import math

import numpy as np

ROW_BLOCK = 1024


# --------------------------------------------------------------------------
# Steps of one head of one (sequence or tile).  Kept as separate functions so
# that each can be checked, and so that tests can plant a mistake in exactly
# one step and show that some pin catches it.
# --------------------------------------------------------------------------

def scores(q_rows: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """S = Q K^T * scale   (§II-A: every query row against every key row)."""
    return (q_rows @ k.T) * scale


def row_logsumexp(s: np.ndarray) -> np.ndarray:
    """Natural-log log-sum-exp of each row of S, with the row max taken out
    first so that exp never overflows."""
    m = s.max(axis=1)
    return m + np.log(np.exp(s - m[:, None]).sum(axis=1))


def probabilities(s: np.ndarray, lse: np.ndarray) -> np.ndarray:
    """P = exp(S - LSE): each row sums to one."""
    return np.exp(s - lse[:, None])


def attention_f64(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float):
    """softmax(Q K^T * scale) V for one head of one sequence or tile.

    q [Lq, d], k [Lk, d], v [Lk, dv]  ->  o [Lq, dv], lse [Lq].
    With Lk == 0 the softmax is empty: o = 0 and lse = -inf.
    """
    lq, lk = q.shape[0], k.shape[0]
    o = np.zeros((lq, v.shape[1]), dtype=np.float64)
    lse = np.full(lq, -np.inf, dtype=np.float64)
    if lq == 0 or lk == 0:
        return o, lse
    for r0 in range(0, lq, ROW_BLOCK):
        r1 = min(lq, r0 + ROW_BLOCK)
        s = scores(q[r0:r1], k, scale)
        l_blk = row_logsumexp(s)
        o[r0:r1] = probabilities(s, l_blk) @ v
        lse[r0:r1] = l_blk
    return o, lse


def default_scale(head_dim: int) -> float:
    """The softmax scale used when none is given: 1/sqrt(d).  The pages print
    no scale; this is the usual scaled dot-product attention, and the tiny
    correctness batch of the workloads states 1/sqrt(64) at head_dim 64."""
    return 1.0 / math.sqrt(head_dim)


# --------------------------------------------------------------------------
# Packed (block-diagonal) forward: §IV-D, one call over all sequences, each
# sequence attends only to itself, outputs in input order.
# --------------------------------------------------------------------------

def varlen_attn_fwd(q, k, v, cu_q, cu_k, scale=None, heads=None):
    """Exact attention of every packed sequence.  Returns o [Tq,H,d], lse [H,Tq].

    `heads` restricts the work to a subset of heads (the others are left at
    o = 0, lse = -inf); used to keep large cases within seconds.
    """
    tq, nh, d = q.shape
    if scale is None:
        scale = default_scale(d)
    o = np.zeros((tq, nh, v.shape[2]), dtype=np.float64)
    lse = np.full((nh, tq), -np.inf, dtype=np.float64)
    hs = range(nh) if heads is None else heads
    for s in range(len(cu_q) - 1):
        qa, qb = int(cu_q[s]), int(cu_q[s + 1])
        ka, kb = int(cu_k[s]), int(cu_k[s + 1])
        for h in hs:
            o_sh, l_sh = attention_f64(q[qa:qb, h], k[ka:kb, h], v[ka:kb, h], scale)
            o[qa:qb, h] = o_sh
            lse[h, qa:qb] = l_sh
    return o, lse


def attention_rows(q, k, v, cu_q, cu_k, seq, head, rows, scale=None):
    """Exact output of selected query rows (relative to sequence `seq`) of one
    head.  Rows are independent, so this is the same value the full call gives
    for them.  Returns o [len(rows), d], lse [len(rows)]."""
    d = q.shape[2]
    if scale is None:
        scale = default_scale(d)
    qa = int(cu_q[seq])
    ka, kb = int(cu_k[seq]), int(cu_k[seq + 1])
    rows = np.asarray(rows, dtype=np.int64)
    return attention_f64(q[qa + rows, head], k[ka:kb, head], v[ka:kb, head], scale)


# --------------------------------------------------------------------------
# Shard tiles and the exact merge (§II-B ring / all-gather accumulation,
# Table II; §IV-D runs such shards alongside whole sequences).
# --------------------------------------------------------------------------

def tile_heads(tile, num_heads: int):
    """The heads a tile covers: [h_start, h_start + h_len), or all of them
    when the tile has no head range or h_len = 0."""
    if len(tile) > 9 and int(tile[9]) > 0:
        return list(range(int(tile[8]), int(tile[8]) + int(tile[9])))
    return list(range(num_heads))


def tile_partial(q, k, v, cu_q, cu_k, tile, scale=None):
    """Attention of one (query-chunk x head-range x KV-chunk) tile of a split
    sequence, restricted to that tile's keys and heads.  Returns the partial
    o [q_len, h, d] and its own log-sum-exp [h, q_len] for the tile's h heads
    (tile_heads order)."""
    seq, q_start, q_len, k_start, k_len = (int(x) for x in tile[:5])
    d = q.shape[2]
    if scale is None:
        scale = default_scale(d)
    qa = int(cu_q[seq]) + q_start
    ka = int(cu_k[seq]) + k_start
    heads = tile_heads(tile, q.shape[1])
    o = np.zeros((q_len, len(heads), v.shape[2]), dtype=np.float64)
    lse = np.full((len(heads), q_len), -np.inf, dtype=np.float64)
    for i, h in enumerate(heads):
        o_h, l_h = attention_f64(q[qa:qa + q_len, h], k[ka:ka + k_len, h],
                                 v[ka:ka + k_len, h], scale)
        o[:, i] = o_h
        lse[i] = l_h
    return o, lse


def tiled_attn_fwd(q, k, v, cu_q, cu_k, tiles, scale=None):
    """The packed forward with some sequences split by a tile table: whole
    sequences as varlen_attn_fwd; for a split sequence every (head range,
    query range) takes the partials of its KV chunks and combines them with
    lse_merge (one chunk passes through).  Returns o [Tq,H,d], lse [H,Tq]."""
    tq, nh, d = q.shape
    if scale is None:
        scale = default_scale(d)
    split = sorted({int(t[0]) for t in tiles})
    whole = [s for s in range(len(cu_q) - 1) if s not in split]
    o = np.zeros((tq, nh, v.shape[2]), dtype=np.float64)
    lse = np.full((nh, tq), -np.inf, dtype=np.float64)
    for s in whole:
        qa, qb = int(cu_q[s]), int(cu_q[s + 1])
        ka, kb = int(cu_k[s]), int(cu_k[s + 1])
        for h in range(nh):
            o[qa:qb, h], lse[h, qa:qb] = attention_f64(q[qa:qb, h], k[ka:kb, h], v[ka:kb, h], scale)
    groups = {}
    for t in tiles:
        key = (int(t[0]), int(t[1]), int(t[2]), tuple(tile_heads(t, nh)))
        groups.setdefault(key, []).append(t)
    for (s, q_start, q_len, heads), ts in groups.items():
        parts = [tile_partial(q, k, v, cu_q, cu_k, t, scale) for t in ts]
        om, lm = lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        r0 = int(cu_q[s]) + q_start
        for i, h in enumerate(heads):
            o[r0:r0 + q_len, h] = om[:, i]
            lse[h, r0:r0 + q_len] = lm[i]
    return o, lse


def lse_merge(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Combine P partial results of the same query rows over disjoint key sets.

    o_parts [P, rows, H, d], lse_parts [P, H, rows]  ->  o [rows,H,d], lse [H,rows]

      lse = log sum_j exp(lse_j)
      o   = sum_j exp(lse_j - lse) * o_j

    A row whose partials are all empty (lse_j = -inf for every j) stays empty:
    o = 0, lse = -inf.
    """
    m = lse_parts.max(axis=0)                                   # [H, rows]
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w_unnorm = np.where(finite[None], np.exp(lse_parts - m_safe[None]), 0.0)
    total = w_unnorm.sum(axis=0)                                # [H, rows]
    lse = np.where(finite, m_safe + np.log(np.where(finite, total, 1.0)), -np.inf)
    w = np.where(finite[None], w_unnorm / np.where(finite, total, 1.0)[None], 0.0)
    o = np.einsum("phr,prhd->rhd", w, o_parts)
    return o, lse


# --------------------------------------------------------------------------
# Analytic backward of O = softmax(Q K^T * scale) V.
# --------------------------------------------------------------------------

def grad_v(p, do_rows):
    """dV contribution of a block of query rows: P^T dO."""
    return p.T @ do_rows


def grad_scores(p, dp, dsum):
    """dS = P * (dP - D), the softmax Jacobian applied row by row."""
    return p * (dp - dsum[:, None])


def grad_q(ds, k, scale):
    """dQ = scale * dS K."""
    return scale * (ds @ k)


def grad_k(ds, q_rows, scale):
    """dK contribution of a block of query rows: scale * dS^T Q."""
    return scale * (ds.T @ q_rows)


def attention_bwd_f64(q, k, v, do, scale):
    """Gradients for one head of one sequence.

    With P = softmax(S), S = Q K^T * scale and upstream dO:
      dV = P^T dO
      dP = dO V^T
      D  = rowsum(dO * O)            (= rowsum(P * dP))
      dS = P * (dP - D)
      dQ = scale * dS K
      dK = scale * dS^T Q
    O and LSE are recomputed here exactly in float64.
    """
    lq, lk = q.shape[0], k.shape[0]
    dq = np.zeros(q.shape, dtype=np.float64)
    dk = np.zeros(k.shape, dtype=np.float64)
    dv = np.zeros(v.shape, dtype=np.float64)
    if lq == 0 or lk == 0:
        return dq, dk, dv
    o, lse = attention_f64(q, k, v, scale)
    dsum = (do * o).sum(axis=1)
    for r0 in range(0, lq, ROW_BLOCK):
        r1 = min(lq, r0 + ROW_BLOCK)
        s = scores(q[r0:r1], k, scale)
        p = probabilities(s, lse[r0:r1])
        dv += grad_v(p, do[r0:r1])
        dp = do[r0:r1] @ v.T
        ds = grad_scores(p, dp, dsum[r0:r1])
        dq[r0:r1] = grad_q(ds, k, scale)
        dk += grad_k(ds, q[r0:r1], scale)
    return dq, dk, dv


def varlen_attn_bwd(q, k, v, do, cu_q, cu_k, scale=None, heads=None, seqs=None):
    """Gradients of the packed block-diagonal attention.  dq [Tq,H,d],
    dk/dv [Tk,H,d].  `heads` / `seqs` restrict the work (others stay 0)."""
    d = q.shape[2]
    if scale is None:
        scale = default_scale(d)
    dq = np.zeros(q.shape, dtype=np.float64)
    dk = np.zeros(k.shape, dtype=np.float64)
    dv = np.zeros(v.shape, dtype=np.float64)
    hs = range(q.shape[1]) if heads is None else heads
    ss = range(len(cu_q) - 1) if seqs is None else seqs
    for s in ss:
        qa, qb = int(cu_q[s]), int(cu_q[s + 1])
        ka, kb = int(cu_k[s]), int(cu_k[s + 1])
        for h in hs:
            g = attention_bwd_f64(q[qa:qb, h], k[ka:kb, h], v[ka:kb, h],
                                  do[qa:qb, h], scale)
            dq[qa:qb, h], dk[ka:kb, h], dv[ka:kb, h] = g
    return dq, dk, dv


def dq_rows(q, k, v, do, cu_q, cu_k, seq, head, rows, scale=None):
    """dQ of selected query rows of one head.  A dQ row depends only on its own
    query row, its own dO row and the full K/V of its sequence, so it can be
    computed row by row.  Returns [len(rows), d]."""
    d = q.shape[2]
    if scale is None:
        scale = default_scale(d)
    qa = int(cu_q[seq])
    ka, kb = int(cu_k[seq]), int(cu_k[seq + 1])
    rows = np.asarray(rows, dtype=np.int64)
    qr = q[qa + rows, head]
    dor = do[qa + rows, head]
    kk, vv = k[ka:kb, head], v[ka:kb, head]
    o_r, lse_r = attention_f64(qr, kk, vv, scale)
    s = scores(qr, kk, scale)
    p = probabilities(s, lse_r)
    dp = dor @ vv.T
    dsum = (dor * o_r).sum(axis=1)
    return grad_q(grad_scores(p, dp, dsum), kk, scale)


def dkdv_rows(q, k, v, do, cu_q, cu_k, seq, head, kv_rows, scale=None):
    """dK and dV of selected key rows (relative to sequence `seq`) of one head.

    A key row's gradients sum over every query row i of its sequence:
      dV_j = sum_i P_ij dO_i,   dK_j = scale * sum_i P_ij (dO_i . v_j - D_i) q_i
    so this first computes LSE and D = rowsum(dO * O) for all query rows (the
    full forward of that head), then only the selected columns of P.
    Returns (dk [len(kv_rows), d], dv [len(kv_rows), d])."""
    d = q.shape[2]
    if scale is None:
        scale = default_scale(d)
    qa, qb = int(cu_q[seq]), int(cu_q[seq + 1])
    ka, kb = int(cu_k[seq]), int(cu_k[seq + 1])
    kv_rows = np.asarray(kv_rows, dtype=np.int64)
    qq, dd = q[qa:qb, head], do[qa:qb, head]
    kk, vv = k[ka:kb, head], v[ka:kb, head]
    o, lse = attention_f64(qq, kk, vv, scale)
    dsum = (dd * o).sum(axis=1)
    s_cols = scores(qq, kk[kv_rows], scale)                # [Lq, |J|]
    p = probabilities(s_cols, lse)
    dv = grad_v(p, dd)
    dp = dd @ vv[kv_rows].T
    ds = grad_scores(p, dp, dsum)
    dk = grad_k(ds, qq, scale)
    return dk, dv


def grads_one_query_row(q, k, v, do_row, cu_q, cu_k, seq, head, row, scale=None):
    """Gradients of one head of sequence `seq` when dO is zero except at query
    row `row` (relative to the sequence), where it is `do_row` [d].

    Then D = rowsum(dO * O) and dP = dO V^T vanish on every other row, so dS is
    zero there and only that row's softmax enters:
      dV_j = P_rj dO_r,   dK_j = scale * dS_rj q_r,   dQ_r = scale * dS_r K,
    with dS_r = P_r * (dO_r V^T - dO_r . O_r); every other dQ row is zero.
    Returns (dq_row [d], dk [Lk, d], dv [Lk, d])."""
    d = q.shape[2]
    if scale is None:
        scale = default_scale(d)
    qa = int(cu_q[seq])
    ka, kb = int(cu_k[seq]), int(cu_k[seq + 1])
    qr = q[qa + row:qa + row + 1, head]
    dor = np.asarray(do_row, dtype=np.float64)[None, :]
    kk, vv = k[ka:kb, head], v[ka:kb, head]
    o_r, lse_r = attention_f64(qr, kk, vv, scale)
    p = probabilities(scores(qr, kk, scale), lse_r)
    ds = grad_scores(p, dor @ vv.T, (dor * o_r).sum(axis=1))
    return grad_q(ds, kk, scale)[0], grad_k(ds, qr, scale), grad_v(p, dor)

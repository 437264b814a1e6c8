"""The workspace-free backward, zl_varlen_attn_bwd_static.

It is for callers that cannot allocate device memory when they need the
gradient (an engine plugin that must not allocate while it runs, code inside
stream capture, a process whose memory is reserved by a pool it may not call).
It keeps its scratch in a fixed array in the library's device image.  These
tests call it twice in a row, the second call on a smaller batch that reuses
the array the first one left behind, and compare every gradient element with
the float64 oracle's analytic gradient and with the regular workspace
backward, within the gradient tolerance; they also cover query and key
lengths that differ (including a sequence with keys but no queries, whose dK
and dV must be zero), more sequences than one launch holds, head_dim 64, and
an oversized batch that is refused before any GPU work.  This file is
collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
import mixed_length_dit_gb300 as zl
from mixed_length_dit_gb300 import _lib
from _helpers import TOL_GRAD_REL_L2, f64, rel_l2

pytestmark = pytest.mark.gpu


def _static_bwd(q, k, v, o, lse, do, cu_q, cu_k, nh, hd, dq, dk, dv):
    lib = _lib.load()
    cq, nq = _lib.int32_array(cu_q)
    ck, _ = _lib.int32_array(cu_k)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.zl_varlen_attn_bwd_static(p(q), p(k), p(v), p(o), p(lse), p(do), cq, ck, nq - 1, nh, hd,
                                         1.0 / hd ** 0.5, p(dq), p(dk), p(dv), stream)


def _check(q, k, v, do, cu_q, cu_k, nh, hd):
    """Runs the forward, the workspace backward and the static backward on one
    batch; every gradient of the static backward must be finite and within the
    gradient tolerance of both the oracle and the workspace backward."""
    o, lse = zl.varlen_attn_fwd(q, k, v, cu_q, cu_k)
    ref_ws = zl.varlen_attn_bwd(q, k, v, o, lse, do, cu_q, cu_k)
    got = [torch.full_like(t, float("nan")) for t in ref_ws]
    st = _static_bwd(q, k, v, o, lse, do, cu_q, cu_k, nh, hd, *got)
    assert st == _lib.ZL_OK, _lib.status_string(st)
    zl.sync_check()
    ref = oracle.varlen_attn_bwd(f64(q), f64(k), f64(v), f64(do), cu_q, cu_k)
    for name, g, r_ws, r in zip(("dq", "dk", "dv"), got, ref_ws, ref):
        assert torch.isfinite(g).all(), name
        e = rel_l2(f64(g), r)
        assert e <= TOL_GRAD_REL_L2, (name, "oracle", e)
        e_ws = rel_l2(f64(g), f64(r_ws))
        assert e_ws <= TOL_GRAD_REL_L2, (name, "workspace backward", e_ws)
    return got


def test_two_calls_in_a_row_match_the_oracle():
    for seed, seqlens in enumerate(([300, 1000, 64, 129, 700], [37, 256, 5])):
        wl = synth.Workload("noalloc", list(seqlens), 4, 128)
        inp = synth.make_inputs(wl, seed=seed, device="cuda")
        cu = wl.cu_seqlens()
        _check(inp["q"], inp["k"], inp["v"], inp["do"], cu, cu, 4, 128)


def test_cross_lengths_and_keys_without_queries():
    cu_q = [0, 0, 130, 200, 521]
    cu_k = [0, 50, 60, 300, 500]
    g = torch.Generator(device="cuda").manual_seed(21)
    mk = lambda n: torch.randn((n, 3, 128), generator=g, device="cuda").to(torch.bfloat16)
    q, k, v, do = mk(521), mk(500), mk(500), mk(521)
    dq, dk, dv = _check(q, k, v, do, cu_q, cu_k, 3, 128)
    assert torch.all(dk[0:50] == 0) and torch.all(dv[0:50] == 0)


def test_more_sequences_than_one_launch_holds_head_dim_64():
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(1, 40, size=700)]
    wl = synth.Workload("many", lens, 2, 64)
    inp = synth.make_inputs(wl, seed=7, device="cuda")
    cu = wl.cu_seqlens()
    _check(inp["q"], inp["k"], inp["v"], inp["do"], cu, cu, 2, 64)


def test_oversized_batch_is_refused():
    wl = synth.Workload("big", [4000], 40, 128)
    t = torch.empty((1, 40, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((40, 1), dtype=torch.float32, device="cuda")
    cu = wl.cu_seqlens()
    st = _static_bwd(t, t, t, t, lse, t, cu, cu, 40, 128, t, t, t)
    assert st == _lib.ZL_EWORKSPACE

"""The workspace-free backward, zl_varlen_attn_bwd_static.

It is for callers that cannot allocate device memory when they need the
gradient (an engine plugin that must not allocate while it runs, code inside
stream capture, a process whose memory is reserved by a pool it may not call).
It keeps its scratch in a fixed array in the library's device image, so these
tests check that two calls in a row, the second on a smaller batch that reuses
the array the first one left behind, both match the regular workspace backward
within the gradient tolerance, and that an oversized batch is refused before
any GPU work.  This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import synth
import mixed_length_dit_gb300 as zl
from mixed_length_dit_gb300 import _lib
from _helpers import TOL_GRAD_REL_L2

pytestmark = pytest.mark.gpu


def _static_bwd(inp, o, lse, cu, nh, hd, dq, dk, dv):
    lib = _lib.load()
    cq, nq = _lib.int32_array(cu)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.zl_varlen_attn_bwd_static(p(inp["q"]), p(inp["k"]), p(inp["v"]), p(o), p(lse), p(inp["do"]),
                                         cq, cq, nq - 1, nh, hd, 1.0 / hd ** 0.5, p(dq), p(dk), p(dv), stream)


def _rel(a, b):
    a, b = a.double(), b.double()
    return ((a - b).norm() / b.norm()).item()


@pytest.mark.parametrize("batches", [([300, 1000, 64, 129, 700], [37, 256, 5])])
def test_two_calls_match_workspace_backward(batches):
    for seqlens in batches:
        wl = synth.Workload("noalloc", list(seqlens), 4, 128)
        inp = synth.make_inputs(wl, seed=len(seqlens), device="cuda")
        cu = wl.cu_seqlens()
        o, lse = zl.varlen_attn_fwd(inp["q"], inp["k"], inp["v"], cu, cu)
        ref = zl.varlen_attn_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], cu, cu)
        got = [torch.full_like(t, float("nan")) for t in ref]
        st = _static_bwd(inp, o, lse, cu, 4, 128, *got)
        assert st == _lib.ZL_OK, _lib.status_string(st)
        zl.sync_check()
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert torch.isfinite(g).all(), name
            assert _rel(g, r) <= TOL_GRAD_REL_L2, (name, _rel(g, r))


def test_oversized_batch_is_refused():
    wl = synth.Workload("big", [4000], 40, 128)
    t = torch.empty((1, 40, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((40, 1), dtype=torch.float32, device="cuda")
    inp = {"q": t, "k": t, "v": t, "do": t}
    st = _static_bwd(inp, t, lse, wl.cu_seqlens(), 40, 128, t, t, t)
    assert st == _lib.ZL_EWORKSPACE

"""Failure detection on the GPU without a fault: every wait inside this
library's kernels is bounded, and a wait that runs out records an error that
the host reads (zl_sync_check -> ZL_ETIMEOUT), ends the other roles of its
CTA, and leaves the context usable.  The Zellige paper's planner either
returns a whole placement or fails as a whole (arXiv 2608.01150v1, §IV-C);
the engine here likewise either finishes a call or reports that it did not.

zl_selftest_wait_timeout makes one wait run out on purpose: an mbarrier that
nothing arrives on, with a short limit, no copies or MMAs in flight.
"""
import time

import pytest
import torch

import synth
import mixed_length_dit_gb300 as zl
from mixed_length_dit_gb300 import _lib
from _helpers import TOL_LSE, TOL_O_BF16, f64

import oracle

pytestmark = pytest.mark.gpu


def _stream():
    import ctypes
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    lib = _lib.load()
    torch.cuda.synchronize()
    assert lib.zl_sync_check(_stream()) == _lib.ZL_OK
    t0 = time.monotonic()
    assert lib.zl_selftest_wait_timeout(20_000_000, _stream()) == _lib.ZL_OK   # 20 ms
    st = lib.zl_sync_check(_stream())
    elapsed = time.monotonic() - t0
    assert st == _lib.ZL_ETIMEOUT, _lib.status_string(st)
    # the second warp, whose own limit is 2 s, left on the abort flag
    assert elapsed < 1.0, elapsed
    assert lib.zl_sync_check(_stream()) == _lib.ZL_OK          # the record was cleared
    # the next call runs normally and matches the oracle
    wl = synth.config(1)
    inp = synth.make_inputs(wl, seed=0, device="cuda", with_grad_out=False)
    cu = wl.cu_seqlens()
    o, lse = zl.varlen_attn_fwd(inp["q"], inp["k"], inp["v"], cu, cu)
    zl.sync_check()
    o_ref, lse_ref = oracle.varlen_attn_fwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), cu, cu)
    assert abs(f64(o) - o_ref).max() <= TOL_O_BF16
    assert abs(f64(lse) - lse_ref).max() <= TOL_LSE


def test_self_test_runs_out_each_time():
    lib = _lib.load()
    for _ in range(3):
        assert lib.zl_selftest_wait_timeout(1_000_000, _stream()) == _lib.ZL_OK
        assert lib.zl_sync_check(_stream()) == _lib.ZL_ETIMEOUT
    assert lib.zl_sync_check(_stream()) == _lib.ZL_OK

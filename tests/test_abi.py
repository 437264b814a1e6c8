"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects malformed calls on the host before any CUDA work
(Zellige arXiv 2608.01150v1 §IV-C: a plan either succeeds or fails as a
whole; here an invalid call returns an error and touches no output)."""
import ctypes
import os
import re

import pytest

from mixed_length_dit_gb300 import _lib
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "zl_attn.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zl_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_lib.EXPORTS)


def test_version_and_strings(lib):
    assert lib.zl_version() >> 16 == 2 and lib.zl_version() & 0xFFFF >= 1
    for code in range(0, -8, -1):
        assert _lib.status_string(code) not in ("", "unknown status")
    assert _lib.status_string(-99) == "unknown status"


def _fwd(lib, cu_q, cu_k, nh=2, hd=64, tiles=None, dtype=_lib.ZL_BF16, scale=0.125,
         ptr=64, ws=None, ws_bytes=0):
    cq, nq = _lib.int32_array(cu_q)
    ck, _ = _lib.int32_array(cu_k)
    ta, nt = _lib.tile_array(tiles)
    p = ctypes.c_void_p(ptr)
    return lib.zl_varlen_attn_fwd(p, p, p, cq, ck, nq - 1, nh, hd, dtype, scale, ta, nt, p, p,
                                  ctypes.c_void_p(ws), ws_bytes, None)


def test_rejects_bad_cu_seqlens(lib):
    assert _fwd(lib, [1, 5], [0, 5]) == _lib.ZL_EINVAL          # does not start at 0
    assert _fwd(lib, [0, 5, 3], [0, 5, 3]) == _lib.ZL_EINVAL    # decreasing
    assert _fwd(lib, [0, 4], [0, 0]) == _lib.ZL_EINVAL          # queries without keys


def test_rejects_bad_shapes_and_types(lib):
    assert _fwd(lib, [0, 5], [0, 5], hd=96) == _lib.ZL_EUNSUPPORTED
    assert _fwd(lib, [0, 5], [0, 5], nh=0) == _lib.ZL_EINVAL
    assert _fwd(lib, [0, 5], [0, 5], dtype=7) == _lib.ZL_EUNSUPPORTED
    assert _fwd(lib, [0, 5], [0, 5], scale=-1.0) == _lib.ZL_EINVAL
    assert _fwd(lib, [0, 5], [0, 5], scale=float("nan")) == _lib.ZL_EINVAL
    assert _fwd(lib, [0, 5], [0, 5], ptr=8) == _lib.ZL_EALIGN
    assert _fwd(lib, [0, 5], [0, 5], ptr=0) == _lib.ZL_EINVAL


def test_empty_batch_is_a_no_op(lib):
    assert _fwd(lib, [0], [0], ptr=0) == _lib.ZL_OK
    assert _fwd(lib, [0, 0, 0], [0, 0, 0], ptr=0) == _lib.ZL_OK


def test_tile_table_validation(lib):
    L = 300
    good = synth.grid_tiles(0, L, L, 2, 3)
    cu = [0, L, L + 10]

    def ws_size(tiles):
        cq, nq = _lib.int32_array(cu)
        ta, nt = _lib.tile_array(tiles)
        out = ctypes.c_size_t(0)
        st = lib.zl_varlen_attn_fwd_workspace_size(cq, cq, nq - 1, 2, 64, ta, nt, ctypes.byref(out))
        return st, out.value

    st, nbytes = ws_size(good)
    assert st == _lib.ZL_OK
    assert nbytes >= 3 * L * 2 * 64 * 4 + 3 * 2 * L * 4
    assert ws_size(list(reversed(good)))[0] == _lib.ZL_OK            # any order
    assert ws_size(good[:-1])[0] == _lib.ZL_EINVAL                   # missing tile
    assert ws_size(good + [good[0]])[0] == _lib.ZL_EINVAL            # duplicate
    bad = list(good)
    t = list(bad[1]); t[4] -= 1; bad[1] = tuple(t)                   # gap in key range
    assert ws_size(bad)[0] == _lib.ZL_EINVAL
    bad = list(good)
    t = list(bad[0]); t[7] = 4; bad[0] = tuple(t)                    # n_kv mismatch
    assert ws_size(bad)[0] == _lib.ZL_EINVAL
    bad = list(good)
    t = list(bad[0]); t[0] = 5; bad[0] = tuple(t)                    # seq out of range
    assert ws_size(bad)[0] == _lib.ZL_EINVAL
    # a full grid whose query chunks do not cover the sequence
    assert ws_size(synth.grid_tiles(0, L - 1, L, 2, 3))[0] == _lib.ZL_EINVAL
    # a sequence with an empty chunk (4 chunks of 1 token over 3 tokens) is rejected
    assert ws_size([(1, 0, 10, 0, 10, 0, 0, 1)])[0] == _lib.ZL_OK
    assert _fwd(lib, cu, cu, tiles=good, ws=0) == _lib.ZL_EWORKSPACE
    assert _fwd(lib, cu, cu, tiles=good, ws=256, ws_bytes=16) == _lib.ZL_EWORKSPACE


def _ws(lib, cu, tiles, nh):
    cq, nq = _lib.int32_array(cu)
    ta, nt = _lib.tile_array(tiles)
    out = ctypes.c_size_t(0)
    st = lib.zl_varlen_attn_fwd_workspace_size(cq, cq, nq - 1, nh, 64, ta, nt, ctypes.byref(out))
    return st, out.value


def _edit(tiles, i, field, value):
    out = list(tiles)
    t = list(out[i])
    t[field] = value
    out[i] = tuple(t)
    return out


def test_head_sharded_tile_validation(lib):
    """(q, h, k) configurations (Zellige §IV-A): head ranges must partition
    [0, H) and every head chunk must repeat the same query x key grid."""
    L, H = 300, 4
    cu = [0, L, L + 10]
    good = synth.grid_tiles(0, L, L, 2, 3, 2, H)             # 2 head chunks x 2 x 3
    assert len(good) == 12
    st, n_heads_split = _ws(lib, cu, good, H)
    assert st == _lib.ZL_OK
    assert n_heads_split == _ws(lib, cu, synth.grid_tiles(0, L, L, 2, 3), H)[1]   # same partials
    assert _ws(lib, cu, list(reversed(good)), H)[0] == _lib.ZL_OK
    assert _ws(lib, cu, good[:6], H)[0] == _lib.ZL_EINVAL            # head chunk 1 missing
    assert _ws(lib, cu, good[:-1], H)[0] == _lib.ZL_EINVAL           # one tile missing
    assert _ws(lib, cu, synth.grid_tiles(0, L, L, 2, 3, 2, H + 2), H)[0] == _lib.ZL_EINVAL  # beyond H
    assert _ws(lib, cu, synth.grid_tiles(0, L, L, 2, 3, 2, H - 1), H)[0] == _lib.ZL_EINVAL  # heads left out
    gap = [t[:8] + (t[8] + (1 if t[10] == 1 else 0), t[9] - (1 if t[10] == 1 else 0), t[10]) for t in good]
    assert _ws(lib, cu, gap, H)[0] == _lib.ZL_EINVAL                 # heads 2 uncovered
    assert _ws(lib, cu, _edit(good, 7, 9, 1), H)[0] == _lib.ZL_EINVAL   # ranges differ in a chunk
    assert _ws(lib, cu, _edit(good, 7, 1, 5), H)[0] == _lib.ZL_EINVAL   # grids differ across chunks
    whole = synth.grid_tiles(0, L, L, 2, 3)
    assert _ws(lib, cu, _edit(whole, 0, 8, 1), H)[0] == _lib.ZL_EINVAL  # h_len 0 needs h_start 0
    assert _ws(lib, cu, _edit(whole, 0, 10, 1), H)[0] == _lib.ZL_EINVAL  # ... and h_chunk 0
    assert _ws(lib, cu, _edit(whole, 0, 9, -1), H)[0] == _lib.ZL_EINVAL
    # key axis not split: no partials, so no workspace
    assert _ws(lib, cu, synth.grid_tiles(0, L, L, 1, 1, 4, H), H) == (_lib.ZL_OK, 0)
    assert _ws(lib, cu, synth.grid_tiles(0, L, L, 3, 1, 2, H), H) == (_lib.ZL_OK, 0)
    mixed = synth.grid_tiles(0, L, L, 3, 1, 2, H) + synth.grid_tiles(1, 10, 10, 1, 2)
    st, nbytes = _ws(lib, cu, mixed, H)
    assert st == _lib.ZL_OK and nbytes >= 2 * 10 * H * 64 * 4 + 2 * H * 10 * 4
    assert nbytes < 2 * L * H * 64 * 4


def test_workspace_size_matches_layout(lib):
    wl = synth.config(4)
    cq, nq = _lib.int32_array(wl.cu_seqlens())
    ta, nt = _lib.tile_array(wl.tiles())
    out = ctypes.c_size_t(0)
    assert lib.zl_varlen_attn_fwd_workspace_size(cq, cq, nq - 1, 40, 128, ta, nt, ctypes.byref(out)) == 0
    R, P = 131072, 4
    counters = 4 * (32768 // 128) * 40          # (query chunk, 128-row block) x head
    assert out.value == P * R * 40 * 128 * 4 + P * 40 * R * 4 + counters * 4
    out2 = ctypes.c_size_t(0)
    assert lib.zl_varlen_attn_bwd_workspace_size(cq, cq, nq - 1, 40, 128, ctypes.byref(out2)) == 0
    T = wl.total_tokens
    assert out2.value >= T * 40 * 128 * 4 + 40 * T * 4


def test_merge_argument_checks(lib):
    p = ctypes.c_void_p(64)
    assert lib.zl_lse_merge(p, p, 0, 10, 2, 64, 10, p, 0, p, 10, None) == _lib.ZL_EINVAL
    assert lib.zl_lse_merge(p, p, 65, 10, 2, 64, 10, p, 0, p, 10, None) == _lib.ZL_EINVAL
    assert lib.zl_lse_merge(p, p, 2, 10, 2, 64, 5, p, 0, p, 10, None) == _lib.ZL_EINVAL
    assert lib.zl_lse_merge(p, p, 2, 10, 2, 32, 10, p, 0, p, 10, None) == _lib.ZL_EUNSUPPORTED
    assert lib.zl_lse_merge(p, p, 2, 0, 2, 64, 0, p, 0, p, 0, None) == _lib.ZL_OK
    # the partial dtype of zl_lse_merge_ex: bf16 or float32 only
    assert lib.zl_lse_merge_ex(p, 7, p, 2, 10, 2, 64, 10, p, 0, p, 10, None) == _lib.ZL_EUNSUPPORTED
    assert lib.zl_lse_merge_ex(p, _lib.ZL_BF16, p, 0, 10, 2, 64, 10, p, 0, p, 10, None) == _lib.ZL_EINVAL
    assert lib.zl_lse_merge_ex(p, _lib.ZL_BF16, p, 2, 0, 2, 64, 0, p, 0, p, 0, None) == _lib.ZL_OK


def test_forward_flags(lib):
    """zl_varlen_attn_fwd_ex accepts exactly the documented flag bits.  The
    head dimension 96 is unsupported, which the library reports only after the
    flags have passed, so no call here can reach a launch."""
    cq, nq = _lib.int32_array([0, 5])
    p = ctypes.c_void_p(64)
    args = [p, p, p, cq, cq, nq - 1, 2, 96, _lib.ZL_BF16, 0.125, None, 0, p, p, None, 0, None]
    assert lib.zl_varlen_attn_fwd_ex(*args, 4) == _lib.ZL_EINVAL
    assert lib.zl_varlen_attn_fwd_ex(*args, 1 << 31) == _lib.ZL_EINVAL
    for ok_flags in (0, _lib.ZL_FWD_FUSED_MERGE, _lib.ZL_FWD_BF16_PARTIALS,
                     _lib.ZL_FWD_FUSED_MERGE | _lib.ZL_FWD_BF16_PARTIALS):
        assert lib.zl_varlen_attn_fwd_ex(*args, ok_flags) == _lib.ZL_EUNSUPPORTED


def test_bwd_argument_checks(lib):
    cq, nq = _lib.int32_array([0, 5])
    p = ctypes.c_void_p(64)
    args = [p] * 6 + [cq, cq, nq - 1, 2, 64]
    tail = [None, 0, p, p, p, p, 1 << 20, None]
    assert lib.zl_varlen_attn_bwd(*args, _lib.ZL_FP32, 0.125, *tail) == _lib.ZL_EUNSUPPORTED
    assert lib.zl_varlen_attn_bwd(*args, _lib.ZL_BF16, 0.0, *tail) == _lib.ZL_EINVAL


def test_static_bwd_applies_the_batch_bounds(lib):
    """The workspace-free backward checks a batch as zl_varlen_attn_bwd does,
    token bounds included, before its scratch limit and before any CUDA call:
    an oversized key count is an invalid argument, not a scratch overflow."""
    p = ctypes.c_void_p(64)
    cq, nq = _lib.int32_array([0, 5])
    for ck_list, nh in (([0, (1 << 31) - 100], 2),          # more keys than int32 row indices allow
                        ([0, (1 << 31) - 300], 4096),       # (Tk + block) * H * d > 2^40
                        ([0, 3000], 8192)):                 # too many heads
        ck, _ = _lib.int32_array(ck_list)
        args = [p] * 6 + [cq, ck, 1, nh, 128, 0.125, p, p, p, None]
        assert lib.zl_varlen_attn_bwd_static(*args) == _lib.ZL_EINVAL, (ck_list, nh)
        wargs = [p] * 6 + [cq, ck, 1, nh, 128, _lib.ZL_BF16, 0.125, None, 0, p, p, p, p, 1 << 40, None]
        assert lib.zl_varlen_attn_bwd(*wargs) == _lib.ZL_EINVAL, (ck_list, nh)
    bad, _ = _lib.int32_array([0, 7, 5])
    assert lib.zl_varlen_attn_bwd_static(*([p] * 6), bad, bad, 2, 2, 64, 0.125, p, p, p, None) == _lib.ZL_EINVAL
    assert lib.zl_varlen_attn_bwd_static(*([p] * 6), cq, cq, 1, 2, 96, 0.125, p, p, p, None) == \
        _lib.ZL_EUNSUPPORTED
    # past the scratch limit: 131,072 query tokens at 40 heads x 128
    big, _ = _lib.int32_array([0, 131072])
    assert lib.zl_varlen_attn_bwd_static(*([p] * 6), big, big, 1, 40, 128, 0.125, p, p, p, None) == \
        _lib.ZL_EWORKSPACE


def test_selftest_limit_is_checked_first(lib):
    """The wait self-test takes limits of 1 ns .. 1 s only, checked before
    any CUDA call."""
    assert lib.zl_selftest_wait_timeout(0, None) == _lib.ZL_EINVAL
    assert lib.zl_selftest_wait_timeout(1_000_000_001, None) == _lib.ZL_EINVAL


def test_no_device_is_reported_not_crashed(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _fwd(lib, [0, 5], [0, 5]) == _lib.ZL_ENODEVICE

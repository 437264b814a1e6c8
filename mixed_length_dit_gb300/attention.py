"""PyTorch-facing wrappers of the C ABI.  torch supplies device memory and the
current CUDA stream; the arithmetic is entirely in libzl_attn.so.

Tensors: q/o [Tq, H, d], k/v [Tk, H, d] contiguous CUDA tensors (bf16 for the
tensor-core path, float32 for the float32 path); lse [H, Tq] float32.
cu_seqlens are host sequences of ints (B+1 entries, starting at 0).
tiles are tuples (seq, q_start, q_len, k_start, k_len, q_chunk, kv_chunk,
n_kv_chunks), see zl_tile_t in include/zl_attn.h.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _lib


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return _lib.ZL_BF16
    if t.dtype == torch.float32:
        return _lib.ZL_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _check_tensor(t, name):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def _last(cu) -> int:
    vals = cu.tolist() if hasattr(cu, "tolist") else list(cu)
    if not vals:
        raise ValueError("cu_seqlens must have at least one entry")
    return int(vals[-1])


def _check_like(t, name, shape, dtype, device):
    """t must have exactly this shape, dtype and device: the library receives
    only its pointer and writes or reads the sizes that the batch implies.
    (Whether it is a contiguous CUDA tensor is checked after every shape.)"""
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or t.device != device:
        raise ValueError(f"{name} must be {tuple(shape)} {dtype} on {device}, "
                         f"got {tuple(t.shape)} {t.dtype} on {t.device}")


def _check_cuda(**tensors):
    for name, t in tensors.items():
        _check_tensor(t, name)


def _check_qkv(q, k, v, cu_seqlens_q, cu_seqlens_k):
    """q [Tq, H, d], k and v [Tk, H, d] of one dtype on one device, with Tq
    and Tk the last entries of the cu_seqlens (the packed layout of the C
    ABI), so that no tensor map or row index reaches past an allocation."""
    if q.dim() != 3:
        raise ValueError("q must be [Tq, H, d]")
    tq, nh, hd = q.shape
    if tq != _last(cu_seqlens_q):
        raise ValueError(f"q has {tq} rows, cu_seqlens_q ends at {_last(cu_seqlens_q)}")
    _check_like(k, "k", (_last(cu_seqlens_k), nh, hd), q.dtype, q.device)
    _check_like(v, "v", k.shape, q.dtype, q.device)
    return tq, nh, hd


def _workspace_bytes(workspace) -> int:
    if workspace is None:
        return 0
    _check_tensor(workspace, "workspace")
    return workspace.numel() * workspace.element_size()


def fwd_workspace_bytes(cu_seqlens_q, cu_seqlens_k, num_heads, head_dim, tiles=None) -> int:
    lib = _lib.load()
    cq, nq = _lib.int32_array(cu_seqlens_q)
    ck, _ = _lib.int32_array(cu_seqlens_k)
    ta, nt = _lib.tile_array(tiles)
    out = ctypes.c_size_t(0)
    _lib.check(lib.zl_varlen_attn_fwd_workspace_size(cq, ck, nq - 1, num_heads, head_dim, ta, nt,
                                                     ctypes.byref(out)), "workspace_size")
    return int(out.value)


def bwd_workspace_bytes(cu_seqlens_q, cu_seqlens_k, num_heads, head_dim) -> int:
    lib = _lib.load()
    cq, nq = _lib.int32_array(cu_seqlens_q)
    ck, _ = _lib.int32_array(cu_seqlens_k)
    out = ctypes.c_size_t(0)
    _lib.check(lib.zl_varlen_attn_bwd_workspace_size(cq, ck, nq - 1, num_heads, head_dim,
                                                     ctypes.byref(out)), "bwd_workspace_size")
    return int(out.value)


def fwd_schedule(cu_seqlens_q, cu_seqlens_k, num_heads, head_dim, tiles=None, dtype=torch.bfloat16):
    """The forward's work items in launch order (host only): a list of
    (launch, seq, tile, head, q_start, q_len, k_start, k_len) tuples, tile
    -1 for a whole sequence (zl_varlen_attn_fwd_schedule)."""
    lib = _lib.load()
    cq, nq = _lib.int32_array(cu_seqlens_q)
    ck, _ = _lib.int32_array(cu_seqlens_k)
    ta, nt = _lib.tile_array(tiles)
    code = _lib.ZL_BF16 if dtype == torch.bfloat16 else _lib.ZL_FP32
    n = ctypes.c_int64(0)
    _lib.check(lib.zl_varlen_attn_fwd_schedule(cq, ck, nq - 1, num_heads, head_dim, code, ta, nt, None, 0,
                                               ctypes.byref(n)), "zl_varlen_attn_fwd_schedule")
    arr = (_lib.WorkItem * max(1, n.value))()
    _lib.check(lib.zl_varlen_attn_fwd_schedule(cq, ck, nq - 1, num_heads, head_dim, code, ta, nt, arr, n.value,
                                               ctypes.byref(n)), "zl_varlen_attn_fwd_schedule")
    return [tuple(getattr(arr[i], f) for f, _ in _lib.WorkItem._fields_) for i in range(n.value)]


def bwd_schedule(cu_seqlens_q, cu_seqlens_k, num_heads, head_dim, tiles=None):
    """The backward's work items in launch order (host only): a list of
    (launch, seq, head, k_start, k_len, q_len) tuples
    (zl_varlen_attn_bwd_schedule)."""
    lib = _lib.load()
    cq, nq = _lib.int32_array(cu_seqlens_q)
    ck, _ = _lib.int32_array(cu_seqlens_k)
    ta, nt = _lib.tile_array(tiles)
    n = ctypes.c_int64(0)
    _lib.check(lib.zl_varlen_attn_bwd_schedule(cq, ck, nq - 1, num_heads, head_dim, ta, nt, None, 0,
                                               ctypes.byref(n)), "zl_varlen_attn_bwd_schedule")
    arr = (_lib.BwdWorkItem * max(1, n.value))()
    _lib.check(lib.zl_varlen_attn_bwd_schedule(cq, ck, nq - 1, num_heads, head_dim, ta, nt, arr, n.value,
                                               ctypes.byref(n)), "zl_varlen_attn_bwd_schedule")
    return [tuple(getattr(arr[i], f) for f, _ in _lib.BwdWorkItem._fields_) for i in range(n.value)]


def alloc_workspace(nbytes: int, device) -> torch.Tensor | None:
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def varlen_attn_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k=None, tiles=None, softmax_scale=None,
                    out=None, lse=None, workspace=None, stream=None, fused_merge=False,
                    bf16_partials=False):
    """Coalesced block-diagonal attention forward.  Returns (o, lse).
    fused_merge merges tile partials inside the forward launch
    (ZL_FWD_FUSED_MERGE); bf16_partials keeps the partial O rows of key-split
    sequences in bf16 (ZL_FWD_BF16_PARTIALS)."""
    lib = _lib.load()
    if cu_seqlens_k is None:
        cu_seqlens_k = cu_seqlens_q
    tq, nh, hd = _check_qkv(q, k, v, cu_seqlens_q, cu_seqlens_k)
    scale = 1.0 / math.sqrt(hd) if softmax_scale is None else float(softmax_scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((nh, tq), dtype=torch.float32, device=q.device)
    _check_like(out, "out", q.shape, q.dtype, q.device)
    _check_like(lse, "lse", (nh, tq), torch.float32, q.device)
    _check_cuda(q=q, k=k, v=v, out=out, lse=lse)
    if workspace is None:
        workspace = alloc_workspace(fwd_workspace_bytes(cu_seqlens_q, cu_seqlens_k, nh, hd, tiles), q.device)
    cq, nq = _lib.int32_array(cu_seqlens_q)
    ck, nk = _lib.int32_array(cu_seqlens_k)
    if nq != nk:
        raise ValueError("cu_seqlens_q and cu_seqlens_k differ in length")
    ta, nt = _lib.tile_array(tiles)
    ws_bytes = _workspace_bytes(workspace)
    flags = (_lib.ZL_FWD_FUSED_MERGE if fused_merge else 0) | (_lib.ZL_FWD_BF16_PARTIALS if bf16_partials else 0)
    st = lib.zl_varlen_attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), cq, ck, nq - 1, nh, hd, _dtype_code(q),
                                   scale, ta, nt, _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                                   _stream_handle(stream), flags)
    _lib.check(st, "zl_varlen_attn_fwd")
    return out, lse


def varlen_attn_bwd(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k=None, tiles=None,
                    softmax_scale=None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward of varlen_attn_fwd.  Returns (dq, dk, dv)."""
    lib = _lib.load()
    if cu_seqlens_k is None:
        cu_seqlens_k = cu_seqlens_q
    tq, nh, hd = _check_qkv(q, k, v, cu_seqlens_q, cu_seqlens_k)
    _check_like(o, "o", q.shape, q.dtype, q.device)
    _check_like(dout, "dout", q.shape, q.dtype, q.device)
    _check_like(lse, "lse", (nh, tq), torch.float32, q.device)
    scale = 1.0 / math.sqrt(hd) if softmax_scale is None else float(softmax_scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_like(dq, "dq", q.shape, q.dtype, q.device)
    _check_like(dk, "dk", k.shape, q.dtype, q.device)
    _check_like(dv, "dv", k.shape, q.dtype, q.device)
    _check_cuda(q=q, k=k, v=v, o=o, lse=lse, dout=dout, dq=dq, dk=dk, dv=dv)
    if workspace is None:
        workspace = alloc_workspace(bwd_workspace_bytes(cu_seqlens_q, cu_seqlens_k, nh, hd), q.device)
    cq, nq = _lib.int32_array(cu_seqlens_q)
    ck, _ = _lib.int32_array(cu_seqlens_k)
    ta, nt = _lib.tile_array(tiles)
    ws_bytes = _workspace_bytes(workspace)
    st = lib.zl_varlen_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), cq, ck,
                                nq - 1, nh, hd, _dtype_code(q), scale, ta, nt, _ptr(dq), _ptr(dk),
                                _ptr(dv), _ptr(workspace), ws_bytes, _stream_handle(stream))
    _lib.check(st, "zl_varlen_attn_bwd")
    return dq, dk, dv


def lse_merge(o_partial, lse_partial, rows=None, out_dtype=torch.bfloat16, out=None, lse=None,
              lse_head_stride=None, stream=None):
    """Exact merge of partials o_partial [P, R, H, d] (float32 or bf16) /
    lse_partial [P, H, R] (float32) into (o [rows, H, d], lse [H, rows])."""
    lib = _lib.load()
    if o_partial.dim() != 4 or o_partial.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("o_partial must be [P, R, H, d] float32 or bf16")
    n_parts, part_rows, nh, hd = o_partial.shape
    dev = o_partial.device
    _check_like(lse_partial, "lse_partial", (n_parts, nh, part_rows), torch.float32, dev)
    rows = part_rows if rows is None else int(rows)
    if not 0 <= rows <= part_rows:
        raise ValueError(f"rows must lie in [0, {part_rows}]")
    if out is None:
        out = torch.empty((rows, nh, hd), dtype=out_dtype, device=dev)
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("out must be bf16 or float32")
    _check_like(out, "out", (rows, nh, hd), out.dtype, dev)
    if lse is None:
        lse = torch.empty((nh, rows), dtype=torch.float32, device=dev)
        lse_head_stride = rows
    stride = rows if lse_head_stride is None else int(lse_head_stride)
    if lse.dtype != torch.float32 or lse.device != dev or stride < rows or \
            (nh > 0 and rows > 0 and lse.numel() < (nh - 1) * stride + rows):
        raise ValueError(f"lse must be float32 on {dev} holding {nh} heads of {rows} rows at stride {stride}")
    _check_cuda(o_partial=o_partial, lse_partial=lse_partial, out=out, lse=lse)
    code = _lib.ZL_BF16 if out.dtype == torch.bfloat16 else _lib.ZL_FP32
    part = _lib.ZL_BF16 if o_partial.dtype == torch.bfloat16 else _lib.ZL_FP32
    st = lib.zl_lse_merge_ex(_ptr(o_partial), part, _ptr(lse_partial), n_parts, rows, nh, hd, part_rows,
                             _ptr(out), code, _ptr(lse), stride,
                             _stream_handle(stream))
    _lib.check(st, "zl_lse_merge_ex")
    return out, lse


def sync_check(stream=None) -> None:
    """Synchronises the stream and raises if a kernel flagged an error."""
    _lib.check(_lib.load().zl_sync_check(_stream_handle(stream)), "zl_sync_check")


def launch_count() -> int:
    return int(_lib.load().zl_launch_count())


def profile_begin() -> None:
    """Starts per-kernel event timing of this library's launches."""
    _lib.check(_lib.load().zl_profile_begin(), "zl_profile_begin")


def profile_end() -> dict:
    """Stops timing; returns {kernel name: (launches, total device ms)}."""
    lib = _lib.load()
    arr = (_lib.ProfileEntry * 32)()
    n = ctypes.c_int32(0)
    _lib.check(lib.zl_profile_end(arr, 32, ctypes.byref(n)), "zl_profile_end")
    return {arr[i].name.decode(): (int(arr[i].launches), float(arr[i].total_ms)) for i in range(n.value)}

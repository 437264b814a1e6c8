"""GB300-native coalesced varlen attention (sm_103a).

The compute lives in libzl_attn.so (C ABI: include/zl_attn.h); this package
holds its sources (csrc/), the build step (build.py) and a thin PyTorch-facing
binding (attention.py).
"""
from .attention import (  # noqa: F401
    alloc_workspace, bwd_schedule, bwd_workspace_bytes, fwd_schedule, fwd_workspace_bytes, launch_count, lse_merge,
    profile_begin, profile_end, sync_check, varlen_attn_bwd, varlen_attn_fwd,
)
from ._lib import ZlError, load  # noqa: F401

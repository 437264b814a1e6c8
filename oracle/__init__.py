"""Float64 CPU oracle (test infrastructure only; see attn_f64)."""
from .attn_f64 import (  # noqa: F401
    ROW_BLOCK, attention_f64, attention_rows, attention_bwd_f64, default_scale,
    dkdv_rows, dq_rows, grad_k, grad_q, grad_scores, grad_v, grads_one_query_row, lse_merge, probabilities,
    row_logsumexp, scores, tile_heads, tile_partial, tiled_attn_fwd,
    varlen_attn_bwd, varlen_attn_fwd,
)

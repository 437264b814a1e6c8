"""The binding's host-side checks (no GPU needed: every check runs before
the first CUDA call).  The C ABI receives pointers only, so the binding
refuses tensors whose shape, dtype or row count disagree with the batch."""
import pytest
import torch

import mixed_length_dit_gb300 as zl


def _t(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


CU_Q = [0, 100, 160]
CU_K = [0, 90, 200]


@pytest.mark.parametrize("q,k,v,match", [
    (_t(150, 2, 64), _t(200, 2, 64), _t(200, 2, 64), "q has 150 rows"),
    (_t(160, 2, 64), _t(208, 2, 64), _t(208, 2, 64), "k must be"),
    (_t(160, 2, 64), _t(200, 1, 64), _t(200, 1, 64), "k must be"),
    (_t(160, 2, 64), _t(200, 2, 64), _t(200, 2, 32), "v must be"),
    (_t(160, 2, 64), _t(200, 2, 64), _t(200, 2, 64, dtype=torch.float32), "v must be"),
    (_t(160, 128), _t(200, 2, 64), _t(200, 2, 64), r"q must be \[Tq, H, d\]"),
])
def test_forward_refuses_inputs_that_disagree_with_the_batch(q, k, v, match):
    with pytest.raises(ValueError, match=match):
        zl.varlen_attn_fwd(q, k, v, CU_Q, CU_K)


def test_forward_refuses_outputs_that_disagree_with_the_batch():
    q, k, v = _t(160, 2, 64), _t(200, 2, 64), _t(200, 2, 64)
    with pytest.raises(ValueError, match="out must be"):
        zl.varlen_attn_fwd(q, k, v, CU_Q, CU_K, out=_t(100, 2, 64), lse=_t(2, 160, dtype=torch.float32))
    with pytest.raises(ValueError, match="lse must be"):
        zl.varlen_attn_fwd(q, k, v, CU_Q, CU_K, out=_t(160, 2, 64), lse=_t(160, 2, dtype=torch.float32))
    # shapes right: host tensors are refused for not being on the GPU
    with pytest.raises(ValueError, match="CUDA tensor"):
        zl.varlen_attn_fwd(q, k, v, CU_Q, CU_K, out=_t(160, 2, 64), lse=_t(2, 160, dtype=torch.float32))


@pytest.mark.parametrize("name,kw,match", [
    ("o", {"o": _t(100, 2, 64)}, "o must be"),
    ("dout", {"dout": _t(160, 2, 32)}, "dout must be"),
    ("lse", {"lse": _t(160, 2, dtype=torch.float32)}, "lse must be"),
    ("dq", {"dq": _t(160, 2, 64, dtype=torch.float32)}, "dq must be"),
    ("dk", {"dk": _t(160, 2, 64)}, "dk must be"),
    ("dv", {"dv": _t(201, 2, 64)}, "dv must be"),
])
def test_backward_refuses_tensors_that_disagree_with_the_batch(name, kw, match):
    args = {"q": _t(160, 2, 64), "k": _t(200, 2, 64), "v": _t(200, 2, 64), "o": _t(160, 2, 64),
            "lse": _t(2, 160, dtype=torch.float32), "dout": _t(160, 2, 64)}
    extra = {}
    for key, val in kw.items():
        (args if key in args else extra)[key] = val
    with pytest.raises(ValueError, match=match):
        zl.varlen_attn_bwd(args["q"], args["k"], args["v"], args["o"], args["lse"], args["dout"], CU_Q, CU_K,
                           **extra)


def test_merge_refuses_partials_that_disagree():
    part = torch.zeros((2, 16, 2, 64))
    with pytest.raises(ValueError, match="lse_partial must be"):
        zl.lse_merge(part, torch.zeros((2, 16, 2)))
    with pytest.raises(ValueError, match="rows must lie"):
        zl.lse_merge(part, torch.zeros((2, 2, 16)), rows=17)
    with pytest.raises(ValueError, match="o_partial must be"):
        zl.lse_merge(part.to(torch.float64), torch.zeros((2, 2, 16)))

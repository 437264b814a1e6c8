"""Shared helpers for the parity tests (no attention arithmetic here)."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances against the float64 oracle (stated for this method: bf16 output
# max-abs 2e-2, LSE 1e-3, gradients relative L2 2e-2, float32 mode 1e-4).
TOL_O_BF16 = 2e-2
TOL_LSE = 1e-3
TOL_GRAD_REL_L2 = 2e-2
TOL_FP32 = 1e-4


def cuda_ok() -> bool:
    return torch.cuda.is_available()


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def cu_from_lens(lens):
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + int(n))
    return cu


def sample_rows(length: int, chunks, n_random: int, rng) -> np.ndarray:
    """Rows of one sequence to check: the first and last row of every chunk,
    the rows around every 128-row block edge inside the first chunk, and
    n_random random rows."""
    rows = set()
    for a, n in chunks:
        if n > 0:
            rows.update({a, a + n - 1, min(a + n - 1, a + 127), min(a + n - 1, a + 128)})
    rows.update(int(x) for x in rng.integers(0, length, size=min(n_random, length)))
    return np.array(sorted(r for r in rows if 0 <= r < length), dtype=np.int64)


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))

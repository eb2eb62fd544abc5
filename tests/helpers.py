"""Shared helpers of the GPU parity tests (no method arithmetic here)."""

import numpy as np
import torch


def to_np(t: torch.Tensor) -> np.ndarray:
    """Exact fp64 copy of a CPU/GPU tensor (bf16 and fp32 upcast exactly)."""
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def sample_rows(BH: int, L: int, n: int, seed: int):
    """(head, t) pairs: first and last token of some heads plus random ones."""
    rng = np.random.default_rng(seed)
    picks = {(0, 0), (BH - 1, L - 1), (0, L - 1), (BH - 1, 0), (BH // 2, min(L - 1, 127)),
             (BH // 2, min(L - 1, 128))}
    while len(picks) < n:
        picks.add((int(rng.integers(BH)), int(rng.integers(L))))
    return sorted(picks)


TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}

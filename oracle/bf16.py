"""bf16 rounding used at the oracle's rounding points (test infrastructure only).

The pages' models are bf16 checkpoints trained in bf16 ("Soup: Fine-Tuning an
8B LLM ...", "Known Limitations and Failure Modes": adapters are created in the
checkpoint dtype).  Wherever the oracle's layer definition says a tensor is
bf16, it is rounded here: round-to-nearest, ties to even, taken directly from
the float64 value (one rounding).  Values stay inside the float32 normal range
in every workload, where bf16 and this rounding agree.
"""
import numpy as np


def round_bf16(x) -> np.ndarray:
    """Nearest bf16 value (ties to even) of x; returned as float64."""
    d = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    u = d.view(np.uint64)
    # bf16 keeps 7 of float64's 52 fraction bits: drop the low 45 with RNE.
    keep = (u >> np.uint64(45)) & np.uint64(1)
    r = ((u + np.uint64((1 << 44) - 1) + keep) >> np.uint64(45)) << np.uint64(45)
    out = r.view(np.float64)
    big = np.abs(d) >= 3.3895313892515355e38  # beyond the largest finite bf16
    if np.any(big) or np.any(~np.isfinite(d)):
        out = np.where(np.isfinite(d) & ~big, out, np.where(np.isnan(d), d, np.copysign(np.inf, d)))
    return out

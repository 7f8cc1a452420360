"""bf16 rounding used at the oracle's rounding points (test infrastructure only).

The pages' models are bf16 checkpoints trained in bf16 ("Soup: Fine-Tuning an
8B LLM ...", "Known Limitations and Failure Modes": adapters are created in the
checkpoint dtype).  Wherever the oracle's layer definition says a tensor is
bf16, it is rounded here: round-to-nearest, ties to even, taken directly from
the float64 value (one rounding), in the bfloat16 format (8 exponent bits as
float32, 7 fraction bits, gradual underflow below 2^-126, overflow to
infinity from the midpoint above the largest finite value (2 - 2^-7) 2^127).
"""
import numpy as np

_MIN_NORMAL = 2.0 ** -126      # smallest normal bf16 (as float32)
_SUB_STEP = 2.0 ** -133        # spacing of the bf16 subnormals
_OVERFLOW = 2.0 ** 128         # first value past the largest finite bf16


def round_bf16(x) -> np.ndarray:
    """Nearest bf16 value (ties to even) of x; returned as float64."""
    d = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    u = d.view(np.uint64)
    # Normal range: bf16 keeps 7 of float64's 52 fraction bits; drop the low
    # 45 with round-to-nearest-even (a carry moves into the next binade).
    keep = (u >> np.uint64(45)) & np.uint64(1)
    r = ((u + np.uint64((1 << 44) - 1) + keep) >> np.uint64(45)) << np.uint64(45)
    out = r.view(np.float64).copy()
    # Below the smallest normal the step is fixed; scaling by a power of two is
    # exact, and np.round takes ties to even.
    tiny = np.abs(d) < _MIN_NORMAL
    if np.any(tiny):
        out[tiny] = np.round(d[tiny] / _SUB_STEP) * _SUB_STEP
    # A value whose rounding reaches 2^128 overflows; NaN stays NaN.
    over = np.isfinite(d) & (np.abs(out) >= _OVERFLOW)
    if np.any(over):
        out[over] = np.copysign(np.inf, d[over])
    nan = np.isnan(d)
    if np.any(nan):
        out[nan] = d[nan]
    return out

"""LoRA linear on a frozen base, forward and backward -- oracle (test infrastructure only).

The method ("Exact Layer Streaming ...", abstract: LoRA fine-tuning with a
frozen, NF4-quantised base; "Soup: Fine-Tuning ...", "Layer Streaming: The
Mechanism Behind the 4 GB Claim": the frozen base never receives an optimizer
step) trains only the adapters A [r, K] and B [N, r] of each frozen linear

    Y = X W^T + s (X A^T) B^T,      s = alpha / r,

the PEFT convention the pages' tool is built on.  The frozen weight W is either
the bf16 dequantisation of the NF4 base or a bf16 base kept in its storage
dtype ("The FP32 Bug and What It Means for Your VRAM").  No bias, no dropout
(the pages name neither).

Backward, for an upstream gradient dY (plain calculus of the line above):

    U  = dY B                  [M, r]
    dX = dY W + s U A          [M, K]
    dA = s U^T X               [r, K]
    dB = s dY^T (X A^T)        [N, r]

All arithmetic here is float64 on the given (bf16-exact) inputs.  The adapter
gradients are reported in fp32 by the library ("Known Limitations and Failure
Modes": the GradScaler needs fp32 adapter gradients); the oracle keeps them in
float64.
"""
import numpy as np


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


def lora_linear_fwd(X, W, A=None, B=None, alpha: float = 0.0):
    """Y = X W^T + (alpha/r) (X A^T) B^T; r = 0 (A or B None) gives the base alone."""
    X, W, A, B = _f64(X), _f64(W), _f64(A), _f64(B)
    Y = X @ W.T
    if A is not None and B is not None and A.shape[0] > 0:
        s = alpha / A.shape[0]
        Y = Y + s * ((X @ A.T) @ B.T)
    return Y


def lora_linear_bwd(X, dY, W, A=None, B=None, alpha: float = 0.0):
    """(dX, dA, dB) of the linear above; dA, dB are None when there is no adapter."""
    X, dY, W, A, B = _f64(X), _f64(dY), _f64(W), _f64(A), _f64(B)
    dX = dY @ W
    if A is None or B is None or A.shape[0] == 0:
        return dX, None, None
    s = alpha / A.shape[0]
    U = dY @ B
    dX = dX + s * (U @ A)
    dA = s * (U.T @ X)
    dB = s * (dY.T @ (X @ A.T))
    return dX, dA, dB

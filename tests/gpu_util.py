"""Helpers shared by the GPU tests: upload seeded numpy inputs, compare against the oracle."""
import numpy as np
import torch


def dev_bf16(x):
    """float32 array of bf16-exact values -> CUDA bf16 tensor (exact)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to("cuda").to(torch.bfloat16)


def host(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_fro(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return np.linalg.norm(got - ref) / (den if den > 0 else 1.0)


BF16_TOL = 1e-2   # relative Frobenius bound for bf16 outputs and all gradients
LOSS_TOL = 1e-3   # relative bound for the fp32 loss

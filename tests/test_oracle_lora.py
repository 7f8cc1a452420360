"""Pins for the LoRA-linear oracle: zero-adapter identities, finite differences, library autograd."""
import numpy as np
import torch

from oracle import lora


def _case(seed, M=5, N=6, K=7, r=3):
    g = np.random.default_rng(seed)
    return (g.standard_normal((M, K)), g.standard_normal((N, K)), g.standard_normal((r, K)),
            g.standard_normal((N, r)), g.standard_normal((M, N)))


def test_zero_B_and_rank_zero_give_base_exactly():
    X, W, A, B, dY = _case(0)
    base = X @ W.T
    assert np.array_equal(lora.lora_linear_fwd(X, W, A, np.zeros_like(B), 16.0), base)
    assert np.array_equal(lora.lora_linear_fwd(X, W, None, None, 16.0), base)
    dX, dA, dB = lora.lora_linear_bwd(X, dY, W, A, np.zeros_like(B), 16.0)
    assert np.array_equal(dX, dY @ W) and np.all(dA == 0) and np.any(dB != 0)


def test_finite_differences():
    X, W, A, B, dY = _case(1)
    alpha = 6.0
    loss = lambda X_, A_, B_: float(np.sum(lora.lora_linear_fwd(X_, W, A_, B_, alpha) * dY))
    dX, dA, dB = lora.lora_linear_bwd(X, dY, W, A, B, alpha)
    h = 1e-6
    for name, arr, grad in (("X", X, dX), ("A", A, dA), ("B", B, dB)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += h
            m[idx] -= h
            args = {"X": (X, A, B), "A": (X, A, B), "B": (X, A, B)}[name]
            ap = [p if n == name else v for n, v in zip("XAB", args)]
            am = [m if n == name else v for n, v in zip("XAB", args)]
            num[idx] = (loss(*ap) - loss(*am)) / (2 * h)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-7)


def test_matches_torch_autograd():
    X, W, A, B, dY = _case(2, M=9, N=11, K=13, r=4)
    alpha = 8.0
    tX, tA, tB = (torch.tensor(a, requires_grad=True) for a in (X, A, B))
    tW = torch.tensor(W)
    y = torch.nn.functional.linear(tX, tW) + (alpha / 4) * torch.nn.functional.linear(
        torch.nn.functional.linear(tX, tA), tB)
    y.backward(torch.tensor(dY))
    np.testing.assert_allclose(lora.lora_linear_fwd(X, W, A, B, alpha), y.detach().numpy(), rtol=1e-12)
    dX, dA, dB = lora.lora_linear_bwd(X, dY, W, A, B, alpha)
    np.testing.assert_allclose(dX, tX.grad.numpy(), rtol=1e-12)
    np.testing.assert_allclose(dA, tA.grad.numpy(), rtol=1e-12)
    np.testing.assert_allclose(dB, tB.grad.numpy(), rtol=1e-12)


def test_scale_is_alpha_over_rank():
    """The adapter scale is s = alpha / r (the PEFT convention the pages' tool follows): padding A and B
    with zero ranks while scaling alpha alike changes nothing, which fails for s = alpha or
    s = alpha / sqrt(r); and one hand-sized case gives the value computed by hand."""
    X, W, A, B, dY = _case(3, r=3)
    A2, B2 = np.vstack([A, np.zeros_like(A)]), np.hstack([B, np.zeros_like(B)])
    np.testing.assert_allclose(lora.lora_linear_fwd(X, W, A2, B2, 12.0), lora.lora_linear_fwd(X, W, A, B, 6.0),
                               rtol=1e-13)
    dX, dA, dB = lora.lora_linear_bwd(X, dY, W, A, B, 6.0)
    dX2, dA2, dB2 = lora.lora_linear_bwd(X, dY, W, A2, B2, 12.0)
    np.testing.assert_allclose(dX2, dX, rtol=1e-13)
    np.testing.assert_allclose(dA2[:3], dA, rtol=1e-13)
    np.testing.assert_allclose(dB2[:, :3], dB, rtol=1e-13)
    assert np.all(dA2[3:] == 0) and np.all(dB2[:, 3:] == 0)
    # X A^T = [1, 2], (X A^T) B^T = 3, s = 4 / 2 = 2: Y = 6 on a zero base
    X1, W1 = np.array([[1.0, 2.0]]), np.zeros((1, 2))
    A1, B1 = np.eye(2), np.array([[1.0, 1.0]])
    assert lora.lora_linear_fwd(X1, W1, A1, B1, 4.0)[0, 0] == 6.0

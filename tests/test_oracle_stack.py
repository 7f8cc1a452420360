"""Pins for the synthetic decoder layer / stack oracle."""
import numpy as np
import torch

from oracle import stack
from oracle.bf16 import round_bf16


def _layers(seed, L, D, Dkv, F, r, std=0.05):
    g = np.random.default_rng(seed)
    shapes = [("q", D, D), ("k", Dkv, D), ("v", Dkv, D), ("o", D, D),
              ("gate", F, D), ("up", F, D), ("down", D, F)]
    return [{n: dict(W=g.standard_normal((N, K)) * std, A=g.standard_normal((r, K)) * std,
                     B=g.standard_normal((N, r)) * std) for n, N, K in shapes} for _ in range(L)]


def _torch_step(h0, dh_top, layers, alpha):
    """The same layer written with torch float64 autograd (library differentiation)."""
    h = torch.tensor(h0, requires_grad=True)
    params = []
    x = h
    for P in layers:
        def lin(z, n):
            A = torch.tensor(P[n]["A"], requires_grad=True)
            B = torch.tensor(P[n]["B"], requires_grad=True)
            params.append((A, B))
            r = A.shape[0]
            return z @ torch.tensor(P[n]["W"]).T + (alpha / r) * (z @ A.T) @ B.T
        rms = lambda z: z / torch.sqrt(torch.mean(z * z, dim=1, keepdim=True) + 1e-5)
        D = x.shape[1]
        x1 = rms(x)
        q, k, v = lin(x1, "q"), lin(x1, "k"), lin(x1, "v")
        g = D // k.shape[1]
        rep = lambda t: t.reshape(t.shape[0], -1, 1, 128).expand(-1, -1, g, -1).reshape(t.shape[0], D)
        a = q * rep(k) + rep(v)
        h1 = x + lin(a, "o")
        x2 = rms(h1)
        m = torch.nn.functional.silu(lin(x2, "gate")) * lin(x2, "up")
        x = h1 + lin(m, "down")
    x.backward(torch.tensor(dh_top))
    return x.detach().numpy(), h.grad.numpy(), params


def test_unrounded_step_matches_torch_autograd():
    L, M, D, Dkv, F, r = 2, 3, 256, 128, 384, 2
    layers = _layers(0, L, D, Dkv, F, r)
    g = np.random.default_rng(1)
    h0, dh = g.standard_normal((M, D)), g.standard_normal((M, D))
    hL, dh0, grads = stack.stack_step(h0, dh, layers, alpha=4.0, rnd=False)
    thL, tdh0, params = _torch_step(h0, dh, layers, 4.0)
    np.testing.assert_allclose(hL, thL, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dh0, tdh0, rtol=1e-9, atol=1e-11)
    it = iter(params)
    for l in range(L):
        for n in ("q", "k", "v", "o", "gate", "up", "down"):
            tA, tB = next(it)
            np.testing.assert_allclose(grads[l][n][0], tA.grad.numpy(), rtol=1e-9, atol=1e-12)
            np.testing.assert_allclose(grads[l][n][1], tB.grad.numpy(), rtol=1e-9, atol=1e-12)


def test_unrounded_step_finite_difference_on_h0():
    L, M, D, Dkv, F, r = 2, 2, 256, 128, 256, 2
    layers = _layers(3, L, D, Dkv, F, r)
    g = np.random.default_rng(4)
    h0, dh = g.standard_normal((M, D)), g.standard_normal((M, D))
    _, dh0, _ = stack.stack_step(h0, dh, layers, alpha=4.0, rnd=False)
    eps = 1e-6
    for idx in [(0, 0), (1, 17), (0, 200)]:
        p, m = h0.copy(), h0.copy()
        p[idx] += eps
        m[idx] -= eps
        fp = np.sum(stack.stack_step(p, dh, layers, 4.0, rnd=False)[0] * dh)
        fm = np.sum(stack.stack_step(m, dh, layers, 4.0, rnd=False)[0] * dh)
        assert abs((fp - fm) / (2 * eps) - dh0[idx]) <= 1e-6 * max(1.0, abs(dh0[idx]))


def test_rms_of_constant_row_and_rep_adjoint():
    h = np.full((1, 256), -3.0)
    y, r = stack.rms_fwd(h)
    np.testing.assert_allclose(y, -3.0 / np.sqrt(9.0 + 1e-5), rtol=1e-15)
    g = np.random.default_rng(2)
    kv, x = g.standard_normal((3, 256)), g.standard_normal((3, 1024))
    # <rep(kv), x> == <kv, rep_sum(x)>
    assert abs(np.sum(stack.rep(kv, 1024) * x) - np.sum(kv * stack.rep_sum(x, 256))) < 1e-10
    # head 5 of q (group 4) reads kv head 1
    np.testing.assert_array_equal(stack.rep(kv, 1024)[:, 5 * 128:6 * 128], kv[:, 128:256])


def test_rounding_points_are_bf16():
    L, M, D, Dkv, F, r = 1, 2, 256, 128, 256, 2
    layers = _layers(5, L, D, Dkv, F, r)
    g = np.random.default_rng(6)
    h0 = g.standard_normal((M, D))
    _, c = stack.layer_forward(h0, layers[0], 4.0, rnd=True)
    for key in ("x1", "q", "k", "v", "a", "x2", "g", "u", "m"):
        assert np.array_equal(round_bf16(c[key]), c[key]), key
    # rounded and unrounded runs stay close (bf16 has 8 significant bits)
    hr, _, _ = stack.stack_step(h0, h0, layers, 4.0, rnd=True)
    hu, _, _ = stack.stack_step(h0, h0, layers, 4.0, rnd=False)
    assert np.linalg.norm(hr - hu) / np.linalg.norm(hu) < 2e-2

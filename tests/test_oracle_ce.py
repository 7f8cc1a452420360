"""Pins for the cross-entropy oracle."""
import math

import numpy as np
import torch

from oracle import ce


def test_matches_torch_cross_entropy():
    g = np.random.default_rng(0)
    M, D, V = 37, 19, 53
    H, W = g.standard_normal((M, D)), g.standard_normal((V, D)) * 0.3
    lab = g.integers(0, V, M)
    lab[[3, 9, 30]] = -100
    loss, dH = ce.ce_fwd_bwd(H, W, lab)
    tH = torch.tensor(H, requires_grad=True)
    tl = torch.nn.functional.cross_entropy(tH @ torch.tensor(W).T, torch.tensor(lab), ignore_index=-100)
    tl.backward()
    assert abs(loss - tl.item()) <= 1e-12 * abs(loss)
    np.testing.assert_allclose(dH, tH.grad.numpy(), rtol=1e-10, atol=1e-14)
    assert np.all(dH[[3, 9, 30]] == 0)


def test_brute_force_small_vocab():
    g = np.random.default_rng(1)
    M, D, V = 6, 3, 7
    H, W = g.standard_normal((M, D)), g.standard_normal((V, D))
    lab = np.array([0, 6, 3, -100, 2, 5])
    loss, dH = ce.ce_fwd_bwd(H, W, lab)
    nv = 5
    tot = 0.0
    ref = np.zeros((M, D))
    for i in range(M):
        if lab[i] == -100:
            continue
        z = [sum(H[i, d] * W[v, d] for d in range(D)) for v in range(V)]
        s = sum(math.exp(t) for t in z)
        tot += math.log(s) - z[lab[i]]
        for d in range(D):
            ref[i, d] = sum((math.exp(z[v]) / s - (v == lab[i])) * W[v, d] for v in range(V)) / nv
    assert abs(loss - tot / nv) < 1e-12
    np.testing.assert_allclose(dH, ref, rtol=1e-10, atol=1e-14)


def test_two_class_sigmoid_and_uniform_logits():
    # V = 2, D = 1: loss = softplus(z_other - z_label)
    H = np.array([[1.5], [-0.7]])
    W = np.array([[0.4], [-1.1]])
    lab = np.array([0, 1])
    loss, _ = ce.ce_fwd_bwd(H, W, lab)
    z = H @ W.T
    sp = lambda t: math.log1p(math.exp(t))
    assert abs(loss - (sp(z[0, 1] - z[0, 0]) + sp(z[1, 0] - z[1, 1])) / 2) < 1e-14
    # all-equal logits: loss = log V, and the softmax term is the mean head row
    V, D = 11, 4
    W = np.tile(np.arange(1, D + 1, dtype=float), (V, 1)) * 0.0 + 0.25
    H = np.ones((3, D))
    loss, dH = ce.ce_fwd_bwd(H, W, np.array([1, 2, 3]))
    assert abs(loss - math.log(V)) < 1e-13
    np.testing.assert_allclose(dH, 0.0, atol=1e-15)


def test_dlogit_rows_sum_to_zero_and_no_valid_rows():
    g = np.random.default_rng(3)
    H, W = g.standard_normal((4, 5)), g.standard_normal((9, 5))
    lab = np.array([1, 2, 3, 4])
    # with W = I-like probe the dH rows are the dlogit rows
    terms, dH, soft = ce.ce_rows(H, np.eye(9)[:, :5] @ np.eye(5), lab, 4, want_soft=True)
    Z = H @ (np.eye(9)[:, :5]).T
    P = np.exp(Z - Z.max(1, keepdims=True))
    P /= P.sum(1, keepdims=True)
    G = P.copy()
    G[np.arange(4), lab] -= 1
    np.testing.assert_allclose(G.sum(1), 0, atol=1e-15)
    loss, dH = ce.ce_fwd_bwd(H, W, np.full(4, -100))
    assert loss == 0.0 and np.all(dH == 0)

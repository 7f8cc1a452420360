"""Pins for the attention / rotary-position / weighted-norm oracle and the attention layer.

Independent checks: torch's float64 scaled_dot_product_attention (causal,
grouped-query) and autograd, torch's rms_norm, closed forms (uniform
attention is a running mean with lse = log(count); position 0 rotates
nothing; a rotation by a known angle), invariants (rotations keep norms and
compose to the identity with their inverse; scores depend on relative
positions only) and finite differences.
"""
import math

import numpy as np
import torch
import torch.nn.functional as Fn

from oracle import attention as at
from oracle import stack

D, DKV = 512, 256          # H = 4 query heads, Hkv = 2 kv heads (group 2)


def _qkv(seed, M, D=D, Dkv=DKV, std=1.0):
    g = np.random.default_rng(seed)
    return g.standard_normal((M, D)) * std, g.standard_normal((M, Dkv)) * std, g.standard_normal((M, Dkv))


def _torch_attn(q, k, v, S):
    """torch SDPA over [nseq, heads, S, 128] views of the row-major inputs."""
    M = q.shape[0]
    to = lambda x: x.reshape(M // S, S, -1, 128).transpose(1, 2)
    o = Fn.scaled_dot_product_attention(to(q), to(k), to(v), is_causal=True, enable_gqa=True,
                                        scale=1.0 / math.sqrt(128))
    return o.transpose(1, 2).reshape(M, -1)


def test_forward_and_backward_match_torch_sdpa_autograd():
    S, M = 24, 48                                     # two sequences
    q, k, v = _qkv(1, M, std=0.3)
    o, lse = at.attention_fwd(q, k, v, S)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    to = _torch_attn(tq, tk, tv, S)
    np.testing.assert_allclose(o, to.detach().numpy(), rtol=1e-12, atol=1e-13)
    do = np.random.default_rng(2).standard_normal(o.shape)
    to.backward(torch.tensor(do))
    dq, dk, dv = at.attention_bwd(q, k, v, o, do, S)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert lse.shape == (M, D // 128)


def test_uniform_attention_is_a_running_mean():
    S, M = 16, 32
    _, k, v = _qkv(3, M)
    q = np.zeros((M, D))                              # every score 0: uniform over the visible keys
    o, lse = at.attention_fwd(q, k, v, S)
    pos = np.arange(M) % S
    np.testing.assert_allclose(lse, np.log(pos + 1.0)[:, None].repeat(D // 128, axis=1), rtol=1e-14)
    for t in range(M):
        s0 = t - pos[t]
        mean = v[s0:t + 1].mean(axis=0)               # [Dkv]
        for h in range(D // 128):
            g = h // (D // DKV)
            np.testing.assert_allclose(o[t, h * 128:(h + 1) * 128], mean[g * 128:(g + 1) * 128], rtol=1e-12,
                                       atol=1e-14)


def test_first_token_of_each_sequence_copies_its_value():
    S, M = 8, 24
    q, k, v = _qkv(4, M)
    o, _ = at.attention_fwd(q, k, v, S)
    for t in range(0, M, S):
        for h in range(D // 128):
            g = h // (D // DKV)
            np.testing.assert_allclose(o[t, h * 128:(h + 1) * 128], v[t, g * 128:(g + 1) * 128], rtol=1e-14)


def test_backward_finite_difference():
    S, M = 6, 12
    q, k, v = _qkv(5, M, std=0.5)
    o, _ = at.attention_fwd(q, k, v, S)
    do = np.random.default_rng(6).standard_normal(o.shape)
    grads = at.attention_bwd(q, k, v, o, do, S)
    eps = 1e-6
    for which, idx in ((0, (3, 130)), (0, (11, 5)), (1, (2, 77)), (1, (7, 200)), (2, (4, 3)), (2, (9, 255))):
        xs = [q.copy(), k.copy(), v.copy()]
        xs[which][idx] += eps
        fp = np.sum(at.attention_fwd(*xs, S)[0] * do)
        xs[which][idx] -= 2 * eps
        fm = np.sum(at.attention_fwd(*xs, S)[0] * do)
        fd = (fp - fm) / (2 * eps)
        assert abs(fd - grads[which][idx]) <= 1e-6 * max(1.0, abs(fd)), (which, idx)


def test_rope_identity_at_zero_known_angles_and_inverse():
    S, theta = 40, 10000.0
    x = np.zeros((S, 256))
    x[:, 0] = 1.0                                      # pair (0, 64): frequency theta^0 = 1
    x[:, 128 + 32] = 1.0                               # pair (32, 96) of head 1: frequency theta^(-1/2) = 0.01
    y = at.rope(x, S, theta)
    np.testing.assert_array_equal(y[0], x[0])          # position 0 rotates nothing
    for p in (1, 7, 39):
        assert abs(y[p, 0] - math.cos(p)) < 1e-15 and abs(y[p, 64] - math.sin(p)) < 1e-15
        assert abs(y[p, 160] - math.cos(0.01 * p)) < 1e-15 and abs(y[p, 224] - math.sin(0.01 * p)) < 1e-15
    z = np.random.default_rng(7).standard_normal((2 * S, 512))
    r = at.rope(z, S, 500000.0)
    np.testing.assert_allclose(at.rope(r, S, 500000.0, inverse=True), z, rtol=1e-13, atol=1e-13)
    pn = lambda a: a.reshape(2 * S, 4, 2, 64)[:, :, 0] ** 2 + a.reshape(2 * S, 4, 2, 64)[:, :, 1] ** 2
    np.testing.assert_allclose(pn(r), pn(z), rtol=1e-12)


def test_rope_scores_depend_on_relative_position_only():
    S, theta = 64, 500000.0
    g = np.random.default_rng(8)
    qv, kv = g.standard_normal(128), g.standard_normal(128)
    X = np.zeros((S, 128))
    Q = at.rope(X + qv, S, theta)
    K = at.rope(X + kv, S, theta)
    for m, n, t in ((5, 2, 17), (30, 30, 9), (40, 1, 20)):
        np.testing.assert_allclose(Q[m] @ K[n], Q[m + t] @ K[n + t], rtol=1e-11)


def test_weighted_rms_matches_torch_rms_norm_autograd():
    g = np.random.default_rng(9)
    h, w, dy = g.standard_normal((5, 256)), g.standard_normal(256), g.standard_normal((5, 256))
    y, r = stack.rms_fwd(h)
    th = torch.tensor(h, requires_grad=True)
    ty = Fn.rms_norm(th, (256,), weight=torch.tensor(w), eps=1e-5)
    np.testing.assert_allclose(y * w, ty.detach().numpy(), rtol=1e-13)
    ty.backward(torch.tensor(dy))
    np.testing.assert_allclose(stack.rms_bwd(y, r, dy, w), th.grad.numpy(), rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(stack.rms_bwd(y, r, dy, np.ones(256)), stack.rms_bwd(y, r, dy), rtol=1e-15)


def _layers(seed, L, Dm, Dkv, F, r, std=0.05):
    g = np.random.default_rng(seed)
    shapes = [("q", Dm, Dm), ("k", Dkv, Dm), ("v", Dkv, Dm), ("o", Dm, Dm),
              ("gate", F, Dm), ("up", F, Dm), ("down", Dm, F)]
    out = []
    for _ in range(L):
        P = {n: dict(W=g.standard_normal((N, K)) * std, A=g.standard_normal((r, K)) * std,
                     B=g.standard_normal((N, r)) * std) for n, N, K in shapes}
        P["norm_attn"] = 1.0 + 0.1 * g.standard_normal(Dm)
        P["norm_mlp"] = 1.0 + 0.1 * g.standard_normal(Dm)
        out.append(P)
    return out


def _torch_attn_step(h0, dh_top, layers, alpha, S, theta):
    """The attention layer with torch float64 autograd: torch SDPA and rms_norm; the
    rotation through rope() of the oracle (pinned above) applied to torch tensors."""
    cos, sin = (torch.tensor(a) for a in at.rope_cos_sin(S, theta))

    def trope(x):
        M, W = x.shape
        c, s = cos[torch.arange(M) % S][:, None, :], sin[torch.arange(M) % S][:, None, :]
        xh = x.reshape(M, W // 128, 128)
        return torch.cat([xh[..., :64] * c - xh[..., 64:] * s, xh[..., 64:] * c + xh[..., :64] * s], 2).reshape(M, W)

    h = torch.tensor(h0, requires_grad=True)
    params, x = [], h
    for P in layers:
        def lin(z, n):
            A = torch.tensor(P[n]["A"], requires_grad=True)
            B = torch.tensor(P[n]["B"], requires_grad=True)
            params.append((A, B))
            return z @ torch.tensor(P[n]["W"]).T + (alpha / A.shape[0]) * (z @ A.T) @ B.T
        Dm = x.shape[1]
        x1 = Fn.rms_norm(x, (Dm,), weight=torch.tensor(P["norm_attn"]), eps=1e-5)
        q, k, v = lin(x1, "q"), lin(x1, "k"), lin(x1, "v")
        a = _torch_attn(trope(q), trope(k), v, S)
        h1 = x + lin(a, "o")
        x2 = Fn.rms_norm(h1, (Dm,), weight=torch.tensor(P["norm_mlp"]), eps=1e-5)
        x = h1 + lin(Fn.silu(lin(x2, "gate")) * lin(x2, "up"), "down")
    x.backward(torch.tensor(dh_top))
    return x.detach().numpy(), h.grad.numpy(), params


def test_attention_stack_matches_torch_autograd():
    L, S, M, Dm, Dkv, F, r = 2, 5, 10, 256, 128, 256, 2
    attn = dict(S=S, theta=500000.0)
    layers = _layers(10, L, Dm, Dkv, F, r)
    g = np.random.default_rng(11)
    h0, dh = g.standard_normal((M, Dm)), g.standard_normal((M, Dm))
    hL, dh0, grads = stack.stack_step(h0, dh, layers, 4.0, rnd=False, attn=attn)
    thL, tdh0, params = _torch_attn_step(h0, dh, layers, 4.0, S, 500000.0)
    np.testing.assert_allclose(hL, thL, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dh0, tdh0, rtol=1e-9, atol=1e-11)
    it = iter(params)
    for l in range(L):
        for n in ("q", "k", "v", "o", "gate", "up", "down"):
            tA, tB = next(it)
            np.testing.assert_allclose(grads[l][n][0], tA.grad.numpy(), rtol=1e-9, atol=1e-12)
            np.testing.assert_allclose(grads[l][n][1], tB.grad.numpy(), rtol=1e-9, atol=1e-12)


def test_sft_step_matches_torch_autograd():
    """Embedding rows, the attention stack, the final weighted norm and the mean CE (ignore -100)."""
    L, S, M, Dm, Dkv, F, r, V = 1, 4, 8, 256, 128, 256, 2, 50
    attn = dict(S=S, theta=10000.0)
    layers = _layers(12, L, Dm, Dkv, F, r)
    g = np.random.default_rng(13)
    embed, W_head = g.standard_normal((V, Dm)), g.standard_normal((V, Dm)) * 0.05
    nf = 1.0 + 0.1 * g.standard_normal(Dm)
    tokens = g.integers(0, V, M)
    labels = g.integers(0, V, M)
    labels[[2, 5]] = -100
    loss, dh0, grads = stack.sft_step(tokens, labels, embed, layers, nf, W_head, 4.0, rnd=False, attn=attn)
    h0 = embed[tokens]
    # torch: forward through the stack, then the head loss and its gradient at hL
    hL_t, _, _ = _torch_attn_step(h0, np.zeros_like(h0), layers, 4.0, S, 10000.0)
    th = torch.tensor(hL_t, requires_grad=True)
    x = Fn.rms_norm(th, (Dm,), weight=torch.tensor(nf), eps=1e-5)
    tl = Fn.cross_entropy(x @ torch.tensor(W_head).T, torch.tensor(labels), ignore_index=-100)
    tl.backward()
    assert abs(loss - tl.item()) <= 1e-12 * max(1.0, abs(loss))
    # dh_top from torch, pushed through the oracle's own stack backward, equals the sft step's dh0
    _, dh0_ref, grads_ref = stack.stack_step(h0, th.grad.numpy(), layers, 4.0, rnd=False, attn=attn)
    np.testing.assert_allclose(dh0, dh0_ref, rtol=1e-10, atol=1e-13)
    for n in ("q", "o", "down"):
        np.testing.assert_allclose(grads[0][n][0], grads_ref[0][n][0], rtol=1e-10, atol=1e-14)


def _moving_reference_softmax(q, k, v, S, tile, tau):
    """Causal attention of one head group, accumulated tile by tile over the keys
    with a per-row reference maximum m (log2 units) that moves only when a
    tile's maximum exceeds it by more than tau; O and l are rescaled only then.
    Returns (o, lse, the largest P formed)."""
    M, D = q.shape
    group = D // k.shape[1]
    c = math.log2(math.e) / math.sqrt(128)
    o = np.zeros((M, D))
    lse = np.zeros((M, D // 128))
    pmax = 0.0
    for h in range(D // 128):
        g = h // group
        for row in range(M):
            b, pos = divmod(row, S)
            qh = q[row, h * 128:(h + 1) * 128]
            m, l, acc = -math.inf, 0.0, np.zeros(128)
            for t0 in range(0, pos + 1, tile):
                keys = range(b * S + t0, b * S + min(t0 + tile, pos + 1))
                s2 = np.array([qh @ k[j, g * 128:(g + 1) * 128] for j in keys]) * c
                mt = s2.max()
                if mt > m + tau:                       # the reference moves; rescale what was summed
                    alpha = 2.0 ** (m - mt) if m > -math.inf else 0.0
                    acc *= alpha
                    l *= alpha
                    m = mt
                p = 2.0 ** (s2 - m)
                pmax = max(pmax, p.max())
                l += p.sum()
                acc += p @ v[list(keys), g * 128:(g + 1) * 128]
            o[row, h * 128:(h + 1) * 128] = acc / l
            lse[row, h] = (m + math.log2(l)) * math.log(2.0)
    return o, lse, pmax


def test_moving_reference_maximum_reproduces_the_softmax():
    """The forward's reading: P = 2^(s c - m) against a reference m that moves only
    when a key tile's maximum exceeds it by more than 8 gives the softmax's O and
    lse exactly (up to float64 rounding), with every P at most 2^8; with key norms
    growing along the sequence the reference does move."""
    S, M, tile = 64, 128, 16
    g = np.random.default_rng(5)
    grow = (1.0 + np.arange(S) / 4.0)[:, None]
    q = g.standard_normal((M, 256)) * 2.0
    k = g.standard_normal((M, 128)) * np.tile(grow, (M // S, 1))
    v = g.standard_normal((M, 128))
    o_ref, lse_ref = at.attention_fwd(q, k, v, S)
    for tau in (0.0, 8.0):
        o, lse, pmax = _moving_reference_softmax(q, k, v, S, tile, tau)
        np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-10)
        assert pmax <= 2.0 ** tau * (1 + 1e-12)
    # inputs where the lazy reference does lag the true running maximum by up to 8
    _, _, pmax8 = _moving_reference_softmax(q, k, v, S, tile, 8.0)
    assert pmax8 > 2.0

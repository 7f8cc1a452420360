"""Causal grouped-query attention with rotary positions -- oracle (test infrastructure only).

The pages stream whole decoder layers of Llama-3.1-8B and Qwen2.5-3B ("Soup
CLI Lets You Fine-Tune an 8B LLM ...", "How Layer Streaming Works") but never
describe the layer's attention.  The reading taken here is the Llama layout
those model names imply:

* H = D / 128 query heads and Hkv = Dkv / 128 key/value heads of width 128;
  query head h reads kv head h // (H / Hkv);
* the M rows are nseq sequences of S consecutive tokens; positions restart at
  0 in every sequence and a token attends to the tokens of its own sequence
  at positions <= its own (causal);
* rotary position embedding on q and k in the rotate-half form: within a
  head, element i < 64 pairs with element i + 64 and the pair is rotated by
  the angle pos * theta^(-i / 64) (theta 500000 for the Llama-3.1 shape; the
  3.1 release's long-context frequency rescaling is not applied);
* softmax over the scores q . k / sqrt(128).

Float64 throughout; the caller decides where bf16 rounding happens.  The
backward is the plain chain rule of that definition.
"""
import numpy as np

HEAD_DIM = 128
HALF = HEAD_DIM // 2


def rope_cos_sin(S: int, theta: float):
    """cos and sin of the rotation angles, [S, 64] float64: angle[p, i] = p * theta^(-i/64)."""
    inv = np.power(float(theta), -np.arange(HALF, dtype=np.float64) / HALF)
    ang = np.arange(S, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang), np.sin(ang)


def rope(x, S: int, theta: float, inverse: bool = False):
    """Rotate every 128-wide head of x [M, n*128] by its token's position (M % S == 0).

    inverse=True rotates by the negative angle: the transpose of the forward
    rotation, which is what the backward applies to the gradients."""
    x = np.asarray(x, dtype=np.float64)
    M, W = x.shape
    c, s = rope_cos_sin(S, theta)
    pos = np.arange(M) % S
    c, s = c[pos][:, None, :], s[pos][:, None, :]
    if inverse:
        s = -s
    xh = x.reshape(M, W // HEAD_DIM, HEAD_DIM)
    x1, x2 = xh[..., :HALF], xh[..., HALF:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=2).reshape(M, W)


def _heads(x, M, S):
    """[M, n*128] -> [nseq, n, S, 128]."""
    n = x.shape[1] // HEAD_DIM
    return np.asarray(x, dtype=np.float64).reshape(M // S, S, n, HEAD_DIM).transpose(0, 2, 1, 3)


def _rows(x):
    """[nseq, n, S, 128] -> [M, n*128]."""
    nseq, n, S, _ = x.shape
    return x.transpose(0, 2, 1, 3).reshape(nseq * S, n * HEAD_DIM)


def _scores(Q, K, group):
    """Causal scores [nseq, H, S, S] for Q [nseq, H, S, d], K [nseq, Hkv, S, d]; -inf above the diagonal."""
    Kq = np.repeat(K, group, axis=1)
    Z = np.einsum("bhid,bhjd->bhij", Q, Kq) / np.sqrt(HEAD_DIM)
    S = Q.shape[2]
    mask = np.triu(np.ones((S, S), dtype=bool), k=1)
    return np.where(mask, -np.inf, Z)


def attention_fwd(q, k, v, S: int):
    """o [M, D] and the natural-log row normaliser lse [M, H] of causal GQA attention."""
    q = np.asarray(q, dtype=np.float64)
    M, D = q.shape
    Dkv = np.asarray(k).shape[1]
    group = D // Dkv
    Q, K, V = _heads(q, M, S), _heads(k, M, S), _heads(v, M, S)
    Z = _scores(Q, K, group)
    zmax = Z.max(axis=3, keepdims=True)
    lse = zmax + np.log(np.exp(Z - zmax).sum(axis=3, keepdims=True))
    P = np.exp(Z - lse)
    O = np.einsum("bhij,bhjd->bhid", P, np.repeat(V, group, axis=1))
    return _rows(O), lse[..., 0].transpose(0, 2, 1).reshape(M, D // HEAD_DIM)


def attention_bwd(q, k, v, o, do, S: int):
    """(dq, dk, dv) of causal GQA attention given the output o and its gradient do.

    dP = dO V^T, dZ = P * (dP - rowsum(dO * O)), dQ = dZ K / sqrt(d),
    dK = sum over the query heads of a kv head of dZ^T Q / sqrt(d), and
    dV = the same sum of P^T dO."""
    q = np.asarray(q, dtype=np.float64)
    M, D = q.shape
    Dkv = np.asarray(k).shape[1]
    group = D // Dkv
    Q, K, V = _heads(q, M, S), _heads(k, M, S), _heads(v, M, S)
    O, dO = _heads(o, M, S), _heads(do, M, S)
    Z = _scores(Q, K, group)
    zmax = Z.max(axis=3, keepdims=True)
    P = np.exp(Z - zmax)
    P /= P.sum(axis=3, keepdims=True)
    Kq, Vq = np.repeat(K, group, axis=1), np.repeat(V, group, axis=1)
    dP = np.einsum("bhid,bhjd->bhij", dO, Vq)
    Di = np.sum(dO * O, axis=3, keepdims=True)
    dZ = P * (dP - Di)
    dQ = np.einsum("bhij,bhjd->bhid", dZ, Kq) / np.sqrt(HEAD_DIM)
    nseq, Hkv = K.shape[0], K.shape[1]
    dKq = np.einsum("bhij,bhid->bhjd", dZ, Q) / np.sqrt(HEAD_DIM)
    dVq = np.einsum("bhij,bhid->bhjd", P, dO)
    dK = dKq.reshape(nseq, Hkv, group, S, HEAD_DIM).sum(axis=2)
    dV = dVq.reshape(nseq, Hkv, group, S, HEAD_DIM).sum(axis=2)
    return _rows(dQ), _rows(dK), _rows(dV)

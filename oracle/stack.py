"""One synthetic decoder layer and the layer-streamed stack step -- oracle (test infrastructure only).

The pages stream whole *decoder layers* ("Exact Layer Streaming ...", abstract;
"Soup CLI Lets You Fine-Tune ...", "How Layer Streaming Works": forward over the
layers, then backward in reverse, each layer's frozen weights fetched from host
RAM) but never state a layer's internals.  Attention's token mixing is outside
this library, so the reading taken here is a pre-norm Llama-shaped layer whose
attention is replaced by a token-local product; all seven LoRA linears stay on
the gradient path:

    x1 = RMS(h)                         RMS(h) = h / sqrt(mean(h^2) + 1e-5)
    q, k, v = L_q(x1), L_k(x1), L_v(x1)
    a  = q * rep(k) + rep(v)            rep: each 128-wide kv head repeated D/Dkv times
    h1 = h + L_o(a)
    x2 = RMS(h1)
    m  = SiLU(L_gate(x2)) * L_up(x2)
    h2 = h1 + L_down(m)

Rounding points (the bf16 training graph of the pages' tool, which trains bf16
checkpoints): every GEMM input and every GEMM output is a bf16 tensor; the
residual stream h, h1, h2 and its gradient stay in fp32 (float64 here); the
elementwise products are formed in high precision from their bf16 operands
and rounded once.  ``rnd=False`` turns every rounding point into the identity,
which makes the backward the exact derivative of the forward (the
finite-difference / autograd pin uses that mode).

The attention variant (``attn=dict(S=..., theta=...)``, oracle/attention.py
for the reading) replaces the token-local product by causal grouped-query
attention with rotary positions:

    qr, kr = R(rope(q)), R(rope(k));   a = R(attention(qr, kr, v))

and both variants take optional RMS-norm weights per layer (P["norm_attn"],
P["norm_mlp"], [D]): x1 = R(RMS(h) * w_attn), x2 = R(RMS(h1) * w_mlp).

The step (forward layers 0..L-1 from h0, backward L-1..0 from dh_top) returns
hL, dh0 and each linear's (dA, dB).  Streaming changes where the frozen weights
live, not what is computed: the streamed and the resident run compute this same
function ("Exact Layer Streaming ...", abstract: bit-exactness against a
resident reference of the same numerics).
"""
import numpy as np

from .attention import attention_bwd, attention_fwd, rope
from .bf16 import round_bf16
from .ce import ce_fwd_bwd
from .lora import lora_linear_bwd, lora_linear_fwd

EPS = 1e-5
HEAD_DIM = 128
PROJ = ("q", "k", "v", "o", "gate", "up", "down")


def _ident(x):
    return x


def rms_fwd(h):
    r = 1.0 / np.sqrt(np.mean(h * h, axis=1) + EPS)
    return h * r[:, None], r


def rms_bwd(y, r, dy, w=None):
    """Gradient wrt h of y * w with y = h * r(h), given y (unrounded), r, the
    weight w ([D], None = no weight) and the output gradient dy."""
    D = y.shape[1]
    if w is not None:
        dy = dy * np.asarray(w, dtype=np.float64)[None, :]
    return r[:, None] * (dy - y * (np.sum(dy * y, axis=1) / D)[:, None])


def _weighted(y, w):
    return y if w is None else y * np.asarray(w, dtype=np.float64)[None, :]


def rep(kv, D):
    """[M, Dkv] -> [M, D]: kv head j//g serves query head j (g = D/Dkv)."""
    M, Dkv = kv.shape
    g = D // Dkv
    return np.broadcast_to(kv.reshape(M, Dkv // HEAD_DIM, 1, HEAD_DIM),
                           (M, Dkv // HEAD_DIM, g, HEAD_DIM)).reshape(M, D)


def rep_sum(x, Dkv):
    """Adjoint of rep: [M, D] -> [M, Dkv], summing over the g query heads of a kv head."""
    M, D = x.shape
    g = D // Dkv
    return x.reshape(M, Dkv // HEAD_DIM, g, HEAD_DIM).sum(axis=2).reshape(M, Dkv)


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def layer_forward(h, P, alpha, rnd=True, attn=None):
    """One layer forward.  P[name] = dict(W=..., A=..., B=...) (float64, bf16 values),
    optional P["norm_attn"], P["norm_mlp"]; attn = None (token-local) or dict(S=, theta=)."""
    R = round_bf16 if rnd else _ident
    lin = lambda x, n: R(lora_linear_fwd(x, P[n]["W"], P[n].get("A"), P[n].get("B"), alpha))
    D = h.shape[1]
    w1, w2 = P.get("norm_attn"), P.get("norm_mlp")
    y1, r1 = rms_fwd(h)
    x1 = R(_weighted(y1, w1))
    q, k, v = lin(x1, "q"), lin(x1, "k"), lin(x1, "v")
    cache = {}
    if attn is None:
        a = R(q * rep(k, D) + rep(v, D))
    else:
        qr, kr = R(rope(q, attn["S"], attn["theta"])), R(rope(k, attn["S"], attn["theta"]))
        o, _ = attention_fwd(qr, kr, v, attn["S"])
        a = R(o)
        cache.update(qr=qr, kr=kr, o=o)
    h1 = h + lin(a, "o")
    y2, r2 = rms_fwd(h1)
    x2 = R(_weighted(y2, w2))
    g, u = lin(x2, "gate"), lin(x2, "up")
    m = R(g * sigmoid(g) * u)
    h2 = h1 + lin(m, "down")
    cache.update(y1=y1, r1=r1, x1=x1, q=q, k=k, v=v, a=a, y2=y2, r2=r2, x2=x2, g=g, u=u, m=m)
    return h2, cache


def layer_backward(cache, dh2, P, alpha, rnd=True, attn=None):
    """One layer backward: returns (dh, {name: (dA, dB)})."""
    R = round_bf16 if rnd else _ident
    c = cache
    grads = {}

    def lin_b(x, dy, n):
        dx, dA, dB = lora_linear_bwd(x, dy, P[n]["W"], P[n].get("A"), P[n].get("B"), alpha)
        grads[n] = (dA, dB)
        return R(dx)

    Dkv = c["k"].shape[1]
    D = c["q"].shape[1]
    dm = lin_b(c["m"], R(dh2), "down")
    sg = sigmoid(c["g"])
    dg = R(dm * c["u"] * sg * (1.0 + c["g"] * (1.0 - sg)))
    du = R(dm * c["g"] * sg)
    dx2 = lin_b(c["x2"], dg, "gate") + lin_b(c["x2"], du, "up")
    dh1 = dh2 + rms_bwd(c["y2"], c["r2"], dx2, P.get("norm_mlp"))
    da = lin_b(c["a"], R(dh1), "o")
    if attn is None:
        dq = R(da * rep(c["k"], D))
        dk = R(rep_sum(da * c["q"], Dkv))
        dv = R(rep_sum(da, Dkv))
    else:
        dqr, dkr, dvr = attention_bwd(c["qr"], c["kr"], c["v"], c["o"], da, attn["S"])
        dq = R(rope(dqr, attn["S"], attn["theta"], inverse=True))
        dk = R(rope(dkr, attn["S"], attn["theta"], inverse=True))
        dv = R(dvr)
    dx1 = lin_b(c["x1"], dq, "q") + lin_b(c["x1"], dk, "k") + lin_b(c["x1"], dv, "v")
    dh = dh1 + rms_bwd(c["y1"], c["r1"], dx1, P.get("norm_attn"))
    return dh, grads


def stack_step(h0, dh_top, layers, alpha, rnd=True, attn=None):
    """Forward layers 0..L-1 from h0, backward L-1..0 from dh_top.

    Returns (hL, dh0, grads) with grads[l][name] = (dA, dB).
    """
    h = np.asarray(h0, dtype=np.float64)
    caches = []
    for P in layers:
        h, c = layer_forward(h, P, alpha, rnd, attn)
        caches.append(c)
    hL = h
    dh = np.asarray(dh_top, dtype=np.float64)
    grads = [None] * len(layers)
    for l in range(len(layers) - 1, -1, -1):
        dh, grads[l] = layer_backward(caches[l], dh, layers[l], alpha, rnd, attn)
    return hL, dh, grads


def sft_step(tokens, labels, embed, layers, norm_final, W_head, alpha, rnd=True, attn=None):
    """One complete supervised fine-tuning step on top of the stack.

    h0 = embed[tokens] (the frozen embedding rows); the stack forward; x =
    R(RMS(hL) * norm_final); the mean cross-entropy of x against the frozen
    head W_head [V, D] (oracle/ce.py: labels aligned with rows, -100
    ignored); its gradient dx (fp32 on the GPU, unrounded here) back through the final norm into
    dh_top; the stack backward.  Returns (loss, dh0, grads)."""
    R = round_bf16 if rnd else _ident
    h = np.asarray(embed, dtype=np.float64)[np.asarray(tokens)]
    caches = []
    for P in layers:
        h, c = layer_forward(h, P, alpha, rnd, attn)
        caches.append(c)
    yf, rf = rms_fwd(h)
    x = R(_weighted(yf, norm_final))
    loss, dx = ce_fwd_bwd(x, W_head, labels)[:2]
    dh = rms_bwd(yf, rf, dx, norm_final)
    grads = [None] * len(layers)
    for l in range(len(layers) - 1, -1, -1):
        dh, grads[l] = layer_backward(caches[l], dh, layers[l], alpha, rnd, attn)
    return loss, dh, grads

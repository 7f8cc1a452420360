"""NF4 quantise / dequantise -- oracle (test infrastructure only).

What the pages fix: the frozen base is held in NF4 (4-bit NormalFloat), the
QLoRA storage type ("Exact Layer Streaming ...", abstract: "Llama-3.1-8B in
NF4"; "Soup CLI Lets You Fine-Tune ...", "Key Takeaways"; "Soup: Fine-Tuning
...", "Who is it for?": QLoRA fine-tunes).  Block size 64 with one fp32 absmax
per block is the problem statement of this library.

What the pages leave open, and the reading taken here:

* The 16 code values are not printed.  NF4 is the published NormalFloat-4 data
  type of the QLoRA paper (Dettmers et al., 2023, section 3 and appendix): the
  normal quantiles at 9 evenly spaced probabilities from
  delta = 1 - (1/30 + 1/32)/2 down to 1/2 (the 1/2 end dropped) give 8
  positive levels; the negated quantiles at 8 evenly spaced probabilities on the
  same interval (1/2 dropped) give 7 negative levels; 0 is added; the 16 values
  are sorted, divided by the largest and rounded to float32 once.
* Rounding rule: the code of an element is the level nearest to
  x = float32(w / absmax) (IEEE round-to-nearest float32 division), ties going
  to the lower level.  A block whose absmax is 0 gets the zero level (code 7).
* Packing: element 2i of a row-major block sits in the HIGH nibble of byte i,
  element 2i+1 in the low nibble.
* Dequantised value: w_hat = float32(T[code] * absmax).  The GEMMs consume
  bf16(w_hat), QLoRA's bf16 compute dtype.
"""
from statistics import NormalDist

import numpy as np

from .bf16 import round_bf16

BLOCK = 64


def normal_quantile(p: float) -> float:
    """Standard normal quantile; the Python standard library's Wichura AS241."""
    return NormalDist().inv_cdf(p)


def code_table() -> np.ndarray:
    """The 16 NF4 levels (float32, ascending), built from the published construction."""
    delta = 1.0 - 0.5 * (1.0 / 30.0 + 1.0 / 32.0)
    positive = [normal_quantile(p) for p in np.linspace(delta, 0.5, 9)[:-1]]
    negative = [-normal_quantile(p) for p in np.linspace(delta, 0.5, 8)[:-1]]
    levels = np.array(sorted(positive + [0.0] + negative), dtype=np.float64)
    return (levels / levels.max()).astype(np.float32)


def nearest_code(x: np.ndarray) -> np.ndarray:
    """Index of the nearest NF4 level to each float32 x; ties go to the lower index.

    Brute force over the 16 levels in float64, where |x - T[i]| is exact for
    float32 operands; numpy's argmin returns the first (lowest) minimiser.
    """
    T = code_table().astype(np.float64)
    x = np.asarray(x, dtype=np.float32).astype(np.float64).ravel()
    out = np.empty(x.size, dtype=np.uint8)
    step = 1 << 20
    for s in range(0, x.size, step):
        xs = x[s:s + step]
        out[s:s + step] = np.argmin(np.abs(xs[:, None] - T[None, :]), axis=1)
    return out


def quantize(W) -> tuple:
    """NF4-quantise W [N, K] (float32 values) -> (codes uint8 [N*K/2], absmax float32 [N*K/64])."""
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 64")
    if not np.all(np.isfinite(W)):
        raise ValueError("non-finite weight")
    blocks = W.reshape(-1, BLOCK)
    absmax = np.max(np.abs(blocks), axis=1).astype(np.float32)
    codes = np.full(blocks.shape, 7, dtype=np.uint8)     # zero level for all-zero blocks
    nz = absmax > 0
    if np.any(nz):
        x = np.divide(blocks[nz], absmax[nz][:, None], dtype=np.float32)
        codes[nz] = nearest_code(x).reshape(x.shape)
    flat = codes.reshape(-1)
    packed = ((flat[0::2] << 4) | flat[1::2]).astype(np.uint8)
    return packed, absmax


def unpack(codes, N: int, K: int) -> np.ndarray:
    """Packed bytes -> per-element codes [N, K] (high nibble first)."""
    c = np.asarray(codes, dtype=np.uint8).reshape(-1)
    out = np.empty(c.size * 2, dtype=np.uint8)
    out[0::2] = c >> 4
    out[1::2] = c & 0xF
    return out.reshape(N, K)


def dequantize(codes, absmax, N: int, K: int) -> np.ndarray:
    """w_hat = float32(T[code] * absmax), [N, K] float32."""
    T = code_table()
    c = unpack(codes, N, K).reshape(-1, BLOCK)
    a = np.asarray(absmax, dtype=np.float32).reshape(-1, 1)
    return (T[c] * a).astype(np.float32).reshape(N, K)


def dequantize_bf16(codes, absmax, N: int, K: int) -> np.ndarray:
    """bf16(w_hat) as float64: the weight the NF4 linear multiplies by."""
    return round_bf16(dequantize(codes, absmax, N, K))


# ------------------------------------------------------ double quantisation
# The pages' base store (3.60 GB pinned, two 113 MB layer buffers for
# Llama-3.1-8B: "Soup: Fine-Tuning ...", "Layer Streaming: The Mechanism
# Behind the 4 GB Claim") fits 4-bit codes plus an 8-bit absmax per block --
# QLoRA's double quantisation.  The pages do not define its format; the
# reading taken here (a plain, fully specified one):
#
# * the fp32 absmax a[n, j] (row n, 64-block j) is stored transposed as
#   q[j, n] (int8), so that the blocks of consecutive rows are contiguous;
# * per 256 consecutive columns of a transposed row (block b of row j):
#     c = float32(sum of the 256 a values in float64, ascending n) / 256),
#     d_n = float32(a_n - c),  s = float32(max |d_n| / 127),
#     q_n = 0 if s == 0 else clip(rint(float32(d_n / s)), -127, 127)
#   (IEEE float32 subtraction and division, rint rounding ties to even);
# * the absmax used is a'_n = fma(s, q_n, c), rounded once to float32.
DQ_BLOCK = 256


def fma32(s, q, c) -> np.ndarray:
    """float32(s * q + c) rounded once: s, c float32, q small integers.

    s * q is exact in float64; TwoSum gives the float64 sum and its exact
    error; rounding the sum to float32 is already correct unless the sum sits
    exactly on a float32 midpoint, where the error's sign decides.
    """
    s = np.asarray(s, np.float32).astype(np.float64)
    c = np.asarray(c, np.float32).astype(np.float64)
    p = s * np.asarray(q, np.float64)
    t = p + c
    bb = t - p
    err = (p - (t - bb)) + (c - bb)
    r = t.astype(np.float32)
    # float32 neighbours of r and the midpoint toward t
    up = np.nextafter(r, np.float32(np.inf))
    dn = np.nextafter(r, np.float32(-np.inf))
    nb = np.where(t > r.astype(np.float64), up, dn)
    mid = (r.astype(np.float64) + nb.astype(np.float64)) / 2
    on_mid = (t == mid) & (err != 0)
    toward = ((err > 0) & (nb > r)) | ((err < 0) & (nb < r))
    return np.where(on_mid & toward, nb, r).astype(np.float32)


def double_quantize(absmax, N: int, K: int) -> tuple:
    """fp32 absmax (row-major [N, K/64]) -> (q int8 [K/64, N], a2 float32 [K/64, N/256, 2] = (c, s))."""
    if N % DQ_BLOCK or K % BLOCK:
        raise ValueError("double quantisation needs N % 256 == 0 and K % 64 == 0")
    a = np.asarray(absmax, np.float32).reshape(N, K // BLOCK).T          # [K/64, N]
    blocks = a.reshape(K // BLOCK, N // DQ_BLOCK, DQ_BLOCK)
    total = np.zeros(blocks.shape[:2], np.float64)
    for i in range(DQ_BLOCK):                                            # ascending n, float64
        total = total + blocks[:, :, i].astype(np.float64)
    c = (total / DQ_BLOCK).astype(np.float32)
    d = np.subtract(blocks, c[:, :, None], dtype=np.float32)
    m = np.max(np.abs(d), axis=2)
    s = np.divide(m, np.float32(127), dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.divide(d, s[:, :, None], dtype=np.float32)
    q = np.where(s[:, :, None] > 0, np.clip(np.rint(r), -127, 127), 0).astype(np.int8)
    a2 = np.stack([c, s], axis=2).astype(np.float32)
    return q.reshape(K // BLOCK, N), a2


def dq_absmax(q, a2, N: int, K: int) -> np.ndarray:
    """The absmax a' = fma(s, q, c) as float32 [N*K/64] (row-major [N, K/64], like `quantize`)."""
    q = np.asarray(q, np.int8).reshape(K // BLOCK, N // DQ_BLOCK, DQ_BLOCK)
    a2 = np.asarray(a2, np.float32).reshape(K // BLOCK, N // DQ_BLOCK, 2)
    ap = fma32(a2[:, :, 1:2], q, a2[:, :, 0:1])
    return ap.reshape(K // BLOCK, N).T.reshape(-1)


def dequantize_dq(codes, q, a2, N: int, K: int) -> np.ndarray:
    """w_hat = float32(T[code] * a') with the double-quantised absmax, [N, K] float32."""
    return dequantize(codes, dq_absmax(q, a2, N, K), N, K)


def dequantize_dq_bf16(codes, q, a2, N: int, K: int) -> np.ndarray:
    return round_bf16(dequantize_dq(codes, q, a2, N, K))

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

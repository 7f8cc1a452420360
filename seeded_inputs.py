"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the bench.

This module holds random draws and dtype rounding only -- none of the arithmetic
of the method (no quantisation, no GEMM, no loss).  Both sides of every parity
test take their inputs from here; nothing here imports the oracle or the CUDA
package.

Recipe (stated once, used everywhere):

* generator: numpy ``Generator(PCG64(seed))``, one generator per tensor, seed =
  ``base_seed * 1000 + tensor_index``;
* normal draws: ``standard_normal(dtype=float32) * std`` then rounded once to
  bf16 (round-to-nearest-even), the checkpoint dtype of every weight and
  activation on the pages (Llama-3.1-8B / Qwen2.5-3B are bf16 checkpoints);
* labels: ``integers(0, V)`` then exactly ``round(0.05 * M)`` rows, picked by a
  seeded permutation, set to ``ignore_index`` (-100);
* RMS-norm weights: ``1 + 0.1 * standard_normal(dtype=float32)`` kept in fp32
  (a trained checkpoint's norm weights sit near 1);
* tokens: ``integers(0, V)`` as int32.

bf16 tensors are carried as float32 arrays whose values are bf16-exact; the
GPU side reinterprets the top 16 bits (``bf16_bits``).
"""
from __future__ import annotations

import numpy as np

IGNORE_INDEX = -100


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed)))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32)
    # NaN stays NaN (never produced by the generators; kept for completeness)
    return np.where(np.isnan(x), x, out)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Top 16 bits of bf16-exact float32 values, as uint16 (for device upload)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Inverse of ``bf16_bits``: uint16 bf16 patterns to float32 values."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(seed: int, shape, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) draw rounded to bf16, returned as float32."""
    g = rng(seed)
    x = g.standard_normal(size=int(np.prod(shape)), dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return round_bf16(x).reshape(shape)


def labels(seed: int, M: int, V: int, ignore_frac: float = 0.05,
           ignore_index: int = IGNORE_INDEX) -> np.ndarray:
    """int32 labels uniform on [0, V); exactly round(ignore_frac*M) rows ignored."""
    g = rng(seed)
    lab = g.integers(0, V, size=M, dtype=np.int64).astype(np.int32)
    n_ign = int(round(ignore_frac * M))
    if n_ign:
        rows = g.permutation(M)[:n_ign]
        lab[rows] = ignore_index
    return lab


# --------------------------------------------------------------------------
# Workload shapes (the pages' models, by shape only; no trained weights)
# --------------------------------------------------------------------------

# Llama-3.1-8B decoder layer: hidden 4096, 8 kv heads of 128, MLP 14336.
LLAMA8B = dict(name="llama-3.1-8b", D=4096, Dkv=1024, F=14336, head_dim=128, layers=32)
# Qwen2.5-3B decoder layer: hidden 2048, 2 kv heads of 128, MLP 11008.
QWEN3B = dict(name="qwen2.5-3b", D=2048, Dkv=256, F=11008, head_dim=128, layers=36)

# projection order used everywhere: (name, out_features N, in_features K)
PROJ_NAMES = ("q", "k", "v", "o", "gate", "up", "down")


def proj_shapes(D: int, Dkv: int, F: int):
    return [("q", D, D), ("k", Dkv, D), ("v", Dkv, D), ("o", D, D),
            ("gate", F, D), ("up", F, D), ("down", D, F)]


def linear_case(seed: int, M: int, N: int, K: int, r: int, w_std=0.02,
                ab_std=0.02):
    """One LoRA linear: W [N,K], X [M,K], A [r,K], B [N,r], dY [M,N] (bf16-exact f32)."""
    return dict(
        W=normal_bf16(seed * 1000 + 0, (N, K), w_std),
        X=normal_bf16(seed * 1000 + 1, (M, K), 1.0),
        A=normal_bf16(seed * 1000 + 2, (r, K), ab_std) if r else None,
        B=normal_bf16(seed * 1000 + 3, (N, r), ab_std) if r else None,
        dY=normal_bf16(seed * 1000 + 4, (M, N), 1.0),
    )


def stack_case(seed: int, L: int, M: int, D: int, Dkv: int, F: int, r: int,
               w_std=0.02, ab_std=0.02):
    """A synthetic stack: per layer 7 weights + 7 (A, B) pairs, h0 and dh_top."""
    layers = []
    for l in range(L):
        lw = {}
        for j, (name, N, K) in enumerate(proj_shapes(D, Dkv, F)):
            base = seed * 1000 + 10 + l * 32 + j * 3
            lw[name] = dict(
                W=normal_bf16(base * 7 + 0, (N, K), w_std),
                A=normal_bf16(base * 7 + 1, (r, K), ab_std) if r else None,
                B=normal_bf16(base * 7 + 2, (N, r), ab_std) if r else None,
            )
        layers.append(lw)
    h0 = normal_bf16(seed * 1000 + 1, (M, D), 1.0)
    dh_top = normal_bf16(seed * 1000 + 2, (M, D), 1.0)
    return dict(layers=layers, h0=h0, dh_top=dh_top)


def ce_case(seed: int, M: int, D: int, V: int, ignore_frac: float = 0.05,
            h_std=1.0, w_std=0.02):
    return dict(
        H=normal_bf16(seed * 1000 + 0, (M, D), h_std),
        W=normal_bf16(seed * 1000 + 1, (V, D), w_std),
        labels=labels(seed * 1000 + 2, M, V, ignore_frac),
    )


def norm_weight(seed: int, D: int) -> np.ndarray:
    """fp32 [D] RMS-norm weight near 1."""
    g = rng(seed)
    return (np.float32(1.0) + np.float32(0.1) * g.standard_normal(size=D, dtype=np.float32)).astype(np.float32)


def tokens(seed: int, M: int, V: int) -> np.ndarray:
    return rng(seed).integers(0, V, size=M, dtype=np.int64).astype(np.int32)


def sft_case(seed: int, M: int, D: int, V: int):
    """Token ids, labels, a bf16 embedding [V, D] ~ N(0, 1), a bf16 head [V, D] ~ N(0, 0.02), a final norm."""
    return dict(tokens=tokens(seed * 1000 + 0, M, V), labels=labels(seed * 1000 + 1, M, V),
                embed=normal_bf16(seed * 1000 + 2, (V, D), 1.0), head=normal_bf16(seed * 1000 + 3, (V, D), 0.02),
                norm_final=norm_weight(seed * 1000 + 4, D))

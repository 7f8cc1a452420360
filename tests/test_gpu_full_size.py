"""Oracle parity at the full sizes of the pages' models.

* One Llama-3.1-8B-shaped layer's seven NF4 LoRA projections (q 4096x4096,
  k/v 1024x4096, o 4096x4096, gate/up 14336x4096, down 4096x14336), r = 16,
  alpha = 32, at M = 2048 tokens, launched the way the 8B layer benchmark and
  the stack launch them: q/k/v and gate/up as projection groups, o and down
  alone ("Soup CLI ...", "Key Takeaways": Llama-3.1-8B-Instruct with an NF4
  base).  This runs the persistent CTA-pair NF4 GEMM at K = 14336 (the down
  forward) and N = 28672 (the gate/up group) and the rank-r passes at those
  widths.  Y, T, dX, dA and dB of every projection are compared with the
  oracle's float64 LoRA linear on the oracle's own NF4 quantisation.
* Two Qwen2.5-3B-shaped decoder layers with a bf16 base (hidden 2048, kv 256,
  MLP 11008) at M = 2048 ("Exact Layer Streaming ...", abstract: Qwen2.5-3B
  with an un-quantised bf16 base) through the streamed stack step, against
  the oracle's layer, and streamed == resident bit for bit over four such
  layers.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from gpu_util import BF16_TOL, dev_bf16, host, rel_fro
from oracle import lora, nf4, stack
from test_gpu_stack import Setup, same_bits

pytestmark = pytest.mark.gpu

LLAMA = si.LLAMA8B
QWEN = si.QWEN3B


def _unit(sl, seed, names, M, r):
    """One launch unit of the layer: its projections' weights quantised by the
    oracle and laid back to back, adapters back to back, shared X."""
    shp = {n: (N, K) for n, N, K in si.proj_shapes(LLAMA["D"], LLAMA["Dkv"], LLAMA["F"])}
    K = shp[names[0]][1]
    X = si.normal_bf16(seed * 100, (M, K), 1.0)
    parts = []
    for g, n in enumerate(names):
        N = shp[n][0]
        W = si.normal_bf16(seed * 100 + 10 + 3 * g, (N, K), 0.02)
        codes, absmax = nf4.quantize(W)
        del W
        parts.append(dict(N=N, codes=codes, absmax=absmax,
                          A=si.normal_bf16(seed * 100 + 11 + 3 * g, (r, K), 0.02),
                          B=si.normal_bf16(seed * 100 + 12 + 3 * g, (N, r), 0.02),
                          dY=si.normal_bf16(seed * 100 + 50 + g, (M, N), 1.0)))
    return X, K, parts


def _run_unit(sl, X, K, parts, r, alpha):
    M, G = X.shape[0], len(parts)
    N_g = [p["N"] for p in parts]
    NN = sum(N_g)
    w = sl.Weight.nf4(torch.from_numpy(np.concatenate([p["codes"] for p in parts])).cuda(),
                      torch.from_numpy(np.concatenate([p["absmax"] for p in parts])).cuda(), NN, K)
    Xd = dev_bf16(X)
    A = dev_bf16(np.concatenate([p["A"] for p in parts]))
    B = dev_bf16(np.concatenate([p["B"] for p in parts]))
    dY = dev_bf16(np.concatenate([p["dY"] for p in parts], axis=1))
    Y = torch.empty(M, NN, dtype=torch.bfloat16, device="cuda")
    T = torch.empty(M, G * r, dtype=torch.float32, device="cuda")
    dX = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    dA = torch.empty(G * r, K, dtype=torch.float32, device="cuda")
    dB = torch.empty(NN, r, dtype=torch.float32, device="cuda")
    if G > 1:
        ws = torch.empty(sl.sl_lora_group_workspace_size(M, G, r), dtype=torch.uint8, device="cuda")
        sl.sl_lora_group_fwd(w, N_g, Xd, A, B, r, alpha, Y, T)
        sl.sl_lora_group_bwd(w, N_g, Xd, dY, A, B, r, alpha, T, dX, dA, dB, False, ws)
    else:
        ws = torch.empty(sl.sl_lora_linear_workspace_size(M, NN, K, r), dtype=torch.uint8, device="cuda")
        sl.sl_lora_linear_fwd(w, Xd, A, B, r, alpha, Y, T, ws)
        sl.sl_lora_linear_bwd(w, Xd, dY, A, B, r, alpha, T, dX, dA, dB, False, ws)
    sl.sl_check_device_errors()
    return host(Y), host(T), host(dX), host(dA), host(dB)


@pytest.mark.parametrize("names", [("q", "k", "v"), ("o",), ("gate", "up"), ("down",)])
def test_llama8b_layer_projections_m2048_match_oracle(gpu_lib, names):
    sl = gpu_lib
    M, r, alpha = 2048, 16, 32.0
    X, K, parts = _unit(sl, 300 + len(names) * 10 + len(names[0]), names, M, r)
    Y, T, dX, dA, dB = _run_unit(sl, X, K, parts, r, alpha)
    errs = {}
    dX_ref = np.zeros((M, K))
    off = 0
    for g, (n, p) in enumerate(zip(names, parts)):
        N = p["N"]
        W_ref = nf4.dequantize_bf16(p["codes"], p["absmax"], N, K)
        errs[f"Y_{n}"] = rel_fro(Y[:, off:off + N], lora.lora_linear_fwd(X, W_ref, p["A"], p["B"], alpha))
        errs[f"T_{n}"] = rel_fro(T[:, g * r:(g + 1) * r], X.astype(np.float64) @ p["A"].T.astype(np.float64))
        dXo, dAo, dBo = lora.lora_linear_bwd(X, p["dY"], W_ref, p["A"], p["B"], alpha)
        dX_ref += dXo
        errs[f"dA_{n}"] = rel_fro(dA[g * r:(g + 1) * r], dAo)
        errs[f"dB_{n}"] = rel_fro(dB[off:off + N], dBo)
        del W_ref, dXo
        off += N
    errs["dX"] = rel_fro(dX, dX_ref)
    print({k: round(float(v), 6) for k, v in errs.items()})
    assert max(errs.values()) <= BF16_TOL, errs


def test_qwen3b_two_bf16_layers_m2048_match_oracle(gpu_lib):
    sl = gpu_lib
    S = Setup(sl, sl.SL_WEIGHT_BF16, L=2, M=2048, D=QWEN["D"], Dkv=QWEN["Dkv"], F=QWEN["F"], r=16, alpha=32.0,
              seed=61)
    hL, dh0, dA, dB = S.run(sl.SL_MODE_STREAMED)
    ohL, odh0, ograds = stack.stack_step(S.h0_np, S.dh_np, S.ref_layers, 32.0, rnd=True)
    errs = {"hL": rel_fro(host(hL), ohL), "dh0": rel_fro(host(dh0), odh0)}
    for l in range(S.L):
        for p, n in enumerate(si.PROJ_NAMES):
            errs[f"dA{l}{n}"] = rel_fro(host(dA[7 * l + p]), ograds[l][n][0])
            errs[f"dB{l}{n}"] = rel_fro(host(dB[7 * l + p]), ograds[l][n][1])
    print({k: round(float(v), 5) for k, v in errs.items()})
    assert max(errs.values()) <= BF16_TOL, errs
    b = S.run(sl.SL_MODE_RESIDENT)
    for x, y in zip((hL, dh0, *dA, *dB), (b[0], b[1], *b[2], *b[3])):
        assert same_bits(x, y)
    S.stack.close()


def test_qwen3b_bf16_stack_m2048_streamed_equals_resident_bitwise(gpu_lib):
    sl = gpu_lib
    S = Setup(sl, sl.SL_WEIGHT_BF16, L=4, M=2048, D=QWEN["D"], Dkv=QWEN["Dkv"], F=QWEN["F"], r=16, alpha=32.0,
              seed=67, with_oracle=False, torch_weights=True)
    a = S.run(sl.SL_MODE_STREAMED)
    h2d, _ = S.stack.last_step_stats()
    assert h2d == (2 * S.L - 2) * S.stack.host_bytes // S.L
    b = S.run(sl.SL_MODE_RESIDENT)
    for x, y in zip((a[0], a[1], *a[2], *a[3]), (b[0], b[1], *b[2], *b[3])):
        assert same_bits(x, y)
    for g in a[2] + a[3]:
        assert torch.isfinite(g).all() and g.abs().sum() > 0
    S.stack.close()


def test_llama8b_layer_split_tail_m1024_matches_oracle(gpu_lib):
    """One Llama-8B-shaped NF4 layer through the stack at M = 1024 with the
    q/k/v and gate/up groups: the persistent GEMMs' last partial waves split
    along K (q/k/v forward: 96 tiles on 74 SM pairs, the 22 tail tiles in 3
    pieces; gate/up forward: 448 tiles, 4 in 4 pieces; down dX: 224 tiles, 2
    in 7 pieces), checked against the oracle's layer."""
    sl = gpu_lib
    S = Setup(sl, sl.SL_WEIGHT_NF4, L=1, M=1024, D=LLAMA["D"], Dkv=LLAMA["Dkv"], F=LLAMA["F"], r=16, alpha=32.0,
              seed=71, packed=True)
    hL, dh0, dA, dB = S.run(sl.SL_MODE_STREAMED)
    ohL, odh0, ograds = stack.stack_step(S.h0_np, S.dh_np, S.ref_layers, 32.0, rnd=True)
    errs = {"hL": rel_fro(host(hL), ohL), "dh0": rel_fro(host(dh0), odh0)}
    for p, n in enumerate(si.PROJ_NAMES):
        errs[f"dA_{n}"] = rel_fro(host(dA[p]), ograds[0][n][0])
        errs[f"dB_{n}"] = rel_fro(host(dB[p]), ograds[0][n][1])
    print({k: round(float(v), 5) for k, v in errs.items()})
    assert max(errs.values()) <= BF16_TOL, errs
    S.stack.close()


def test_llama8b_stack_split_tail_m1024_streamed_equals_resident_bitwise(gpu_lib):
    """Three 8B-shaped NF4 layers at the headline M = 1024 (every split tail
    of the step) streamed and resident: bitwise equal, and repeatable."""
    sl = gpu_lib
    S = Setup(sl, sl.SL_WEIGHT_NF4, L=3, M=1024, D=LLAMA["D"], Dkv=LLAMA["Dkv"], F=LLAMA["F"], r=16, alpha=32.0,
              seed=73, with_oracle=False, torch_weights=True, packed=True)
    a = S.run(sl.SL_MODE_STREAMED)
    b = S.run(sl.SL_MODE_RESIDENT)
    c = S.run(sl.SL_MODE_STREAMED)
    for x, y, z in zip((a[0], a[1], *a[2], *a[3]), (b[0], b[1], *b[2], *b[3]), (c[0], c[1], *c[2], *c[3])):
        assert same_bits(x, y) and same_bits(x, z)
    for g in a[2] + a[3]:
        assert torch.isfinite(g).all() and g.abs().sum() > 0
    S.stack.close()

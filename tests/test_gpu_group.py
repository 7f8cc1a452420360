"""Projection groups (q/k/v- and gate/up-like) on the GPU against the oracle,
projection by projection: one fused NF4 GEMM and one rank-r pass of each
kind for G LoRA linears that read the same input."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import lora, nf4
from gpu_util import BF16_TOL, dev_bf16, host, rel_fro

pytestmark = pytest.mark.gpu


def make_group(seed, M, K, N_g, r):
    X = si.normal_bf16(seed * 100, (M, K), 1.0)
    parts = []
    for g, N in enumerate(N_g):
        c = si.linear_case(seed * 100 + 10 + g, M, N, K, r)
        oc, oa = nf4.quantize(c["W"])
        parts.append(dict(W_ref=nf4.dequantize_bf16(oc, oa, N, K), codes=oc, absmax=oa, A=c["A"], B=c["B"],
                          dY=c["dY"]))
    return X, parts


def run_group(sl, X, parts, N_g, K, r, alpha, accumulate=False, dA0=None, dB0=None):
    M, G, NN = X.shape[0], len(N_g), sum(N_g)
    codes = torch.from_numpy(np.concatenate([p["codes"] for p in parts])).cuda()
    absmax = torch.from_numpy(np.concatenate([p["absmax"] for p in parts])).cuda()
    w = sl.Weight.nf4(codes, absmax, NN, K)
    Xd = dev_bf16(X)
    A_cat = dev_bf16(np.concatenate([p["A"] for p in parts]))
    B_cat = dev_bf16(np.concatenate([p["B"] for p in parts]))
    dY_cat = dev_bf16(np.concatenate([p["dY"] for p in parts], axis=1))
    Y = torch.empty(M, NN, dtype=torch.bfloat16, device="cuda")
    T = torch.empty(M, G * r, dtype=torch.float32, device="cuda")
    sl.sl_lora_group_fwd(w, N_g, Xd, A_cat, B_cat, r, alpha, Y, T)
    dX = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    dA = dA0.clone() if dA0 is not None else torch.empty(G * r, K, dtype=torch.float32, device="cuda")
    dB = dB0.clone() if dB0 is not None else torch.empty(NN, r, dtype=torch.float32, device="cuda")
    ws = torch.empty(sl.sl_lora_group_workspace_size(M, G, r), dtype=torch.uint8, device="cuda")
    sl.sl_lora_group_bwd(w, N_g, Xd, dY_cat, A_cat, B_cat, r, alpha, T, dX, dA, dB, accumulate, ws)
    sl.sl_check_device_errors()
    return Y, T, dX, dA, dB


GROUPS = [
    # (M, K, N_g, r, alpha): q/k/v-like (G = 3), gate/up-like at the largest fold (G r = 64), four projections
    (300, 512, (512, 256, 256), 16, 32.0),
    (260, 512, (768, 768), 32, 16.0),
    (400, 768, (256, 256, 512, 256), 8, 16.0),
]


@pytest.mark.parametrize("M,K,N_g,r,alpha", GROUPS)
def test_group_matches_oracle_per_projection(gpu_lib, M, K, N_g, r, alpha):
    X, parts = make_group(5 + len(N_g), M, K, N_g, r)
    Y, T, dX, dA, dB = run_group(gpu_lib, X, parts, N_g, K, r, alpha)
    Yh, Th, dAh, dBh = host(Y), host(T), host(dA), host(dB)
    dX_ref = np.zeros((M, K))
    off = 0
    for g, (N, p) in enumerate(zip(N_g, parts)):
        Yo = lora.lora_linear_fwd(X, p["W_ref"], p["A"], p["B"], alpha)
        dXo, dAo, dBo = lora.lora_linear_bwd(X, p["dY"], p["W_ref"], p["A"], p["B"], alpha)
        dX_ref += dXo
        assert rel_fro(Yh[:, off:off + N], Yo) <= BF16_TOL
        assert rel_fro(Th[:, g * r:(g + 1) * r], X.astype(np.float64) @ p["A"].T) <= BF16_TOL
        assert rel_fro(dAh[g * r:(g + 1) * r], dAo) <= BF16_TOL
        assert rel_fro(dBh[off:off + N], dBo) <= BF16_TOL
        off += N
    assert rel_fro(host(dX), dX_ref) <= BF16_TOL


def test_group_deterministic_and_accumulate(gpu_lib):
    M, K, N_g, r, alpha = 300, 512, (512, 256, 256), 16, 32.0
    X, parts = make_group(3, M, K, N_g, r)
    a = run_group(gpu_lib, X, parts, N_g, K, r, alpha)
    b = run_group(gpu_lib, X, parts, N_g, K, r, alpha)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    acc = run_group(gpu_lib, X, parts, N_g, K, r, alpha, accumulate=True, dA0=a[3], dB0=a[4])
    assert torch.allclose(acc[3], 2 * a[3], rtol=1e-6, atol=0)
    assert torch.allclose(acc[4], 2 * a[4], rtol=1e-6, atol=0)


def test_group_rejects_bad_layouts(gpu_lib):
    M, K, r = 300, 512, 16
    X, parts = make_group(4, M, K, (512, 256), r)
    codes = torch.from_numpy(np.concatenate([p["codes"] for p in parts])).cuda()
    absmax = torch.from_numpy(np.concatenate([p["absmax"] for p in parts])).cuda()
    w = gpu_lib.Weight.nf4(codes, absmax, 768, K)
    Xd = dev_bf16(X)
    A = torch.zeros(2 * r, K, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(768, r, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(M, 768, dtype=torch.bfloat16, device="cuda")
    T = torch.empty(M, 2 * r, dtype=torch.float32, device="cuda")
    for N_g in ((512, 255), (500, 268), (512, 512)):   # not multiples of 256 / wrong total
        with pytest.raises(gpu_lib.SLError) as e:
            gpu_lib.sl_lora_group_fwd(w, N_g, Xd, A, B, r, 32.0, Y, T)
        assert e.value.status == gpu_lib.SL_ERR_INVALID
    with pytest.raises(gpu_lib.SLError):                 # G r > 64
        gpu_lib.sl_lora_group_fwd(w, (256, 256, 256), Xd, A, B, 32, 32.0, Y, T)

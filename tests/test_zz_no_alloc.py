"""The allocation-free forward (sl_lora_linear_fwd_noalloc) against the workspace forward.

For callers that cannot allocate device memory, libsl keeps this forward's
scratch in a fixed 4 MiB device array.  This file is collected last so that a
failure here leaves every other test already run; it passes alone in a fresh
process and after the others.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from gpu_util import BF16_TOL, dev_bf16, host, rel_fro

pytestmark = pytest.mark.gpu


def _weight(sl, kind, W):
    if kind == "nf4":
        N, K = W.shape
        codes = torch.empty(N * K // 2, dtype=torch.uint8, device="cuda")
        absmax = torch.empty(N * K // 64, dtype=torch.float32, device="cuda")
        sl.sl_nf4_quantize(W, codes, absmax)
        return sl.Weight.nf4(codes, absmax, N, K)
    return sl.Weight.bf16(W)


def test_noalloc_forward_matches_workspace_forward_twice(gpu_lib):
    sl = gpu_lib
    # two calls in a row with different shapes; both need the scratch (K > 512)
    for seed, (M, N, K, r, kind) in enumerate([(300, 512, 2048, 16, "nf4"), (128, 1024, 4096, 8, "bf16")]):
        c = si.linear_case(40 + seed, M, N, K, r)
        w = _weight(sl, kind, dev_bf16(c["W"]))
        X, A, B = dev_bf16(c["X"]), dev_bf16(c["A"]), dev_bf16(c["B"])
        Y0 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        T0 = torch.empty(M, r, dtype=torch.float32, device="cuda")
        ws = torch.empty(sl.sl_lora_linear_workspace_size(M, N, K, r), dtype=torch.uint8, device="cuda")
        sl.sl_lora_linear_fwd(w, X, A, B, r, 2.0 * r, Y0, T0, ws)
        Y1 = torch.full_like(Y0, float("nan"))
        T1 = torch.full_like(T0, float("nan"))
        sl.sl_lora_linear_fwd_noalloc(w, X, A, B, r, 2.0 * r, Y1, T1)
        sl.sl_check_device_errors()
        assert rel_fro(host(Y1), host(Y0)) <= BF16_TOL
        assert rel_fro(host(T1), host(T0)) <= BF16_TOL
        assert torch.isfinite(Y1.float()).all() and torch.isfinite(T1).all()


def test_noalloc_rejects_scratch_above_maximum(gpu_lib):
    sl = gpu_lib
    M, N, K, r = 8192, 256, 14336, 32          # 28 splits x 8192 x 32 x 4 B = 29 MiB > 4 MiB
    W = torch.zeros(N, K, dtype=torch.bfloat16, device="cuda")
    w = sl.Weight.bf16(W)
    X = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    A = torch.zeros(r, K, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(N, r, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    T = torch.empty(M, r, dtype=torch.float32, device="cuda")
    with pytest.raises(sl.SLError) as e:
        sl.sl_lora_linear_fwd_noalloc(w, X, A, B, r, 16.0, Y, T)
    assert e.value.status == sl.SL_ERR_INVALID and "maximum" in str(e.value)

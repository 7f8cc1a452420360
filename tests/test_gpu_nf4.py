"""NF4 quantise / dequantise on the GPU against the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import nf4
from gpu_util import dev_bf16

pytestmark = pytest.mark.gpu


def gpu_quantize(sl, W_t):
    N, K = W_t.shape
    codes = torch.empty(N * K // 2, dtype=torch.uint8, device="cuda")
    absmax = torch.empty(N * K // 64, dtype=torch.float32, device="cuda")
    sl.sl_nf4_quantize(W_t, codes, absmax)
    return codes, absmax


@pytest.mark.parametrize("N,K", [(512, 512), (96, 1024), (1, 64)])
def test_quantize_bitexact_bf16(gpu_lib, N, K):
    W = si.normal_bf16(11 + N, (N, K), 0.02)
    c, a = gpu_quantize(gpu_lib, dev_bf16(W))
    oc, oa = nf4.quantize(W)
    assert np.array_equal(c.cpu().numpy(), oc)
    assert np.array_equal(a.cpu().numpy().view(np.uint32), oa.view(np.uint32))


def test_quantize_special_values_fp32(gpu_lib):
    T = nf4.code_table().astype(np.float64)
    rows = []
    for j in range(15):            # values around every exact midpoint, absmax pinned to 1 by the last element
        mid = (T[j] + T[j + 1]) / 2
        m32 = np.float32(mid)
        vals = [np.nextafter(m32, np.float32(-2)), m32, np.nextafter(m32, np.float32(2)), np.float32(T[j]),
                np.float32(T[j + 1])]
        row = np.zeros(64, np.float32)
        row[:len(vals)] = vals
        row[63] = 1.0
        rows.append(row)
    rows.append(np.zeros(64, np.float32))                      # all-zero block
    rows.append(np.linspace(-3.0, 7.0, 64).astype(np.float32))  # absmax = 7, hits +1 exactly
    W = np.stack(rows)
    Wt = torch.from_numpy(W).cuda()
    c, a = gpu_quantize(gpu_lib, Wt)
    oc, oa = nf4.quantize(W)
    assert np.array_equal(c.cpu().numpy(), oc)
    assert np.array_equal(a.cpu().numpy(), oa)


def test_quantize_full_size_sampled_rows(gpu_lib):
    """Full 14336 x 4096 gate projection; the quantiser is block-local, so sampled rows suffice."""
    N, K = 14336, 4096
    W = si.normal_bf16(7, (N, K), 0.02)
    c, a = gpu_quantize(gpu_lib, dev_bf16(W))
    rows = np.random.default_rng(0).choice(N, 48, replace=False)
    oc, oa = nf4.quantize(W[rows])
    cg = c.view(N, K // 2)[torch.from_numpy(rows).cuda()].cpu().numpy().reshape(-1)
    ag = a.view(N, K // 64)[torch.from_numpy(rows).cuda()].cpu().numpy().reshape(-1)
    assert np.array_equal(cg, oc)
    assert np.array_equal(ag, oa)


def test_dequantize_bitexact(gpu_lib):
    N, K = 256, 512
    W = si.normal_bf16(3, (N, K), 0.02)
    oc, oa = nf4.quantize(W)
    c = torch.from_numpy(oc).cuda()
    a = torch.from_numpy(oa).cuda()
    out32 = torch.empty(N, K, dtype=torch.float32, device="cuda")
    out16 = torch.empty(N, K, dtype=torch.bfloat16, device="cuda")
    gpu_lib.sl_nf4_dequantize(c, a, N, K, out32)
    gpu_lib.sl_nf4_dequantize(c, a, N, K, out16)
    ref = nf4.dequantize(oc, oa, N, K)
    assert np.array_equal(out32.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(out16.float().cpu().numpy(), nf4.dequantize_bf16(oc, oa, N, K).astype(np.float32))


def test_nonfinite_rejected(gpu_lib):
    W = np.zeros((2, 64), np.float32)
    W[1, 5] = np.nan
    with pytest.raises(gpu_lib.SLError) as e:
        gpu_quantize(gpu_lib, torch.from_numpy(W).cuda())
    assert e.value.status == gpu_lib.SL_ERR_NONFINITE
    with pytest.raises(gpu_lib.SLError):
        gpu_quantize(gpu_lib, torch.zeros(2, 96, device="cuda"))

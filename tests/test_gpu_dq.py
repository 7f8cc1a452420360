"""Double-quantised NF4 absmax on the GPU against the oracle.

The 8-bit absmax and its (offset, scale) pairs are integer / IEEE-exact work:
the quantiser and the dequantised weight are compared bit for bit.  The LoRA
linear and the projection group on NF4_DQ weights are compared with the
oracle on the double-quantised weight, and bit for bit with the same kernels
fed a plain fp32 absmax equal to fma(s, q, c).
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import lora, nf4
from gpu_util import BF16_TOL, dev_bf16, host, rel_fro

pytestmark = pytest.mark.gpu


def quantized(seed, N, K):
    W = si.normal_bf16(seed, (N, K), 0.02)
    codes, absmax = nf4.quantize(W)
    return codes, absmax


def device_dq(gpu_lib, absmax, N, K, q_pad=0, a2_pad=0):
    """Run the library's quantiser; return (qabsmax, absmax2) device tensors."""
    am = torch.from_numpy(absmax).cuda()
    a2_ld = 2 * (N // 256) + a2_pad
    a2_ld += (-a2_ld) % 4
    q = torch.full((K // 64, N + q_pad), 99, dtype=torch.int8, device="cuda")
    a2 = torch.full((K // 64, a2_ld), 7.0, dtype=torch.float32, device="cuda")
    gpu_lib.sl_nf4_double_quantize(am, N, K, q, a2)
    torch.cuda.synchronize()
    return q, a2


@pytest.mark.parametrize("N,K,q_pad,a2_pad", [(256, 64, 0, 0), (768, 512, 16, 4), (2048, 256, 0, 0)])
def test_double_quantize_bit_exact(gpu_lib, N, K, q_pad, a2_pad):
    rng = np.random.default_rng(N + K)
    absmax = (np.abs(rng.standard_normal(N * K // 64)) * 0.05 + 1e-3).astype(np.float32)
    # a constant 256-block (s = 0: every q is 0, a' = c exactly) and a block of wide range
    am2 = absmax.reshape(N, K // 64)
    am2[:256, 0] = np.float32(0.0371)
    if N >= 512:
        am2[256:512, -1] *= np.float32(40.0)
    q, a2 = device_dq(gpu_lib, absmax, N, K, q_pad, a2_pad)
    oq, oa2 = nf4.double_quantize(absmax, N, K)
    qh = q.cpu().numpy()
    a2h = a2.cpu().numpy()
    assert np.array_equal(qh[:, :N], oq)
    assert np.all(qh[:, N:] == 99)                       # the padding is untouched
    got = a2h[:, :2 * (N // 256)].reshape(K // 64, N // 256, 2)
    assert np.array_equal(got.view(np.uint32), oa2.view(np.uint32))
    assert np.all(a2h[:, 2 * (N // 256):] == 7.0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_dq_weight_dequantize_bit_exact(gpu_lib, dtype):
    N, K = 768, 512
    codes, absmax = quantized(71, N, K)
    q, a2 = device_dq(gpu_lib, absmax, N, K)
    oq, oa2 = nf4.double_quantize(absmax, N, K)
    w = gpu_lib.Weight.nf4_dq(torch.from_numpy(codes).cuda(), q, a2, N, K)
    out = torch.empty(N, K, dtype=dtype, device="cuda")
    gpu_lib.sl_weight_dequantize(w, out)
    torch.cuda.synchronize()
    ref = nf4.dequantize_dq(codes, oq, oa2, N, K) if dtype == torch.float32 else \
        nf4.dequantize_dq_bf16(codes, oq, oa2, N, K)
    got = out.float().cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.astype(np.float32).view(np.uint32))


def dq_arrays(gpu_lib, absmax, N, K):
    """(qabsmax, absmax2) on the device and the plain fp32 absmax a' = fma(s, q, c) they stand for."""
    q, a2 = device_dq(gpu_lib, absmax, N, K)
    oq, oa2 = nf4.double_quantize(absmax, N, K)
    return q, a2, oq, oa2, nf4.dq_absmax(oq, oa2, N, K)


@pytest.mark.parametrize("M,N,K,r,alpha", [(300, 512, 768, 16, 32.0), (1000, 1536, 512, 32, 16.0),
                                           (129, 256, 256, 8, 16.0)])
def test_dq_linear_matches_oracle_and_plain_absmax(gpu_lib, M, N, K, r, alpha):
    c = si.linear_case(900 + M, M, N, K, r)
    codes, absmax = nf4.quantize(c["W"])
    q, a2, oq, oa2, ap = dq_arrays(gpu_lib, absmax, N, K)
    W_ref = nf4.dequantize_dq_bf16(codes, oq, oa2, N, K)
    cd = torch.from_numpy(codes).cuda()
    w_dq = gpu_lib.Weight.nf4_dq(cd, q, a2, N, K)
    X, A, B, dY = dev_bf16(c["X"]), dev_bf16(c["A"]), dev_bf16(c["B"]), dev_bf16(c["dY"])

    def run(w):
        Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        T = torch.empty(M, r, dtype=torch.float32, device="cuda")
        ws = torch.empty(gpu_lib.sl_lora_linear_workspace_size(M, N, K, r), dtype=torch.uint8, device="cuda")
        gpu_lib.sl_lora_linear_fwd(w, X, A, B, r, alpha, Y, T, ws)
        dX = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
        dA = torch.empty(r, K, dtype=torch.float32, device="cuda")
        dB = torch.empty(N, r, dtype=torch.float32, device="cuda")
        gpu_lib.sl_lora_linear_bwd(w, X, dY, A, B, r, alpha, T, dX, dA, dB, False, ws)
        gpu_lib.sl_check_device_errors()
        return Y, dX, dA, dB

    Y, dX, dA, dB = run(w_dq)
    Yo = lora.lora_linear_fwd(c["X"], W_ref, c["A"], c["B"], alpha)
    dXo, dAo, dBo = lora.lora_linear_bwd(c["X"], c["dY"], W_ref, c["A"], c["B"], alpha)
    assert rel_fro(host(Y), Yo) <= BF16_TOL
    assert rel_fro(host(dX), dXo) <= BF16_TOL
    assert rel_fro(host(dA), dAo) <= BF16_TOL
    assert rel_fro(host(dB), dBo) <= BF16_TOL
    # the weight the GEMM dequantises is exactly the oracle's: same result as a plain absmax a'
    # (a plain absmax of one wave of tiles takes the non-persistent pair kernel,
    # whose LoRA fold may sum in another order: equal up to fp32 rounding)
    Yp, dXp, dAp, dBp = run(gpu_lib.Weight.nf4(cd, torch.from_numpy(ap).cuda(), N, K))
    assert rel_fro(host(Yp), host(Y)) <= 1e-3
    assert rel_fro(host(dXp), host(dX)) <= 1e-3
    assert torch.equal(dA, dAp) and torch.equal(dB, dBp)


def test_dq_group_bit_identical_to_plain_absmax(gpu_lib):
    """Groups always run the persistent kernel: NF4_DQ and the plain absmax a' agree bit for bit."""
    M, K, N_g, r, alpha = 300, 512, (512, 256, 256), 16, 32.0
    NN, G = sum(N_g), len(N_g)
    X = si.normal_bf16(41, (M, K), 1.0)
    cases = [si.linear_case(420 + g, M, N, K, r) for g, N in enumerate(N_g)]
    W = np.concatenate([cs["W"] for cs in cases])
    codes, absmax = nf4.quantize(W)
    q, a2, oq, oa2, ap = dq_arrays(gpu_lib, absmax, NN, K)
    cd = torch.from_numpy(codes).cuda()
    Xd = dev_bf16(X)
    A_cat = dev_bf16(np.concatenate([cs["A"] for cs in cases]))
    B_cat = dev_bf16(np.concatenate([cs["B"] for cs in cases]))
    dY_cat = dev_bf16(np.concatenate([cs["dY"] for cs in cases], axis=1))

    def run(w):
        Y = torch.empty(M, NN, dtype=torch.bfloat16, device="cuda")
        T = torch.empty(M, G * r, dtype=torch.float32, device="cuda")
        gpu_lib.sl_lora_group_fwd(w, N_g, Xd, A_cat, B_cat, r, alpha, Y, T)
        dX = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
        dA = torch.empty(G * r, K, dtype=torch.float32, device="cuda")
        dB = torch.empty(NN, r, dtype=torch.float32, device="cuda")
        ws = torch.empty(gpu_lib.sl_lora_group_workspace_size(M, G, r), dtype=torch.uint8, device="cuda")
        gpu_lib.sl_lora_group_bwd(w, N_g, Xd, dY_cat, A_cat, B_cat, r, alpha, T, dX, dA, dB, False, ws)
        gpu_lib.sl_check_device_errors()
        return Y, dX, dA, dB

    got = run(gpu_lib.Weight.nf4_dq(cd, q, a2, NN, K))
    plain = run(gpu_lib.Weight.nf4(cd, torch.from_numpy(ap).cuda(), NN, K))
    for x, y in zip(got, plain):
        assert torch.equal(x, y)
    W_ref = nf4.dequantize_dq_bf16(codes, oq, oa2, NN, K)
    Yo = lora.lora_linear_fwd(X, W_ref[:N_g[0]], cases[0]["A"], cases[0]["B"], alpha)
    assert rel_fro(host(got[0])[:, :N_g[0]], Yo) <= BF16_TOL


def test_dq_column_range_of_shared_arrays(gpu_lib):
    """A weight that is columns dq_col0 .. dq_col0 + N of arrays quantised for a larger N."""
    M, K, r, alpha = 300, 512, 8, 16.0
    N_all, col0, N = 1280, 512, 512
    c = si.linear_case(77, M, N_all, K, r)
    codes, absmax = nf4.quantize(c["W"])
    q, a2, oq, oa2, _ = dq_arrays(gpu_lib, absmax, N_all, K)
    W_ref = nf4.dequantize_dq_bf16(codes, oq, oa2, N_all, K)[col0:col0 + N]
    # codes of rows col0 .. col0 + N (K / 2 bytes per row)
    cd = torch.from_numpy(np.ascontiguousarray(codes.reshape(N_all, K // 2)[col0:col0 + N])).cuda()
    w = gpu_lib.Weight.nf4_dq(cd, q, a2, N, K, col0=col0)
    out = torch.empty(N, K, dtype=torch.bfloat16, device="cuda")
    gpu_lib.sl_weight_dequantize(w, out)
    assert np.array_equal(host(out), W_ref)
    X, A, B, dY = dev_bf16(c["X"]), dev_bf16(c["A"][:, :]), dev_bf16(c["B"][col0:col0 + N]), \
        dev_bf16(c["dY"][:, col0:col0 + N])
    Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    T = torch.empty(M, r, dtype=torch.float32, device="cuda")
    ws = torch.empty(gpu_lib.sl_lora_linear_workspace_size(M, N, K, r), dtype=torch.uint8, device="cuda")
    gpu_lib.sl_lora_linear_fwd(w, X, A, B, r, alpha, Y, T, ws)
    dX = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    dA = torch.empty(r, K, dtype=torch.float32, device="cuda")
    dB = torch.empty(N, r, dtype=torch.float32, device="cuda")
    gpu_lib.sl_lora_linear_bwd(w, X, dY, A, B, r, alpha, T, dX, dA, dB, False, ws)
    gpu_lib.sl_check_device_errors()
    Bn, dYn = c["B"][col0:col0 + N], c["dY"][:, col0:col0 + N]
    assert rel_fro(host(Y), lora.lora_linear_fwd(c["X"], W_ref, c["A"], Bn, alpha)) <= BF16_TOL
    dXo, _, _ = lora.lora_linear_bwd(c["X"], dYn, W_ref, c["A"], Bn, alpha)
    assert rel_fro(host(dX), dXo) <= BF16_TOL


def test_dq_rejects_small_m_and_bad_layouts(gpu_lib):
    N, K, r = 512, 256, 8
    codes, absmax = quantized(5, N, K)
    q, a2 = device_dq(gpu_lib, absmax, N, K)
    cd = torch.from_numpy(codes).cuda()
    X = torch.zeros(128, K, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(128, N, dtype=torch.bfloat16, device="cuda")
    w = gpu_lib.Weight.nf4_dq(cd, q, a2, N, K)
    with pytest.raises(gpu_lib.SLError) as e:                       # M <= 128: one-CTA kernels read fp32 absmax only
        gpu_lib.sl_lora_linear_fwd(w, X, None, None, 0, 1.0, Y, None)
    assert e.value.status == gpu_lib.SL_ERR_UNSUPPORTED
    X2 = torch.zeros(200, K, dtype=torch.bfloat16, device="cuda")
    Y2 = torch.empty(200, N, dtype=torch.bfloat16, device="cuda")
    for bad in (gpu_lib.Weight.nf4_dq(cd, q, a2, N, K, col0=128),            # column offset not a multiple of 256
                gpu_lib.Weight.nf4_dq(cd, q[:, :256], a2, N, K),             # qabsmax rows shorter than N
                gpu_lib.Weight.nf4_dq(cd, q, a2[:, :2], N, K)):              # absmax2 rows shorter than 2 N / 256
        with pytest.raises(gpu_lib.SLError) as e:
            gpu_lib.sl_lora_linear_fwd(bad, X2, None, None, 0, 1.0, Y2, None)
        assert e.value.status == gpu_lib.SL_ERR_INVALID

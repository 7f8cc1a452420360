"""Causal GQA attention with rotary positions on the GPU against the oracle."""
import numpy as np
import pytest
import torch

from oracle import attention as at
from oracle.bf16 import round_bf16
from gpu_util import BF16_TOL, dev_bf16, host, rel_fro

pytestmark = pytest.mark.gpu


def bf16_inputs(seed, M, D, Dkv, std=1.0):
    g = np.random.default_rng(seed)
    return [round_bf16(g.standard_normal((M, n)) * std).astype(np.float32) for n in (D, Dkv, Dkv)]


def table(gpu_lib, S, theta):
    t = torch.empty(S, 128, dtype=torch.float32, device="cuda")
    gpu_lib.sl_rope_table(S, theta, t)
    return t


def test_rope_table_is_the_rounded_fp64_angles(gpu_lib):
    S, theta = 1024, 500000.0
    t = table(gpu_lib, S, theta).cpu().numpy()
    c, s = at.rope_cos_sin(S, theta)
    for got, ref in ((t[:, :64], c), (t[:, 64:], s)):
        ulp = np.abs(got.view(np.int32).astype(np.int64) - ref.astype(np.float32).view(np.int32).astype(np.int64))
        assert ulp.max() <= 1


@pytest.mark.parametrize("inverse", [False, True])
def test_rope_apply_matches_oracle(gpu_lib, inverse):
    S, theta, M = 256, 10000.0, 512
    x = bf16_inputs(3, M, 512, 128)[0]
    buf = torch.zeros(M, 640, dtype=torch.bfloat16, device="cuda")     # a strided view, as in a q/k/v region
    view = buf[:, 64:576]
    view.copy_(dev_bf16(x))
    gpu_lib.sl_rope_apply(view, S, table(gpu_lib, S, theta), inverse=inverse)
    ref = round_bf16(at.rope(x, S, theta, inverse=inverse))
    got = host(view)
    assert rel_fro(got, ref) <= 2e-3
    assert np.abs(got - ref).max() <= np.abs(ref).max() * 2.0 ** -7
    assert np.all(host(buf[:, :64]) == 0) and np.all(host(buf[:, 576:]) == 0)


CASES = [
    # (M, S, H, Hkv): GQA group 2, MQA with two sequences, MHA, Llama-3.1-8B heads at one sequence of 512
    (256, 128, 4, 2),
    (768, 384, 4, 1),
    (512, 256, 2, 2),
    (512, 512, 32, 8),
    # 16 sequences: (S/128) Hkv nseq = 256 CTAs fill the GPU, so dK/dV sum their kv head's query heads in-CTA
    (4096, 256, 16, 8),
    # one 2048-token sequence: 16 query tiles, the longest causal loops
    (2048, 2048, 4, 1),
]


def run_attention(gpu_lib, M, S, H, Hkv, seed, packed=True, rope=None):
    D, Dkv = H * 128, Hkv * 128
    q, k, v = bf16_inputs(seed, M, D, Dkv)
    if packed:   # q, k, v as column blocks of one [M, D + 2 Dkv] region (the grouped projection's output)
        qkv = torch.empty(M, D + 2 * Dkv, dtype=torch.bfloat16, device="cuda")
        qd, kd, vd = qkv[:, :D], qkv[:, D:D + Dkv], qkv[:, D + Dkv:]
        qd.copy_(dev_bf16(q))
        kd.copy_(dev_bf16(k))
        vd.copy_(dev_bf16(v))
    else:
        qd, kd, vd = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    o = torch.empty(M, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(H, M, dtype=torch.float32, device="cuda")
    gpu_lib.sl_attention_fwd(qd, kd, vd, S, o, lse)
    gpu_lib.sl_check_device_errors()
    dO = dev_bf16(bf16_inputs(seed + 1, M, D, Dkv)[0])
    dq = torch.empty(M, D, dtype=torch.bfloat16, device="cuda")
    dk = torch.empty(M, Dkv, dtype=torch.bfloat16, device="cuda")
    dv = torch.empty(M, Dkv, dtype=torch.bfloat16, device="cuda")
    gpu_lib.sl_attention_bwd(qd, kd, vd, o, dO, lse, S, dq, dk, dv, rope_table=rope)
    gpu_lib.sl_check_device_errors()
    return (q, k, v, host(dO)), (o, lse, dq, dk, dv)


@pytest.mark.parametrize("M,S,H,Hkv", CASES)
def test_attention_fwd_bwd_matches_oracle(gpu_lib, M, S, H, Hkv):
    (q, k, v, dO), (o, lse, dq, dk, dv) = run_attention(gpu_lib, M, S, H, Hkv, seed=M + H)
    o_ref, lse_ref = at.attention_fwd(q, k, v, S)
    assert rel_fro(host(o), o_ref) <= BF16_TOL
    np.testing.assert_allclose(host(lse).T, lse_ref, rtol=2e-5, atol=2e-5)
    # the backward of the oracle at the forward output the kernels saw (bf16 o)
    dq_ref, dk_ref, dv_ref = at.attention_bwd(q, k, v, o_ref, dO, S)
    assert rel_fro(host(dq), dq_ref) <= BF16_TOL
    assert rel_fro(host(dk), dk_ref) <= BF16_TOL
    assert rel_fro(host(dv), dv_ref) <= BF16_TOL


def test_attention_first_rows_and_determinism(gpu_lib):
    M, S, H, Hkv = 512, 256, 4, 2
    a_in, a = run_attention(gpu_lib, M, S, H, Hkv, seed=9, packed=False)
    _, b = run_attention(gpu_lib, M, S, H, Hkv, seed=9, packed=True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)                          # strided or dense inputs, same bits; reruns identical
    q, k, v, _ = a_in
    o = host(a[0])
    for t in (0, S):                                      # the first token of each sequence copies its value
        for h in range(H):
            g = h // (H // Hkv)
            np.testing.assert_array_equal(o[t, h * 128:(h + 1) * 128], v[t, g * 128:(g + 1) * 128])


@pytest.mark.parametrize("M,S,H,Hkv", [(512, 256, 4, 2), (4096, 256, 16, 8)])
def test_attention_bwd_rotates_gradients_back(gpu_lib, M, S, H, Hkv):
    """With the rotary table, dq and dk leave as the gradients of the unrotated q and k
    (per-query-head partials and the in-CTA head sum)."""
    theta = 500000.0
    (q, k, v, dO), (o, lse, dq, dk, dv) = run_attention(gpu_lib, M, S, H, Hkv, seed=13, rope=table(gpu_lib, S, theta))
    o_ref, _ = at.attention_fwd(q, k, v, S)
    dq_ref, dk_ref, dv_ref = at.attention_bwd(q, k, v, o_ref, dO, S)
    assert rel_fro(host(dq), at.rope(dq_ref, S, theta, inverse=True)) <= BF16_TOL
    assert rel_fro(host(dk), at.rope(dk_ref, S, theta, inverse=True)) <= BF16_TOL
    assert rel_fro(host(dv), dv_ref) <= BF16_TOL


def test_attention_rejects_bad_shapes(gpu_lib):
    q = torch.zeros(200, 256, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(200, 128, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(2, 200, dtype=torch.float32, device="cuda")
    with pytest.raises(gpu_lib.SLError) as e:            # S not a multiple of 128
        gpu_lib.sl_attention_fwd(q, k, k, 100, o, lse)
    assert e.value.status == gpu_lib.SL_ERR_INVALID
    q3 = torch.zeros(256, 384, dtype=torch.bfloat16, device="cuda")
    k2 = torch.zeros(256, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(gpu_lib.SLError):                  # 3 query heads over 2 kv heads
        gpu_lib.sl_attention_fwd(q3, k2, k2, 128, torch.empty_like(q3), torch.empty(3, 256, device="cuda"))


def test_attention_rescales_when_the_row_maximum_grows(gpu_lib):
    """Key norms that grow along the sequence make a row's maximum score rise by
    more than 2^8 between 128-key tiles, so the forward has to rescale O
    (checked on the inputs below); o, lse and the gradients still match."""
    M, S, H, Hkv = 1024, 1024, 4, 2
    D, Dkv = H * 128, Hkv * 128
    g = np.random.default_rng(21)
    grow = (1.0 + np.arange(S) / 64.0)[:, None]
    q = round_bf16(g.standard_normal((M, D)) * 2.0).astype(np.float32)
    k = round_bf16(g.standard_normal((M, Dkv)) * grow).astype(np.float32)
    v = round_bf16(g.standard_normal((M, Dkv))).astype(np.float32)
    dO = round_bf16(g.standard_normal((M, D))).astype(np.float32)
    # the inputs exercise the rescale: per row, the running maximum (log2 units)
    # grows by more than 8 at a later tile for most rows of the later query tiles
    moved = 0
    for h in range(H):
        s2 = (q[:, h * 128:(h + 1) * 128].astype(np.float64) @ k[:, (h // 2) * 128:(h // 2 + 1) * 128].T.astype(np.float64))
        s2 *= np.log2(np.e) / np.sqrt(128.0)
        s2[np.triu_indices(S, 1)] = -np.inf
        tile_max = s2.reshape(S, S // 128, 128).max(axis=2)
        run = np.maximum.accumulate(tile_max, axis=1)
        moved += int(np.sum(np.any(tile_max[:, 1:] > run[:, :-1] + 8.0, axis=1)))
    assert moved > H * S // 2
    qd, kd, vd = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    o = torch.empty(M, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(H, M, dtype=torch.float32, device="cuda")
    gpu_lib.sl_attention_fwd(qd, kd, vd, S, o, lse)
    dq = torch.empty(M, D, dtype=torch.bfloat16, device="cuda")
    dk = torch.empty(M, Dkv, dtype=torch.bfloat16, device="cuda")
    dv = torch.empty(M, Dkv, dtype=torch.bfloat16, device="cuda")
    gpu_lib.sl_attention_bwd(qd, kd, vd, o, dev_bf16(dO), lse, S, dq, dk, dv)
    gpu_lib.sl_check_device_errors()
    o_ref, lse_ref = at.attention_fwd(q, k, v, S)
    assert rel_fro(host(o), o_ref) <= BF16_TOL
    np.testing.assert_allclose(host(lse).T, lse_ref, rtol=2e-5, atol=2e-5)
    dq_ref, dk_ref, dv_ref = at.attention_bwd(q, k, v, o_ref, dO, S)
    assert rel_fro(host(dq), dq_ref) <= BF16_TOL
    assert rel_fro(host(dk), dk_ref) <= BF16_TOL
    assert rel_fro(host(dv), dv_ref) <= BF16_TOL


def test_attention_full_bench_shape_sampled_sequences(gpu_lib):
    """The launch the attention bench times (8 sequences of 1024 tokens, 32 query
    heads over 8 kv heads, rotary table on), sampled: in two sequences, every
    row of o, lse and dq of one kv head's four query heads, and every row of
    that kv head's dk and dv, against the oracle run on just those heads."""
    M, S, H, Hkv, theta = 8192, 1024, 32, 8, 500000.0
    (q, k, v, dO), (o, lse, dq, dk, dv) = run_attention(gpu_lib, M, S, H, Hkv, seed=77, rope=table(gpu_lib, S, theta))
    o, lse, dq, dk, dv = host(o), host(lse).T, host(dq), host(dk), host(dv)
    grp = H // Hkv
    for b, g in ((0, 0), (5, 6)):
        rows = slice(b * S, (b + 1) * S)
        qc = slice(g * grp * 128, (g + 1) * grp * 128)   # the query heads of kv head g
        kc = slice(g * 128, (g + 1) * 128)
        o_ref, lse_ref = at.attention_fwd(q[rows, qc], k[rows, kc], v[rows, kc], S)
        assert rel_fro(o[rows, qc], o_ref) <= BF16_TOL
        np.testing.assert_allclose(lse[rows, g * grp:(g + 1) * grp], lse_ref, rtol=2e-5, atol=2e-5)
        dq_ref, dk_ref, dv_ref = at.attention_bwd(q[rows, qc], k[rows, kc], v[rows, kc], o_ref, dO[rows, qc], S)
        assert rel_fro(dq[rows, qc], at.rope(dq_ref, S, theta, inverse=True)) <= BF16_TOL
        assert rel_fro(dk[rows, kc], at.rope(dk_ref, S, theta, inverse=True)) <= BF16_TOL
        assert rel_fro(dv[rows, kc], dv_ref) <= BF16_TOL

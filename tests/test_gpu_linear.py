"""The fused NF4 / bf16 LoRA linear (forward and backward) on the GPU against the oracle."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import lora, nf4
from gpu_util import BF16_TOL, dev_bf16, host, rel_fro

pytestmark = pytest.mark.gpu


def make(sl, seed, M, N, K, r, kind):
    c = si.linear_case(seed, M, N, K, r)
    if kind == "nf4":
        oc, oa = nf4.quantize(c["W"])
        W_ref = nf4.dequantize_bf16(oc, oa, N, K)
        codes, absmax = torch.from_numpy(oc).cuda(), torch.from_numpy(oa).cuda()
        w = sl.Weight.nf4(codes, absmax, N, K)
    else:
        W_ref = c["W"].astype(np.float64)
        w = sl.Weight.bf16(dev_bf16(c["W"]))
    t = {k: (dev_bf16(v) if v is not None else None) for k, v in c.items() if k != "W"}
    return c, W_ref, w, t


def run(sl, w, t, M, N, K, r, alpha, accumulate=False, dA0=None, dB0=None):
    Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    T = torch.empty(M, max(r, 1), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(sl.sl_lora_linear_workspace_size(M, N, K, r), 1), dtype=torch.uint8, device="cuda")
    sl.sl_lora_linear_fwd(w, t["X"], t["A"], t["B"], r, alpha, Y, T, ws)
    dX = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    dA = dA0.clone() if dA0 is not None else torch.empty(r, K, dtype=torch.float32, device="cuda")
    dB = dB0.clone() if dB0 is not None else torch.empty(N, r, dtype=torch.float32, device="cuda")
    sl.sl_lora_linear_bwd(w, t["X"], t["dY"], t["A"], t["B"], r, alpha, T, dX, dA, dB, accumulate, ws)
    sl.sl_check_device_errors()
    return Y, T, dX, dA, dB


CASES = [
    # (M, N, K, r, alpha, kind)  -- first row: the single 512x512 NF4 linear, r=8, alpha=16
    (64, 512, 512, 8, 16.0, "nf4"),
    (300, 768, 1024, 16, 32.0, "nf4"),     # several tiles in M and N, ragged M tail
    (200, 512, 768, 16, 32.0, "bf16"),
    (130, 1024, 512, 32, 16.0, "nf4"),     # rank 32: two extra K-steps
    (70, 352, 128, 8, 16.0, "bf16"),       # fewer K-blocks than stages, partial N tile
    (150, 96, 256, 16, 32.0, "nf4"),       # N < one tile; dX reduction ends mid-block
    # CTA-pair edges: M = 129 (the pair's second CTA holds one row), M = 257 (a second
    # pair of one row), N = 32, one k-block of a bf16 weight, ranks 24 and 32
    (129, 32, 256, 8, 16.0, "nf4"),
    (129, 288, 64, 32, 8.0, "bf16"),
    (257, 256, 512, 16, 32.0, "bf16"),
    (256, 256, 256, 24, 48.0, "nf4"),
]


@pytest.mark.parametrize("M,N,K,r,alpha,kind", CASES)
def test_linear_matches_oracle(gpu_lib, M, N, K, r, alpha, kind):
    c, W_ref, w, t = make(gpu_lib, 100 + M, M, N, K, r, kind)
    Y, T, dX, dA, dB = run(gpu_lib, w, t, M, N, K, r, alpha)
    Yo = lora.lora_linear_fwd(c["X"], W_ref, c["A"], c["B"], alpha)
    dXo, dAo, dBo = lora.lora_linear_bwd(c["X"], c["dY"], W_ref, c["A"], c["B"], alpha)
    assert rel_fro(host(Y), Yo) <= BF16_TOL
    assert rel_fro(host(T), c["X"].astype(np.float64) @ c["A"].T) <= BF16_TOL
    assert rel_fro(host(dX), dXo) <= BF16_TOL
    assert rel_fro(host(dA), dAo) <= BF16_TOL
    assert rel_fro(host(dB), dBo) <= BF16_TOL


def test_zero_B_equals_base_and_rank_zero(gpu_lib):
    M, N, K, r = 96, 512, 512, 16
    c, W_ref, w, t = make(gpu_lib, 7, M, N, K, r, "nf4")
    t["B"] = torch.zeros_like(t["B"])
    Y1 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    Y0 = torch.empty_like(Y1)
    T = torch.empty(M, r, dtype=torch.float32, device="cuda")
    ws = torch.empty(gpu_lib.sl_lora_linear_workspace_size(M, N, K, r), dtype=torch.uint8, device="cuda")
    gpu_lib.sl_lora_linear_fwd(w, t["X"], t["A"], t["B"], r, 32.0, Y1, T, ws)
    gpu_lib.sl_lora_linear_fwd(w, t["X"], None, None, 0, 32.0, Y0, None)
    assert torch.equal(Y1.float(), Y0.float())
    assert rel_fro(host(Y0), c["X"].astype(np.float64) @ W_ref.T) <= BF16_TOL


def test_deterministic_and_accumulate(gpu_lib):
    M, N, K, r = 260, 512, 1024, 16
    c, W_ref, w, t = make(gpu_lib, 9, M, N, K, r, "nf4")
    a = run(gpu_lib, w, t, M, N, K, r, 32.0)
    b = run(gpu_lib, w, t, M, N, K, r, 32.0)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    acc = run(gpu_lib, w, t, M, N, K, r, 32.0, accumulate=True, dA0=a[3], dB0=a[4])
    assert torch.allclose(acc[3], 2 * a[3], rtol=1e-6, atol=0)
    assert torch.allclose(acc[4], 2 * a[4], rtol=1e-6, atol=0)


def test_bounded_wait_times_out_without_fault(gpu_lib):
    for mbar in (False, True):
        gpu_lib.sl_debug_timeout_probe(2_000_000, mbarrier=mbar)
        with pytest.raises(gpu_lib.SLError) as e:
            gpu_lib.sl_check_device_errors()
        assert e.value.status == gpu_lib.SL_ERR_TIMEOUT
        gpu_lib.sl_check_device_errors()          # cleared; the context is still usable
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0


@pytest.mark.parametrize("M,N,K,kind", [(2048, 2560, 2560, "nf4"), (300, 1248, 2048, "nf4"), (1024, 4864, 4096, "nf4"),
                                        (1024, 4096, 4864, "nf4"), (2048, 2560, 2560, "bf16"), (300, 1248, 2048, "bf16"),
                                        (1024, 4096, 4864, "bf16")])
def test_pair_gemm_tile_walk_matches_oracle(gpu_lib, M, N, K, kind):
    """The CTA-pair GEMM (NF4 weights dequantised in the kernel, or bf16
    weights loaded by TMA) at sizes where tiles outnumber the SM pairs
    (80 pair tiles on 74: some clusters run two tiles, alternating their
    TMEM accumulators and LoRA staging) and with a ragged M pair and a
    partial N tile. With a workspace the persistent kernel splits its last
    partial wave along K (80 tiles: the 6 tail tiles in 3 pieces; 76 tiles
    in the forward of N = 4864 or the dX of K = 4864: 2 tail tiles in 4
    pieces, the partial sums added in piece order): bitwise repeatable, and
    within rounding of the forward without a workspace (no split)."""
    r, alpha = 16, 32.0
    c, W_ref, w, t = make(gpu_lib, 11, M, N, K, r, kind)
    a = run(gpu_lib, w, t, M, N, K, r, alpha)
    b = run(gpu_lib, w, t, M, N, K, r, alpha)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    T = torch.empty(M, r, dtype=torch.float32, device="cuda")
    gpu_lib.sl_lora_linear_fwd(w, t["X"], t["A"], t["B"], r, alpha, Y, T, None)
    gpu_lib.sl_check_device_errors()
    assert torch.equal(T, a[1]) and rel_fro(host(Y), host(a[0])) <= 2e-3
    Yo = lora.lora_linear_fwd(c["X"], W_ref, c["A"], c["B"], alpha)
    dXo, dAo, dBo = lora.lora_linear_bwd(c["X"], c["dY"], W_ref, c["A"], c["B"], alpha)
    assert rel_fro(host(a[0]), Yo) <= BF16_TOL
    assert rel_fro(host(a[2]), dXo) <= BF16_TOL
    assert rel_fro(host(a[3]), dAo) <= BF16_TOL
    assert rel_fro(host(a[4]), dBo) <= BF16_TOL


def test_kernel_timing_on_the_device_clock(gpu_lib):
    """A timed GEMM launch records its own span on the device clock; with no
    copy in flight it is within the CUDA-event pair around the launch."""
    sl = gpu_lib
    M, N, K, r = 300, 768, 1024, 16
    c, W_ref, w, t = make(sl, 13, M, N, K, r, "nf4")
    Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    T = torch.empty(M, r, dtype=torch.float32, device="cuda")
    sl.sl_lora_linear_fwd(w, t["X"], t["A"], t["B"], r, 32.0, Y, T, None)
    sl.sl_kernel_timing(True)
    for _ in range(3):
        sl.sl_lora_linear_fwd(w, t["X"], t["A"], t["B"], r, 32.0, Y, T, None)
    sl.sl_kernel_timing(False)
    n_ev, ms_ev, flops = sl.sl_kernel_timing_read(0)
    n_ck, ms_ck = sl.sl_kernel_timing_read_clock(0)
    assert n_ev == 3 and n_ck == 3 and flops > 0
    assert 0 < ms_ck <= ms_ev * 1.05, (ms_ck, ms_ev)
    sl.sl_check_device_errors()

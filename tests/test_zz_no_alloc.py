"""The allocation-free forward (sl_lora_linear_fwd_noalloc).

Some callers cannot allocate device memory: code that runs under a memory
manager owning all of it (a framework's caching allocator with a hard budget,
an application that forbids cudaMalloc because it synchronises the device and
fragments its pool).  For them libsl keeps this forward's scratch in a fixed
4 MiB device array.  These tests check that entry point against the oracle and
against the workspace forward, at and just past the array's limit, with
misaligned pointers, and -- in a fresh process whose first libsl call that
touches the error word or the scratch is this one -- that it leaves the
device's free memory unchanged.

This file is collected last so that a failure here leaves every other test
already run; it passes alone in a fresh process and after the others.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import seeded_inputs as si
from gpu_util import BF16_TOL, dev_bf16, host, rel_fro
from oracle import lora, nf4

pytestmark = pytest.mark.gpu

LIMIT = 4 << 20   # bytes of the fixed scratch array


def _weight(sl, kind, W32):
    """(library weight, the oracle's bf16 view of it) for a bf16-exact float32 W."""
    N, K = W32.shape
    if kind == "nf4":
        oc, oa = nf4.quantize(W32)
        w = sl.Weight.nf4(torch.from_numpy(oc).cuda(), torch.from_numpy(oa).cuda(), N, K)
        return w, nf4.dequantize_bf16(oc, oa, N, K)
    return sl.Weight.bf16(dev_bf16(W32)), W32.astype(np.float64)


def _need(M, K, r):
    splits = -(-K // 512)
    return splits * M * r * 4 if splits > 1 else 0


@pytest.mark.parametrize("M,N,K,r,kind", [
    (300, 512, 2048, 16, "nf4"),    # ragged M (not a multiple of 32 or 128), four K splits
    (77, 768, 1536, 8, "bf16"),     # ragged M below one tile
    (200, 256, 4096, 24, "nf4"),    # rank 24: the 32-wide kernel with its last 8 rank rows unused
    (130, 512, 1024, 32, "bf16"),   # rank 32
    (64, 512, 512, 8, "nf4"),       # one split: no scratch at all
])
def test_noalloc_forward_matches_oracle(gpu_lib, M, N, K, r, kind):
    sl = gpu_lib
    c = si.linear_case(60 + M, M, N, K, r)
    w, W_ref = _weight(sl, kind, c["W"])
    X, A, B = dev_bf16(c["X"]), dev_bf16(c["A"]), dev_bf16(c["B"])
    alpha = 2.0 * r
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    T = torch.full((M, r), float("nan"), dtype=torch.float32, device="cuda")
    sl.sl_lora_linear_fwd_noalloc(w, X, A, B, r, alpha, Y, T)
    sl.sl_check_device_errors()
    assert rel_fro(host(Y), lora.lora_linear_fwd(c["X"], W_ref, c["A"], c["B"], alpha)) <= BF16_TOL
    assert rel_fro(host(T), c["X"].astype(np.float64) @ c["A"].T.astype(np.float64)) <= BF16_TOL


def test_noalloc_forward_matches_workspace_forward_twice(gpu_lib):
    sl = gpu_lib
    # two calls in a row with different shapes; both need the scratch (K > 512)
    for seed, (M, N, K, r, kind) in enumerate([(300, 512, 2048, 16, "nf4"), (128, 1024, 4096, 8, "bf16")]):
        c = si.linear_case(40 + seed, M, N, K, r)
        w, _ = _weight(sl, kind, c["W"])
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


def test_noalloc_scratch_exactly_at_the_limit_and_one_row_over(gpu_lib):
    sl = gpu_lib
    M, N, K, r = 4096, 256, 4096, 32           # 8 splits x 4096 x 32 x 4 B = 4 MiB exactly
    assert _need(M, K, r) == LIMIT and _need(M + 1, K, r) > LIMIT
    c = si.linear_case(77, M + 1, N, K, r)
    w, W_ref = _weight(sl, "bf16", c["W"])
    X, A, B = dev_bf16(c["X"]), dev_bf16(c["A"]), dev_bf16(c["B"])
    Y = torch.full((M + 1, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    T = torch.full((M + 1, r), float("nan"), dtype=torch.float32, device="cuda")
    # need == maximum: accepted, and correct
    sl.sl_lora_linear_fwd_noalloc(w, X[:M], A, B, r, 32.0, Y[:M], T[:M])
    sl.sl_check_device_errors()
    Xo = c["X"][:M]
    assert rel_fro(host(Y[:M]), lora.lora_linear_fwd(Xo, W_ref, c["A"], c["B"], 32.0)) <= BF16_TOL
    assert rel_fro(host(T[:M]), Xo.astype(np.float64) @ c["A"].T.astype(np.float64)) <= BF16_TOL
    # one row more: rejected before anything is launched
    n0 = sl.lib().sl_launch_count()
    with pytest.raises(sl.SLError) as e:
        sl.sl_lora_linear_fwd_noalloc(w, X, A, B, r, 32.0, Y, T)
    assert e.value.status == sl.SL_ERR_INVALID and "maximum" in str(e.value)
    assert sl.lib().sl_launch_count() == n0


def test_noalloc_rejects_misaligned_pointers_before_launching(gpu_lib):
    sl = gpu_lib
    M, N, K, r = 64, 256, 1024, 16
    c = si.linear_case(5, M, N, K, r)
    w, _ = _weight(sl, "bf16", c["W"])
    Xb = torch.zeros(M * K + 8, dtype=torch.bfloat16, device="cuda")
    Ab = torch.zeros(r * K + 8, dtype=torch.bfloat16, device="cuda")
    X, A, B = Xb[:M * K].view(M, K), Ab[:r * K].view(r, K), dev_bf16(c["B"])
    Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    T = torch.empty(M, r, dtype=torch.float32, device="cuda")
    X_off = Xb[1:1 + M * K].view(M, K)      # 2 bytes past a 16-byte boundary
    A_off = Ab[4:4 + r * K].view(r, K)      # 8 bytes past
    for args in [(X_off, A, B), (X, A_off, B)]:
        n0 = sl.lib().sl_launch_count()
        with pytest.raises(sl.SLError) as e:
            sl.sl_lora_linear_fwd_noalloc(w, *args, r, 32.0, Y, T)
        assert e.value.status == sl.SL_ERR_INVALID and "aligned" in str(e.value)
        assert sl.lib().sl_launch_count() == n0
    sl.sl_check_device_errors()


# A fresh process that touches the GPU only through the CUDA runtime (for its
# inputs) and libsl.  Modules load eagerly, and one libsl call that uses
# neither the error word nor any scratch (the rotary table) brings libsl's
# modules in first, so the free-memory readings around the allocation-free
# forward see only what that forward allocates.
_FRESH = r"""
import ctypes, json, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
import layer_streamed_qlora_linear_b300 as sl
import seeded_inputs as si
rt = ctypes.CDLL("libcudart.so")
P = ctypes.c_void_p
def ok(e, what):
    if e != 0:
        raise RuntimeError(what + " failed: %d" % e)
def dev(a):
    a = np.ascontiguousarray(a)
    p = P()
    ok(rt.cudaMalloc(ctypes.byref(p), ctypes.c_size_t(max(a.nbytes, 16))), "cudaMalloc")
    ok(rt.cudaMemcpy(p, a.ctypes.data_as(P), ctypes.c_size_t(a.nbytes), 1), "cudaMemcpy")
    return p
def free_bytes():
    f, t = ctypes.c_size_t(), ctypes.c_size_t()
    ok(rt.cudaDeviceSynchronize(), "sync")
    ok(rt.cudaMemGetInfo(ctypes.byref(f), ctypes.byref(t)), "cudaMemGetInfo")
    return f.value
M, N, K, r = 300, 512, 2048, 16
c = si.linear_case(91, M, N, K, r)
X, A, B = (dev(si.bf16_bits(c[k])) for k in ("X", "A", "B"))
Wd = dev(si.bf16_bits(c["W"]))
Y = [dev(np.zeros(M * N, np.uint16)) for _ in range(3)]
T = [dev(np.zeros(M * r, np.float32)) for _ in range(3)]
rope = dev(np.zeros(128 * 128, np.float32))
L = sl.lib()
ok(L.sl_rope_table(128, ctypes.c_double(10000.0), rope, None), "sl_rope_table")
w = sl.sl_weight(kind=sl.SL_WEIGHT_BF16, N=N, K=K, w=Wd.value)
before = free_bytes()
for i in range(2):
    ok(L.sl_lora_linear_fwd_noalloc(ctypes.byref(w), X, M, A, B, r, ctypes.c_float(32.0), Y[i], T[i], None),
       "sl_lora_linear_fwd_noalloc")
after = free_bytes()
ws = dev(np.zeros(sl.lib().sl_lora_linear_workspace_size(M, N, K, r) // 4 + 1, np.float32))
ok(L.sl_lora_linear_fwd(ctypes.byref(w), X, M, A, B, r, ctypes.c_float(32.0), Y[2], T[2], ws,
                        ctypes.c_size_t(sl.lib().sl_lora_linear_workspace_size(M, N, K, r)), None), "fwd")
ok(L.sl_check_device_errors(None), "device errors")
def get(p, n, dt):
    out = np.empty(n, dt)
    ok(rt.cudaMemcpy(out.ctypes.data_as(P), p, ctypes.c_size_t(out.nbytes), 2), "cudaMemcpy D2H")
    return out
ys = [si.bits_to_f32(get(Y[i], M * N, np.uint16)).astype(np.float64) for i in range(3)]
ts = [get(T[i], M * r, np.float32).astype(np.float64) for i in range(3)]
def rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))
print(json.dumps(dict(before=before, after=after, y=[rel(ys[i], ys[2]) for i in range(2)],
                      t=[rel(ts[i], ts[2]) for i in range(2)])))
"""


def test_noalloc_first_call_in_a_fresh_process_allocates_nothing(gpu_lib):
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, CUDA_MODULE_LOADING="EAGER")
    p = subprocess.run([sys.executable, "-c", _FRESH, root], capture_output=True, text=True, timeout=300,
                       env=env, cwd=root)
    assert p.returncode == 0, p.stderr[-2000:]
    res = json.loads(p.stdout.strip().splitlines()[-1])
    assert res["after"] == res["before"], res
    assert max(res["y"]) <= BF16_TOL and max(res["t"]) <= BF16_TOL, res

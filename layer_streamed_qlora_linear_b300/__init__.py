"""Python binding of libsl (the layer-streamed NF4 LoRA library for B300).

Argument marshalling only: every function below forwards torch tensors' device
pointers (and the current CUDA stream) to the C ABI declared in
``include/sl.h`` under the same name.  All arithmetic runs in libsl's CUDA
kernels; there is no CPU or PyTorch fallback -- if ``libsl.so`` is missing or
cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsl.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "sl.h")

SL_OK, SL_ERR_INVALID, SL_ERR_CUDA, SL_ERR_UNSUPPORTED, SL_ERR_TIMEOUT, SL_ERR_NONFINITE, SL_ERR_OOM = range(7)
SL_DTYPE_BF16, SL_DTYPE_F32 = 0, 1
SL_WEIGHT_NF4, SL_WEIGHT_BF16, SL_WEIGHT_NF4_DQ = 0, 1, 2
SL_MODE_STREAMED, SL_MODE_RESIDENT = 0, 1
SL_MIX_TOKEN_LOCAL, SL_MIX_ATTENTION = 0, 1
STATUS_NAMES = {0: "SL_OK", 1: "SL_ERR_INVALID", 2: "SL_ERR_CUDA", 3: "SL_ERR_UNSUPPORTED",
                4: "SL_ERR_TIMEOUT", 5: "SL_ERR_NONFINITE", 6: "SL_ERR_OOM"}


class SLError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class sl_weight(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("codes", ctypes.c_void_p), ("absmax", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("qabsmax", ctypes.c_void_p), ("qabsmax_ld", ctypes.c_int64),
                ("absmax2", ctypes.c_void_p), ("absmax2_ld", ctypes.c_int64), ("dq_col0", ctypes.c_int64)]


class sl_stack_desc(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int32), ("kind", ctypes.c_int32), ("D", ctypes.c_int64),
                ("Dkv", ctypes.c_int64), ("F", ctypes.c_int64),
                ("host_blobs", ctypes.POINTER(ctypes.c_void_p)),
                ("device_blobs", ctypes.POINTER(ctypes.c_void_p)),
                ("mixer", ctypes.c_int32), ("seq_len", ctypes.c_int64), ("rope_theta", ctypes.c_double)]


_lib = None
_P, _I32, _I64, _SZ, _F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_SIGS = {
    "sl_last_error": (ctypes.c_char_p, []),
    "sl_version": (_I32, []),
    "sl_launch_count": (ctypes.c_uint64, []),
    "sl_nf4_code_table": (None, [_P]),
    "sl_check_device_errors": (_I32, [_P]),
    "sl_debug_timeout_probe": (_I32, [_I64, _I32, _P]),
    "sl_kernel_timing": (_I32, [_I32]),
    "sl_kernel_timing_read": (_I32, [_I32, _P, _P, _P]),
    "sl_kernel_timing_read_clock": (_I32, [_I32, _P, _P]),
    "sl_nf4_quantize": (_I32, [_P, _I32, _I64, _I64, _P, _P, _P]),
    "sl_nf4_dequantize": (_I32, [_P, _P, _I64, _I64, _I32, _P, _P]),
    "sl_nf4_double_quantize": (_I32, [_P, _I64, _I64, _P, _I64, _P, _I64, _P]),
    "sl_weight_dequantize": (_I32, [ctypes.POINTER(sl_weight), _I32, _P, _P]),
    "sl_lora_linear_fwd": (_I32, [ctypes.POINTER(sl_weight), _P, _I64, _P, _P, _I32, _F, _P, _P, _P, _SZ, _P]),
    "sl_lora_linear_bwd": (_I32, [ctypes.POINTER(sl_weight), _P, _P, _I64, _P, _P, _I32, _F, _P, _P, _P, _P,
                                  _I32, _P, _SZ, _P]),
    "sl_lora_linear_workspace_size": (_SZ, [_I64, _I64, _I64, _I32]),
    "sl_lora_linear_fwd_noalloc": (_I32, [ctypes.POINTER(sl_weight), _P, _I64, _P, _P, _I32, _F, _P, _P, _P]),
    "sl_lora_group_fwd": (_I32, [ctypes.POINTER(sl_weight), _I32, _P, _P, _I64, _P, _P, _I32, _F, _P, _P, _P]),
    "sl_lora_group_bwd": (_I32, [ctypes.POINTER(sl_weight), _I32, _P, _P, _P, _I64, _P, _P, _I32, _F, _P, _P,
                                 _P, _P, _I32, _P, _SZ, _P]),
    "sl_lora_group_workspace_size": (_SZ, [_I64, _I32, _I32]),
    "sl_stack_blob_layout": (_I32, [_I32, _I64, _I64, _I64, _P, _P]),
    "sl_stack_dq_layout": (_I32, [_I64, _I64, _I64, _P, _P, _P, _P, _P]),
    "sl_sft_step": (_I32, [_P, _I32, _P, _P, _I64, _P, _I64, _P, _P, _I64, _P, _P, _I32, _F, _P, _P, _P, _I32,
                           _P, _SZ, _P]),
    "sl_sft_workspace_size": (_SZ, [_P, _I64, _I32, _I64, _I64]),
    "sl_rope_table": (_I32, [_I64, ctypes.c_double, _P, _P]),
    "sl_rope_apply": (_I32, [_P, _I64, _I64, _I32, _I64, _P, _I32, _P]),
    "sl_attention_fwd": (_I32, [_P, _I64, _P, _I64, _P, _I64, _I64, _I64, _I32, _I32, _P, _I64, _P, _P]),
    "sl_attention_workspace_size": (_SZ, [_I64, _I32]),
    "sl_attention_bwd": (_I32, [_P, _I64, _P, _I64, _P, _I64, _P, _I64, _P, _I64, _P, _I64, _I64, _I32, _I32,
                                _P, _I64, _P, _I64, _P, _I64, _P, _P, _SZ, _P]),
    "sl_stack_create": (_I32, [ctypes.POINTER(sl_stack_desc), _P, _P, _P]),
    "sl_stack_destroy": (_I32, [_P]),
    "sl_stack_workspace_size": (_SZ, [_P, _I64, _I32]),
    "sl_stream_stack_step": (_I32, [_P, _I32, _P, _I64, _P, _P, _P, _I32, _F, _P, _P, _P, _P, _I32, _P, _SZ,
                                    _P]),
    "sl_stack_last_step_stats": (_I32, [_P, _P, _P]),
    "sl_ce_fwd_bwd": (_I32, [_P, _I64, _I64, _P, _I64, _P, _I32, _I64, _P, _P, _P, _SZ, _P]),
    "sl_ce_workspace_size": (_SZ, [_I64, _I64, _I64, _I64]),
}


def lib() -> ctypes.CDLL:
    """The loaded libsl; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libsl.so not found at {LIB_PATH}: run __graft_entry__.build() "
                               "(python -m layer_streamed_qlora_linear_b300.build)")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            if hasattr(l, name):
                f = getattr(l, name)
                f.restype = res
                f.argtypes = args
        _lib = l
    return _lib


def header_functions() -> list:
    """Names of every function declared in include/sl.h."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sl_[a-z0-9_]+)\s*\(", text)))


def _check(status: int):
    if status != SL_OK:
        raise SLError(status, lib().sl_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


# ------------------------------------------------------------------ library
def sl_version() -> int:
    return lib().sl_version()


def sl_nf4_code_table():
    buf = (ctypes.c_float * 16)()
    lib().sl_nf4_code_table(buf)
    return list(buf)


def sl_check_device_errors(stream=None):
    _check(lib().sl_check_device_errors(_stream(stream)))


def sl_debug_timeout_probe(limit_ns: int, mbarrier: bool = False, stream=None):
    _check(lib().sl_debug_timeout_probe(int(limit_ns), int(bool(mbarrier)), _stream(stream)))


def sl_launch_count() -> int:
    """libsl kernel launches so far in this process."""
    return int(lib().sl_launch_count())


GEMM_VARIANTS = ("nf4_fwd", "nf4_dx", "bf16_fwd", "bf16_dx", "ce_logits", "ce_dh")
RANK_R_VARIANTS = ("rank_t", "rank_u", "rank_grad")  # timing variants 6, 7, 8 (work in bytes)
ATTN_VARIANTS = ("attn_fwd", "attn_bwd")              # timing variants 9, 10 (work in FLOPs)
TIMED_VARIANTS = GEMM_VARIANTS + RANK_R_VARIANTS + ATTN_VARIANTS


def sl_kernel_timing(enable: bool):
    _check(lib().sl_kernel_timing(int(bool(enable))))


def sl_kernel_timing_read_clock(variant: int):
    """(launches, ms) of one GEMM variant (0-5) on the device clock since timing was enabled."""
    n, ms = ctypes.c_uint64(0), ctypes.c_double(0)
    _check(lib().sl_kernel_timing_read_clock(int(variant), ctypes.byref(n), ctypes.byref(ms)))
    return n.value, ms.value


def sl_kernel_timing_read(variant: int):
    """(launches, ms, work) of one timed variant since timing was enabled:
    work is FLOPs for GEMM variants 0-5 and bytes for rank-r variants 6-8."""
    n, ms, fl = ctypes.c_uint64(0), ctypes.c_double(0), ctypes.c_double(0)
    _check(lib().sl_kernel_timing_read(int(variant), ctypes.byref(n), ctypes.byref(ms), ctypes.byref(fl)))
    return n.value, ms.value, fl.value


# ---------------------------------------------------------------------- NF4
def sl_nf4_quantize(W, codes, absmax, stream=None):
    """W [N, K] bf16/fp32 -> codes uint8 [N*K/2], absmax fp32 [N*K/64] (synchronises)."""
    import torch
    N, K = W.shape
    dt = SL_DTYPE_F32 if W.dtype == torch.float32 else SL_DTYPE_BF16
    _check(lib().sl_nf4_quantize(_ptr(W), dt, N, K, _ptr(codes), _ptr(absmax), _stream(stream)))


def sl_nf4_dequantize(codes, absmax, N, K, out, stream=None):
    import torch
    dt = SL_DTYPE_F32 if out.dtype == torch.float32 else SL_DTYPE_BF16
    _check(lib().sl_nf4_dequantize(_ptr(codes), _ptr(absmax), N, K, dt, _ptr(out), _stream(stream)))


def sl_nf4_double_quantize(absmax, N, K, qabsmax, absmax2, qabsmax_ld=None, absmax2_ld=None, stream=None):
    """absmax [N*K/64] fp32 -> qabsmax int8 [K/64, >= N] and absmax2 fp32 [K/64, >= 2 N/256] (see include/sl.h)."""
    q_ld = qabsmax.shape[-1] if qabsmax_ld is None else qabsmax_ld
    a2_ld = absmax2.shape[-1] if absmax2_ld is None else absmax2_ld
    _check(lib().sl_nf4_double_quantize(_ptr(absmax), N, K, _ptr(qabsmax), q_ld, _ptr(absmax2), a2_ld,
                                        _stream(stream)))


def sl_weight_dequantize(weight, out, stream=None):
    import torch
    dt = SL_DTYPE_F32 if out.dtype == torch.float32 else SL_DTYPE_BF16
    _check(lib().sl_weight_dequantize(ctypes.byref(weight.desc), dt, _ptr(out), _stream(stream)))


# ---------------------------------------------------------------- weights
class Weight:
    """An sl_weight descriptor that keeps its tensors alive."""

    def __init__(self, kind, N, K, codes=None, absmax=None, w=None, qabsmax=None, absmax2=None, col0=0):
        self.tensors = (codes, absmax, w, qabsmax, absmax2)
        self.desc = sl_weight(kind, N, K, codes.data_ptr() if codes is not None else None,
                              absmax.data_ptr() if absmax is not None else None,
                              w.data_ptr() if w is not None else None,
                              qabsmax.data_ptr() if qabsmax is not None else None,
                              qabsmax.shape[-1] if qabsmax is not None else 0,
                              absmax2.data_ptr() if absmax2 is not None else None,
                              absmax2.shape[-1] if absmax2 is not None else 0, int(col0))

    @staticmethod
    def nf4(codes, absmax, N, K):
        return Weight(SL_WEIGHT_NF4, N, K, codes=codes, absmax=absmax)

    @staticmethod
    def nf4_dq(codes, qabsmax, absmax2, N, K, col0=0):
        """Double-quantised NF4: qabsmax int8 [K/64, ld], absmax2 fp32 [K/64, ld2]; columns col0 .. col0+N."""
        return Weight(SL_WEIGHT_NF4_DQ, N, K, codes=codes, qabsmax=qabsmax, absmax2=absmax2, col0=col0)

    @staticmethod
    def bf16(w):
        return Weight(SL_WEIGHT_BF16, w.shape[0], w.shape[1], w=w)


# ------------------------------------------------------------- LoRA linear
def sl_lora_linear_fwd(weight: Weight, X, A, B, r, alpha, Y, T_save, ws=None, stream=None):
    M = X.shape[0]
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(lib().sl_lora_linear_fwd(ctypes.byref(weight.desc), _ptr(X), M, _ptr(A), _ptr(B), int(r),
                                    float(alpha), _ptr(Y), _ptr(T_save), _ptr(ws), ws_bytes, _stream(stream)))


def sl_lora_linear_fwd_noalloc(weight: Weight, X, A, B, r, alpha, Y, T_save, stream=None):
    """The forward without a workspace argument: its scratch is a fixed 4 MiB device array in libsl.

    For callers that cannot allocate device memory; calls overlapping on the GPU race on the array."""
    M = X.shape[0]
    _check(lib().sl_lora_linear_fwd_noalloc(ctypes.byref(weight.desc), _ptr(X), M, _ptr(A), _ptr(B), int(r),
                                            float(alpha), _ptr(Y), _ptr(T_save), _stream(stream)))


def sl_lora_linear_workspace_size(M, N, K, r) -> int:
    return lib().sl_lora_linear_workspace_size(M, N, K, r)


def sl_lora_linear_bwd(weight: Weight, X, dY, A, B, r, alpha, T_save, dX, dA, dB, accumulate=False,
                       ws=None, stream=None):
    M = dY.shape[0]
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(lib().sl_lora_linear_bwd(ctypes.byref(weight.desc), _ptr(X), _ptr(dY), M, _ptr(A), _ptr(B), int(r),
                                    float(alpha), _ptr(T_save), _ptr(dX), _ptr(dA), _ptr(dB),
                                    int(bool(accumulate)), _ptr(ws), ws_bytes, _stream(stream)))


# ---------------------------------------------------------- projection groups
def _n_array(N_g):
    arr = (ctypes.c_int64 * len(N_g))(*[int(n) for n in N_g])
    return arr


def sl_lora_group_fwd(weight: Weight, N_g, X, A_cat, B_cat, r, alpha, Y_cat, T_cat, stream=None):
    """G projections reading X, weights/adapters back to back (see include/sl.h)."""
    n = _n_array(N_g)
    _check(lib().sl_lora_group_fwd(ctypes.byref(weight.desc), len(N_g), n, _ptr(X), X.shape[0], _ptr(A_cat),
                                   _ptr(B_cat), int(r), float(alpha), _ptr(Y_cat), _ptr(T_cat), _stream(stream)))


def sl_lora_group_bwd(weight: Weight, N_g, X, dY_cat, A_cat, B_cat, r, alpha, T_cat, dX, dA_cat, dB_cat,
                      accumulate=False, ws=None, stream=None):
    n = _n_array(N_g)
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(lib().sl_lora_group_bwd(ctypes.byref(weight.desc), len(N_g), n, _ptr(X), _ptr(dY_cat), dY_cat.shape[0],
                                   _ptr(A_cat), _ptr(B_cat), int(r), float(alpha), _ptr(T_cat), _ptr(dX),
                                   _ptr(dA_cat), _ptr(dB_cat), int(bool(accumulate)), _ptr(ws), ws_bytes,
                                   _stream(stream)))


def sl_lora_group_workspace_size(M, G, r):
    return int(lib().sl_lora_group_workspace_size(int(M), int(G), int(r)))


# ---------------------------------------------------------------- attention
def _ld(t):
    """Row stride (elements) of a 2-D row-major view."""
    return int(t.stride(0))


def sl_rope_table(S, theta, table, stream=None):
    """table fp32 [S, 128]: cos / sin of p * theta^(-i/64)."""
    _check(lib().sl_rope_table(int(S), float(theta), _ptr(table), _stream(stream)))


def sl_rope_apply(x, S, table, inverse=False, stream=None):
    """In place on the bf16 2-D view x [M, nheads*128] (any row stride)."""
    _check(lib().sl_rope_apply(_ptr(x), _ld(x), x.shape[0], x.shape[1] // 128, int(S), _ptr(table), int(inverse),
                               _stream(stream)))


def sl_attention_fwd(q, k, v, S, o, lse, stream=None):
    """Causal GQA attention on 2-D bf16 views q [M, H*128], k, v [M, Hkv*128]; o [M, H*128], lse fp32 [H, M]."""
    M, H, Hkv = q.shape[0], q.shape[1] // 128, k.shape[1] // 128
    _check(lib().sl_attention_fwd(_ptr(q), _ld(q), _ptr(k), _ld(k), _ptr(v), _ld(v), M, int(S), H, Hkv, _ptr(o),
                                  _ld(o), _ptr(lse), _stream(stream)))


def sl_attention_workspace_size(M, H):
    return int(lib().sl_attention_workspace_size(int(M), int(H)))


def sl_attention_bwd(q, k, v, o, dO, lse, S, dq, dk, dv, rope_table=None, ws=None, stream=None):
    import torch
    M, H, Hkv = q.shape[0], q.shape[1] // 128, k.shape[1] // 128
    if ws is None:
        ws = torch.empty(sl_attention_workspace_size(M, H), dtype=torch.uint8, device=q.device)
    _check(lib().sl_attention_bwd(_ptr(q), _ld(q), _ptr(k), _ld(k), _ptr(v), _ld(v), _ptr(o), _ld(o), _ptr(dO),
                                  _ld(dO), _ptr(lse), M, int(S), H, Hkv, _ptr(dq), _ld(dq), _ptr(dk), _ld(dk),
                                  _ptr(dv), _ld(dv), _ptr(rope_table), _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(stream)))


# -------------------------------------------------------------------- stack
def sl_stack_blob_layout(kind, D, Dkv, F):
    offs = (ctypes.c_size_t * 16)()
    total = ctypes.c_size_t(0)
    _check(lib().sl_stack_blob_layout(kind, D, Dkv, F, offs, ctypes.byref(total)))
    return list(offs), total.value


def sl_stack_dq_layout(D, Dkv, F):
    """Per projection of an NF4_DQ blob: dict(q_off, q_ld, a2_off, a2_ld, col0) (see include/sl.h)."""
    arrs = [(ctypes.c_size_t * 7)(), (ctypes.c_int64 * 7)(), (ctypes.c_size_t * 7)(), (ctypes.c_int64 * 7)(),
            (ctypes.c_int64 * 7)()]
    _check(lib().sl_stack_dq_layout(D, Dkv, F, *arrs))
    keys = ("q_off", "q_ld", "a2_off", "a2_ld", "col0")
    return [{k: int(a[p]) for k, a in zip(keys, arrs)} for p in range(7)]


PROJ_NAMES = ("q", "k", "v", "o", "gate", "up", "down")
# projections whose absmax a double-quantised blob keeps in one 8-bit array
DQ_GROUPS = ((0, 1, 2), (3,), (4, 5), (6,))


def proj_shapes(D, Dkv, F):
    """(N, K) of the seven projections of a layer, in blob order."""
    return [(D, D), (Dkv, D), (Dkv, D), (D, D), (F, D), (F, D), (D, F)]


def build_layer_blob(kind, D, Dkv, F, weights, stream=None, norms=None):
    """One layer blob on the device from its seven bf16 weights [N, K] (device tensors)
    and its two RMS-norm weights (fp32 [D] each; None: ones).

    NF4 blobs are filled by sl_nf4_quantize directly at the layout offsets;
    NF4_DQ blobs take the codes the same way and the absmax of each group
    (DQ_GROUPS) through sl_nf4_double_quantize; bf16 blobs hold the weights
    as they are (the storage dtype).
    """
    import torch
    offs, total = sl_stack_blob_layout(kind, D, Dkv, F)
    blob = torch.zeros(total, dtype=torch.uint8, device="cuda")
    shapes = proj_shapes(D, Dkv, F)
    for i in range(2):
        dst = blob[offs[14 + i]: offs[14 + i] + D * 4].view(torch.float32)
        dst.copy_(norms[i].reshape(-1).to(dst.device, torch.float32) if norms is not None else torch.ones(D))
    if kind == SL_WEIGHT_NF4_DQ:
        dq = sl_stack_dq_layout(D, Dkv, F)
        for group in DQ_GROUPS:
            K = shapes[group[0]][1]
            Ng = sum(shapes[p][0] for p in group)
            am = torch.empty(Ng * K // 64, dtype=torch.float32, device="cuda")
            for p in group:
                N = shapes[p][0]
                assert tuple(weights[p].shape) == (N, K)
                c0 = dq[p]["col0"] * K // 64
                sl_nf4_quantize(weights[p], blob[offs[2 * p]: offs[2 * p] + N * K // 2], am[c0: c0 + N * K // 64],
                                stream)
            d = dq[group[0]]
            rows = K // 64
            q = blob[d["q_off"]: d["q_off"] + rows * d["q_ld"]].view(torch.int8).view(rows, d["q_ld"])
            a2 = blob[d["a2_off"]: d["a2_off"] + rows * d["a2_ld"] * 4].view(torch.float32).view(rows, d["a2_ld"])
            sl_nf4_double_quantize(am, Ng, K, q, a2, stream=stream)
        torch.cuda.synchronize()   # the fp32 absmax `am` is freed on return
        return blob
    for p, ((N, K), W) in enumerate(zip(shapes, weights)):
        assert tuple(W.shape) == (N, K)
        if kind == SL_WEIGHT_NF4:
            codes = blob[offs[2 * p]: offs[2 * p] + N * K // 2]
            absmax = blob[offs[2 * p + 1]: offs[2 * p + 1] + N * K // 64 * 4].view(torch.float32)
            sl_nf4_quantize(W, codes, absmax, stream)
        else:
            blob[offs[2 * p]: offs[2 * p] + N * K * 2].view(torch.bfloat16).copy_(W.reshape(-1))
    return blob


def packed_views(shapes, dtype, device="cuda"):
    """Tensors of the given 2-D shapes back to back in one allocation (views, in order).

    Adapters of a layer allocated this way (A: [r, K_p], B: [N_p, r] in
    projection order) let the stack run q/k/v and gate/up as projection groups.
    """
    import torch
    total = sum(int(a) * int(b) for a, b in shapes)
    buf = torch.empty(total, dtype=dtype, device=device)
    views, off = [], 0
    for a, b in shapes:
        views.append(buf[off:off + a * b].view(a, b))
        off += a * b
    return views


def adapter_shapes(D, Dkv, F, r):
    """([r, K_p]) and ([N_p, r]) of the seven projections, in blob order."""
    shp = proj_shapes(D, Dkv, F)
    return [(r, K) for N, K in shp], [(N, r) for N, K in shp]


class Stack:
    """Owns an sl_stack handle (two device layer buffers, copy stream, events)."""

    def __init__(self, kind, D, Dkv, F, host_blobs, device_blobs=None, mixer=SL_MIX_TOKEN_LOCAL, seq_len=0,
                 rope_theta=0.0):
        """mixer=SL_MIX_ATTENTION: causal GQA attention over sequences of seq_len tokens."""
        self.L = len(host_blobs)
        self._host = host_blobs
        self._dev = device_blobs
        self._hp = (ctypes.c_void_p * self.L)(*[b.data_ptr() for b in host_blobs])
        self._dp = (ctypes.c_void_p * self.L)(*[b.data_ptr() for b in device_blobs]) if device_blobs else None
        self.desc = sl_stack_desc(self.L, kind, D, Dkv, F, self._hp, self._dp, int(mixer), int(seq_len),
                                  float(rope_theta))
        self.handle = ctypes.c_void_p()
        hb, bb = ctypes.c_size_t(0), ctypes.c_size_t(0)
        _check(lib().sl_stack_create(ctypes.byref(self.desc), ctypes.byref(self.handle), ctypes.byref(hb),
                                     ctypes.byref(bb)))
        self.host_bytes, self.buffer_bytes = hb.value, bb.value

    def workspace_size(self, M, r):
        return lib().sl_stack_workspace_size(self.handle, M, r)

    def step(self, mode, h0, dh_top, A, B, r, alpha, hL, dh0, dA, dB, ws, accumulate=False, stream=None):
        """One fwd+bwd step; A, B, dA, dB are lists of 7*L tensors (or None when r == 0)."""
        n = 7 * self.L
        arr = lambda ts: (ctypes.c_void_p * n)(*[t.data_ptr() for t in ts]) if ts is not None else None
        M = h0.shape[0]
        _check(lib().sl_stream_stack_step(self.handle, mode, _ptr(h0), M, _ptr(dh_top), arr(A), arr(B), int(r),
                                          float(alpha), _ptr(hL), _ptr(dh0), arr(dA), arr(dB),
                                          int(bool(accumulate)), _ptr(ws), ws.numel() * ws.element_size(),
                                          _stream(stream)))

    def sft_workspace_size(self, M, r, V, chunk_V):
        return int(lib().sl_sft_workspace_size(self.handle, int(M), int(r), int(V), int(chunk_V)))

    def sft_step(self, mode, tokens, labels, embed, norm_final, W_head, chunk_V, A, B, r, alpha, loss, dA, dB, ws,
                 accumulate=False, stream=None):
        """One complete SFT step (embedding, stack, final norm, head CE, backward); loss: fp32 [1] on the device."""
        n = 7 * self.L
        arr = lambda ts: (ctypes.c_void_p * n)(*[t.data_ptr() for t in ts]) if ts is not None else None
        _check(lib().sl_sft_step(self.handle, mode, _ptr(tokens), _ptr(labels), tokens.shape[0], _ptr(embed),
                                 embed.shape[0], _ptr(norm_final), _ptr(W_head), int(chunk_V), arr(A), arr(B),
                                 int(r), float(alpha), _ptr(loss), arr(dA), arr(dB), int(bool(accumulate)), _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(stream)))

    def last_step_stats(self):
        a, b = ctypes.c_uint64(0), ctypes.c_uint64(0)
        _check(lib().sl_stack_last_step_stats(self.handle, ctypes.byref(a), ctypes.byref(b)))
        return a.value, b.value

    def close(self):
        if self.handle:
            _check(lib().sl_stack_destroy(self.handle))
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------ cross-entropy
def sl_ce_workspace_size(M, D, V, chunk_V) -> int:
    return lib().sl_ce_workspace_size(M, D, V, chunk_V)


def sl_ce_fwd_bwd(H, W_head, labels, loss, dH, ws, chunk_V=8192, ignore_index=-100, stream=None):
    """loss: 1-element fp32 device tensor; dH: [M, D] fp32 device tensor."""
    M, D = H.shape
    V = W_head.shape[0]
    _check(lib().sl_ce_fwd_bwd(_ptr(H), M, D, _ptr(W_head), V, _ptr(labels), int(ignore_index), int(chunk_V),
                               _ptr(loss), _ptr(dH), _ptr(ws), ws.numel() * ws.element_size(),
                               _stream(stream)))

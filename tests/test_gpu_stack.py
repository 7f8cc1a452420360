"""The layer-streamed stack step on the GPU: oracle parity and streamed == resident bitwise."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import nf4, stack
from gpu_util import BF16_TOL, LOSS_TOL, dev_bf16, host, rel_fro

pytestmark = pytest.mark.gpu


class Setup:
    """Blobs (pinned host + device copies), adapters and grads for one synthetic stack."""

    def __init__(self, sl, kind, L, M, D, Dkv, F, r, alpha, seed, with_oracle=True, torch_weights=False,
                 packed=False, attn=None, norms=False):
        """packed: each layer's adapters (and gradients) back to back, so that
        NF4 stacks with M > 128 run q/k/v and gate/up as projection groups;
        attn = (S, theta): causal GQA attention over sequences of S tokens;
        norms: random RMS-norm weights (ones otherwise)."""
        self.attn = None if attn is None else dict(S=attn[0], theta=attn[1])
        self.sl, self.kind, self.L, self.M, self.D, self.Dkv, self.F, self.r, self.alpha = \
            sl, kind, L, M, D, Dkv, F, r, alpha
        self.packed = packed
        shapes = sl.proj_shapes(D, Dkv, F)
        self.host_blobs, self.dev_blobs, self.A, self.B, self.ref_layers = [], [], [], [], []
        if torch_weights:   # large stacks: weights drawn on the device from a seeded torch generator
            gen = torch.Generator(device="cuda").manual_seed(seed)
            rnd = lambda shape, std: (torch.randn(*shape, generator=gen, device="cuda") * std).to(torch.bfloat16)
            for l in range(L):
                Ws = [rnd((N, K), 0.02) for N, K in shapes]
                blob = sl.build_layer_blob(kind, D, Dkv, F, Ws)
                self._add_blob(blob)
                for N, K in shapes:
                    self.A.append(rnd((r, K), 0.02))
                    self.B.append(rnd((N, r), 0.02))
            self.h0 = torch.randn(M, D, generator=gen, device="cuda").to(torch.bfloat16).float()
            self.dh = torch.randn(M, D, generator=gen, device="cuda").to(torch.bfloat16).float()
        else:
            c = si.stack_case(seed, L, M, D, Dkv, F, r)
            for l in range(L):
                lw = c["layers"][l]
                Ws = [dev_bf16(lw[n]["W"]) for n in si.PROJ_NAMES]
                nw = [si.norm_weight(seed * 1000 + 500 + 2 * l + i, D) for i in range(2)] if norms else None
                blob = sl.build_layer_blob(kind, D, Dkv, F, Ws,
                                           norms=[torch.from_numpy(w) for w in nw] if norms else None)
                self._add_blob(blob)
                ref = {}
                if norms:
                    ref["norm_attn"], ref["norm_mlp"] = nw[0].astype(np.float64), nw[1].astype(np.float64)
                Wdq = dq_ref_weights(sl, lw) if with_oracle and kind == sl.SL_WEIGHT_NF4_DQ else None
                for n in si.PROJ_NAMES:
                    W = lw[n]["W"]
                    if with_oracle:
                        if kind == sl.SL_WEIGHT_NF4:
                            Wr = nf4.dequantize_bf16(*nf4.quantize(W), *W.shape)
                        elif kind == sl.SL_WEIGHT_NF4_DQ:
                            Wr = Wdq[n]
                        else:
                            Wr = W.astype(np.float64)
                        ref[n] = dict(W=Wr, A=lw[n]["A"].astype(np.float64), B=lw[n]["B"].astype(np.float64))
                    self.A.append(dev_bf16(lw[n]["A"]))
                    self.B.append(dev_bf16(lw[n]["B"]))
                self.ref_layers.append(ref)
            self.h0_np, self.dh_np = c["h0"], c["dh_top"]
            self.h0 = torch.from_numpy(c["h0"]).cuda()
            self.dh = torch.from_numpy(c["dh_top"]).cuda()
        if packed:
            sa, sb = sl.adapter_shapes(D, Dkv, F, r)
            for l in range(L):
                for views, src in ((sl.packed_views(sa, torch.bfloat16), self.A), (sl.packed_views(sb, torch.bfloat16), self.B)):
                    for p in range(7):
                        views[p].copy_(src[7 * l + p])
                        src[7 * l + p] = views[p]
        mix = dict(mixer=sl.SL_MIX_ATTENTION, seq_len=attn[0], rope_theta=attn[1]) if attn else {}
        self.stack = sl.Stack(kind, D, Dkv, F, self.host_blobs, self.dev_blobs, **mix)
        self.ws = torch.empty(self.stack.workspace_size(M, r), dtype=torch.uint8, device="cuda")

    def grads(self):
        """NaN-filled gradient buffers shaped like the adapters (packed like them)."""
        if not self.packed:
            return ([torch.full_like(a, float("nan"), dtype=torch.float32) for a in self.A],
                    [torch.full_like(b, float("nan"), dtype=torch.float32) for b in self.B])
        sa, sb = self.sl.adapter_shapes(self.D, self.Dkv, self.F, self.r)
        dA, dB = [], []
        for _ in range(self.L):
            dA += self.sl.packed_views(sa, torch.float32)
            dB += self.sl.packed_views(sb, torch.float32)
        for t in dA + dB:
            t.fill_(float("nan"))
        return dA, dB

    def _add_blob(self, blob):
        h = torch.empty(blob.numel(), dtype=torch.uint8, pin_memory=True)
        h.copy_(blob)
        self.host_blobs.append(h)
        self.dev_blobs.append(blob)

    def run(self, mode):
        sl = self.sl
        hL = torch.empty(self.M, self.D, device="cuda")
        dh0 = torch.empty_like(hL)
        dA, dB = self.grads()
        self.stack.step(mode, self.h0, self.dh, self.A, self.B, self.r, self.alpha, hL, dh0, dA, dB, self.ws)
        sl.sl_check_device_errors()
        return hL, dh0, dA, dB


def dq_ref_weights(sl, lw):
    """The oracle's bf16 weights of a double-quantised layer: each absmax group
    (q/k/v, o, gate/up, down) double-quantised as one [K/64, N_group] array."""
    out = {}
    for group in sl.DQ_GROUPS:
        names = [si.PROJ_NAMES[p] for p in group]
        qs = [nf4.quantize(lw[n]["W"]) for n in names]
        K = lw[names[0]]["W"].shape[1]
        Ns = [lw[n]["W"].shape[0] for n in names]
        q, a2 = nf4.double_quantize(np.concatenate([a for _, a in qs]), sum(Ns), K)
        ap = nf4.dq_absmax(q, a2, sum(Ns), K)
        off = 0
        for n, (codes, _), N in zip(names, qs, Ns):
            out[n] = nf4.dequantize_bf16(codes, ap[off * K // 64:(off + N) * K // 64], N, K)
            off += N
    return out


def same_bits(a, b):
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("kind_name", ["nf4", "bf16"])
def test_small_stack_matches_oracle_and_resident(gpu_lib, kind_name):
    sl = gpu_lib
    kind = sl.SL_WEIGHT_NF4 if kind_name == "nf4" else sl.SL_WEIGHT_BF16
    S = Setup(sl, kind, L=3, M=96, D=256, Dkv=128, F=512, r=16, alpha=32.0, seed=21)
    hL, dh0, dA, dB = S.run(sl.SL_MODE_STREAMED)
    h2d, kernels = S.stack.last_step_stats()
    assert h2d == (2 * S.L - 2) * S.stack.host_bytes // S.L and kernels > 0
    ohL, odh0, ograds = stack.stack_step(S.h0_np, S.dh_np, S.ref_layers, 32.0, rnd=True)
    assert rel_fro(host(hL), ohL) <= BF16_TOL
    assert rel_fro(host(dh0), odh0) <= BF16_TOL
    for l in range(S.L):
        for p, n in enumerate(si.PROJ_NAMES):
            assert rel_fro(host(dA[7 * l + p]), ograds[l][n][0]) <= BF16_TOL, (l, n)
            assert rel_fro(host(dB[7 * l + p]), ograds[l][n][1]) <= BF16_TOL, (l, n)
    # the streamed run equals the resident run bit for bit, and re-runs are identical
    r_ = S.run(sl.SL_MODE_RESIDENT)
    s2 = S.run(sl.SL_MODE_STREAMED)
    h2d2, _ = S.stack.last_step_stats()
    assert h2d2 == (2 * S.L - 4) * S.stack.host_bytes // S.L     # layers 0 and 1 still resident
    for x, y, z in zip((hL, dh0, *dA, *dB), (r_[0], r_[1], *r_[2], *r_[3]), (s2[0], s2[1], *s2[2], *s2[3])):
        assert same_bits(x, y) and same_bits(x, z)
    S.stack.close()


def test_grouped_stack_matches_oracle_and_resident(gpu_lib):
    """NF4, M > 128, adapters back to back: q/k/v and gate/up run as projection
    groups; same oracle tolerance, streamed == resident bit for bit, and close
    to the per-projection run of the same stack."""
    sl = gpu_lib
    S = Setup(sl, sl.SL_WEIGHT_NF4, L=3, M=160, D=512, Dkv=256, F=768, r=16, alpha=32.0, seed=23, packed=True)
    hL, dh0, dA, dB = S.run(sl.SL_MODE_STREAMED)
    ohL, odh0, ograds = stack.stack_step(S.h0_np, S.dh_np, S.ref_layers, 32.0, rnd=True)
    assert rel_fro(host(hL), ohL) <= BF16_TOL
    assert rel_fro(host(dh0), odh0) <= BF16_TOL
    for l in range(S.L):
        for p, n in enumerate(si.PROJ_NAMES):
            assert rel_fro(host(dA[7 * l + p]), ograds[l][n][0]) <= BF16_TOL, (l, n)
            assert rel_fro(host(dB[7 * l + p]), ograds[l][n][1]) <= BF16_TOL, (l, n)
    r_ = S.run(sl.SL_MODE_RESIDENT)
    for x, y in zip((hL, dh0, *dA, *dB), (r_[0], r_[1], *r_[2], *r_[3])):
        assert same_bits(x, y)
    # the same stack with separately allocated adapters runs projection by projection
    hL_u, dh0_u = torch.empty_like(hL), torch.empty_like(dh0)
    dA_u = [torch.empty(a.shape, device="cuda") for a in S.A]
    dB_u = [torch.empty(b.shape, device="cuda") for b in S.B]
    A_u = [a.clone() for a in S.A]
    B_u = [b.clone() for b in S.B]
    S.stack.step(sl.SL_MODE_STREAMED, S.h0, S.dh, A_u, B_u, 16, 32.0, hL_u, dh0_u, dA_u, dB_u, S.ws)
    sl.sl_check_device_errors()
    assert rel_fro(host(hL_u), host(hL)) <= 2e-3 and rel_fro(host(dh0_u), host(dh0)) <= 5e-3
    S.stack.close()


def test_two_full_width_layers_match_oracle(gpu_lib):
    """Llama-3.1-8B layer widths (bf16 base so the oracle needs no 218M-element quantisation), M=64."""
    sl = gpu_lib
    S = Setup(sl, sl.SL_WEIGHT_BF16, L=2, M=64, D=4096, Dkv=1024, F=14336, r=16, alpha=32.0, seed=5)
    hL, dh0, dA, dB = S.run(sl.SL_MODE_STREAMED)
    ohL, odh0, ograds = stack.stack_step(S.h0_np, S.dh_np, S.ref_layers, 32.0, rnd=True)
    errs = {"hL": rel_fro(host(hL), ohL), "dh0": rel_fro(host(dh0), odh0)}
    for l in range(2):
        for p, n in enumerate(si.PROJ_NAMES):
            errs[f"dA{l}{n}"] = rel_fro(host(dA[7 * l + p]), ograds[l][n][0])
            errs[f"dB{l}{n}"] = rel_fro(host(dB[7 * l + p]), ograds[l][n][1])
    print({k: round(float(v), 5) for k, v in errs.items()})
    assert max(errs.values()) <= BF16_TOL, errs
    S.stack.close()


@pytest.mark.parametrize("kind_name,L,packed", [("nf4", 6, False), ("nf4", 4, True), ("bf16", 4, False)])
def test_full_width_streamed_equals_resident_bitwise(gpu_lib, kind_name, L, packed):
    """8B-shaped layers (bf16 layers are 416 MiB, above the ~165 MiB size of the pages' NF4 bug);
    packed adapters run the NF4 layers' q/k/v and gate/up as projection groups."""
    sl = gpu_lib
    kind = sl.SL_WEIGHT_NF4 if kind_name == "nf4" else sl.SL_WEIGHT_BF16
    S = Setup(sl, kind, L=L, M=160, D=4096, Dkv=1024, F=14336, r=16, alpha=32.0, seed=77,
              with_oracle=False, torch_weights=True, packed=packed)
    a = S.run(sl.SL_MODE_STREAMED)
    b = S.run(sl.SL_MODE_RESIDENT)
    for x, y in zip((a[0], a[1], *a[2], *a[3]), (b[0], b[1], *b[2], *b[3])):
        assert same_bits(x, y)
    for g in a[2] + a[3]:            # every adapter received a finite, non-zero gradient
        assert torch.isfinite(g).all() and g.abs().sum() > 0
    S.stack.close()


def test_pageable_host_memory_rejected(gpu_lib):
    sl = gpu_lib
    offs, total = sl.sl_stack_blob_layout(sl.SL_WEIGHT_BF16, 256, 128, 512)
    pageable = torch.zeros(total, dtype=torch.uint8)
    with pytest.raises(sl.SLError) as e:
        sl.Stack(sl.SL_WEIGHT_BF16, 256, 128, 512, [pageable])
    assert e.value.status == sl.SL_ERR_INVALID


def test_gradient_accumulation_over_micro_batches(gpu_lib):
    """accumulate=1 adds each micro-batch's adapter gradients; bytes streamed per token stay the same."""
    sl = gpu_lib
    S = Setup(sl, sl.SL_WEIGHT_NF4, L=3, M=64, D=256, Dkv=128, F=512, r=16, alpha=32.0, seed=31, with_oracle=False)
    g = torch.Generator(device="cuda").manual_seed(5)
    batches = [(torch.randn(64, 256, generator=g, device="cuda"), torch.randn(64, 256, generator=g, device="cuda"))
               for _ in range(2)]
    hL, dh0 = torch.empty(64, 256, device="cuda"), torch.empty(64, 256, device="cuda")
    S.run(sl.SL_MODE_STREAMED)                   # warm: layers 0 and 1 stay resident from here on
    single = []
    for h0, dh in batches:
        dA = [torch.empty(a.shape, device="cuda") for a in S.A]
        dB = [torch.empty(b.shape, device="cuda") for b in S.B]
        S.stack.step(sl.SL_MODE_STREAMED, h0, dh, S.A, S.B, 16, 32.0, hL, dh0, dA, dB, S.ws)
        single.append((dA, dB, S.stack.last_step_stats()[0]))
    accA = [torch.empty(a.shape, device="cuda") for a in S.A]
    accB = [torch.empty(b.shape, device="cuda") for b in S.B]
    for i, (h0, dh) in enumerate(batches):
        S.stack.step(sl.SL_MODE_STREAMED, h0, dh, S.A, S.B, 16, 32.0, hL, dh0, accA, accB, S.ws, accumulate=i > 0)
    sl.sl_check_device_errors()
    for j in range(len(S.A)):
        assert torch.equal(accA[j], single[0][0][j] + single[1][0][j])
        assert torch.equal(accB[j], single[0][1][j] + single[1][1][j])
    assert single[0][2] == single[1][2]          # same streamed bytes for every micro-batch of M tokens
    S.stack.close()


def test_adapters_off_pass_equals_zero_B(gpu_lib):
    """r = 0 runs the frozen base alone: the same hL and dh0 as adapters whose B is zero."""
    sl = gpu_lib
    S = Setup(sl, sl.SL_WEIGHT_NF4, L=2, M=96, D=256, Dkv=128, F=512, r=16, alpha=32.0, seed=41, with_oracle=False)
    hL0, dh00 = torch.empty(96, 256, device="cuda"), torch.empty(96, 256, device="cuda")
    S.stack.step(sl.SL_MODE_STREAMED, S.h0, S.dh, None, None, 0, 32.0, hL0, dh00, None, None, S.ws)
    S.B = [torch.zeros_like(b) for b in S.B]
    hL1, dh01, dA, dB = S.run(sl.SL_MODE_STREAMED)
    assert torch.equal(hL0, hL1) and torch.equal(dh00, dh01)
    assert all(torch.count_nonzero(a) == 0 for a in dA)      # dA = s (dY B)^T X = 0 when B = 0
    assert all(torch.count_nonzero(b) > 0 for b in dB)
    S.stack.close()


@pytest.mark.parametrize("packed", [True, False])
def test_dq_stack_matches_oracle_and_resident(gpu_lib, packed):
    """Double-quantised absmax (8-bit, per absmax group): oracle parity on the
    grouped (packed adapters) and per-projection paths, streamed == resident
    bit for bit, and the blob is the smaller one that streams."""
    sl = gpu_lib
    S = Setup(sl, sl.SL_WEIGHT_NF4_DQ, L=3, M=160, D=512, Dkv=256, F=768, r=16, alpha=32.0, seed=29, packed=packed)
    hL, dh0, dA, dB = S.run(sl.SL_MODE_STREAMED)
    ohL, odh0, ograds = stack.stack_step(S.h0_np, S.dh_np, S.ref_layers, 32.0, rnd=True)
    assert rel_fro(host(hL), ohL) <= BF16_TOL
    assert rel_fro(host(dh0), odh0) <= BF16_TOL
    for l in range(S.L):
        for p, n in enumerate(si.PROJ_NAMES):
            assert rel_fro(host(dA[7 * l + p]), ograds[l][n][0]) <= BF16_TOL, (l, n)
            assert rel_fro(host(dB[7 * l + p]), ograds[l][n][1]) <= BF16_TOL, (l, n)
    r_ = S.run(sl.SL_MODE_RESIDENT)
    for x, y in zip((hL, dh0, *dA, *dB), (r_[0], r_[1], *r_[2], *r_[3])):
        assert same_bits(x, y)
    _, nf4_bytes = sl.sl_stack_blob_layout(sl.SL_WEIGHT_NF4, 512, 256, 768)
    assert S.stack.host_bytes // S.L < nf4_bytes
    S.stack.close()


def test_dq_stack_rejects_small_m(gpu_lib):
    sl = gpu_lib
    S = Setup(sl, sl.SL_WEIGHT_NF4_DQ, L=2, M=128, D=256, Dkv=256, F=512, r=8, alpha=16.0, seed=31,
              with_oracle=False)
    with pytest.raises(sl.SLError) as e:
        S.run(sl.SL_MODE_STREAMED)
    assert e.value.status == sl.SL_ERR_UNSUPPORTED
    S.stack.close()


@pytest.mark.parametrize("kind_name,packed", [("nf4", True), ("nf4", False), ("bf16", False)])
def test_attention_stack_matches_oracle_and_resident(gpu_lib, kind_name, packed):
    """The full decoder layer: weighted RMS norms, causal GQA attention with
    rotary positions over two sequences, SiLU-gated MLP; grouped (packed) and
    per-projection paths; streamed == resident bit for bit."""
    sl = gpu_lib
    kind = sl.SL_WEIGHT_NF4 if kind_name == "nf4" else sl.SL_WEIGHT_BF16
    S = Setup(sl, kind, L=2, M=256, D=512, Dkv=256, F=768, r=16, alpha=32.0, seed=37, packed=packed,
              attn=(128, 500000.0), norms=True)
    hL, dh0, dA, dB = S.run(sl.SL_MODE_STREAMED)
    ohL, odh0, ograds = stack.stack_step(S.h0_np, S.dh_np, S.ref_layers, 32.0, rnd=True, attn=S.attn)
    assert rel_fro(host(hL), ohL) <= BF16_TOL
    assert rel_fro(host(dh0), odh0) <= BF16_TOL
    for l in range(S.L):
        for p, n in enumerate(si.PROJ_NAMES):
            assert rel_fro(host(dA[7 * l + p]), ograds[l][n][0]) <= BF16_TOL, (l, n)
            assert rel_fro(host(dB[7 * l + p]), ograds[l][n][1]) <= BF16_TOL, (l, n)
    r_ = S.run(sl.SL_MODE_RESIDENT)
    for x, y in zip((hL, dh0, *dA, *dB), (r_[0], r_[1], *r_[2], *r_[3])):
        assert same_bits(x, y)
    S.stack.close()


def test_sft_step_matches_oracle_and_resident(gpu_lib):
    """One complete step: embedding rows, the streamed attention stack, the
    final weighted norm, the vocab-chunked head cross-entropy and the backward
    into every adapter."""
    sl = gpu_lib
    M, D, Dkv, F, V, r, alpha = 256, 512, 256, 768, 1536, 16, 32.0
    S = Setup(sl, sl.SL_WEIGHT_NF4, L=2, M=M, D=D, Dkv=Dkv, F=F, r=r, alpha=alpha, seed=43, packed=True,
              attn=(128, 500000.0), norms=True)
    c = si.sft_case(7, M, D, V)
    tok, lab = torch.from_numpy(c["tokens"]).cuda(), torch.from_numpy(c["labels"]).cuda()
    emb, head = dev_bf16(c["embed"]), dev_bf16(c["head"])
    nf = torch.from_numpy(c["norm_final"]).cuda()
    ws = torch.empty(S.stack.sft_workspace_size(M, r, V, 512), dtype=torch.uint8, device="cuda")

    def run(mode):
        loss = torch.empty(1, device="cuda")
        dA, dB = S.grads()
        S.stack.sft_step(mode, tok, lab, emb, nf, head, 512, S.A, S.B, r, alpha, loss, dA, dB, ws)
        sl.sl_check_device_errors()
        return loss, dA, dB

    loss, dA, dB = run(sl.SL_MODE_STREAMED)
    oloss, _, ograds = stack.sft_step(c["tokens"], c["labels"], c["embed"].astype(np.float64), S.ref_layers,
                                      c["norm_final"].astype(np.float64), c["head"].astype(np.float64), alpha,
                                      rnd=True, attn=S.attn)
    assert abs(loss.item() - oloss) <= LOSS_TOL * abs(oloss)
    for l in range(S.L):
        for p, n in enumerate(si.PROJ_NAMES):
            assert rel_fro(host(dA[7 * l + p]), ograds[l][n][0]) <= BF16_TOL, (l, n)
            assert rel_fro(host(dB[7 * l + p]), ograds[l][n][1]) <= BF16_TOL, (l, n)
    loss_r, dA_r, dB_r = run(sl.SL_MODE_RESIDENT)
    assert same_bits(loss, loss_r)
    for x, y in zip(dA + dB, dA_r + dB_r):
        assert same_bits(x, y)
    S.stack.close()


def test_sft_step_on_double_quantised_per_projection_stack(gpu_lib):
    """The SFT step on an 8-bit-absmax stack with separately allocated adapters
    (every projection its own GEMM): oracle parity and streamed == resident."""
    sl = gpu_lib
    M, D, Dkv, F, V, r, alpha = 256, 512, 256, 768, 1024, 8, 16.0
    S = Setup(sl, sl.SL_WEIGHT_NF4_DQ, L=2, M=M, D=D, Dkv=Dkv, F=F, r=r, alpha=alpha, seed=47, packed=False,
              attn=(256, 10000.0), norms=True)
    c = si.sft_case(9, M, D, V)
    tok, lab = torch.from_numpy(c["tokens"]).cuda(), torch.from_numpy(c["labels"]).cuda()
    emb, head = dev_bf16(c["embed"]), dev_bf16(c["head"])
    nf = torch.from_numpy(c["norm_final"]).cuda()
    ws = torch.empty(S.stack.sft_workspace_size(M, r, V, 256), dtype=torch.uint8, device="cuda")
    outs = []
    for mode in (sl.SL_MODE_STREAMED, sl.SL_MODE_RESIDENT):
        loss = torch.empty(1, device="cuda")
        dA, dB = S.grads()
        S.stack.sft_step(mode, tok, lab, emb, nf, head, 256, S.A, S.B, r, alpha, loss, dA, dB, ws)
        sl.sl_check_device_errors()
        outs.append((loss, dA, dB))
    oloss, _, ograds = stack.sft_step(c["tokens"], c["labels"], c["embed"].astype(np.float64), S.ref_layers,
                                      c["norm_final"].astype(np.float64), c["head"].astype(np.float64), alpha,
                                      rnd=True, attn=S.attn)
    loss, dA, dB = outs[0]
    assert abs(loss.item() - oloss) <= LOSS_TOL * abs(oloss)
    for l in range(S.L):
        for p, n in enumerate(si.PROJ_NAMES):
            assert rel_fro(host(dA[7 * l + p]), ograds[l][n][0]) <= BF16_TOL, (l, n)
            assert rel_fro(host(dB[7 * l + p]), ograds[l][n][1]) <= BF16_TOL, (l, n)
    assert same_bits(outs[0][0], outs[1][0])
    for x, y in zip(outs[0][1] + outs[0][2], outs[1][1] + outs[1][2]):
        assert same_bits(x, y)
    S.stack.close()

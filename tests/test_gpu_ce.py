"""Chunked LM-head cross-entropy on the GPU against the oracle."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import ce
from gpu_util import BF16_TOL, LOSS_TOL, dev_bf16, host, rel_fro

pytestmark = pytest.mark.gpu


def run(sl, H, W, lab, chunk):
    M, D = H.shape
    V = W.shape[0]
    loss = torch.empty(1, device="cuda")
    dH = torch.empty(M, D, device="cuda")
    ws = torch.empty(sl.sl_ce_workspace_size(M, D, V, chunk), dtype=torch.uint8, device="cuda")
    sl.sl_ce_fwd_bwd(H, W, lab, loss, dH, ws, chunk_V=chunk)
    sl.sl_check_device_errors()
    return float(loss.item()), dH


@pytest.mark.parametrize("M,D,V,chunk,w_std", [
    (200, 256, 1056, 512, 0.05),     # ragged last chunk (32 columns, one empty half tile)
    (130, 512, 4096, 1024, 0.05),
    (64, 256, 256, 8192, 0.05),      # one chunk larger than the vocabulary
    (192, 256, 2048, 256, 0.5),      # logits spread ~ +-25: the running max moves across 8 chunks
    (1280, 1024, 8192, 8192, 0.05),  # CTA pairs: 160 logits tiles on 74 clusters, the 12 tail tiles split along K
    (129, 256, 768, 512, 0.05),      # CTA pairs with one row in the second CTA; last chunk 256 wide
])
def test_ce_matches_oracle(gpu_lib, M, D, V, chunk, w_std):
    c = si.ce_case(3 + M, M, D, V, h_std=1.0, w_std=w_std)
    loss, dH = run(gpu_lib, dev_bf16(c["H"]), dev_bf16(c["W"]), torch.from_numpy(c["labels"]).cuda(), chunk)
    ol, odH, osoft = ce.ce_fwd_bwd(c["H"], c["W"], c["labels"], want_soft=True)
    assert abs(loss - ol) <= LOSS_TOL * abs(ol)
    assert rel_fro(host(dH), odH) <= BF16_TOL
    nv = int(np.sum(c["labels"] != -100))
    valid = c["labels"] != -100
    gsoft = host(dH)
    gsoft[valid] += c["W"][c["labels"][valid]] / nv
    assert rel_fro(gsoft, osoft) <= BF16_TOL
    assert np.all(host(dH)[~valid] == 0)


def test_ce_no_valid_rows(gpu_lib):
    c = si.ce_case(9, 64, 256, 512)
    lab = torch.full((64,), -100, dtype=torch.int32, device="cuda")
    loss, dH = run(gpu_lib, dev_bf16(c["H"]), dev_bf16(c["W"]), lab, 256)
    assert loss == 0.0 and torch.count_nonzero(dH) == 0


def test_ce_full_size(gpu_lib):
    """LM head of Llama-3.1-8B: M=2048, D=4096, V=128256, 5% ignored, chunk 8192.

    The loss is checked against the oracle over all rows; dH on 24 sampled rows."""
    M, D, V = 2048, 4096, 128256
    c = si.ce_case(5, M, D, V)
    loss, dH = run(gpu_lib, dev_bf16(c["H"]), dev_bf16(c["W"]), torch.from_numpy(c["labels"]).cuda(), 8192)
    lab = c["labels"]
    nv = int(np.sum(lab != -100))
    W64 = c["W"].astype(np.float64)
    terms, _, _ = ce.ce_rows(c["H"], W64, lab, nv, want_grad=False)
    ol = terms.sum() / nv
    assert abs(loss - ol) <= LOSS_TOL * abs(ol)
    rows = np.random.default_rng(1).choice(M, 24, replace=False)
    _, odH, osoft = ce.ce_rows(c["H"][rows], W64, lab[rows], nv, want_soft=True)
    g = host(dH)[rows]
    assert rel_fro(g, odH) <= BF16_TOL
    v = lab[rows] != -100
    g[v] += c["W"][lab[rows][v]] / nv
    assert rel_fro(g, osoft) <= BF16_TOL

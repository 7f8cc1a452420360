"""CPU-side checks of the workspace-size calls (host arithmetic only, no GPU):
every size covers what the header says the workspace holds, is a multiple of
256 bytes where the header asks for 256-byte alignment, and is zero when the
call needs no workspace."""
import pytest

import layer_streamed_qlora_linear_b300 as sl


@pytest.mark.parametrize("M,r", [(1, 8), (1024, 16), (2048, 32), (4097, 24)])
def test_linear_and_group_workspaces_hold_U(M, r):
    lin = sl.sl_lora_linear_workspace_size(M, 4096, 4096, r)
    assert lin >= M * r * 4 and lin % 256 == 0             # U [M, r] fp32
    for G in (1, 2, 3):
        grp = sl.sl_lora_group_workspace_size(M, G, r)
        assert grp >= M * G * r * 4 and grp % 256 == 0     # U_cat [M, G r] fp32
    assert sl.sl_lora_linear_workspace_size(M, 4096, 4096, 0) == 0   # no adapter, no side product
    assert sl.sl_lora_group_workspace_size(M, 3, 0) == 0


@pytest.mark.parametrize("M,H", [(128, 4), (1024, 32), (8192, 32)])
def test_attention_workspace_holds_di_and_the_head_partials(M, H):
    ws = sl.sl_attention_workspace_size(M, H)
    assert ws >= M * H * 4 + 2 * M * H * 128 * 4             # Di [H, M]; dK, dV partials [H, M, 128]
    assert ws >= sl.sl_attention_workspace_size(M // 2, H)
    assert sl.sl_attention_workspace_size(0, H) == 0


@pytest.mark.parametrize("M,V,chunk", [(2048, 128256, 8192), (64, 1000, 256), (300, 5000, 2048)])
def test_ce_workspace_holds_one_chunk_and_its_partials(M, V, chunk):
    ws = sl.sl_ce_workspace_size(M, 4096, V, chunk)
    halves = 2 * -(-chunk // 256)
    assert ws >= M * chunk * 2 + 2 * M * halves * 4 + 7 * M * 4  # bf16 exp chunk, (max, sum) partials, row state
    assert ws % 256 == 0
    # never the logits: the size does not depend on the vocabulary (for M > 128 it
    # includes a fixed split-K scratch of the CTA-pair GEMMs), far below them at full size
    assert sl.sl_ce_workspace_size(M, 4096, 4 * V, chunk) == ws
    if V >= 100000:
        assert ws < M * V * 2 // 8
    assert sl.sl_ce_workspace_size(0, 4096, V, chunk) == 0

"""Host logic of the layer blob layouts (no GPU): regions are disjoint and
aligned, and the double-quantised blob of a Llama-3.1-8B-shaped layer has
the size the pages give for one streamed layer buffer."""
import layer_streamed_qlora_linear_b300 as sl

LLAMA8B = (4096, 1024, 14336)


def regions(kind, D, Dkv, F):
    offs, total = sl.sl_stack_blob_layout(kind, D, Dkv, F)
    shapes = sl.proj_shapes(D, Dkv, F)
    out = []
    for p, (N, K) in enumerate(shapes):
        if kind == sl.SL_WEIGHT_BF16:
            out.append((offs[2 * p], N * K * 2))
        else:
            out.append((offs[2 * p], N * K // 2))
            if kind == sl.SL_WEIGHT_NF4:
                out.append((offs[2 * p + 1], N * K // 64 * 4))
    if kind == sl.SL_WEIGHT_NF4_DQ:
        dq = sl.sl_stack_dq_layout(D, Dkv, F)
        for group in sl.DQ_GROUPS:
            d = dq[group[0]]
            rows = shapes[group[0]][1] // 64
            out.append((d["q_off"], rows * d["q_ld"]))
            out.append((d["a2_off"], rows * d["a2_ld"] * 4))
    return out, total


def test_regions_disjoint_aligned_and_inside():
    for kind in (sl.SL_WEIGHT_NF4, sl.SL_WEIGHT_BF16, sl.SL_WEIGHT_NF4_DQ):
        for dims in (LLAMA8B, (512, 256, 768), (3584, 512, 18944)):
            regs, total = regions(kind, *dims)
            regs.sort()
            for (o, n), (o2, _) in zip(regs, regs[1:]):
                assert o % 256 == 0 and o + n <= o2
            assert regs[-1][0] + regs[-1][1] <= total


def test_dq_groups_share_arrays_with_column_offsets():
    D, Dkv, F = LLAMA8B
    dq = sl.sl_stack_dq_layout(D, Dkv, F)
    shapes = sl.proj_shapes(D, Dkv, F)
    for group in sl.DQ_GROUPS:
        col = 0
        Ng = sum(shapes[p][0] for p in group)
        for p in group:
            assert dq[p]["q_off"] == dq[group[0]]["q_off"] and dq[p]["a2_off"] == dq[group[0]]["a2_off"]
            assert dq[p]["col0"] == col and col % 256 == 0
            assert dq[p]["q_ld"] == Ng and dq[p]["a2_ld"] >= 2 * Ng // 256 and dq[p]["a2_ld"] % 4 == 0
            col += shapes[p][0]


def test_dq_blob_is_the_pages_layer_buffer():
    _, dq_total = sl.sl_stack_blob_layout(sl.SL_WEIGHT_NF4_DQ, *LLAMA8B)
    _, nf4_total = sl.sl_stack_blob_layout(sl.SL_WEIGHT_NF4, *LLAMA8B)
    # two 113 MB layer buffers and a 3.60 GB pinned store of 32 layers
    assert abs(dq_total / 1e6 - 113) / 113 < 0.01
    assert abs(32 * dq_total / 1e9 - 3.60) / 3.60 < 0.01
    assert 0.91 < dq_total / nf4_total < 0.92          # the 8-bit absmax saves about 8 % of the stream


def test_dq_layout_rejects_narrow_kv():
    import pytest
    with pytest.raises(sl.SLError):
        sl.sl_stack_blob_layout(sl.SL_WEIGHT_NF4_DQ, 256, 128, 512)

"""bench.py's host-side staging for the end-to-end step (no GPU): the inputs of
a step are packed back to back into one buffer at 256-byte aligned offsets and
viewed back as the original tensors, so one copy moves them all."""
import torch

import bench
import workloads


def test_staging_layout_is_aligned_and_round_trips():
    batch = workloads.make_batch(workloads.WORKLOADS["tiny_bf16_1x4k"])
    ins = [batch.q, batch.page_table, batch.slot_ids, batch.row_lens,
           torch.rand(batch.R, batch.M)]
    offs, total = bench._layout(ins)
    assert total % 256 == 0
    end = 0
    for t, (o, nb) in zip(ins, offs):
        assert o % 256 == 0 and o >= end          # aligned, no overlap
        assert nb == t.numel() * t.element_size()
        end = o + nb
    assert end <= total
    buf = torch.zeros(total, dtype=torch.uint8)
    views = bench._views(buf, ins, offs)
    for v, t in zip(views, ins):
        v.copy_(t)
    for v, t in zip(bench._views(buf, ins, offs), ins):
        assert v.dtype == t.dtype and v.shape == t.shape and v.is_contiguous()
        assert torch.equal(v.view(torch.uint8), t.contiguous().view(torch.uint8))


def test_staging_views_share_the_buffer():
    a = torch.arange(10, dtype=torch.int32)
    b = torch.ones(3, 5, dtype=torch.float32)
    offs, total = bench._layout([a, b])
    buf = torch.zeros(total, dtype=torch.uint8)
    va, vb = bench._views(buf, [a, b], offs)
    va.copy_(a)
    vb.copy_(b)
    # writing through the views lands in the one buffer a single copy moves
    assert torch.equal(buf[offs[0][0]:offs[0][0] + 40].view(torch.int32), a)
    assert torch.equal(buf[offs[1][0]:offs[1][0] + 60].view(torch.float32).view(3, 5), b)


def test_kernel_hash_ignores_comments_and_layout_only():
    a = 'int a = 1; // note\n/* block\n note */ const char* s = "x // kept \\" /* kept */";\n'
    b = 'int a = 1;\nconst char* s = "x // kept \\" /* kept */";  // other note\n'
    assert bench.code_only(a) == bench.code_only(b)
    # a change of code, or of a literal's contents, is a change
    assert bench.code_only(a) != bench.code_only(a.replace("a = 1", "a = 2"))
    assert bench.code_only(a) != bench.code_only(a.replace("// kept", "//  kept"))

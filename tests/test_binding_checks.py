"""The Python binding's extent checks (no GPU needed).

The C ABI takes bare addresses, so it cannot see how large a buffer is; the
binding can. Every wrapper refuses, with ValueError and before any CUDA or
library call, a tensor smaller than the bytes the call would touch under the
plan (T, the padded T, T/P and the row width), parts of one argument that
differ in shape or dtype, and index outputs that are not int32. Tensors of
the right size pass these checks and reach the library, which here refuses a
stand-in plan whose handle is NULL.
"""
import pytest
import torch

BF16, F32, I32 = torch.bfloat16, torch.float32, torch.int32


def _plan(cpt, P=4, n=2, T=64, Tpad=None, layout=0):
    return cpt.Plan(0, None, layout, P, n, T, T if Tpad is None else Tpad)


def _reaches_library(cpt, fn):
    with pytest.raises(cpt.CptError) as ei:
        fn()
    assert ei.value.status == cpt.CPT_ERR_INVALID_ARG
    return str(ei.value)


def _refused(fn, match):
    with pytest.raises(ValueError, match=match):
        fn()


def test_grad_return_extents(cpt):
    plan = _plan(cpt)
    w, o = torch.zeros((4, 64, 16), dtype=BF16), torch.zeros((4, 16, 16), dtype=BF16)
    assert "plan is NULL" in _reaches_library(cpt, lambda: cpt.cpt_grad_return(plan, w, None, o, None, stream=0))
    _refused(lambda: cpt.cpt_grad_return(plan, w[:, :63], None, o, None, stream=0), "contiguous")
    _refused(lambda: cpt.cpt_grad_return(plan, torch.zeros((4, 63, 16), dtype=BF16), None, o, None, stream=0),
             "dk_writers")
    _refused(lambda: cpt.cpt_grad_return(plan, w, None, torch.zeros((4, 15, 16), dtype=BF16), None, stream=0),
             "dk_owners")
    _refused(lambda: cpt.cpt_grad_return(plan, w, None, torch.zeros((4, 32, 8), dtype=BF16), None, stream=0),
             "rows have")
    short = [torch.zeros((64, 16), dtype=BF16) for _ in range(3)] + [torch.zeros((32, 16), dtype=BF16)]
    _refused(lambda: cpt.cpt_grad_return(plan, short, None, o, None, stream=0), "differ")
    _refused(lambda: cpt.cpt_grad_return(plan, w, w.float(), o, o, stream=0), "dV pair")
    _refused(lambda: cpt.cpt_grad_return_accumulate(plan, w, None, torch.zeros((4, 15, 16), dtype=BF16), None,
                                                    stream=0), "dk_owners")
    _refused(lambda: cpt.cpt_grad_return_rows(plan, w[:, :60].contiguous(), None, o, None, 0, 8, stream=0),
             "dk_writers")
    # float32 owners of bf16 writers hold twice the bytes: right size passes
    _reaches_library(cpt, lambda: cpt.cpt_grad_return(plan, w, None, o.float(), None, stream=0))


def test_padded_plan_sizes_by_the_padded_total(cpt):
    plan = _plan(cpt, T=60, Tpad=64, layout=cpt.CPT_LAYOUT_DUAL_CHUNK_SWAP_PADDED)
    o = torch.zeros((4, 16, 16), dtype=BF16)
    _refused(lambda: cpt.cpt_grad_return(plan, torch.zeros((4, 60, 16), dtype=BF16), None, o, None, stream=0),
             "dk_writers")
    _reaches_library(cpt, lambda: cpt.cpt_grad_return(plan, torch.zeros((4, 64, 16), dtype=BF16), None, o, None,
                                                      stream=0))
    q = torch.zeros((60, 16), dtype=BF16)
    _reaches_library(cpt, lambda: cpt.cpt_partition(plan, [q], [torch.zeros((4, 16, 16), dtype=BF16)], stream=0))
    _refused(lambda: cpt.cpt_partition(plan, [q], [torch.zeros((4, 15, 16), dtype=BF16)], stream=0), "dsts")
    _reaches_library(cpt, lambda: cpt.cpt_restore(plan, [torch.zeros((4, 16, 16), dtype=BF16)], [q], stream=0))
    _refused(lambda: cpt.cpt_restore(plan, [torch.zeros((4, 15, 16), dtype=BF16)], [q], stream=0), "srcs")


def test_partition_and_restore_extents(cpt):
    plan = _plan(cpt)
    q, loc = torch.zeros((64, 16), dtype=BF16), torch.zeros((4, 16, 16), dtype=BF16)
    _reaches_library(cpt, lambda: cpt.cpt_partition(plan, [q, q], [loc, loc.clone()], stream=0))
    _refused(lambda: cpt.cpt_partition(plan, [q], [loc, loc], stream=0), "differ in length")
    _refused(lambda: cpt.cpt_partition(plan, [q[:63]], [loc], stream=0), "srcs")
    _refused(lambda: cpt.cpt_partition(plan, [q], [loc[:3]], stream=0), "dsts")
    _refused(lambda: cpt.cpt_partition(plan, [q], [loc.float()], stream=0), "dtype")
    _refused(lambda: cpt.cpt_partition_rows(plan, [q[:32]], [loc], 0, 16, stream=0), "srcs")
    _refused(lambda: cpt.cpt_restore(plan, [loc[:3]], [q], stream=0), "srcs")
    _refused(lambda: cpt.cpt_restore(plan, [loc], [q[:63]], stream=0), "dsts")


def test_map_metadata_and_lengths_extents(cpt):
    plan = _plan(cpt, P=4, n=3, T=64)
    _reaches_library(cpt, lambda: cpt.cpt_index_map(plan, torch.zeros(64, dtype=I32), torch.zeros(64, dtype=I32),
                                                    stream=0))
    _refused(lambda: cpt.cpt_index_map(plan, torch.zeros(63, dtype=I32), stream=0), "l2g")
    _refused(lambda: cpt.cpt_index_map(plan, torch.zeros(64, dtype=torch.int64), stream=0), "dtype")
    _refused(lambda: cpt.cpt_index_map(plan, torch.zeros(64, dtype=I32), torch.zeros(32, dtype=I32), stream=0),
             "g2l")
    ok = [torch.zeros(4, dtype=I32), torch.zeros(4, dtype=I32), torch.zeros((4, 4), dtype=I32),
          torch.zeros(5, dtype=I32)]
    _reaches_library(cpt, lambda: cpt.cpt_thd_metadata(plan, *ok, stream=0))
    _refused(lambda: cpt.cpt_thd_metadata(plan, ok[0], ok[1], torch.zeros((4, 3), dtype=I32), ok[3], stream=0),
             "cu_local")
    _refused(lambda: cpt.cpt_thd_metadata(plan, ok[0], ok[1], ok[2], torch.zeros(4, dtype=I32), stream=0),
             "seg_offsets")
    _reaches_library(cpt, lambda: cpt.cpt_thd_real_lengths(plan, torch.zeros((4, 3), dtype=I32), stream=0))
    _refused(lambda: cpt.cpt_thd_real_lengths(plan, torch.zeros((4, 2), dtype=I32), stream=0), "real_len")


def test_scatter_and_slot_reduce_extents(cpt):
    plan = _plan(cpt)
    src = torch.zeros((64, 16), dtype=BF16)
    slots = [torch.zeros((16, 16), dtype=BF16) for _ in range(4)]
    _reaches_library(cpt, lambda: cpt.cpt_grad_scatter(plan, 1, src, slots, slots[1], stream=0))
    _refused(lambda: cpt.cpt_grad_scatter(plan, 1, src[:63], slots, slots[1], stream=0), "src")
    _refused(lambda: cpt.cpt_grad_scatter(plan, 1, src, [s.float() for s in slots], slots[1], stream=0), "dtype")
    _refused(lambda: cpt.cpt_grad_scatter(plan, 1, src, [s[:15] for s in slots], slots[1], stream=0), "slots")
    dst = torch.zeros((16, 16), dtype=F32)
    with pytest.raises(cpt.CptError):  # CPU memory: the library's device check refuses it
        cpt.cpt_slot_reduce(slots, dst, stream=0)
    _refused(lambda: cpt.cpt_slot_reduce(slots, dst[:15], stream=0), "dst")
    _refused(lambda: cpt.cpt_slot_reduce(slots, dst, torch.zeros(1, dtype=torch.int64), stream=0), "status")


def test_noalloc_checks_only_batches_within_its_limits(cpt):
    w, o = torch.zeros((2, 8, 8), dtype=BF16), torch.zeros((2, 4, 8), dtype=BF16)
    _refused(lambda: cpt.cpt_grad_return_noalloc(0, 2, [0, 12], 12, w, None, o, None, stream=0), "dk_writers")
    # padded layout: [0, 5] pads to 8 rows, which these buffers hold
    with pytest.raises(cpt.CptError):  # CPU memory: the library's device check refuses it
        cpt.cpt_grad_return_noalloc(3, 2, [0, 5], 5, w, None, o, None, stream=0)
    big = cpt.CPT_NOALLOC_MAX_TOKENS + 4
    msg = _reaches_library(cpt, lambda: cpt.cpt_grad_return_noalloc(0, 2, [0, big], big, w, None, o, None, stream=0))
    assert "no-allocation limit" in msg

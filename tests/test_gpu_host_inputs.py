"""Host inputs that the library copies to the device: the plan calls take
cu_seqlens from host memory, and the caller may reuse that buffer as soon as
the call returns, even when it is pinned (a pinned source would otherwise
still be read by a copy in flight behind earlier work on the stream).

Each test keeps the stream busy with a bounded spin kernel, calls the C ABI
with cu_seqlens in pinned host memory, overwrites the buffer at once, and
checks the result against the oracle's map or the plan-based call. A copy
that read the overwritten buffer would build the map of all-zero
boundaries, whose entries stay in range, so a failure shows as wrong values
and never as a fault.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from context_attention_token_gb300 import synth
from gpu_helpers import bits, to_dev, to_host

pytestmark = pytest.mark.gpu

SPIN_CYCLES = 40_000_000  # about 20 ms at GB300 clocks, long enough to hold the copy


def _pinned_cu(lens):
    cu = synth.cu_from_lengths(lens)
    return cu, torch.tensor(cu, dtype=torch.int32).pin_memory()


@pytest.mark.parametrize("layout", [0, 1, 3], ids=["per_document", "packed", "padded"])
def test_plan_create_copies_pinned_cu_seqlens_before_returning(cpt, cuda_device, layout):
    P = 4
    lens = [40, 8, 72, 24] if layout != 3 else [37, 5, 70, 21]
    cu, pinned = _pinned_cu(lens)
    T, n = int(cu[-1]), len(lens)
    ws = torch.empty(max(cpt.cpt_plan_workspace_bytes(layout, P, n, T), 256), dtype=torch.uint8,
                     device="cuda")
    stream = torch.cuda.current_stream()
    torch.cuda._sleep(SPIN_CYCLES)
    h = ctypes.c_void_p()
    st = cpt._lib.cpt_plan_create(layout, P, ctypes.c_void_p(pinned.data_ptr()), n, T,
                                  ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                  ctypes.c_void_p(stream.cuda_stream), ctypes.byref(h))
    assert st == 0, cpt._lib.cpt_last_error_string()
    pinned.zero_()  # the caller reuses its buffer at once
    tpad = ctypes.c_int64()
    assert cpt._lib.cpt_plan_padded_tokens(h.value, ctypes.byref(tpad)) == 0
    plan = cpt.Plan(h.value, ws, layout, P, n, T, tpad.value)
    l2g = torch.empty(tpad.value, dtype=torch.int32, device="cuda")
    g2l = torch.empty_like(l2g)
    cpt.cpt_index_map(plan, l2g, g2l)
    # the metadata too: the packed map is the identity whatever cu_seqlens holds
    meta = [torch.empty(P, dtype=torch.int32, device="cuda"), torch.empty(P, dtype=torch.int32, device="cuda"),
            torch.empty((P, n + 1), dtype=torch.int32, device="cuda"),
            torch.empty(P + 1, dtype=torch.int32, device="cuda")]
    cpt.cpt_thd_metadata(plan, *meta)
    torch.cuda.synchronize()
    if layout == 3:
        cup, want_l2g, want_g2l = oracle.padded_index_map(P, cu)
        want_meta = oracle.thd_metadata(0, P, cup, tpad.value)
    else:
        want_l2g, want_g2l = oracle.index_map(layout, P, cu, T)
        want_meta = oracle.thd_metadata(layout, P, cu, T)
    assert np.array_equal(to_host(l2g), want_l2g)
    assert np.array_equal(to_host(g2l), want_g2l)
    for got_m, want_m in zip(meta, want_meta):
        assert np.array_equal(to_host(got_m), want_m)
    cpt.cpt_plan_destroy(plan)


def test_noalloc_copies_pinned_cu_seqlens_before_returning(cpt, cuda_device):
    P, row = 4, 256
    lens = [48, 16, 96, 32]
    cu, pinned = _pinned_cu(lens)
    T, n = int(cu[-1]), len(lens)
    rng = np.random.default_rng(4242)
    dkw = torch.stack([to_dev(synth.uniform_bf16(rng, (T, row))) for _ in range(P)])
    got = torch.empty((P, T // P, row), dtype=torch.bfloat16, device="cuda")
    want = torch.empty_like(got)
    plan = cpt.cpt_plan_create(0, P, cu, T)
    cpt.cpt_grad_return(plan, dkw, None, want, None)
    w, o = cpt._Parts(dkw, P), cpt._Parts(got, P)
    stream = torch.cuda.current_stream()
    torch.cuda._sleep(SPIN_CYCLES)
    st = cpt._lib.cpt_grad_return_noalloc(0, P, ctypes.c_void_p(pinned.data_ptr()), n, T, w.array(), None,
                                          o.array(), None, w.row_elems(), w.code(), o.code(),
                                          ctypes.c_void_p(stream.cuda_stream))
    assert st == 0, cpt._lib.cpt_last_error_string()
    pinned.zero_()
    torch.cuda.synchronize()
    assert np.array_equal(bits(to_host(got)), bits(to_host(want)))

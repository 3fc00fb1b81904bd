"""The bounded waits of the bulk-copy kernels, made to run out on purpose.

A test switch makes every bulk-copy mbarrier announce 16 bytes more than its
copies deliver. Every copy still completes and nothing faults, but no wait
can finish, so each one gives up after its budget of about a second. The
gradient return, the row gather and the slot reduce must count those
timeouts and return, leaving the context usable (the row gather in both its
forms: row blocks for a permuted map, a straight copy for the identity). With the switch off again,
the same calls must give the oracle's bits and count nothing.
"""
import numpy as np
import pytest
import torch

import oracle
from context_attention_token_gb300 import synth
from gpu_helpers import bits, to_dev, to_host

pytestmark = pytest.mark.gpu


def _run_all(cpt, plan, q, part, dkw, dko, slots, red, plan_packed, part_packed):
    cpt.cpt_partition(plan, [q], [part])
    cpt.cpt_partition(plan_packed, [q], [part_packed])  # identity map: the straight copy
    cpt.cpt_grad_return(plan, dkw, None, dko, None)
    cpt.cpt_slot_reduce(slots, red)
    torch.cuda.synchronize()


def test_bulk_waits_that_run_out_are_counted_and_the_context_recovers(cpt, cuda_device):
    P, T, row = 4, 64, 512  # 1 KB bf16 rows
    cu = synth.cu_from_lengths([T])
    rng = np.random.default_rng(9900)
    xq = synth.uniform_bf16(rng, (T, row))
    xw = [synth.uniform_bf16(rng, (T, row)) for _ in range(P)]
    xs = [synth.uniform_f32(rng, (4096,)) for _ in range(3)]  # 16 KB slots: four 4 KB chunks
    plan = cpt.cpt_plan_create(0, P, cu, T)
    plan_packed = cpt.cpt_plan_create(1, P, cu, T)
    q = to_dev(xq)
    part = torch.empty((P, T // P, row), dtype=torch.bfloat16, device="cuda")
    part_packed = torch.empty_like(part)
    dkw = torch.stack([to_dev(w) for w in xw])
    dko = torch.empty((P, T // P, row), dtype=torch.bfloat16, device="cuda")
    slots = [to_dev(x) for x in xs]
    red = torch.empty(4096, device="cuda")

    cpt.cpt_kernel_wait_timeouts(reset=True)
    cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_BULK)
    try:
        cpt.cpt_test_stall_bulk_waits(True)
        try:
            _run_all(cpt, plan, q, part, dkw, dko, slots, red, plan_packed, part_packed)
        finally:
            cpt.cpt_test_stall_bulk_waits(False)
        stalled = cpt.cpt_kernel_wait_timeouts(reset=True)
        # at least one give-up in each of the four kernels
        assert stalled >= 4, stalled

        _run_all(cpt, plan, q, part, dkw, dko, slots, red, plan_packed, part_packed)
        assert cpt.cpt_kernel_wait_timeouts() == 0
    finally:
        cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_AUTO)
    l2g, _ = oracle.index_map(0, P, cu, T)
    assert np.array_equal(to_host(part).reshape(T, row), oracle.partition(l2g, xq))
    assert np.array_equal(to_host(part_packed).reshape(T, row), xq)
    want = oracle.grad_return(l2g, xw, oracle.BF16)
    got = to_host(dko)
    for o in range(P):
        assert np.array_equal(got[o], want[o])
    assert np.array_equal(bits(to_host(red)), bits(oracle.slot_reduce(xs, oracle.F32)))

"""Staged owner-gradient return on one GPU: P writer streams scatter and
publish their epoch, P owner streams wait and reduce ("Add stream-ordered CP
gradient return primitive", TransformerEngine PR 3235, sequence diagram).

The staged result must equal the fused kernel and the oracle bit for bit.
Failures are injected without any GPU fault: a publish the host never
enqueues (caught on the host), and a flag row that nothing sets after it is
cleared on the owner's own stream (the bounded device check runs out of time
and the reduce is skipped).
"""
import numpy as np
import pytest
import torch

import oracle
from context_attention_token_gb300 import synth
from gpu_helpers import to_dev, to_host

pytestmark = pytest.mark.gpu


def _setup(cpt, P, layout, lens, row_shape=(4, 32), seed=0):
    cu = synth.cu_from_lengths(lens)
    T = int(cu[-1])
    rng = np.random.default_rng(seed)
    host = [synth.normal_bf16(rng, (T,) + row_shape) for _ in range(P)]
    plan = cpt.cpt_plan_create(layout, P, cu, T)
    writers = [to_dev(h) for h in host]
    return cu, T, host, plan, writers


def _run_staged(cpt, plan, writers, P, T, row_shape, ep, mode, rounds=1, skip_publish=None,
                clear_owner_flags=None, timeout_ns=2_000_000_000):
    Tp = T // P
    slots = torch.empty((P, P, Tp) + row_shape, dtype=torch.bfloat16, device="cuda")
    out = torch.full((P, Tp) + row_shape, 9.0, dtype=torch.bfloat16, device="cuda")
    main = torch.cuda.current_stream()
    wstreams = [torch.cuda.Stream() for _ in range(P)]
    ostreams = [torch.cuda.Stream() for _ in range(P)]
    results = []
    for _ in range(rounds):
        cpt.cpt_epoch_advance(ep)
        for w in range(P):
            wstreams[w].wait_stream(main)
            cpt.cpt_grad_scatter(plan, w, writers[w], [slots[o][w] for o in range(P)], slots[w][w],
                                 stream=wstreams[w])
            if w != skip_publish:
                cpt.cpt_epoch_publish(ep, w, stream=wstreams[w])
        for o in range(P):
            ostreams[o].wait_stream(main)
            if clear_owner_flags is not None and o == clear_owner_flags:
                for w in range(P):
                    ostreams[o].wait_stream(wstreams[w])
                with torch.cuda.stream(ostreams[o]):
                    ep.flags.view(P, P)[o].zero_()
            try:
                cpt.cpt_epoch_wait(ep, o, timeout_ns, mode, stream=ostreams[o])
                results.append(cpt.CPT_OK)
            except cpt.CptError as e:
                results.append(e.status)
            cpt.cpt_slot_reduce([slots[o][w] for w in range(P)], out[o], ep.status_ptr(o),
                                stream=ostreams[o])
        for s in wstreams + ostreams:
            main.wait_stream(s)
    torch.cuda.synchronize()
    status = [cpt.cpt_epoch_status(ep, o) for o in range(P)]
    return out, results, status


@pytest.mark.parametrize("P,layout,lens", [
    (2, 0, [16, 24, 24]),
    (3, 0, [6 * 50, 6 * 7]),
    (4, 0, [8 * 256]),
    (4, 1, [5, 1000, 27]),
    (8, 0, [16 * 40, 0, 16 * 3]),
])
@pytest.mark.parametrize("mode", [0, 1], ids=["bounded", "driver"])
def test_staged_equals_fused_and_oracle(cpt, cuda_device, P, layout, lens, mode):
    row_shape = (4, 32)
    cu, T, host, plan, writers = _setup(cpt, P, layout, lens, row_shape)
    ep = cpt.cpt_epoch_create(P)
    out, results, status = _run_staged(cpt, plan, writers, P, T, row_shape, ep, mode, rounds=3)
    assert results == [cpt.CPT_OK] * (3 * P)
    assert status == [0] * P
    fused = torch.empty_like(out)
    cpt.cpt_grad_return(plan, writers, None, fused, None)
    torch.cuda.synchronize()
    assert torch.equal(fused.view(torch.int16), out.view(torch.int16))
    l2g, _ = oracle.index_map(layout, P, cu, T)
    want = oracle.grad_return(l2g, host, oracle.BF16)
    got = to_host(out)
    for o in range(P):
        assert np.array_equal(got[o], want[o])
    # epoch flags hold the last epoch from every writer
    assert bool((ep.flags == 3).all().item())


def test_scatter_matches_oracle(cpt, cuda_device):
    P = 4
    cu, T, host, plan, writers = _setup(cpt, P, 0, [8 * 100, 8 * 9], (2, 64), seed=3)
    slots = torch.empty((P, T // P, 2, 64), dtype=torch.bfloat16, device="cuda")
    cpt.cpt_grad_scatter(plan, 2, writers[2], [slots[o] for o in range(P)], slots[2])
    torch.cuda.synchronize()
    l2g, _ = oracle.index_map(0, P, cu, T)
    want = oracle.grad_scatter(l2g, host[2], P)
    got = to_host(slots)
    for o in range(P):
        assert np.array_equal(got[o], want[o])


def test_missing_publish_is_refused_on_host(cpt, cuda_device):
    P = 4
    cu, T, host, plan, writers = _setup(cpt, P, 0, [8 * 64])
    ep = cpt.cpt_epoch_create(P)
    out, results, status = _run_staged(cpt, plan, writers, P, T, (4, 32), ep, 0, skip_publish=2)
    assert results == [cpt.CPT_ERR_NOT_PUBLISHED] * P
    assert status == [cpt.CPT_ERR_NOT_PUBLISHED] * P
    # every reduce saw the failed status and wrote nothing
    assert bool((out == 9.0).all().item())


def test_flag_that_nothing_sets_times_out(cpt, cuda_device):
    P = 4
    cu, T, host, plan, writers = _setup(cpt, P, 0, [8 * 64])
    ep = cpt.cpt_epoch_create(P)
    out, results, status = _run_staged(cpt, plan, writers, P, T, (4, 32), ep, 0,
                                       clear_owner_flags=1, timeout_ns=2_000_000)
    assert results == [cpt.CPT_OK] * P  # the host saw every publish enqueued
    assert status == [0, cpt.CPT_ERR_TIMEOUT, 0, 0]
    assert bool((out[1] == 9.0).all().item())
    assert not bool((out[0] == 9.0).all().item())
    # the context is still usable afterwards
    x = torch.ones(4, device="cuda") + 1
    assert x.sum().item() == 8.0


def test_epoch_api_errors(cpt, cuda_device):
    ep = cpt.cpt_epoch_create(2)
    with pytest.raises(cpt.CptError) as ei:
        cpt.cpt_epoch_publish(ep, 0)  # no epoch started
    assert ei.value.status == cpt.CPT_ERR_INVALID_ARG
    cpt.cpt_epoch_advance(ep)
    with pytest.raises(cpt.CptError):
        cpt.cpt_epoch_publish(ep, 2)
    with pytest.raises(cpt.CptError):
        cpt.cpt_epoch_wait(ep, 0, timeout_ns=20 * 10**9)
    with pytest.raises(cpt.CptError):
        cpt.cpt_epoch_create(9)
    host = torch.zeros(4, dtype=torch.int32).pin_memory()
    with pytest.raises(cpt.CptError) as ei:
        cpt.cpt_epoch_create(2, flags=host)
    assert ei.value.status == cpt.CPT_ERR_DEVICE


def _staged_round(cpt, plan, writers, slots, out, ep, P, wstreams, ostreams, main,
                  clear_flags_to=None, timeout_ns=2_000_000_000):
    for w in range(P):
        wstreams[w].wait_stream(main)
        cpt.cpt_grad_scatter(plan, w, writers[w], [slots[o][w] for o in range(P)], slots[w][w],
                             stream=wstreams[w])
        cpt.cpt_epoch_publish(ep, w, stream=wstreams[w])
    for o in range(P):
        ostreams[o].wait_stream(main)
        if clear_flags_to is not None:
            for w in range(P):
                ostreams[o].wait_stream(wstreams[w])
            with torch.cuda.stream(ostreams[o]):
                ep.flags.view(P, P)[o].fill_(clear_flags_to)
        cpt.cpt_epoch_wait(ep, o, timeout_ns, 0, stream=ostreams[o])
        cpt.cpt_slot_reduce([slots[o][w] for w in range(P)], out[o], ep.status_ptr(o), stream=ostreams[o])
    for st in wstreams + ostreams:
        main.wait_stream(st)
    torch.cuda.synchronize()
    return [cpt.cpt_epoch_status(ep, o) for o in range(P)]


def test_epoch_count_wraps_around(cpt, cuda_device):
    """Epochs run through 2^32 and wrap to 1 (0 is skipped); the flag test is
    (int32)(flag - epoch) >= 0, so a stale pre-wrap flag 0xFFFFFFFF does not
    satisfy epoch 1 although it is larger as an unsigned number."""
    P = 2
    cu, T, host, plan, writers = _setup(cpt, P, 0, [4 * 32])
    slots = torch.empty((P, P, T // P, 4, 32), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((P, T // P, 4, 32), dtype=torch.bfloat16, device="cuda")
    fused = torch.empty_like(out)
    cpt.cpt_grad_return(plan, writers, None, fused, None)
    ep = cpt.cpt_epoch_create(P)
    main = torch.cuda.current_stream()
    ws = [torch.cuda.Stream() for _ in range(P)]
    os_ = [torch.cuda.Stream() for _ in range(P)]
    cpt.cpt_epoch_set(ep, 0xFFFFFFFE)
    assert _staged_round(cpt, plan, writers, slots, out, ep, P, ws, os_, main) == [0, 0]
    assert cpt.cpt_epoch_advance(ep) == 0xFFFFFFFF
    assert _staged_round(cpt, plan, writers, slots, out, ep, P, ws, os_, main) == [0, 0]
    assert bool((ep.flags == -1).all().item())  # 0xFFFFFFFF in every flag
    assert cpt.cpt_epoch_advance(ep) == 1  # wrapped, 0 skipped
    assert _staged_round(cpt, plan, writers, slots, out, ep, P, ws, os_, main) == [0, 0]
    assert torch.equal(out.view(torch.int16), fused.view(torch.int16))
    # a stale pre-wrap value in the flags must not pass for epoch 2
    assert cpt.cpt_epoch_advance(ep) == 2
    out.fill_(9.0)
    st = _staged_round(cpt, plan, writers, slots, out, ep, P, ws, os_, main,
                       clear_flags_to=-1, timeout_ns=2_000_000)
    assert st == [cpt.CPT_ERR_TIMEOUT] * P
    assert bool((out == 9.0).all().item())
    with pytest.raises(cpt.CptError):
        cpt.cpt_epoch_set(ep, 0)


def test_writers_publish_from_host_threads(cpt, cuda_device):
    """Each writer rank is a host thread with its own stream; the C ABI is
    called concurrently (the binding releases the GIL) and the epoch state
    keeps its bookkeeping consistent."""
    import threading

    P = 4
    cu, T, host, plan, writers = _setup(cpt, P, 0, [8 * 256], seed=9)
    slots = torch.empty((P, P, T // P, 4, 32), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((P, T // P, 4, 32), dtype=torch.bfloat16, device="cuda")
    fused = torch.empty_like(out)
    cpt.cpt_grad_return(plan, writers, None, fused, None)
    ep = cpt.cpt_epoch_create(P)
    main = torch.cuda.current_stream()
    wstreams = [torch.cuda.Stream() for _ in range(P)]
    ostreams = [torch.cuda.Stream() for _ in range(P)]
    errors = []

    def writer(w):
        try:
            cpt.cpt_grad_scatter(plan, w, writers[w], [slots[o][w] for o in range(P)], slots[w][w],
                                 stream=wstreams[w])
            cpt.cpt_epoch_publish(ep, w, stream=wstreams[w])
        except Exception as e:  # reported below
            errors.append(e)

    for _ in range(5):
        cpt.cpt_epoch_advance(ep)
        for s in wstreams:
            s.wait_stream(main)
        threads = [threading.Thread(target=writer, args=(w,)) for w in range(P)]
        for t in threads:
            t.start()
        for t in threads:
            t.join()
        assert not errors, errors
        for o in range(P):
            ostreams[o].wait_stream(main)
            cpt.cpt_epoch_wait(ep, o, 2_000_000_000, 0, stream=ostreams[o])
            cpt.cpt_slot_reduce([slots[o][w] for w in range(P)], out[o], ep.status_ptr(o),
                                stream=ostreams[o])
        for s in wstreams + ostreams:
            main.wait_stream(s)
        torch.cuda.synchronize()
        assert [cpt.cpt_epoch_status(ep, o) for o in range(P)] == [0] * P
        assert torch.equal(out.view(torch.int16), fused.view(torch.int16))

"""CUDA graphs: a training step records the layout calls once and replays
them every iteration, so the kernel-only calls must capture and replay
correctly, and the calls that act on host state must refuse capture
("[PyTorch] Add experimental packed-contiguous THD all-gather CP",
TransformerEngine PR 3221, "Scope and constraints": graph capture is
rejected on the experimental path).
"""
import numpy as np
import pytest
import torch

import oracle
from context_attention_token_gb300 import synth
from gpu_helpers import to_dev, to_host

pytestmark = pytest.mark.gpu


def test_captured_step_replays_with_new_inputs(cpt, cuda_device):
    P, lens, row = 4, [8 * 300, 0, 8 * 97], (4, 64)
    cu = synth.cu_from_lengths(lens)
    T = int(cu[-1])
    plan = cpt.cpt_plan_create(0, P, cu, T)  # plans are built outside capture
    l2g, _ = oracle.index_map(0, P, cu, T)
    q = torch.empty((T,) + row, dtype=torch.bfloat16, device="cuda")
    qloc = torch.empty((P, T // P) + row, dtype=torch.bfloat16, device="cuda")
    qback = torch.empty_like(q)
    w = torch.empty((P, T) + row, dtype=torch.bfloat16, device="cuda")
    o = torch.empty((P, T // P) + row, dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        cpt.cpt_partition(plan, [q], [qloc])
        cpt.cpt_restore(plan, [qloc], [qback])
        cpt.cpt_grad_return(plan, w, None, o, None)
    for seed in (1, 2):
        rng = np.random.default_rng(seed)
        hq = synth.normal_bf16(rng, (T,) + row)
        hw = [synth.normal_bf16(rng, (T,) + row) for _ in range(P)]
        q.copy_(to_dev(hq))
        w.copy_(torch.stack([to_dev(x) for x in hw]))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(to_host(qloc).reshape((T,) + row), oracle.partition(l2g, hq))
        assert np.array_equal(to_host(qback), hq)
        want = oracle.grad_return(l2g, hw, oracle.BF16)
        got = to_host(o)
        for r in range(P):
            assert np.array_equal(got[r], want[r])


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_host_state_calls_refuse_capture(cpt, cuda_device):
    P = 2
    cu = [0, 16]
    ep = cpt.cpt_epoch_create(P)
    cpt.cpt_epoch_advance(ep)
    ws = torch.empty(cpt.cpt_plan_workspace_bytes(0, P, 1, 16), dtype=torch.uint8, device="cuda")
    w = torch.ones((P, 16, 8), dtype=torch.bfloat16, device="cuda")
    o = torch.full((P, 8, 8), 3.0, dtype=torch.bfloat16, device="cuda")
    cpt.cpt_grad_return_noalloc(0, P, cu, 16, w, None, o, None)  # one-time set-up, outside capture
    torch.cuda.synchronize()
    o.fill_(3.0)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    errors = []
    with torch.cuda.graph(g, stream=side):
        for fn in (lambda: cpt.cpt_plan_create(0, P, cu, 16, workspace=ws),
                   lambda: cpt.cpt_epoch_publish(ep, 0),
                   lambda: cpt.cpt_epoch_wait(ep, 0),
                   lambda: cpt.cpt_grad_return_noalloc(0, P, cu, 16, w, None, o, None)):
            try:
                fn()
            except cpt.CptError as e:
                errors.append((e.status, str(e)))
    assert [s for s, _ in errors] == [cpt.CPT_ERR_UNSUPPORTED] * 4
    assert all("stream capture" in m for _, m in errors)
    # the refused allocation-free call enqueued nothing
    torch.cuda.synchronize()
    assert bool((o == 3.0).all().item())
    # the epoch bookkeeping is untouched: still nothing published
    torch.cuda.synchronize()
    with pytest.raises(cpt.CptError) as ei:
        cpt.cpt_epoch_wait(ep, 0)
    assert ei.value.status == cpt.CPT_ERR_NOT_PUBLISHED

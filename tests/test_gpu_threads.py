"""Calls from several host threads at once, each on its own stream.

The header promises thread-safe calls. The launchers keep per-device caches
(function attributes, occupancy, the SM count) that the first calls fill
in; here four threads race through them under each kernel-path setting, and
every thread's results must still equal the oracle's. Each thread runs a
different layout and batch (per-document, packed-contiguous, padded) through
the plan, the partition, the restore and the gradient return, three times.
"""
import threading

import numpy as np
import pytest
import torch

import oracle
from context_attention_token_gb300 import synth
from gpu_helpers import to_dev, to_host

pytestmark = pytest.mark.gpu

CASES = [
    (0, 4, [8 * 700, 0, 8 * 333], (4, 64)),
    (1, 3, [500, 12, 2000, 8], (8, 32)),
    (3, 8, [13, 400, 1, 77], (2, 128)),
    (0, 2, [4 * 5000], (16, 16)),
]


def _run(cpt, case, seed, out, errors):
    try:
        layout, P, lens, row = case
        cu = synth.cu_from_lengths(lens)
        T = int(cu[-1])
        rng = np.random.default_rng(seed)
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            plan = cpt.cpt_plan_create(layout, P, cu, T, stream=stream)
            Tpad = plan.padded_tokens
            hq = synth.normal_bf16(rng, (T,) + row)
            hw = [synth.normal_bf16(rng, (Tpad,) + row) for _ in range(P)]
            q = to_dev(hq)
            w = torch.stack([to_dev(x) for x in hw])
            loc = torch.empty((P, Tpad // P) + row, dtype=torch.bfloat16, device="cuda")
            back = torch.empty_like(q)
            own = torch.empty((P, Tpad // P) + row, dtype=torch.bfloat16, device="cuda")
            for _ in range(3):
                cpt.cpt_partition(plan, [q], [loc], stream=stream)
                cpt.cpt_restore(plan, [loc], [back], stream=stream)
                cpt.cpt_grad_return(plan, w, None, own, None, stream=stream)
            stream.synchronize()
        out[seed] = (case, cu, T, Tpad, hq, hw, to_host(loc), to_host(back), to_host(own))
    except Exception as e:  # reported by the main thread
        errors.append(repr(e))


@pytest.mark.parametrize("path", ["auto", "bulk", "loads"])
def test_threads_calling_at_once_match_the_oracle(cpt, cuda_device, path):
    code = {"auto": cpt.CPT_KERNEL_AUTO, "bulk": cpt.CPT_KERNEL_BULK, "loads": cpt.CPT_KERNEL_LOADS}[path]
    cpt.cpt_set_kernel_path(code)
    try:
        out, errors = {}, []
        threads = [threading.Thread(target=_run, args=(cpt, c, 100 + i, out, errors))
                   for i, c in enumerate(CASES)]
        for t in threads:
            t.start()
        for t in threads:
            t.join(timeout=300)
        assert not errors, errors
        assert len(out) == len(CASES)
    finally:
        cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_AUTO)
    for seed, (case, cu, T, Tpad, hq, hw, loc, back, own) in out.items():
        layout, P, lens, row = case
        if layout == 3:
            want_loc = oracle.partition_padded(P, cu, hq)
            _, l2g, _ = oracle.padded_index_map(P, cu)
        else:
            l2g, _ = oracle.index_map(layout, P, cu, T)
            want_loc = oracle.partition(l2g, hq)
        assert np.array_equal(loc.reshape((Tpad,) + row), want_loc), (seed, case)
        assert np.array_equal(back, hq), (seed, case)
        want = oracle.grad_return(l2g, hw, oracle.BF16)
        for o in range(P):
            assert np.array_equal(own[o], want[o]), (seed, case, o)
    assert cpt.cpt_kernel_wait_timeouts() == 0

"""Parity of the two slot-reduce kernels.

With equal input and output types, the ordered slot sum can run either of
two kernels: 16-byte loads into registers, or bulk copies that stage 4 KB
chunks of every slot in shared memory. The bulk kernel takes the whole
chunks and the loads kernel the tail. Each case runs under the measured
rule and with each kernel forced. Sizes straddle the chunk: below one chunk,
exactly one, whole chunks plus a ragged tail of odd length. Every output is
compared bit for bit with the oracle, with canary bands. The status gate
must stop both kernels, and no bulk-copy wait may run out.
"""
import numpy as np
import pytest
import torch

import oracle
from context_attention_token_gb300 import synth
from gpu_helpers import Guarded, bits, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["auto", "loads", "bulk"])
def kernel(cpt, request):
    code = {"auto": cpt.CPT_KERNEL_AUTO, "loads": cpt.CPT_KERNEL_LOADS,
            "bulk": cpt.CPT_KERNEL_BULK}[request.param]
    cpt.cpt_set_kernel_path(code)
    yield request.param
    cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_AUTO)


def _elems(nbytes, dt):
    return nbytes // (4 if dt == "f32" else 2)


# bytes per slot: under a chunk, one chunk, chunks + 16 B, chunks + an odd tail
SIZES = [4080, 4096, 3 * 4096 + 16, 37 * 4096 + 6, (1 << 20) + 4096 * 5 + 10]


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("nbytes", SIZES)
def test_slot_reduce_kernels_match_oracle(cpt, cuda_device, kernel, P, dt, nbytes):
    n = _elems(nbytes, dt)
    rng = np.random.default_rng(8000 + 10 * P + len(dt))
    gen = synth.uniform_f32 if dt == "f32" else synth.uniform_bf16
    slots = [gen(rng, (n,)) for _ in range(P)]
    dst = Guarded((n,), torch.float32 if dt == "f32" else torch.bfloat16)
    cpt.cpt_slot_reduce([to_dev(s) for s in slots], dst.t)
    torch.cuda.synchronize()
    want = oracle.slot_reduce(slots, oracle.F32 if dt == "f32" else oracle.BF16)
    assert np.array_equal(bits(to_host(dst.t)), bits(want))
    assert dst.bands_intact()


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_slot_reduce_status_gate_stops_both_kernels(cpt, cuda_device, kernel, dt):
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    n = _elems(5 * 4096 + 48, dt)
    slots = [torch.ones(n, dtype=tdt, device="cuda") for _ in range(3)]
    dst = torch.full((n,), 5.0, dtype=tdt, device="cuda")
    status = torch.tensor([7], dtype=torch.int32, device="cuda")
    cpt.cpt_slot_reduce(slots, dst, status)
    torch.cuda.synchronize()
    assert bool((dst == 5.0).all().item())
    status.zero_()
    cpt.cpt_slot_reduce(slots, dst, status)
    torch.cuda.synchronize()
    assert bool((dst == 3.0).all().item())


def test_slot_reduce_no_bulk_wait_ran_out(cpt, cuda_device):
    torch.cuda.synchronize()
    assert cpt.cpt_kernel_wait_timeouts() == 0

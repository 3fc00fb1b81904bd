"""Parity of the two row-gather kernels (partition, restore, row ranges).

The gather can run either of two kernels: 16-byte loads per row, or blocks of
consecutive rows moved through shared memory with bulk copies. Each case runs
under the measured rule and with each kernel forced, bit for bit against the
oracle, with canary bands around every output. The cases exercise the
blocks kernel's paths: one contiguous source run per block (large
documents), several runs per block (many short documents), zero-filled
padding rows (padded layout), blocks split across two rank pieces (row
ranges), and rows at and just past its shared-memory limit. Where the map is
the identity and the destination contiguous (packed-contiguous partition,
restore and scatter), the bulk path is a straight copy: those cases cover a
ring that wraps many times, a short last block, row ranges and slots that
are not contiguous.
"""
import numpy as np
import pytest
import torch

import oracle
from context_attention_token_gb300 import synth
from gpu_helpers import Guarded, bits, to_dev, to_host

pytestmark = pytest.mark.gpu

DSC, PACKED, PADDED = 0, 1, 3


@pytest.fixture(params=["auto", "loads", "bulk"])
def kernel(cpt, request):
    code = {"auto": cpt.CPT_KERNEL_AUTO, "loads": cpt.CPT_KERNEL_LOADS,
            "bulk": cpt.CPT_KERNEL_BULK}[request.param]
    cpt.cpt_set_kernel_path(code)
    yield request.param
    cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_AUTO)


# (layout, P, document lengths, row elements, element type)
CASES = [
    (DSC, 4, [2048, 1024], 2560, "bf16"),               # long runs: one bulk load per block
    (DSC, 4, [8] * 30 + [64, 16], 2560, "bf16"),        # 1-row chunks: many runs per block
    (DSC, 1, [40, 24], 512, "bf16"),
    (DSC, 2, [12, 36, 4], 1024, "f32"),
    (DSC, 3, [6, 60, 12], 1536, "bf16"),
    (DSC, 5, [10, 30, 200], 600, "bf16"),               # 1200-byte rows
    (DSC, 8, [16, 160, 48], 256, "f32"),
    (DSC, 4, [8, 16], 8, "bf16"),                       # 16-byte rows: 32-row blocks
    (DSC, 2, [4, 8], 25600, "bf16"),                    # 50 KB rows: one per block, 200 KB of stages
    (DSC, 2, [4, 8], 25608, "bf16"),                    # 16 bytes more: the 16-byte-load kernel
    (PACKED, 3, [5, 50, 17, 3, 9], 2048, "bf16"),
    (PACKED, 8, [0, 77, 19], 640, "f32"),
    (PADDED, 4, [5, 33, 1, 12], 2560, "bf16"),          # zero-filled padding rows
    (PADDED, 8, [3, 17, 100], 512, "f32"),
    (PACKED, 4, [70000, 60000, 1072], 512, "bf16"),     # straight copy: 4096 blocks, the ring wraps
    (PACKED, 2, [7, 9], 8, "bf16"),                     # straight copy of 16-byte rows, one short block
]


def _ids(c):
    return f"L{c[0]}-P{c[1]}-n{len(c[2])}-row{c[3]}-{c[4]}"


def _case(case, seed):
    layout, P, lens, row, dt = case
    cu = synth.cu_from_lengths(lens)
    T = int(cu[-1])
    if layout != PADDED:
        assert oracle.check_layout(layout, P, cu, T) == 0
    rng = np.random.default_rng(seed)
    gen = synth.uniform_f32 if dt == "f32" else synth.uniform_bf16
    return layout, P, cu, T, [gen(rng, (T, row)) for _ in range(3)]


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_partition_and_restore_both_kernels(cpt, cuda_device, kernel, case):
    layout, P, cu, T, xs = _case(case, 9100 + case[1] + case[3])
    row, tdt = case[3], torch.float32 if case[4] == "f32" else torch.bfloat16
    plan = cpt.cpt_plan_create(layout, P, cu, T)
    Tpad = plan.padded_tokens
    src = [to_dev(x) for x in xs]
    parts = [Guarded((P, Tpad // P, row), tdt) for _ in xs]
    cpt.cpt_partition(plan, src, [g.t for g in parts])
    backs = [Guarded((T, row), tdt) for _ in xs]
    cpt.cpt_restore(plan, [g.t for g in parts], [g.t for g in backs])
    torch.cuda.synchronize()
    if layout == PADDED:
        want = [oracle.partition_padded(P, cu, x) for x in xs]
    else:
        l2g, _ = oracle.index_map(layout, P, cu, T)
        want = [oracle.partition(l2g, x) for x in xs]
    for x, w, g, bk in zip(xs, want, parts, backs):
        assert np.array_equal(bits(to_host(g.t)).reshape(Tpad, row), bits(w))
        assert np.array_equal(bits(to_host(bk.t)), bits(x))
        assert g.bands_intact() and bk.bands_intact()


@pytest.mark.parametrize("case", [CASES[0], CASES[1], CASES[5], CASES[10], CASES[12], CASES[14]], ids=_ids)
def test_partition_row_ranges_both_kernels(cpt, cuda_device, kernel, case):
    """Ranges that start and end inside rank pieces, so blocks straddle two
    ranks, and a range of one row."""
    layout, P, cu, T, xs = _case(case, 9200 + case[1])
    row, tdt = case[3], torch.float32 if case[4] == "f32" else torch.bfloat16
    plan = cpt.cpt_plan_create(layout, P, cu, T)
    Tpad = plan.padded_tokens
    Tp = Tpad // P
    src = [to_dev(x) for x in xs]
    whole = [torch.empty((P, Tp, row), dtype=tdt, device="cuda") for _ in xs]
    cpt.cpt_partition(plan, src, whole)
    pieces = [torch.full((P, Tp, row), 9.0, dtype=tdt, device="cuda") for _ in xs]
    cuts = sorted({0, 1, max(1, Tp - 3), min(Tpad, Tp + 5), min(Tpad, 2 * Tp + 1), Tpad})
    for a, b in zip(cuts, cuts[1:]):
        cpt.cpt_partition_rows(plan, src, pieces, a, b - a)
    torch.cuda.synchronize()
    for w, pc in zip(whole, pieces):
        assert np.array_equal(bits(to_host(w)), bits(to_host(pc)))


@pytest.mark.parametrize("contiguous", [True, False])
def test_packed_scatter_into_slots(cpt, cuda_device, kernel, contiguous):
    """The staged scatter with the identity map: slots laid end to end make
    it a straight copy, separate slots keep it a gather; both give the
    oracle's slots."""
    P, lens, row = 4, [70000, 61072], 512
    cu = synth.cu_from_lengths(lens)
    T = int(cu[-1])
    plan = cpt.cpt_plan_create(PACKED, P, cu, T)
    x = synth.uniform_bf16(np.random.default_rng(9300), (T, row))
    if contiguous:
        buf = torch.empty((P, T // P, row), dtype=torch.bfloat16, device="cuda")
        slots = [buf[o] for o in range(P)]
    else:  # 16 rows of gap between slots, so they are never laid end to end
        buf = torch.empty((P, T // P + 16, row), dtype=torch.bfloat16, device="cuda")
        slots = [buf[o, : T // P] for o in range(P)]
    w = 1
    cpt.cpt_grad_scatter(plan, w, to_dev(x), slots, slots[w])
    torch.cuda.synchronize()
    l2g, _ = oracle.index_map(PACKED, P, cu, T)
    want = oracle.grad_scatter(l2g, x, P)
    for o in range(P):
        assert np.array_equal(to_host(slots[o]), want[o])


def test_no_gather_wait_ran_out(cpt, cuda_device):
    torch.cuda.synchronize()
    assert cpt.cpt_kernel_wait_timeouts() == 0

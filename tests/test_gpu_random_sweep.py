"""Seeded random sweep: many small batches of random shape through every
call of the C ABI, each output compared with the oracle bit for bit.

Each case draws a layout, P in 1..8, a document mix (zero-length documents
included), a row width that is a multiple of 16 bytes but not of a warp's
512 bytes, and a dtype pair, and runs once under the measured kernel rule
and once with the bulk-copy kernels forced. A second, wider sweep draws up to
40 documents, batches of up to about 10^6 tokens and rows of up to 4096
elements (16 KB of float32), and runs each case with either kernel family
forced. The fixed cases elsewhere pin known corners; these sweeps look for
the corners nobody thought of.
"""
import numpy as np
import pytest
import torch

import oracle
from context_attention_token_gb300 import synth
from gpu_helpers import bits, to_dev, to_host

pytestmark = pytest.mark.gpu

DSC, PACKED, PADDED = 0, 1, 3


def _case(seed):
    rng = np.random.default_rng(9000 + seed)
    layout = int(rng.choice([DSC, PACKED, PADDED]))
    P = int(rng.integers(1, 9))
    n = int(rng.integers(1, 9))
    if layout == DSC:
        lens = (rng.integers(0, 40, size=n) * 2 * P).tolist()
    else:
        lens = rng.integers(0, 300, size=n).tolist()
    if layout == PACKED:
        lens[-1] += (-sum(lens)) % P
    if sum(lens) == 0:
        lens[0] = 2 * P
    din = rng.choice(["f32", "bf16"])
    dout = rng.choice(["f32", "bf16"])
    # row elements: a multiple of 8 keeps both dtypes at 16-byte rows
    row = int(rng.integers(1, 41)) * 8
    return rng, layout, P, lens, row, str(din), str(dout)


def _wide_case(seed):
    """Longer batches and wider rows: many bulk-copy blocks and row
    pipelines per case, runs of source rows across block edges, and blocks
    split across rank pieces. About 64 MB of writer rows at most."""
    rng = np.random.default_rng(77000 + seed)
    layout = int(rng.choice([DSC, PACKED, PADDED]))
    P = int(rng.integers(1, 9))
    n = int(rng.integers(1, 41))
    din = str(rng.choice(["f32", "bf16"]))
    dout = str(rng.choice(["f32", "bf16"]))
    lo, hi = [(1, 41), (40, 161), (160, 513)][int(rng.integers(0, 3))]
    row = int(rng.integers(lo, hi)) * 8
    esz = 4 if din == "f32" else 2
    max_T = max(2 * P * n, (48 << 20) // (row * esz * (P + 1)))
    per = max(1, max_T // n)
    if layout == DSC:
        lens = (rng.integers(0, max(2, per // (2 * P)) + 1, size=n) * 2 * P).tolist()
    else:
        lens = rng.integers(0, per + 1, size=n).tolist()
    if layout == PACKED:
        lens[-1] += (-sum(lens)) % P
    if sum(lens) == 0:
        lens[0] = 2 * P
    return rng, layout, P, lens, row, din, dout


def _rand(rng, shape, dt):
    return synth.uniform_f32(rng, shape) if dt == "f32" else synth.uniform_bf16(rng, shape)


def _tdt(dt):
    return torch.float32 if dt == "f32" else torch.bfloat16


@pytest.fixture(params=["auto", "bulk"])
def kernel_path(cpt, request):
    """Each case runs under the measured kernel rule, and again with the
    bulk-copy kernels forced wherever they can run, so that they also meet
    rows of any width from 16 bytes up."""
    cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_AUTO if request.param == "auto"
                                   else cpt.CPT_KERNEL_BULK)
    yield request.param
    cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_AUTO)


@pytest.mark.parametrize("seed", range(100))
def test_random_case_every_call(cpt, cuda_device, seed, kernel_path):
    _run_case(cpt, seed, _case(seed))


@pytest.fixture(params=["loads", "bulk"])
def forced_path(cpt, request):
    """One kernel family forced for the whole case, then the default back."""
    cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_LOADS if request.param == "loads" else cpt.CPT_KERNEL_BULK)
    yield request.param
    cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_AUTO)


@pytest.mark.parametrize("seed", range(60))
def test_wide_random_case_every_call(cpt, cuda_device, seed, forced_path):
    _run_case(cpt, seed, _wide_case(seed))


def _run_case(cpt, seed, case):
    rng, layout, P, lens, row, din, dout = case
    cu = synth.cu_from_lengths(lens)
    T = int(cu[-1])
    n = len(lens)
    plan = cpt.cpt_plan_create(layout, P, cu, T)
    if layout == PADDED:
        cup, l2g, g2l = oracle.padded_index_map(P, cu)
        meta_layout, meta_cu = DSC, cup
    else:
        l2g, g2l = oracle.index_map(layout, P, cu, T)
        cup, meta_layout, meta_cu = cu, layout, cu
    Tpad = int(cup[-1])
    assert plan.padded_tokens == Tpad
    assert cpt.cpt_layout_padded_tokens(layout, P, cu, T) == Tpad  # the host query agrees with the plan

    # maps, metadata, real lengths
    d_l2g = torch.empty(Tpad, dtype=torch.int32, device="cuda")
    d_g2l = torch.empty(Tpad, dtype=torch.int32, device="cuda")
    cpt.cpt_index_map(plan, d_l2g, d_g2l)
    ns = torch.empty(P, dtype=torch.int32, device="cuda")
    first = torch.empty(P, dtype=torch.int32, device="cuda")
    cul = torch.empty((P, n + 1), dtype=torch.int32, device="cuda")
    offs = torch.empty(P + 1, dtype=torch.int32, device="cuda")
    cpt.cpt_thd_metadata(plan, ns, first, cul, offs)
    rl = torch.empty((P, n), dtype=torch.int32, device="cuda")
    cpt.cpt_thd_real_lengths(plan, rl)

    # partition, restore, grad_return, accumulate, row ranges
    x = _rand(rng, (T, row), din)
    src = to_dev(x)
    part = torch.empty((P, Tpad // P, row), dtype=src.dtype, device="cuda")
    cpt.cpt_partition(plan, [src], [part])
    back = torch.empty_like(src)
    cpt.cpt_restore(plan, [part], [back])
    writers = [_rand(rng, (Tpad, row), din) for _ in range(P)]
    dw = torch.stack([to_dev(w) for w in writers])
    owners = torch.empty((P, Tpad // P, row), dtype=_tdt(dout), device="cuda")
    cpt.cpt_grad_return(plan, dw, None, owners, None)
    starts = [_rand(rng, (Tpad // P, row), dout) for _ in range(P)]
    acc = torch.stack([to_dev(s) for s in starts])
    cpt.cpt_grad_return_accumulate(plan, dw, None, acc, None)
    cut = int(rng.integers(0, Tpad + 1))
    pieces = torch.empty_like(owners)
    cpt.cpt_grad_return_rows(plan, dw, None, pieces, None, 0, cut)
    cpt.cpt_grad_return_rows(plan, dw, None, pieces, None, cut, Tpad - cut)
    torch.cuda.synchronize()

    assert np.array_equal(to_host(d_l2g), l2g) and np.array_equal(to_host(d_g2l), g2l)
    for got, want in zip((ns, first, cul, offs), oracle.thd_metadata(meta_layout, P, meta_cu, Tpad)):
        assert np.array_equal(to_host(got), want)
    assert np.array_equal(to_host(rl), oracle.real_lengths(layout if layout != PADDED else DSC, P, cu,
                                                           padded=layout == PADDED))
    if layout == PADDED:
        want_part = oracle.partition_padded(P, cu, x)
    else:
        want_part = oracle.partition(l2g, x)
    assert np.array_equal(bits(to_host(part)).reshape(Tpad, row), bits(want_part))
    assert np.array_equal(bits(to_host(back)), bits(x))
    code = oracle.F32 if dout == "f32" else oracle.BF16
    want = oracle.grad_return(l2g, writers, code)
    want_acc = oracle.grad_return_accumulate(l2g, writers, starts)
    got, got_acc, got_pieces = to_host(owners), to_host(acc), to_host(pieces)
    for o in range(P):
        assert np.array_equal(bits(got[o]), bits(want[o])), (seed, o)
        assert np.array_equal(bits(got_acc[o]), bits(want_acc[o])), (seed, o)
        assert np.array_equal(bits(got_pieces[o]), bits(want[o])), (seed, o)


def test_random_sweep_no_bulk_wait_ran_out(cpt, cuda_device):
    torch.cuda.synchronize()
    assert cpt.cpt_kernel_wait_timeouts() == 0

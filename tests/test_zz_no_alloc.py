"""The allocation-free gradient return, through the C ABI.

Some callers cannot allocate device memory: a plugin whose host application
owns all device memory through its own pool, or a step whose memory plan is
fixed in advance. They cannot hand cpt_plan_create a workspace, so
cpt_grad_return_noalloc keeps its ownership map in a fixed-size array inside
the library. Its output must equal the plan-based cpt_grad_return bit for bit
(tolerance 0, as everywhere in these tests), over two calls in a row that
reuse the shared array with different layouts and sizes.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test; it also passes on its own.
"""
import numpy as np
import pytest
import torch

from context_attention_token_gb300 import synth
from gpu_helpers import to_dev

pytestmark = pytest.mark.gpu


def _case(P, layout, lens, row_shape, dt, seed):
    cu = synth.cu_from_lengths(lens)
    T = int(cu[-1])
    rng = np.random.default_rng(seed)
    if dt == "bf16":
        mk = lambda: synth.normal_bf16(rng, (T,) + row_shape)  # noqa: E731
    else:
        mk = lambda: synth.uniform_f32(rng, (T,) + row_shape)  # noqa: E731
    dkw = torch.stack([to_dev(mk()) for _ in range(P)])
    dvw = torch.stack([to_dev(mk()) for _ in range(P)])
    return cu, T, dkw, dvw


def test_noalloc_matches_plan_path_on_two_calls_in_a_row(cpt, cuda_device):
    # two different batches back to back on one stream: the second call must
    # rebuild the shared map (other layout, other P, other document split)
    cases = [
        (4, cpt.CPT_LAYOUT_DUAL_CHUNK_SWAP, [8 * 1024, 0, 8 * 3072], (8, 128), "bf16", 11),
        (3, cpt.CPT_LAYOUT_PACKED_CONTIGUOUS, [5, 7000, 1, 2993], (2, 64), "f32", 12),
    ]
    data = [_case(*c) for c in cases]
    outs = []
    for (P, layout, lens, row_shape, dt, _), (cu, T, dkw, dvw) in zip(cases, data):
        dko = torch.full((P, T // P) + row_shape, 7.0, dtype=dkw.dtype, device="cuda")
        dvo = torch.full_like(dko, 7.0)
        cpt.cpt_grad_return_noalloc(layout, P, cu, T, dkw, dvw, dko, dvo)
        outs.append((dko, dvo))
    torch.cuda.synchronize()
    for (P, layout, lens, row_shape, dt, _), (cu, T, dkw, dvw), (dko, dvo) in zip(cases, data, outs):
        plan = cpt.cpt_plan_create(layout, P, cu, T)
        rk = torch.empty_like(dko)
        rv = torch.empty_like(dvo)
        cpt.cpt_grad_return(plan, dkw, dvw, rk, rv)
        torch.cuda.synchronize()
        iv = torch.int16 if dko.dtype == torch.bfloat16 else torch.int32
        assert torch.equal(dko.view(iv), rk.view(iv))
        assert torch.equal(dvo.view(iv), rv.view(iv))


def test_noalloc_allocates_nothing_after_setup(cpt, cuda_device):
    P, cu = 2, synth.cu_from_lengths([4 * 512])
    T = int(cu[-1])
    w = torch.ones((P, T, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty((P, T // P, 64), dtype=torch.bfloat16, device="cuda")
    cpt.cpt_grad_return_noalloc(0, P, cu, T, w, None, o, None)  # first call: set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        cpt.cpt_grad_return_noalloc(0, P, cu, T, w, None, o, None)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert bool((o == 2).all().item())


def test_noalloc_rejects_batches_beyond_its_limit(cpt, cuda_device):
    P = 2
    T = cpt.CPT_NOALLOC_MAX_TOKENS + 4
    cu = [0, T]
    w = torch.empty((P, 1, 8), dtype=torch.bfloat16, device="cuda")
    o = torch.full((P, 1, 8), 3.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cpt.CptError) as ei:
        cpt.cpt_grad_return_noalloc(0, P, cu, T, w, None, o, None)
    assert ei.value.status == cpt.CPT_ERR_INVALID_ARG
    assert "no-allocation limit" in str(ei.value)
    many = list(range(0, 2 * (cpt.CPT_NOALLOC_MAX_DOCS + 1) + 1, 2))
    with pytest.raises(cpt.CptError) as ei:
        cpt.cpt_grad_return_noalloc(1, P, many, many[-1], w, None, o, None)
    assert "no-allocation limit" in str(ei.value)
    torch.cuda.synchronize()
    assert bool((o == 3.0).all().item())


def test_noalloc_limit_applies_to_the_padded_total(cpt, cuda_device):
    # 40,000 documents of 17 tokens: 680,000 raw tokens, within the limit,
    # but each pads to 32 at P=8, so the map would cover 1,280,000 tokens
    P, n, L = 8, 40000, 17
    PAD = cpt.CPT_LAYOUT_DUAL_CHUNK_SWAP_PADDED
    cu = list(range(0, n * L + 1, L))
    T = cu[-1]
    assert T <= cpt.CPT_NOALLOC_MAX_TOKENS
    assert cpt.cpt_layout_padded_tokens(PAD, P, cu, T) == n * 32 > cpt.CPT_NOALLOC_MAX_TOKENS
    w = torch.empty((P, 1, 8), dtype=torch.bfloat16, device="cuda")
    o = torch.full((P, 1, 8), 3.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cpt.CptError) as ei:
        cpt.cpt_grad_return_noalloc(PAD, P, cu, T, w, None, o, None)
    assert ei.value.status == cpt.CPT_ERR_INVALID_ARG
    assert "padded total 1280000" in str(ei.value)
    torch.cuda.synchronize()
    assert bool((o == 3.0).all().item())


def test_noalloc_padded_layout_matches_plan_path(cpt, cuda_device):
    P, lens = 4, [13, 0, 1000, 7]
    cu = synth.cu_from_lengths(lens)
    T = int(cu[-1])
    plan = cpt.cpt_plan_create(cpt.CPT_LAYOUT_DUAL_CHUNK_SWAP_PADDED, P, cu, T)
    Tpad = plan.padded_tokens
    rng = np.random.default_rng(5)
    w = torch.stack([to_dev(synth.normal_bf16(rng, (Tpad, 2, 64))) for _ in range(P)])
    a = torch.empty((P, Tpad // P, 2, 64), dtype=torch.bfloat16, device="cuda")
    b = torch.empty_like(a)
    cpt.cpt_grad_return_noalloc(cpt.CPT_LAYOUT_DUAL_CHUNK_SWAP_PADDED, P, cu, T, w, None, a, None)
    cpt.cpt_grad_return(plan, w, None, b, None)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))

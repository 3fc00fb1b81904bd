"""GPU parity: every C-ABI call against the CPU oracle, bit for bit.

Index and metadata outputs are integers; partition and scatter are bit
copies; gradient sums are binary32 in writer order 0..P-1 on both sides, with
one round-to-nearest-even to bf16, so every comparison here has tolerance 0.
Sizes span many grid-stride passes of each kernel and ragged row tails.
"""
import numpy as np
import pytest
import torch

import oracle
from context_attention_token_gb300 import synth
from gpu_helpers import Guarded, bits, to_dev, to_host

pytestmark = pytest.mark.gpu

DSC, PACKED = 0, 1


def _cu(lens):
    return synth.cu_from_lengths(lens)


# (layout, P, document lengths): tiny configuration, zero-length documents,
# P=1 and P=8, a single document, many short documents, uneven packed docs.
MAP_CASES = [
    (DSC, 2, [16, 24, 24]),
    (PACKED, 2, [16, 24, 24]),
    (DSC, 1, [10, 0, 6, 2]),
    (PACKED, 1, [3, 0, 7]),
    (DSC, 8, [0, 16, 0, 160, 32, 0]),
    (PACKED, 8, [1, 5, 0, 90, 24]),
    (DSC, 3, [6 * 7, 6 * 1, 6 * 40, 0, 6 * 3]),
    (PACKED, 3, [5, 50, 1, 40]),
    (DSC, 4, [32768]),
    (DSC, 4, [8] * 700),
    (PACKED, 4, list(range(1, 64)) + [4 * 1000 - sum(range(1, 64))]),
]


def _lognormal_case(layout):
    rng = synth.rng_for(2, 0)
    lens = synth.lognormal_doc_lengths(131072, rng, multiple=8 if layout == DSC else 1)
    return lens


@pytest.mark.parametrize("case", MAP_CASES + [(DSC, 4, None), (PACKED, 4, None)],
                         ids=lambda c: f"L{c[0]}P{c[1]}n{len(c[2]) if c[2] else 'lognormal'}")
def test_index_map_and_metadata(cpt, cuda_device, case):
    layout, P, lens = case
    if lens is None:
        lens = _lognormal_case(layout)
    cu = _cu(lens)
    T = int(cu[-1])
    n = len(lens)
    plan = cpt.cpt_plan_create(layout, P, cu, T)
    l2g = Guarded((T,), torch.int32)
    g2l = Guarded((T,), torch.int32)
    cpt.cpt_index_map(plan, l2g.t, g2l.t)
    ns = torch.full((P,), -7, dtype=torch.int32, device="cuda")
    first = torch.full((P,), -7, dtype=torch.int32, device="cuda")
    cul = torch.full((P, n + 1), -7, dtype=torch.int32, device="cuda")
    offs = torch.full((P + 1,), -7, dtype=torch.int32, device="cuda")
    cpt.cpt_thd_metadata(plan, ns, first, cul, offs)
    torch.cuda.synchronize()

    ol2g, og2l = oracle.index_map(layout, P, cu, T)
    assert np.array_equal(to_host(l2g.t), ol2g)
    assert np.array_equal(to_host(g2l.t), og2l)
    assert l2g.bands_intact() and g2l.bands_intact()
    ons, ofirst, ocul, ooffs = oracle.thd_metadata(layout, P, cu, T)
    assert np.array_equal(to_host(ns), ons)
    assert np.array_equal(to_host(first), ofirst)
    assert np.array_equal(to_host(cul), ocul)
    assert np.array_equal(to_host(offs), ooffs)
    # the plan's own copy (used by the gather kernels) equals the exported map
    assert cpt.cpt_plan_info(plan) == (T, P, n)


def test_empty_batch(cpt, cuda_device):
    for layout in (DSC, PACKED):
        plan = cpt.cpt_plan_create(layout, 4, [0], 0)
        e = torch.empty(0, dtype=torch.int32, device="cuda")
        cpt.cpt_index_map(plan, e, e)
        w = torch.empty((4, 0, 8, 16), dtype=torch.bfloat16, device="cuda")
        o = torch.empty((4, 0, 8, 16), dtype=torch.bfloat16, device="cuda")
        cpt.cpt_grad_return(plan, w, w, o, o)
        q = torch.empty((0, 8, 16), dtype=torch.bfloat16, device="cuda")
        cpt.cpt_partition(plan, [q], [torch.empty((4, 0, 8, 16), dtype=torch.bfloat16, device="cuda")])
        ns = torch.full((4,), -7, dtype=torch.int32, device="cuda")
        first = torch.full((4,), -7, dtype=torch.int32, device="cuda")
        cul = torch.full((4, 1), -7, dtype=torch.int32, device="cuda")
        offs = torch.full((5,), -7, dtype=torch.int32, device="cuda")
        cpt.cpt_thd_metadata(plan, ns, first, cul, offs)
        torch.cuda.synchronize()
        assert to_host(ns).tolist() == [0] * 4
        assert to_host(first).tolist() == [-1] * 4
        assert to_host(cul).tolist() == [[0]] * 4
        assert to_host(offs).tolist() == [0] * 5


# ---------------------------------------------------------------- partition


def _rand_rows(rng, T, row_shape, dt):
    if dt == "f32":
        return synth.uniform_f32(rng, (T,) + row_shape)
    return synth.normal_bf16(rng, (T,) + row_shape)


@pytest.mark.parametrize("layout,P,lens,row_shape,dt", [
    (DSC, 2, [16, 24, 24], (2, 8), "f32"),
    (PACKED, 2, [16, 24, 24], (2, 8), "f32"),
    (DSC, 4, [8 * 3, 8 * 500, 0, 8 * 211], (3, 40), "bf16"),   # 240-byte rows: ragged lanes
    (PACKED, 3, [7, 1000, 3, 2590], (8, 16), "bf16"),
    (DSC, 8, [16 * 64, 16 * 3], (20, 128), "bf16"),
    (DSC, 1, [10, 0, 22], (1, 4), "f32"),
])
def test_partition_matches_oracle(cpt, cuda_device, layout, P, lens, row_shape, dt):
    cu = _cu(lens)
    T = int(cu[-1])
    rng = np.random.default_rng(7)
    xs = [_rand_rows(rng, T, row_shape, dt) for _ in range(3)]
    plan = cpt.cpt_plan_create(layout, P, cu, T)
    src = [to_dev(x) for x in xs]
    dst = [Guarded((P, T // P) + row_shape, src[0].dtype) for _ in range(3)]
    cpt.cpt_partition(plan, src, [d.t for d in dst])
    torch.cuda.synchronize()
    l2g, _ = oracle.index_map(layout, P, cu, T)
    for x, d in zip(xs, dst):
        want = oracle.partition(l2g, x).reshape((P, T // P) + row_shape)
        assert np.array_equal(bits(to_host(d.t)), bits(want))
        assert d.bands_intact()


@pytest.mark.parametrize("layout,P,lens,row_shape,dt", [
    (DSC, 2, [16, 24, 24], (2, 8), "f32"),
    (PACKED, 2, [16, 24, 24], (2, 8), "f32"),
    (DSC, 4, [8 * 3, 8 * 500, 0, 8 * 211], (3, 40), "bf16"),
    (PACKED, 3, [7, 1000, 3, 2590], (8, 16), "bf16"),
    (DSC, 8, [16 * 64, 16 * 3], (20, 128), "bf16"),
    (DSC, 1, [10, 0, 22], (1, 4), "f32"),
])
def test_restore_matches_oracle(cpt, cuda_device, layout, P, lens, row_shape, dt):
    """All-gather restore: rank-local [P, T/P, ...] back to global order."""
    cu = _cu(lens)
    T = int(cu[-1])
    rng = np.random.default_rng(17)
    locs = [_rand_rows(rng, T, row_shape, dt) for _ in range(3)]
    plan = cpt.cpt_plan_create(layout, P, cu, T)
    src = [to_dev(x).view((P, T // P) + row_shape) for x in locs]
    dst = [Guarded((T,) + row_shape, src[0].dtype) for _ in range(3)]
    cpt.cpt_restore(plan, src, [d.t for d in dst])
    torch.cuda.synchronize()
    l2g, _ = oracle.index_map(layout, P, cu, T)
    for x, d in zip(locs, dst):
        assert np.array_equal(bits(to_host(d.t)), bits(oracle.restore(l2g, x)))
        assert d.bands_intact()


def test_partition_row_ids(cpt, cuda_device):
    """Rows carry their global id in every 16-bit word: the output shows the map."""
    P, cu = 4, _cu([8 * 11, 8 * 40, 8 * 5])
    T = int(cu[-1])
    ids = np.repeat(np.arange(T, dtype=np.uint16)[:, None], 64, axis=1)
    plan = cpt.cpt_plan_create(DSC, P, cu, T)
    src = to_dev(ids)
    dst = torch.empty((P, T // P, 64), dtype=torch.bfloat16, device="cuda")
    cpt.cpt_partition(plan, [src], [dst])
    torch.cuda.synchronize()
    got = to_host(dst).reshape(T, 64)
    l2g, _ = oracle.index_map(DSC, P, cu, T)
    assert np.array_equal(got[:, 0], l2g.astype(np.uint16))
    assert np.all(got == got[:, :1])


@pytest.mark.parametrize("layout", [DSC, PACKED])
def test_partition_lognormal_full(cpt, cuda_device, layout):
    """Packed THD workload: T=131072 from lognormal documents, Q/K/V [T,16,128] bf16."""
    lens = _lognormal_case(layout)
    cu = _cu(lens)
    T = int(cu[-1])
    xs = [synth.normal_bf16(synth.rng_for(2, 1 + t), (T, 16, 128)) for t in range(3)]
    plan = cpt.cpt_plan_create(layout, 4, cu, T)
    src = [to_dev(x) for x in xs]
    dst = [torch.empty((4, T // 4, 16, 128), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    cpt.cpt_partition(plan, src, dst)
    torch.cuda.synchronize()
    l2g, _ = oracle.index_map(layout, 4, cu, T)
    for x, d in zip(xs, dst):
        assert np.array_equal(to_host(d).reshape(T, 16, 128), oracle.partition(l2g, x))


# ---------------------------------------------------------------- grad return


def _writers(rng, P, T, row_shape, dt, sigma=1.0):
    if dt == "f32":
        return [synth.uniform_f32(rng, (T,) + row_shape) for _ in range(P)]
    return [synth.normal_bf16(rng, (T,) + row_shape, sigma) for _ in range(P)]


GR_CASES = [
    # tiny configuration: P=2, T=64 from [16,24,24], H=2, D=8, float32
    (DSC, 2, [16, 24, 24], (2, 8), "f32", "f32"),
    (PACKED, 2, [16, 24, 24], (2, 8), "f32", "f32"),
    (DSC, 1, [8, 0, 24], (2, 8), "bf16", "bf16"),
    (DSC, 3, [6 * 100, 0, 6 * 301], (3, 8), "bf16", "bf16"),     # 48-byte rows
    (DSC, 4, [8 * 257, 8 * 3], (5, 40), "bf16", "f32"),
    (PACKED, 5, [1, 2003, 996], (2, 8), "f32", "bf16"),
    (PACKED, 6, [6 * 512], (4, 24), "f32", "f32"),
    (DSC, 7, [14 * 70, 14 * 5], (1, 24), "bf16", "bf16"),
    (DSC, 8, [16 * 128, 0, 16 * 9], (20, 128), "bf16", "bf16"),
    (PACKED, 8, [5, 1019], (8, 128), "bf16", "f32"),
]


@pytest.mark.parametrize("case", GR_CASES, ids=lambda c: f"L{c[0]}P{c[1]}{c[4]}to{c[5]}")
@pytest.mark.parametrize("with_dv", [True, False])
def test_grad_return_matches_oracle(cpt, cuda_device, case, with_dv):
    layout, P, lens, row_shape, din, dout = case
    cu = _cu(lens)
    T = int(cu[-1])
    rng = np.random.default_rng(1000 + P)
    wk = _writers(rng, P, T, row_shape, din)
    wv = _writers(rng, P, T, row_shape, din)
    plan = cpt.cpt_plan_create(layout, P, cu, T)
    odt = torch.float32 if dout == "f32" else torch.bfloat16
    ok = [Guarded((T // P,) + row_shape, odt) for _ in range(P)]
    ov = [Guarded((T // P,) + row_shape, odt) for _ in range(P)]
    cpt.cpt_grad_return(plan, [to_dev(w) for w in wk], [to_dev(w) for w in wv] if with_dv else None,
                        [o.t for o in ok], [o.t for o in ov] if with_dv else None)
    torch.cuda.synchronize()
    l2g, _ = oracle.index_map(layout, P, cu, T)
    code = oracle.F32 if dout == "f32" else oracle.BF16
    for ws, outs in ((wk, ok), (wv, ov)) if with_dv else ((wk, ok),):
        want = oracle.grad_return(l2g, ws, code)
        for o in range(P):
            assert np.array_equal(bits(to_host(outs[o].t)), bits(want[o])), f"owner {o}"
            assert outs[o].bands_intact()
    if not with_dv:
        for o in ov:
            assert (o.raw == 0x5A).all()


def test_grad_return_single_doc_config(cpt, cuda_device):
    """Single-document gradient return: P=4, S=32768, H=8, D=128, bf16 N(0,1),
    8 chunks of 4096 tokens, dK and dV in one launch, every output compared."""
    P, S = 4, 32768
    cu = _cu([S])
    wk = [synth.normal_bf16(synth.rng_for(1, w), (S, 8, 128)) for w in range(P)]
    wv = [synth.normal_bf16(synth.rng_for(1, 10 + w), (S, 8, 128)) for w in range(P)]
    plan = cpt.cpt_plan_create(DSC, P, cu, S)
    dkw = torch.stack([to_dev(w) for w in wk])
    dvw = torch.stack([to_dev(w) for w in wv])
    dko = torch.empty((P, S // P, 8, 128), dtype=torch.bfloat16, device="cuda")
    dvo = torch.empty_like(dko)
    cpt.cpt_grad_return(plan, dkw, dvw, dko, dvo)
    torch.cuda.synchronize()
    l2g, _ = oracle.index_map(DSC, P, cu, S)
    for ws, out in ((wk, dko), (wv, dvo)):
        want = oracle.grad_return(l2g, ws, oracle.BF16)
        got = to_host(out)
        for o in range(P):
            assert np.array_equal(got[o], want[o])
    # owner r holds chunks r and 7-r: spot-check one row of each half directly
    h = to_host(dko)
    for r in range(P):
        for j, g in ((0, r * 4096), (4096, (7 - r) * 4096)):
            acc = np.float32(0)
            vals = [(wk[w][g].astype(np.uint32) << 16).view(np.float32) for w in range(P)]
            acc = vals[0].copy()
            for v in vals[1:]:
                acc = np.add(acc, v, dtype=np.float32)
            assert np.array_equal(h[r][j], oracle.f32_to_bf16_array(acc))


@pytest.mark.parametrize("case", GR_CASES, ids=lambda c: f"L{c[0]}P{c[1]}{c[4]}to{c[5]}")
def test_grad_return_accumulate_matches_oracle(cpt, cuda_device, case):
    """Accumulate-into mode: the owners' current values start the ordered sums."""
    layout, P, lens, row_shape, din, dout = case
    cu = _cu(lens)
    T = int(cu[-1])
    rng = np.random.default_rng(3000 + P)
    wk = _writers(rng, P, T, row_shape, din)
    wv = _writers(rng, P, T, row_shape, din)
    if dout == "f32":
        sk = [synth.uniform_f32(rng, (T // P,) + row_shape, -3, 3) for _ in range(P)]
        sv = [synth.uniform_f32(rng, (T // P,) + row_shape, -3, 3) for _ in range(P)]
    else:
        sk = [synth.uniform_bf16(rng, (T // P,) + row_shape, -3, 3) for _ in range(P)]
        sv = [synth.uniform_bf16(rng, (T // P,) + row_shape, -3, 3) for _ in range(P)]
    plan = cpt.cpt_plan_create(layout, P, cu, T)
    ok = [to_dev(x) for x in sk]
    ov = [to_dev(x) for x in sv]
    cpt.cpt_grad_return_accumulate(plan, [to_dev(w) for w in wk], [to_dev(w) for w in wv], ok, ov)
    torch.cuda.synchronize()
    l2g, _ = oracle.index_map(layout, P, cu, T)
    for ws, starts, outs in ((wk, sk, ok), (wv, sv, ov)):
        want = oracle.grad_return_accumulate(l2g, ws, starts)
        for o in range(P):
            assert np.array_equal(bits(to_host(outs[o])), bits(want[o])), f"owner {o}"


@pytest.mark.parametrize("P", [2, 4, 8])
def test_grad_return_accumulate_closed_forms(cpt, cuda_device, P):
    cu = _cu([2 * P * 64])
    T = int(cu[-1])
    plan = cpt.cpt_plan_create(DSC, P, cu, T)
    w = torch.ones((P, T, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.ones((P, T // P, 64), dtype=torch.bfloat16, device="cuda")
    cpt.cpt_grad_return_accumulate(plan, w, None, o, None)
    cpt.cpt_grad_return_accumulate(plan, w, None, o, None)
    torch.cuda.synchronize()
    assert bool((o == 2 * P + 1).all().item())


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_grad_return_closed_forms(cpt, cuda_device, P, dt):
    """All-ones writers give exactly P; the order canary gives 1, not 0 or 2."""
    cu = _cu([2 * P * 96])
    T = int(cu[-1])
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    plan = cpt.cpt_plan_create(DSC, P, cu, T)
    w = torch.ones((P, T, 64), dtype=tdt, device="cuda")
    o = torch.empty((P, T // P, 64), dtype=tdt, device="cuda")
    cpt.cpt_grad_return(plan, w, None, o, None)
    torch.cuda.synchronize()
    assert bool((o == P).all().item())
    if P == 4:
        canary = torch.tensor([2.0**24, 1.0, -(2.0**24), 1.0], dtype=tdt, device="cuda")
        w = canary.view(4, 1, 1).expand(4, T, 64).contiguous()
        cpt.cpt_grad_return(plan, w, None, o, None)
        torch.cuda.synchronize()
        assert bool((o == 1.0).all().item())
    nz = torch.full((P, T, 64), -0.0, dtype=tdt, device="cuda")
    cpt.cpt_grad_return(plan, nz, None, o, None)
    torch.cuda.synchronize()
    assert bool(torch.signbit(o).all().item()) and bool((o == 0).all().item())


# ---------------------------------------------------------------- slot reduce


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("din,dout", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32"), ("f32", "bf16")])
@pytest.mark.parametrize("n", [1, 7, 8, 1000, 4096 * 37 + 5, 1 << 20])
def test_slot_reduce_matches_oracle(cpt, cuda_device, P, din, dout, n):
    rng = np.random.default_rng(n + P)
    slots = [synth.uniform_f32(rng, (n,)) if din == "f32" else synth.uniform_bf16(rng, (n,))
             for _ in range(P)]
    odt = torch.float32 if dout == "f32" else torch.bfloat16
    dst = Guarded((n,), odt)
    cpt.cpt_slot_reduce([to_dev(s) for s in slots], dst.t)
    torch.cuda.synchronize()
    want = oracle.slot_reduce(slots, oracle.F32 if dout == "f32" else oracle.BF16)
    assert np.array_equal(bits(to_host(dst.t)), bits(want))
    assert dst.bands_intact()


def test_slot_reduce_status_gate(cpt, cuda_device):
    slots = [torch.ones(1000, device="cuda") for _ in range(3)]
    dst = torch.full((1000,), 5.0, device="cuda")
    status = torch.tensor([7], dtype=torch.int32, device="cuda")
    cpt.cpt_slot_reduce(slots, dst, status)
    torch.cuda.synchronize()
    assert bool((dst == 5.0).all().item())
    status.zero_()
    cpt.cpt_slot_reduce(slots, dst, status)
    torch.cuda.synchronize()
    assert bool((dst == 3.0).all().item())


# ---------------------------------------------------------------- validation


def test_rejections_leave_outputs_untouched(cpt, cuda_device):
    P, cu = 4, _cu([64])
    plan = cpt.cpt_plan_create(DSC, P, cu, 64)
    w = torch.randn((P, 64, 16), device="cuda").to(torch.bfloat16)
    o = torch.full((P, 16, 16), 3.0, dtype=torch.bfloat16, device="cuda")

    def expect(status, fn):
        with pytest.raises(cpt.CptError) as ei:
            fn()
        assert ei.value.status == status, str(ei.value)

    host = torch.empty((P, 64, 16), dtype=torch.bfloat16).pin_memory()
    expect(cpt.CPT_ERR_DEVICE, lambda: cpt.cpt_grad_return(plan, host, None, o, None))
    expect(cpt.CPT_ERR_ALIAS, lambda: cpt.cpt_grad_return(plan, w, None, [o[0], o[0], o[1], o[2]], None))
    expect(cpt.CPT_ERR_ALIAS, lambda: cpt.cpt_grad_return(plan, w, None, [w[0][:16]] + [o[i] for i in range(1, 4)], None))
    expect(cpt.CPT_ERR_INVALID_ARG, lambda: cpt.cpt_grad_return(plan, w, w, o, None))
    mis = torch.empty(P * 16 * 16 + 8, dtype=torch.bfloat16, device="cuda")[1:1 + P * 16 * 16].view(P, 16, 16)
    expect(cpt.CPT_ERR_ALIGNMENT, lambda: cpt.cpt_grad_return(plan, w, None, mis, None))
    w3 = torch.randn((P, 64, 3), device="cuda")  # 12-byte rows
    o3 = torch.empty((P, 16, 3), device="cuda")
    expect(cpt.CPT_ERR_ALIGNMENT, lambda: cpt.cpt_grad_return(plan, w3, None, o3, None))
    slots = [torch.empty((16, 16), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    expect(cpt.CPT_ERR_ALIAS, lambda: cpt.cpt_grad_scatter(plan, 1, w[1], slots, slots[0]))
    expect(cpt.CPT_ERR_INVALID_ARG, lambda: cpt.cpt_grad_scatter(plan, 4, w[1], slots, slots[0]))
    expect(cpt.CPT_ERR_NOT_DIVISIBLE, lambda: cpt.cpt_plan_create(DSC, 4, [0, 12], 12))
    expect(cpt.CPT_ERR_NOT_DIVISIBLE, lambda: cpt.cpt_plan_create(PACKED, 3, [0, 10], 10))
    expect(cpt.CPT_ERR_INVALID_ARG, lambda: cpt.cpt_plan_create(DSC, 9, [0, 18], 18))
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    expect(cpt.CPT_ERR_WORKSPACE, lambda: cpt.cpt_plan_create(DSC, 4, cu, 64, workspace=small))
    q = torch.randn((64, 16), device="cuda")
    expect(cpt.CPT_ERR_ALIAS, lambda: cpt.cpt_partition(plan, [q], [q.view(P, 16, 16)]))
    torch.cuda.synchronize()
    assert bool((o == 3.0).all().item())


# ---------------------------------------------------------------- padded layout

PADDED = 3
PAD_CASES = [
    (2, [5, 0, 7], (2, 8), "f32"),
    (4, [1, 8, 13, 0, 2047, 3], (3, 40), "bf16"),
    (8, [100, 17], (20, 128), "bf16"),
    (3, [6, 7, 11, 1], (1, 8), "bf16"),
    (1, [3, 0, 4], (1, 4), "f32"),
]


@pytest.mark.parametrize("P,lens,row_shape,dt", PAD_CASES)
def test_padded_layout_matches_oracle(cpt, cuda_device, P, lens, row_shape, dt):
    cu = _cu(lens)
    T = int(cu[-1])
    n = len(lens)
    cup, ol2g, og2l = oracle.padded_index_map(P, cu)
    Tpad = int(cup[-1])
    plan = cpt.cpt_plan_create(PADDED, P, cu, T)
    assert cpt.cpt_plan_padded_tokens(plan) == Tpad and plan.local_tokens == Tpad // P

    # maps and metadata over the padded boundaries, real-token counts
    l2g = torch.empty(Tpad, dtype=torch.int32, device="cuda")
    g2l = torch.empty(Tpad, dtype=torch.int32, device="cuda")
    cpt.cpt_index_map(plan, l2g, g2l)
    ns = torch.empty(P, dtype=torch.int32, device="cuda")
    first = torch.empty(P, dtype=torch.int32, device="cuda")
    cul = torch.empty((P, n + 1), dtype=torch.int32, device="cuda")
    offs = torch.empty(P + 1, dtype=torch.int32, device="cuda")
    cpt.cpt_thd_metadata(plan, ns, first, cul, offs)
    rl = torch.full((P, n), -1, dtype=torch.int32, device="cuda")
    cpt.cpt_thd_real_lengths(plan, rl)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(l2g), ol2g) and np.array_equal(to_host(g2l), og2l)
    for got, want in zip((ns, first, cul, offs), oracle.thd_metadata(DSC, P, cup, Tpad)):
        assert np.array_equal(to_host(got), want)
    assert np.array_equal(to_host(rl), oracle.real_lengths(DSC, P, cu, padded=True))

    # partition pads on the fly, restore drops the padding
    rng = np.random.default_rng(P + 70)
    xs = [_rand_rows(rng, T, row_shape, dt) for _ in range(3)]
    src = [to_dev(x) for x in xs]
    dst = [Guarded((P, Tpad // P) + row_shape, src[0].dtype) for _ in range(3)]
    for d in dst:
        d.t.fill_(7.0)  # padding rows must come back as zeros
    cpt.cpt_partition(plan, src, [d.t for d in dst])
    back = [Guarded((T,) + row_shape, src[0].dtype) for _ in range(3)]
    cpt.cpt_restore(plan, [d.t for d in dst], [b.t for b in back])
    torch.cuda.synchronize()
    for x, d, b in zip(xs, dst, back):
        want = oracle.partition_padded(P, cu, x).reshape((P, Tpad // P) + row_shape)
        assert np.array_equal(bits(to_host(d.t)), bits(want))
        assert np.array_equal(bits(to_host(b.t)), bits(x))
        assert d.bands_intact() and b.bands_intact()

    # gradient return over the padded global buffer
    wk = _writers(rng, P, Tpad, row_shape, dt)
    ok = [Guarded((Tpad // P,) + row_shape, src[0].dtype) for _ in range(P)]
    cpt.cpt_grad_return(plan, [to_dev(w) for w in wk], None, [o.t for o in ok], None)
    torch.cuda.synchronize()
    want = oracle.grad_return(ol2g, wk, oracle.F32 if dt == "f32" else oracle.BF16)
    for o in range(P):
        assert np.array_equal(bits(to_host(ok[o].t)), bits(want[o]))
        assert ok[o].bands_intact()


@pytest.mark.parametrize("layout,P,lens", [(DSC, 4, [8 * 3, 8 * 500, 0, 8 * 211]),
                                           (PACKED, 3, [7, 1000, 3, 2590]),
                                           (PACKED, 8, [1, 5, 0, 90, 24])])
def test_real_lengths_unpadded(cpt, cuda_device, layout, P, lens):
    cu = _cu(lens)
    T = int(cu[-1])
    plan = cpt.cpt_plan_create(layout, P, cu, T)
    rl = torch.full((P, len(lens)), -1, dtype=torch.int32, device="cuda")
    cpt.cpt_thd_real_lengths(plan, rl)
    torch.cuda.synchronize()
    want = oracle.real_lengths(layout, P, cu)
    assert np.array_equal(to_host(rl), want)
    assert np.array_equal(want.sum(axis=0), np.diff(cu))


# ---------------------------------------------------------------- row ranges


@pytest.mark.parametrize("layout,P,lens", [(DSC, 4, [8 * 300, 0, 8 * 97]), (PACKED, 3, [7, 1000, 3, 2590]),
                                           (PADDED, 4, [13, 0, 1000, 7])])
def test_row_range_calls_cover_the_full_calls(cpt, cuda_device, layout, P, lens):
    """Ragged row pieces that together cover the batch give the full result;
    rows outside a single piece are not touched."""
    cu = _cu(lens)
    T = int(cu[-1])
    row = (2, 64)
    plan = cpt.cpt_plan_create(layout, P, cu, T)
    Tpad = plan.padded_tokens
    rng = np.random.default_rng(31)
    hq = synth.normal_bf16(rng, (T,) + row)
    hw = [synth.normal_bf16(rng, (Tpad,) + row) for _ in range(P)]
    q = to_dev(hq)
    w = torch.stack([to_dev(x) for x in hw])
    full_q = torch.empty((P, Tpad // P) + row, dtype=torch.bfloat16, device="cuda")
    full_o = torch.empty((P, Tpad // P) + row, dtype=torch.bfloat16, device="cuda")
    cpt.cpt_partition(plan, [q], [full_q])
    cpt.cpt_grad_return(plan, w, None, full_o, None)
    cuts = sorted(set([0, Tpad] + rng.integers(0, Tpad, size=9).tolist()))
    part_q = torch.full_like(full_q, 5.0)
    part_o = torch.full_like(full_o, 5.0)
    for a, b in zip(cuts[:-1], cuts[1:]):
        cpt.cpt_partition_rows(plan, [q], [part_q], a, b - a)
        cpt.cpt_grad_return_rows(plan, w, None, part_o, None, a, b - a)
    one_q = torch.full_like(full_q, 5.0)
    a, b = Tpad // 3, Tpad // 3 + 101
    cpt.cpt_partition_rows(plan, [q], [one_q], a, b - a)
    torch.cuda.synchronize()
    assert torch.equal(part_q.view(torch.int16), full_q.view(torch.int16))
    assert torch.equal(part_o.view(torch.int16), full_o.view(torch.int16))
    flat = one_q.view(Tpad, -1)
    assert torch.equal(flat[a:b].view(torch.int16), full_q.view(Tpad, -1)[a:b].view(torch.int16))
    assert bool((flat[:a] == 5.0).all().item()) and bool((flat[b:] == 5.0).all().item())
    with pytest.raises(cpt.CptError) as ei:
        cpt.cpt_grad_return_rows(plan, w, None, part_o, None, Tpad - 1, 2)
    assert ei.value.status == cpt.CPT_ERR_INVALID_ARG

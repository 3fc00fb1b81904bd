"""Full-size parity at the pages' training shape ("Add stream-ordered CP
gradient return primitive", TransformerEngine PR 3235, "Validation": CP=4,
S=262144, 20 heads of dimension 128), in the launch configuration the
benchmark times: one fused dK+dV grad_return launch and one three-tensor
partition launch.

Every output element is compared with the oracle: the writers are copied
back to the host and the oracle redoes all 13.4 GB of the fused launch's
sums (and the whole lognormal batch and both 1 GB slot reduces), with its
calls spread over host threads (ctypes releases the GIL; each thread runs
the unmodified oracle on its own part). Properties that hold at any size are
checked on the whole output as well.
"""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import oracle
from context_attention_token_gb300 import synth
from gpu_helpers import bits, to_host

pytestmark = pytest.mark.gpu

P, S, H, D = 4, 262144, 20, 128
TP = S // P
M = S // (2 * P)  # chunk length 32768


def _host_threads():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_grad_return_all(l2g, writer_sets, out_dtype):
    """oracle.grad_return of each writer set (dK, dV, ...), one host thread each."""
    with cf.ThreadPoolExecutor(max_workers=len(writer_sets)) as ex:
        return list(ex.map(lambda ws: oracle.grad_return(l2g, ws, out_dtype), writer_sets))


def _oracle_slot_reduce_chunked(slots, out_dtype, parts):
    """oracle.slot_reduce over `parts` contiguous element ranges in parallel;
    each range is an independent ordered sum of the same slots."""
    n = slots[0].shape[0]
    cuts = [n * i // parts for i in range(parts + 1)]
    with cf.ThreadPoolExecutor(max_workers=parts) as ex:
        pieces = list(ex.map(lambda ab: oracle.slot_reduce([s[ab[0]:ab[1]] for s in slots], out_dtype),
                             zip(cuts, cuts[1:])))
    return np.concatenate(pieces)


@pytest.fixture(scope="module")
def big_plan(cpt, cuda_device):
    cu = np.array([0, S], np.int32)
    plan = cpt.cpt_plan_create(0, P, cu, S)
    l2g, _ = oracle.index_map(0, P, cu, S)
    return plan, l2g


def test_grad_return_pages_shape_whole_output(cpt, big_plan):
    """The benched launch (dK and dV fused, P=4, S=262144, 20x128 bf16):
    every one of the 2 x 4 x 65536 owner rows equals the oracle bit for bit."""
    plan, l2g = big_plan
    dkw = synth.device_normal_bf16((P, S, H, D), 4001, 0.02, "cuda")
    dvw = synth.device_normal_bf16((P, S, H, D), 4002, 0.02, "cuda")
    dko = torch.empty((P, TP, H, D), dtype=torch.bfloat16, device="cuda")
    dvo = torch.empty_like(dko)
    cpt.cpt_grad_return(plan, dkw, dvw, dko, dvo)
    torch.cuda.synchronize()
    assert cpt.cpt_kernel_wait_timeouts() == 0
    sets = [[to_host(w_all[w]) for w in range(P)] for w_all in (dkw, dvw)]
    got = [to_host(dko), to_host(dvo)]
    del dkw, dvw, dko, dvo
    torch.cuda.empty_cache()
    want = _oracle_grad_return_all(l2g, sets, oracle.BF16)
    for g, w in zip(got, want):
        for o in range(P):
            assert np.array_equal(g[o], w[o]), f"owner {o} differs"


def test_grad_return_pages_shape_closed_forms(cpt, big_plan):
    plan, _ = big_plan
    w = torch.ones((P, S, H, D), dtype=torch.bfloat16, device="cuda")
    o = torch.empty((P, TP, H, D), dtype=torch.bfloat16, device="cuda")
    cpt.cpt_grad_return(plan, w, None, o, None)
    torch.cuda.synchronize()
    assert bool((o == P).all().item())
    # writer w holds the value 2^w at every token: every owner element is
    # 1 + 2 + 4 + 8 = 15 exactly, and each writer's contribution is visible
    w.copy_(torch.tensor([1.0, 2.0, 4.0, 8.0], dtype=torch.bfloat16, device="cuda").view(P, 1, 1, 1)
            .expand(P, S, H, D))
    cpt.cpt_grad_return(plan, w, None, o, None)
    torch.cuda.synchronize()
    assert bool((o == 15.0).all().item())
    # row-id payload in writer 0 (others zero): owner o row j must hold l2g[o*TP+j]
    # as a bf16-exact small integer pattern: encode (g mod 256)
    gid = (torch.arange(S, device="cuda") % 256).to(torch.bfloat16).view(S, 1, 1)
    w.zero_()
    w[0].copy_(gid.expand(S, H, D))
    cpt.cpt_grad_return(plan, w, None, o, None)
    torch.cuda.synchronize()
    cu = np.array([0, S], np.int32)
    l2g, _ = oracle.index_map(0, P, cu, S)
    want = torch.from_numpy((l2g % 256).astype(np.float32)).cuda().to(torch.bfloat16).view(P, TP)
    assert torch.equal(o[:, :, 0, 0], want)
    assert bool((o == o[:, :, :1, :1]).all().item())
    del w, o
    torch.cuda.empty_cache()


def test_partition_pages_shape_whole_output(cpt, big_plan):
    plan, l2g = big_plan
    qkv = [synth.device_normal_bf16((S, H, D), 4010 + t, 1.0, "cuda") for t in range(3)]
    dst = [torch.empty((P, TP, H, D), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    cpt.cpt_partition(plan, qkv, dst)
    torch.cuda.synchronize()
    # the oracle's row copy through its own map, over the whole of Q, K and V
    for x, d in zip(qkv, dst):
        want = oracle.partition(l2g, to_host(x))
        assert np.array_equal(to_host(d).reshape(S, H, D), want)
        del want
    # whole tensors: the oracle's map applied by torch's own row gather
    # (a library routine, not this library's kernel) must equal the output
    gi = torch.from_numpy(l2g.astype(np.int64)).cuda()
    for x, d in zip(qkv, dst):
        assert torch.equal(d.view(S, H, D).view(torch.int16), x.index_select(0, gi).view(torch.int16))
    # all-gather restore of K and V gives back the inputs bit for bit
    back = [torch.empty((S, H, D), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    cpt.cpt_restore(plan, dst[1:], back)
    torch.cuda.synchronize()
    for x, b in zip(qkv[1:], back):
        assert torch.equal(b.view(torch.int16), x.view(torch.int16))
    del qkv, dst, back
    torch.cuda.empty_cache()


def test_largest_batch_the_maps_allow(cpt, cuda_device):
    """T = 2^31 - 8 tokens (one document, P=4, 16-byte rows): the int32 maps
    and every 64-bit offset in the kernels at their limit."""
    T, Pm = 2**31 - 8, 4
    m = T // (2 * Pm)
    Tp = T // Pm
    plan = cpt.cpt_plan_create(0, Pm, [0, T], T)
    l2g = torch.empty(T, dtype=torch.int32, device="cuda")
    g2l = torch.empty(T, dtype=torch.int32, device="cuda")
    cpt.cpt_index_map(plan, l2g, g2l)
    torch.cuda.synchronize()
    # the ownership rule: rank r holds chunk r, then chunk 2P-1-r
    for r in range(Pm):
        for j in (0, 1, m - 1, m, m + 1, Tp - 1):
            want = r * m + j if j < m else (2 * Pm - 1 - r) * m + (j - m)
            assert int(l2g[r * Tp + j].item()) == want
    step = 1 << 27
    for a in range(0, T, step):
        b = min(a + step, T)
        idx = l2g[a:b].long()
        assert torch.equal(g2l[idx].long(), torch.arange(a, b, device="cuda"))
    del g2l, idx
    # row-id payload: global row g holds g in all four words; after the
    # partition local row q must hold l2g[q]
    src = torch.arange(T, dtype=torch.int32, device="cuda").view(T, 1).expand(T, 4).contiguous()
    dst = torch.empty((Pm, Tp, 4), dtype=torch.int32, device="cuda")
    cpt.cpt_partition(plan, [src.view(torch.float32)], [dst.view(torch.float32)])
    torch.cuda.synchronize()
    flat = dst.view(T, 4)
    for a in range(0, T, step):
        b = min(a + step, T)
        blk = flat[a:b]
        assert torch.equal(blk[:, 0], l2g[a:b]) and bool((blk == blk[:, :1]).all().item())
    del src, dst, flat, l2g
    torch.cuda.empty_cache()


@pytest.mark.parametrize("layout", [0, 1])
def test_grad_return_lognormal_batch_whole_output(cpt, cuda_device, layout):
    """Packed THD configuration: T=131072 from lognormal documents, writers
    [4, T, 16, 128] bf16 N(0,1), both layouts, every owner row against the
    oracle."""
    Pl, Tl, Hl = 4, 131072, 16
    lens = synth.lognormal_doc_lengths(Tl, synth.rng_for(2, 0), multiple=8 if layout == 0 else 1)
    cu = synth.cu_from_lengths(lens)
    plan = cpt.cpt_plan_create(layout, Pl, cu, Tl)
    l2g, _ = oracle.index_map(layout, Pl, cu, Tl)
    wk = synth.device_normal_bf16((Pl, Tl, Hl, D), 4101 + layout, 1.0, "cuda")
    wv = synth.device_normal_bf16((Pl, Tl, Hl, D), 4111 + layout, 1.0, "cuda")
    ok = torch.empty((Pl, Tl // Pl, Hl, D), dtype=torch.bfloat16, device="cuda")
    ov = torch.empty_like(ok)
    cpt.cpt_grad_return(plan, wk, wv, ok, ov)
    torch.cuda.synchronize()
    assert cpt.cpt_kernel_wait_timeouts() == 0
    sets = [[to_host(w_all[w]) for w in range(Pl)] for w_all in (wk, wv)]
    got = [to_host(ok), to_host(ov)]
    del wk, wv, ok, ov
    torch.cuda.empty_cache()
    want = _oracle_grad_return_all(l2g, sets, oracle.BF16)
    for g, w in zip(got, want):
        for o in range(Pl):
            assert np.array_equal(g[o], w[o]), f"owner {o} differs"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_slot_reduce_one_gigabyte_slots_whole_output(cpt, cuda_device, dtype):
    """Slot-reduce configuration at its largest message: 8 slots of 1 GB
    (plus a ragged tail of 3 elements), every element against the oracle."""
    esz = torch.tensor([], dtype=dtype).element_size()
    n = (1 << 30) // esz + 3
    gen = torch.Generator(device="cuda")
    gen.manual_seed(4200 + esz)
    slots = [(torch.rand(n, device="cuda", generator=gen) * 2 - 1).to(dtype) for _ in range(8)]
    dst = torch.empty(n, dtype=dtype, device="cuda")
    cpt.cpt_slot_reduce(slots, dst)
    torch.cuda.synchronize()
    assert cpt.cpt_kernel_wait_timeouts() == 0
    hs = [to_host(s) for s in slots]
    got = to_host(dst)
    del slots, dst
    torch.cuda.empty_cache()
    want = _oracle_slot_reduce_chunked(hs, oracle.BF16 if dtype == torch.bfloat16 else oracle.F32,
                                       min(16, _host_threads()))
    assert np.array_equal(bits(got), bits(want))


def test_packed_partition_and_restore_pages_shape_whole_output(cpt, cuda_device):
    """The packed-contiguous policy at the pages' shape (P=4, S=262144, one
    document, 20x128 bf16): the whole Q/K/V partition against the oracle's
    packed map, and the restore back to the inputs. At this size the bulk path
    runs its straight copy."""
    cu = np.array([0, S], np.int32)
    plan = cpt.cpt_plan_create(1, P, cu, S)
    l2g, _ = oracle.index_map(1, P, cu, S)
    qkv = [synth.device_normal_bf16((S, H, D), 4020 + t, 1.0, "cuda") for t in range(3)]
    dst = [torch.empty((P, TP, H, D), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    cpt.cpt_partition(plan, qkv, dst)
    torch.cuda.synchronize()
    for x, d in zip(qkv, dst):
        assert np.array_equal(to_host(d).reshape(S, H, D), oracle.partition(l2g, to_host(x)))
    back = [torch.empty((S, H, D), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    cpt.cpt_restore(plan, dst, back)
    torch.cuda.synchronize()
    for x, b in zip(qkv, back):
        assert torch.equal(b.view(torch.int16), x.view(torch.int16))
    assert cpt.cpt_kernel_wait_timeouts() == 0
    del qkv, dst, back
    torch.cuda.empty_cache()


def test_staged_path_equals_fused_pages_shape(cpt, big_plan):
    """The staged gradient return at the pages' shape (P writer streams
    scatter into owner slots and publish an epoch, P owner streams wait and
    reduce their slots in writer order) equals the fused launch bit for bit;
    the fused launch equals the oracle on every element (above)."""
    plan, _ = big_plan
    dkw = synth.device_normal_bf16((P, S, H, D), 4001, 0.02, "cuda")
    fused = torch.empty((P, TP, H, D), dtype=torch.bfloat16, device="cuda")
    cpt.cpt_grad_return(plan, dkw, None, fused, None)
    slots = torch.empty((P, P, TP, H, D), dtype=torch.bfloat16, device="cuda")
    staged = torch.full((P, TP, H, D), 9.0, dtype=torch.bfloat16, device="cuda")
    ep = cpt.cpt_epoch_create(P)
    main = torch.cuda.current_stream()
    wst = [torch.cuda.Stream() for _ in range(P)]
    ost = [torch.cuda.Stream() for _ in range(P)]
    cpt.cpt_epoch_advance(ep)
    for w in range(P):
        wst[w].wait_stream(main)
        cpt.cpt_grad_scatter(plan, w, dkw[w], [slots[o, w] for o in range(P)], slots[w, w], stream=wst[w])
        cpt.cpt_epoch_publish(ep, w, stream=wst[w])
    for o in range(P):
        ost[o].wait_stream(main)
        cpt.cpt_epoch_wait(ep, o, 2_000_000_000, cpt.CPT_WAIT_BOUNDED, stream=ost[o])
        cpt.cpt_slot_reduce(slots[o], staged[o], ep.status_ptr(o), stream=ost[o])
    for st in wst + ost:
        main.wait_stream(st)
    torch.cuda.synchronize()
    assert [cpt.cpt_epoch_status(ep, o) for o in range(P)] == [0] * P
    assert torch.equal(staged.view(torch.int16), fused.view(torch.int16))
    assert cpt.cpt_kernel_wait_timeouts() == 0
    del dkw, fused, slots, staged
    torch.cuda.empty_cache()

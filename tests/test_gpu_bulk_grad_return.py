"""Parity of the bulk-copy gradient return kernel.

With equal input and output types and overwrite mode, the gradient return
can run either of two kernels: 16-byte loads into registers, or bulk copies
that stage the P writer rows in shared memory. Each case here runs three
times: under the measured rule, and with each kernel forced. The cases span
every cp_size and both sides of each edge of the rule: the smallest bulk row
at P = 3 and P = 4, float32 rows at P = 4, and rows at P = 8 just inside and
just outside the bulk kernel's shared-memory limit (outside it, forcing bulk
runs the loads kernel). Every
output is compared bit for bit with the oracle, with canary bands around
each owner's buffer. The last test checks that no bulk-copy wait ran out of
its budget in any of them.
"""
import numpy as np
import pytest
import torch

import oracle
from context_attention_token_gb300 import synth
from gpu_helpers import Guarded, bits, to_dev, to_host

pytestmark = pytest.mark.gpu

DSC, PACKED, PADDED = 0, 1, 3

# (layout, P, document lengths, row elements, element type); the comment
# names the kernel that the row-size part of the rule picks. These launches
# are small, so under "auto" the launch-size part (at least 2 GiB for P <= 6)
# keeps P <= 6 on the 16-byte loads; the forced runs cover both kernels.
CASES = [
    (DSC, 1, [64, 32], 2560, "bf16"),        # 16-byte loads: P = 1
    (DSC, 2, [40, 24], 2560, "bf16"),        # 16-byte loads: P = 2
    (DSC, 3, [30, 6, 66], 1536, "bf16"),     # bulk: 3 KB rows, the smallest at P = 3
    (DSC, 3, [30, 6], 1024, "bf16"),         # 16-byte loads: 2 KB rows at P = 3
    (DSC, 4, [8, 56, 200], 2560, "bf16"),    # bulk: the pages' 20x128 rows
    (DSC, 4, [24, 8], 1024, "bf16"),         # bulk: 2 KB rows, the smallest at P = 4
    (DSC, 4, [24], 504, "bf16"),             # 16-byte loads: 1008-byte rows
    (DSC, 4, [16, 8], 512, "f32"),           # bulk: 2 KB float32 rows
    (DSC, 4, [16, 8], 1024, "f32"),          # 16-byte loads: 4 KB float32 rows
    (DSC, 5, [10, 90], 256, "f32"),          # bulk: 1 KB rows
    (DSC, 6, [12, 12, 36], 300, "f32"),      # bulk: 1200-byte rows, not a multiple of 512
    (DSC, 7, [14, 70], 520, "bf16"),         # bulk: 1040-byte rows
    (DSC, 8, [16, 48, 160], 2560, "bf16"),   # bulk
    (DSC, 8, [16], 1592, "f32"),             # bulk: 2 x 9 x 6368 B, at the shared-memory limit
    (DSC, 8, [16], 1596, "f32"),             # 16-byte loads: 16 bytes more per row
    (PACKED, 3, [5, 50, 17, 3, 9], 1536, "bf16"),
    (PACKED, 8, [0, 77, 19], 2560, "bf16"),
    (PADDED, 4, [5, 33, 1, 12], 2560, "bf16"),
    (PADDED, 8, [3, 17], 1024, "f32"),
]


KERNELS = ["auto", "loads", "bulk"]


@pytest.fixture
def kernel(cpt, request):
    """Run the test with the requested kernel choice, then restore the default."""
    code = {"auto": cpt.CPT_KERNEL_AUTO, "loads": cpt.CPT_KERNEL_LOADS,
            "bulk": cpt.CPT_KERNEL_BULK}[request.param]
    cpt.cpt_set_kernel_path(code)
    yield request.param
    cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_AUTO)


def _ids(c):
    return f"L{c[0]}-P{c[1]}-n{len(c[2])}-row{c[3]}-{c[4]}"


def _setup(case, seed):
    layout, P, lens, row, dt = case
    cu = synth.cu_from_lengths(lens)
    T = int(cu[-1])
    if layout == PADDED:
        cup, l2g, _ = oracle.padded_index_map(P, cu)
        Tpad = int(cup[-1])
    else:
        assert oracle.check_layout(layout, P, cu, T) == 0
        l2g, _ = oracle.index_map(layout, P, cu, T)
        Tpad = T
    rng = np.random.default_rng(seed)
    gen = synth.uniform_f32 if dt == "f32" else synth.uniform_bf16
    wk = [gen(rng, (Tpad, row)) for _ in range(P)]
    wv = [gen(rng, (Tpad, row)) for _ in range(P)]
    return layout, P, cu, T, Tpad, l2g, wk, wv, (oracle.F32 if dt == "f32" else oracle.BF16)


@pytest.mark.parametrize("kernel", KERNELS, indirect=True)
@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_bulk_grad_return_matches_oracle(cpt, cuda_device, case, kernel):
    layout, P, cu, T, Tpad, l2g, wk, wv, code = _setup(case, 7100 + case[1])
    odt = torch.float32 if case[4] == "f32" else torch.bfloat16
    row = case[3]
    plan = cpt.cpt_plan_create(layout, P, cu, T)
    ok = [Guarded((Tpad // P, row), odt) for _ in range(P)]
    ov = [Guarded((Tpad // P, row), odt) for _ in range(P)]
    cpt.cpt_grad_return(plan, torch.stack([to_dev(w) for w in wk]), torch.stack([to_dev(w) for w in wv]),
                        [o.t for o in ok], [o.t for o in ov])
    torch.cuda.synchronize()
    for ws, outs in ((wk, ok), (wv, ov)):
        want = oracle.grad_return(l2g, ws, code)
        for o in range(P):
            assert np.array_equal(bits(to_host(outs[o].t)), bits(want[o])), f"owner {o}"
            assert outs[o].bands_intact(), f"owner {o}"


ROW_RANGE_CASES = [c for c in CASES if c[3] * (4 if c[4] == "f32" else 2) >= 4096]


@pytest.mark.parametrize("kernel", KERNELS, indirect=True)
@pytest.mark.parametrize("case", ROW_RANGE_CASES, ids=_ids)
def test_bulk_grad_return_dk_only_and_row_ranges(cpt, cuda_device, case, kernel):
    """dK alone (no dV pair), then the same sums as three row ranges, then
    dK and dV together over three other row ranges (the launch's row index
    crosses from the dK half to the dV half, and the range offset applies to
    both)."""
    layout, P, cu, T, Tpad, l2g, wk, wv, code = _setup(case, 7200 + case[1])
    odt = torch.float32 if case[4] == "f32" else torch.bfloat16
    row = case[3]
    plan = cpt.cpt_plan_create(layout, P, cu, T)
    dkw = torch.stack([to_dev(w) for w in wk])
    whole = torch.empty((P, Tpad // P, row), dtype=odt, device="cuda")
    cpt.cpt_grad_return(plan, dkw, None, whole, None)
    pieces = torch.full((P, Tpad // P, row), 7.0, dtype=odt, device="cuda")
    cuts = [0, Tpad // 3, (2 * Tpad) // 3 + 1, Tpad]
    for a, b in zip(cuts, cuts[1:]):
        cpt.cpt_grad_return_rows(plan, dkw, None, pieces, None, a, b - a)
    torch.cuda.synchronize()
    dvw = torch.stack([to_dev(w) for w in wv])
    pk = torch.full((P, Tpad // P, row), 3.0, dtype=odt, device="cuda")
    pv = torch.full((P, Tpad // P, row), 5.0, dtype=odt, device="cuda")
    cuts2 = [0, 1, Tpad // 2, Tpad]
    for a, b in zip(cuts2, cuts2[1:]):
        cpt.cpt_grad_return_rows(plan, dkw, dvw, pk, pv, a, b - a)
    torch.cuda.synchronize()
    want = oracle.grad_return(l2g, wk, code)
    want_v = oracle.grad_return(l2g, wv, code)
    got_w, got_p = to_host(whole), to_host(pieces)
    got_k2, got_v2 = to_host(pk), to_host(pv)
    for o in range(P):
        assert np.array_equal(bits(got_w[o]), bits(want[o])), f"owner {o}"
        assert np.array_equal(bits(got_p[o]), bits(want[o])), f"owner {o}"
        assert np.array_equal(bits(got_k2[o]), bits(want[o])), f"owner {o}"
        assert np.array_equal(bits(got_v2[o]), bits(want_v[o])), f"owner {o}"


@pytest.mark.parametrize("kernel", KERNELS, indirect=True)
@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_bulk_grad_return_accumulate(cpt, cuda_device, case, kernel):
    """Accumulate mode: the owners' current rows start the ordered sums (the
    bulk kernel loads them into its output stage with the writer rows)."""
    layout, P, cu, T, Tpad, l2g, wk, wv, code = _setup(case, 7500 + case[1])
    row, dt = case[3], case[4]
    odt = torch.float32 if dt == "f32" else torch.bfloat16
    rng = np.random.default_rng(7600 + P)
    gen = synth.uniform_f32 if dt == "f32" else synth.uniform_bf16
    starts_k = [gen(rng, (Tpad // P, row)) for _ in range(P)]
    starts_v = [gen(rng, (Tpad // P, row)) for _ in range(P)]
    plan = cpt.cpt_plan_create(layout, P, cu, T)
    ok = torch.stack([to_dev(x) for x in starts_k])
    ov = torch.stack([to_dev(x) for x in starts_v])
    cpt.cpt_grad_return_accumulate(plan, torch.stack([to_dev(w) for w in wk]),
                                   torch.stack([to_dev(w) for w in wv]), ok, ov)
    torch.cuda.synchronize()
    for ws, st, out in ((wk, starts_k, ok), (wv, starts_v, ov)):
        want = oracle.grad_return_accumulate(l2g, ws, st)
        got = to_host(out)
        for o in range(P):
            assert np.array_equal(bits(got[o]), bits(want[o])), f"owner {o}"


MIXED = [
    (DSC, 4, [8, 56, 200], 2560, "bf16", "f32"),     # bf16 writers into float32 owners
    (DSC, 8, [16, 48], 1024, "bf16", "f32"),
    (DSC, 4, [8, 56, 200], 1280, "f32", "bf16"),     # float32 writers into bf16 owners
    (PADDED, 3, [5, 33, 1, 12], 512, "f32", "bf16"),
    (PACKED, 5, [0, 77, 23], 520, "bf16", "f32"),
]


@pytest.mark.parametrize("kernel", KERNELS, indirect=True)
@pytest.mark.parametrize("accumulate", [False, True], ids=["overwrite", "accumulate"])
@pytest.mark.parametrize("case", MIXED, ids=lambda c: f"L{c[0]}-P{c[1]}-row{c[3]}-{c[4]}to{c[5]}")
def test_bulk_grad_return_mixed_types(cpt, cuda_device, case, accumulate, kernel):
    """Writers and owners of different element types; the bulk kernel stages
    output rows of the output type."""
    layout, P, lens, row, din, dout = case
    cu = synth.cu_from_lengths(lens)
    T = int(cu[-1])
    if layout == PADDED:
        cup, l2g, _ = oracle.padded_index_map(P, cu)
        Tpad = int(cup[-1])
    else:
        l2g, _ = oracle.index_map(layout, P, cu, T)
        Tpad = T
    rng = np.random.default_rng(7700 + P + row)
    gin = synth.uniform_f32 if din == "f32" else synth.uniform_bf16
    gout = synth.uniform_f32 if dout == "f32" else synth.uniform_bf16
    wk = [gin(rng, (Tpad, row)) for _ in range(P)]
    wv = [gin(rng, (Tpad, row)) for _ in range(P)]
    plan = cpt.cpt_plan_create(layout, P, cu, T)
    code = oracle.F32 if dout == "f32" else oracle.BF16
    if accumulate:
        sk = [gout(rng, (Tpad // P, row)) for _ in range(P)]
        sv = [gout(rng, (Tpad // P, row)) for _ in range(P)]
        ok = torch.stack([to_dev(x) for x in sk])
        ov = torch.stack([to_dev(x) for x in sv])
        cpt.cpt_grad_return_accumulate(plan, torch.stack([to_dev(w) for w in wk]),
                                       torch.stack([to_dev(w) for w in wv]), ok, ov)
        wants = (oracle.grad_return_accumulate(l2g, wk, sk), oracle.grad_return_accumulate(l2g, wv, sv))
    else:
        odt = torch.float32 if dout == "f32" else torch.bfloat16
        ok = torch.empty((P, Tpad // P, row), dtype=odt, device="cuda")
        ov = torch.empty_like(ok)
        cpt.cpt_grad_return(plan, torch.stack([to_dev(w) for w in wk]), torch.stack([to_dev(w) for w in wv]),
                            ok, ov)
        wants = (oracle.grad_return(l2g, wk, code), oracle.grad_return(l2g, wv, code))
    torch.cuda.synchronize()
    for want, out in zip(wants, (ok, ov)):
        got = to_host(out)
        for o in range(P):
            assert np.array_equal(bits(got[o]), bits(want[o])), f"owner {o}"


@pytest.mark.parametrize("kernel", ["loads", "bulk"], indirect=True)
@pytest.mark.parametrize("case", [CASES[4], CASES[17]], ids=_ids)
def test_bulk_grad_return_noalloc(cpt, cuda_device, case, kernel):
    layout, P, cu, T, Tpad, l2g, wk, wv, code = _setup(case, 7300 + case[1])
    row = case[3]
    dkw = torch.stack([to_dev(w) for w in wk])
    dvw = torch.stack([to_dev(w) for w in wv])
    dko = torch.empty((P, Tpad // P, row), dtype=torch.bfloat16, device="cuda")
    dvo = torch.empty_like(dko)
    cpt.cpt_grad_return_noalloc(layout, P, cu, T, dkw, dvw, dko, dvo)
    torch.cuda.synchronize()
    for ws, out in ((wk, dko), (wv, dvo)):
        want = oracle.grad_return(l2g, ws, code)
        got = to_host(out)
        for o in range(P):
            assert np.array_equal(got[o], want[o]), f"owner {o}"


def test_bulk_kernel_from_concurrent_host_threads(cpt, cuda_device):
    """Four host threads, each on its own stream, launch the bulk kernel over
    and over with different row sizes, so the launcher's per-size occupancy
    cache keeps changing under them. Every result equals the oracle's."""
    import threading

    cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_BULK)
    try:
        jobs = []
        for k, row in enumerate((512, 1024, 2560, 640)):
            layout, P, cu, T, Tpad, l2g, wk, wv, code = _setup((DSC, 4, [8, 56, 200], row, "bf16"), 7400 + k)
            plan = cpt.cpt_plan_create(layout, P, cu, T)
            dkw = torch.stack([to_dev(w) for w in wk])
            dvw = torch.stack([to_dev(w) for w in wv])
            outs = [(torch.empty((P, Tpad // P, row), dtype=torch.bfloat16, device="cuda"),
                     torch.empty((P, Tpad // P, row), dtype=torch.bfloat16, device="cuda")) for _ in range(3)]
            want = (oracle.grad_return(l2g, wk, code), oracle.grad_return(l2g, wv, code))
            jobs.append((plan, dkw, dvw, outs, want, torch.cuda.Stream()))
        torch.cuda.synchronize()
        errors = []

        def run(job):
            plan, dkw, dvw, outs, _, stream = job
            try:
                for it in range(30):
                    ko, vo = outs[it % 3]
                    cpt.cpt_grad_return(plan, dkw, dvw, ko, vo, stream=stream)
            except Exception as e:  # reported on the main thread
                errors.append(e)

        threads = [threading.Thread(target=run, args=(j,)) for j in jobs]
        for t in threads:
            t.start()
        for t in threads:
            t.join()
        torch.cuda.synchronize()
        assert not errors, errors
        for plan, dkw, dvw, outs, want, _ in jobs:
            for ko, vo in outs:
                got_k, got_v = to_host(ko), to_host(vo)
                for o in range(4):
                    assert np.array_equal(got_k[o], want[0][o]) and np.array_equal(got_v[o], want[1][o])
    finally:
        cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_AUTO)


def test_no_bulk_copy_wait_ran_out(cpt, cuda_device):
    """Every bulk-copy wait above completed within its budget."""
    torch.cuda.synchronize()
    assert cpt.cpt_kernel_wait_timeouts() == 0
    assert cpt.cpt_kernel_wait_timeouts(reset=True) == 0

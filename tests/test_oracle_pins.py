"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these re-types the oracle's own formulas: the map is checked against
an ownership-then-sort brute force and a hand-derived worked example, the
sums against integer closed forms, an order canary, IEEE special cases and
numpy's own binary32 adds, and the bf16 rounding against hand-written IEEE
canaries and torch's CPU conversion.
"""
import os

import numpy as np
import pytest
import torch

import bruteforce as bf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    kv = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            kv[key] = vals
    return kv


# ---------------------------------------------------------------- maps


def test_worked_example_tiny(oracle_lib):
    o = oracle_lib
    g = _read_golden("dsc_tiny_worked_example.txt")
    P, T = int(g["P"][0]), int(g["T"][0])
    cu = [int(v) for v in g["cu_seqlens"]]
    l2g, g2l = o.index_map(o.LAYOUT_DSC, P, cu, T)
    for r in range(P):
        assert l2g[r * T // P:(r + 1) * T // P].tolist() == [int(v) for v in g[f"dsc_l2g_rank{r}"]]
    for tag, layout in (("dsc", o.LAYOUT_DSC), ("packed", o.LAYOUT_PACKED)):
        ns, first, cul, offs = o.thd_metadata(layout, P, cu, T)
        assert ns.tolist() == [int(v) for v in g[f"{tag}_num_segs"]]
        assert first.tolist() == [int(v) for v in g[f"{tag}_seg_doc_first"]]
        for r in range(P):
            assert cul[r].tolist() == [int(v) for v in g[f"{tag}_cu_local_rank{r}"]]
        assert offs.tolist() == [int(v) for v in g[f"{tag}_seg_offsets"]]


@pytest.mark.parametrize("P", [1, 2, 3, 4])
def test_dsc_map_matches_bruteforce_exhaustive(oracle_lib, P):
    o = oracle_lib
    for T in range(0, 25, 2 * P):
        for lens in bf.compositions(T, 2 * P, max_docs=4):
            cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
            l2g, g2l = o.index_map(o.LAYOUT_DSC, P, cu, T)
            want = bf.l2g_by_ownership(0, cu.tolist(), P, T)
            assert l2g.tolist() == want, (P, lens)
            assert all(g2l[want[q]] == q for q in range(T))
            meta = o.thd_metadata(o.LAYOUT_DSC, P, cu, T)
            ns, first, rows, offs = bf.metadata_by_runs(0, cu.tolist(), P, T)
            assert meta[0].tolist() == ns and meta[1].tolist() == first
            assert meta[2].tolist() == rows and meta[3].tolist() == offs


@pytest.mark.parametrize("P", [1, 2, 3, 4])
def test_packed_map_and_metadata_match_bruteforce(oracle_lib, P):
    o = oracle_lib
    for T in range(0, 13, P):
        for lens in bf.compositions(T, 1, max_docs=4):
            cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
            l2g, g2l = o.index_map(o.LAYOUT_PACKED, P, cu, T)
            assert l2g.tolist() == bf.l2g_by_ownership(1, cu.tolist(), P, T)
            meta = o.thd_metadata(o.LAYOUT_PACKED, P, cu, T)
            ns, first, rows, offs = bf.metadata_by_runs(1, cu.tolist(), P, T)
            assert meta[0].tolist() == ns, (P, lens)
            assert meta[1].tolist() == first, (P, lens)
            assert meta[2].tolist() == rows, (P, lens)
            assert meta[3].tolist() == offs


def _random_cu(rng, P, n_docs, max_units, divisible):
    unit = 2 * P if divisible else 1
    lens = rng.integers(0, max_units + 1, size=n_docs) * unit
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
def test_map_invariants_random(oracle_lib, P):
    o = oracle_lib
    rng = np.random.default_rng(77 + P)
    for _ in range(20):
        cu = _random_cu(rng, P, int(rng.integers(1, 12)), 60, True)
        T = int(cu[-1])
        l2g, g2l = o.index_map(o.LAYOUT_DSC, P, cu, T)
        # bijection on [0, T) and inverse round trip
        assert np.array_equal(np.sort(l2g), np.arange(T))
        assert np.array_equal(g2l[l2g], np.arange(T))
        assert np.array_equal(l2g[g2l], np.arange(T))
        Tp = T // P
        for r in range(P):
            mine = l2g[r * Tp:(r + 1) * Tp]
            for i in range(len(cu) - 1):
                L = int(cu[i + 1] - cu[i])
                if L == 0:
                    continue
                m = L // (2 * P)
                in_doc = mine[(mine >= cu[i]) & (mine < cu[i + 1])]
                chunks = sorted(set(((in_doc - cu[i]) // m).tolist()))
                # owner r holds exactly chunks r and 2P-1-r of every document
                assert chunks == sorted({r, 2 * P - 1 - r})
                # load balance: its two chunk ids sum to 2P-1
                assert sum(chunks) == 2 * P - 1 or P == 0
                # chunk r lies before chunk 2P-1-r in local order
                assert np.all(np.diff(in_doc) > 0)
        if P == 1:
            assert np.array_equal(l2g, np.arange(T))
        if T % P == 0:
            pl2g, pg2l = o.index_map(o.LAYOUT_PACKED, P, cu, T)
            assert np.array_equal(pl2g, np.arange(T)) and np.array_equal(pg2l, np.arange(T))


@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_metadata_invariants_random(oracle_lib, P):
    o = oracle_lib
    rng = np.random.default_rng(99 + P)
    for _ in range(20):
        n = int(rng.integers(1, 15))
        cu = _random_cu(rng, P, n, 50, False)
        T = int(cu[-1])
        T -= T % P
        if T == 0:
            continue
        cu = np.minimum(cu, T)
        ns, first, cul, offs = o.thd_metadata(o.LAYOUT_PACKED, P, cu, T)
        Tp = T // P
        assert offs[0] == 0 and np.array_equal(np.diff(offs), ns)
        piece = np.zeros(n, np.int64)
        total = 0
        for r in range(P):
            k = ns[r]
            assert cul[r][k] == Tp and np.all(cul[r][k:] == Tp)
            assert cul[r][0] == 0 and np.all(np.diff(cul[r][:k + 1]) > 0)
            seg_lens = np.diff(cul[r][:k + 1])
            total += seg_lens.sum()
            docs = [bf.doc_of_token(cu.tolist(), r * Tp + int(cul[r][s])) for s in range(k)]
            assert (docs[0] if k else -1) == first[r]
            assert docs == sorted(set(docs))  # document order, one piece each
            for s in range(k):
                piece[docs[s]] += seg_lens[s]
        assert total == T
        # each document's pieces over the ranks add back to its length
        assert np.array_equal(piece, np.diff(cu))


def test_layout_preconditions(oracle_lib):
    o = oracle_lib
    assert o.check_layout(o.LAYOUT_DSC, 2, [0, 16, 40, 64], 64) == 0
    assert o.check_layout(o.LAYOUT_DSC, 2, [0, 18, 40, 64], 64) == 2  # 18 % 4
    assert o.check_layout(o.LAYOUT_PACKED, 2, [0, 18, 40, 64], 64) == 0
    assert o.check_layout(o.LAYOUT_PACKED, 3, [0, 18, 40, 64], 64) == 2  # 64 % 3
    assert o.check_layout(o.LAYOUT_DSC, 2, [0, 40, 16, 64], 64) == 1  # decreasing
    assert o.check_layout(o.LAYOUT_DSC, 2, [1, 16, 40, 64], 64) == 1  # not from 0
    assert o.check_layout(o.LAYOUT_DSC, 2, [0, 16, 40, 64], 65) == 1  # wrong end
    assert o.check_layout(o.LAYOUT_DSC, 0, [0, 16], 16) == 1
    with pytest.raises(o.OracleError):
        o.index_map(o.LAYOUT_DSC, 2, [0, 18, 40, 64], 64)


# ---------------------------------------------------------------- partition


@pytest.mark.parametrize("layout", [0, 1])
def test_partition_row_ids(oracle_lib, layout):
    o = oracle_lib
    P, cu = 4, [0, 8, 8, 48, 96]
    T = 96
    l2g, _ = o.index_map(layout, P, cu, T)
    # each row carries its global row id in every 16-bit word
    src = np.repeat(np.arange(T, dtype=np.uint16)[:, None], 24, axis=1).reshape(T, 3, 8)
    dst = o.partition(l2g, src)
    want = bf.l2g_by_ownership(layout, cu, P, T)
    assert np.array_equal(dst[:, 0, 0], np.array(want, np.uint16))
    assert np.all(dst == dst[:, :1, :1])
    scat = o.grad_scatter(l2g, src, P)
    for r in range(P):
        assert np.array_equal(scat[r][:, 0, 0], np.array(want[r * T // P:(r + 1) * T // P], np.uint16))


@pytest.mark.parametrize("layout,P,cu", [(0, 4, [0, 8, 8, 48, 96]), (1, 3, [0, 5, 50, 51, 96]),
                                          (0, 1, [0, 10, 12])])
def test_restore_inverts_partition(oracle_lib, layout, P, cu):
    o = oracle_lib
    T = cu[-1]
    l2g, _ = o.index_map(layout, P, cu, T)
    rng = np.random.default_rng(2)
    x = rng.integers(0, 2**16, size=(T, 2, 8), dtype=np.uint16)
    local = o.partition(l2g, x)
    assert np.array_equal(o.restore(l2g, local), x)
    # row ids: global row g of the restored buffer comes from local row g2l[g]
    ids = np.repeat(np.arange(T, dtype=np.uint16)[:, None], 8, axis=1)
    want_map = bf.l2g_by_ownership(layout, cu, P, T)
    back = o.restore(l2g, ids)
    for q, g in enumerate(want_map):
        assert back[g, 0] == q


# ---------------------------------------------------------------- bf16


def test_rne_canaries(oracle_lib):
    o = oracle_lib
    rows = []
    with open(os.path.join(GOLDEN, "bf16_rne_canaries.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                a, b = line.split()[:2]
                rows.append((int(a, 16), int(b, 16)))
    bits = np.array([a for a, _ in rows], np.uint32)
    got = o.f32_to_bf16_array(bits.view(np.float32))
    assert [hex(v) for v in got.tolist()] == [hex(b) for _, b in rows]
    for a, b in rows:
        assert o.f32_to_bf16(np.uint32(a).view(np.float32)) == b


def test_rne_matches_torch_cpu(oracle_lib):
    o = oracle_lib
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    exp = (bits >> 23) & 0xFF
    bits = bits[exp != 0xFF]  # finite only (NaN is outside the contract)
    # plus every tie pattern in a few binades
    ties = (np.arange(0, 1 << 12, dtype=np.uint32) << 16) | 0x8000
    bits = np.concatenate([bits, ties[((ties >> 23) & 0xFF) != 0xFF]])
    x = bits.view(np.float32)
    got = o.f32_to_bf16_array(x)
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    # widening is exact: bf16 bits shifted into the top half
    h = rng.integers(0, 2**16, size=5000).astype(np.uint16)
    h = h[((h >> 7) & 0xFF) != 0xFF]
    wide = torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    assert all(o.bf16_to_f32(int(v)) == w for v, w in zip(h[:500], wide[:500]))


# ---------------------------------------------------------------- sums


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_all_ones_give_P(oracle_lib, P, dt):
    o = oracle_lib
    one = np.ones((5, 16), np.float32)
    slots = [one if dt == "f32" else o.f32_to_bf16_array(one) for _ in range(P)]
    out32 = o.slot_reduce(slots, o.F32)
    assert np.all(out32 == P)
    out16 = o.slot_reduce(slots, o.BF16)
    assert np.all(out16 == o.f32_to_bf16(float(P)))


def test_integer_sums_exact(oracle_lib):
    o = oracle_lib
    rng = np.random.default_rng(3)
    for P in (2, 3, 5, 8):
        ints = rng.integers(-100, 101, size=(P, 1000))
        slots = [ints[w].astype(np.float32) for w in range(P)]
        out = o.slot_reduce(slots, o.F32)
        assert np.array_equal(out.astype(np.int64), ints.sum(axis=0))
        # |sum| <= 800 < 256 does not hold, so compare bf16 on small values only
        small = rng.integers(-30, 31, size=(P, 1000))
        sb = [o.f32_to_bf16_array(small[w].astype(np.float32)) for w in range(P)]
        ob = o.slot_reduce(sb, o.F32)
        assert np.array_equal(ob.astype(np.int64), small.sum(axis=0))


def test_order_canary(oracle_lib):
    o = oracle_lib
    big = np.float32(2.0**24)
    a = [np.array([v], np.float32) for v in (big, 1.0, -big, 1.0)]
    b = [np.array([v], np.float32) for v in (1.0, 1.0, big, -big)]
    # ((2^24 + 1) + -2^24) + 1: 2^24 + 1 ties to 2^24, so the ordered sum is 1
    assert o.slot_reduce(a, o.F32)[0] == 1.0
    assert o.slot_reduce(b, o.F32)[0] == 2.0
    ab = [o.f32_to_bf16_array(s) for s in a]
    assert o.slot_reduce(ab, o.F32)[0] == 1.0


def test_negative_zero_survives(oracle_lib):
    o = oracle_lib
    nz = np.full(4, -0.0, np.float32)
    out = o.slot_reduce([nz, nz, nz], o.F32)
    assert np.all(out.view(np.uint32) == 0x80000000)
    out16 = o.slot_reduce([nz, nz], o.BF16)
    assert np.all(out16 == 0x8000)
    mixed = o.slot_reduce([nz, np.zeros(4, np.float32)], o.F32)
    assert np.all(mixed.view(np.uint32) == 0)  # -0 + +0 = +0 under round-to-nearest


def test_single_slot_roundtrip(oracle_lib):
    o = oracle_lib
    rng = np.random.default_rng(8)
    x = o.f32_to_bf16_array(rng.standard_normal(4096).astype(np.float32))
    assert np.array_equal(o.slot_reduce([x], o.BF16), x)
    y = rng.standard_normal(4096).astype(np.float32)
    assert np.array_equal(o.slot_reduce([y], o.F32).view(np.uint32), y.view(np.uint32))


def _numpy_ordered_sum(slots_f32):
    acc = slots_f32[0].astype(np.float32).copy()
    for s in slots_f32[1:]:
        acc = np.add(acc, s.astype(np.float32), dtype=np.float32)
    return acc


def _bf16_to_f32_np(h):
    return (h.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("P", [2, 4, 8])
def test_random_sums_match_numpy_binary32(oracle_lib, P):
    o = oracle_lib
    rng = np.random.default_rng(11 + P)
    s32 = [rng.standard_normal(20000).astype(np.float32) * np.float32(0.02) for _ in range(P)]
    assert np.array_equal(o.slot_reduce(s32, o.F32).view(np.uint32),
                          _numpy_ordered_sum(s32).view(np.uint32))
    s16 = [o.f32_to_bf16_array(s) for s in s32]
    ref = _numpy_ordered_sum([_bf16_to_f32_np(s) for s in s16])
    want16 = torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(o.slot_reduce(s16, o.BF16), want16)


@pytest.mark.parametrize("layout,P,cu", [
    (0, 2, [0, 16, 40, 64]),
    (1, 2, [0, 16, 40, 64]),
    (0, 4, [0, 32, 32, 96]),
    (1, 3, [0, 5, 50, 51, 96]),
    (0, 1, [0, 10, 12]),
])
@pytest.mark.parametrize("din,dout", [("f32", 0), ("bf16", 1), ("bf16", 0), ("f32", 1)])
def test_grad_return_matches_numpy(oracle_lib, layout, P, cu, din, dout):
    o = oracle_lib
    T = cu[-1]
    rng = np.random.default_rng(1)
    w32 = [rng.uniform(-1, 1, size=(T, 2, 8)).astype(np.float32) for _ in range(P)]
    writers = w32 if din == "f32" else [o.f32_to_bf16_array(w) for w in w32]
    l2g, _ = o.index_map(layout, P, cu, T)
    owners = o.grad_return(l2g, writers, dout)
    want_map = np.array(bf.l2g_by_ownership(layout, cu, P, T), np.int64)
    wf = [w if din == "f32" else _bf16_to_f32_np(w) for w in writers]
    Tp = T // P
    for r in range(P):
        rows = want_map[r * Tp:(r + 1) * Tp]
        ref = _numpy_ordered_sum([w[rows] for w in wf])
        if dout == 0:
            assert np.array_equal(owners[r].view(np.uint32), ref.view(np.uint32))
        else:
            want = torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(owners[r], want)


@pytest.mark.parametrize("din,dout", [("f32", 0), ("bf16", 1), ("bf16", 0)])
def test_grad_return_accumulate_matches_numpy(oracle_lib, din, dout):
    o = oracle_lib
    P, cu = 4, [0, 32, 32, 96]
    T = cu[-1]
    rng = np.random.default_rng(9)
    w32 = [rng.uniform(-1, 1, size=(T, 16)).astype(np.float32) for _ in range(P)]
    writers = w32 if din == "f32" else [o.f32_to_bf16_array(w) for w in w32]
    start32 = [rng.uniform(-4, 4, size=(T // P, 16)).astype(np.float32) for _ in range(P)]
    start = start32 if dout == 0 else [o.f32_to_bf16_array(x) for x in start32]
    l2g, _ = o.index_map(0, P, cu, T)
    got = o.grad_return_accumulate(l2g, writers, start)
    want_map = np.array(bf.l2g_by_ownership(0, cu, P, T), np.int64)
    wf = [w if din == "f32" else _bf16_to_f32_np(w) for w in writers]
    for r in range(P):
        rows = want_map[r * (T // P):(r + 1) * (T // P)]
        s0 = start[r] if dout == 0 else _bf16_to_f32_np(start[r])
        ref = _numpy_ordered_sum([s0] + [w[rows] for w in wf])
        if dout == 0:
            assert np.array_equal(got[r].view(np.uint32), ref.view(np.uint32))
        else:
            want = torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(got[r], want)
        # the inputs are not modified
        assert np.array_equal(start[r], start32[r] if dout == 0 else o.f32_to_bf16_array(start32[r]))


def test_grad_return_accumulate_closed_forms(oracle_lib):
    o = oracle_lib
    P, cu = 3, [0, 12]
    l2g, _ = o.index_map(0, P, cu, 12)
    ones = [np.ones((12, 4), np.float32) for _ in range(P)]
    out = o.grad_return_accumulate(l2g, ones, [np.ones((4, 4), np.float32) for _ in range(P)])
    assert all(np.all(x == P + 1) for x in out)
    # order canary: start 2^24, writers (1, -2^24, 1): ((2^24+1)-2^24)+1 = 1,
    # while adding the start last would give 2
    big = np.float32(2.0**24)
    ws = [np.full((12, 4), v, np.float32) for v in (1.0, -big, 1.0)]
    out = o.grad_return_accumulate(l2g, ws, [np.full((4, 4), big, np.float32) for _ in range(P)])
    assert all(np.all(x == 1.0) for x in out)


# ---------------------------------------------------------------- padded layout


def _real_len_closed_form(P, lens):
    """Real tokens of each document on each rank: the rank's chunks r and
    2P-1-r of the padded document, each clipped to the real length."""
    out = np.zeros((P, len(lens)), np.int64)
    for i, L in enumerate(lens):
        Lp = -(-L // (2 * P)) * (2 * P)
        mp = Lp // (2 * P)
        for r in range(P):
            for k in (r, 2 * P - 1 - r):
                out[r, i] += min(max(L - k * mp, 0), mp)
    return out


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
def test_padded_layout_pins(oracle_lib, P):
    o = oracle_lib
    rng = np.random.default_rng(50 + P)
    for _ in range(15):
        lens = rng.integers(0, 40, size=int(rng.integers(1, 7))).tolist()
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        T = int(cu[-1])
        cup = o.pad_cu(P, cu)
        Lp = np.diff(cup)
        assert np.all(Lp % (2 * P) == 0) and np.all(Lp >= np.diff(cu)) and np.all(Lp - np.diff(cu) < 2 * P)
        # row ids + 1 as payload: zero marks padding
        ids = (np.arange(T, dtype=np.uint16) + 1)[:, None].repeat(4, axis=1)
        local = o.partition_padded(P, cu, ids)
        assert local.shape[0] == int(cup[-1])
        nz = local[:, 0][local[:, 0] != 0]
        assert sorted(nz.tolist()) == list(range(1, T + 1))          # each raw row exactly once
        assert np.all(local[local[:, 0] == 0] == 0)                    # padding rows all zero
        assert np.array_equal(o.restore_padded(P, cu, local), ids)     # un-pad inverts
        rl = o.real_lengths(0, P, cu, padded=True)
        assert np.array_equal(rl, _real_len_closed_form(P, lens))
        assert np.array_equal(rl.sum(axis=0), np.diff(cu))
        Tp = int(cup[-1]) // P
        for r in range(P):
            assert rl[r].sum() == np.count_nonzero(local[r * Tp:(r + 1) * Tp, 0])


def test_padded_layout_reduces_to_plain_when_divisible(oracle_lib):
    o = oracle_lib
    P, cu = 4, [0, 16, 16, 48, 96]
    assert np.array_equal(o.pad_cu(P, cu), np.array(cu, np.int32))
    rng = np.random.default_rng(4)
    x = rng.integers(0, 2**16, size=(96, 8), dtype=np.uint16)
    l2g, _ = o.index_map(0, P, cu, 96)
    assert np.array_equal(o.partition_padded(P, cu, x), o.partition(l2g, x))
    assert np.array_equal(o.real_lengths(0, P, cu, padded=True), o.real_lengths(0, P, cu))
    assert np.array_equal(o.real_lengths(0, P, cu), np.tile(np.diff(cu) // P, (P, 1)))

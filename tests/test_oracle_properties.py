"""Property-based pins (hypothesis): generated document mixes, shrunk to a
minimal counterexample on failure.

  * the oracle's maps and metadata equal the brute-force restatements for
    every layout, the padded one included;
  * the library's host-side validation agrees with the oracle's precondition
    check on arbitrary, often malformed, inputs.
Skipped where hypothesis is not installed.
"""
import numpy as np
import pytest

import bruteforce as bf

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402


@st.composite
def dsc_batches(draw):
    P = draw(st.integers(1, 6))
    units = draw(st.lists(st.integers(0, 4), min_size=1, max_size=5))
    return P, [u * 2 * P for u in units]


@st.composite
def packed_batches(draw):
    P = draw(st.integers(1, 6))
    lens = draw(st.lists(st.integers(0, 12), min_size=1, max_size=5))
    lens[-1] += (-sum(lens)) % P
    return P, lens


@st.composite
def raw_batches(draw):
    P = draw(st.integers(1, 5))
    lens = draw(st.lists(st.integers(0, 15), min_size=1, max_size=4))
    return P, lens


def _cu(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


@settings(max_examples=150, deadline=None)
@given(dsc_batches())
def test_dsc_oracle_equals_bruteforce(oracle_lib, batch):
    P, lens = batch
    cu = _cu(lens)
    T = int(cu[-1])
    l2g, g2l = oracle_lib.index_map(0, P, cu, T)
    assert l2g.tolist() == bf.l2g_by_ownership(0, cu.tolist(), P, T)
    assert np.array_equal(g2l[l2g], np.arange(T))
    got = oracle_lib.thd_metadata(0, P, cu, T)
    want = bf.metadata_by_runs(0, cu.tolist(), P, T)
    assert [x.tolist() for x in got] == [want[0], want[1], want[2], want[3]]


@settings(max_examples=150, deadline=None)
@given(packed_batches())
def test_packed_oracle_equals_bruteforce(oracle_lib, batch):
    P, lens = batch
    cu = _cu(lens)
    T = int(cu[-1])
    l2g, _ = oracle_lib.index_map(1, P, cu, T)
    assert l2g.tolist() == list(range(T))
    got = oracle_lib.thd_metadata(1, P, cu, T)
    want = bf.metadata_by_runs(1, cu.tolist(), P, T)
    assert [x.tolist() for x in got] == [want[0], want[1], want[2], want[3]]
    rl = oracle_lib.real_lengths(1, P, cu)
    assert np.array_equal(rl.sum(axis=0), np.diff(cu))


@settings(max_examples=150, deadline=None)
@given(raw_batches())
def test_padded_oracle_properties(oracle_lib, batch):
    P, lens = batch
    cu = _cu(lens)
    T = int(cu[-1])
    cup = oracle_lib.pad_cu(P, cu)
    # padding: smallest multiple of 2P at or above each length
    assert all(int(b) == -(-L // (2 * P)) * (2 * P) for b, L in zip(np.diff(cup), lens))
    ids = (np.arange(T, dtype=np.uint16) + 1)[:, None]
    local = oracle_lib.partition_padded(P, cu, ids)
    assert sorted(local[local[:, 0] != 0, 0].tolist()) == list(range(1, T + 1))
    assert np.array_equal(oracle_lib.restore_padded(P, cu, local), ids)
    # every real token sits on the rank the brute-force owner rule of the
    # padded buffer names
    _, l2g, _ = oracle_lib.padded_index_map(P, cu)
    Tp = int(cup[-1]) // P
    for q in range(int(cup[-1])):
        if local[q, 0]:
            assert bf.owner_dsc(cup.tolist(), P, int(l2g[q])) == q // Tp


@settings(max_examples=300, deadline=None)
@given(st.integers(0, 2), st.integers(0, 9), st.lists(st.integers(-3, 20), min_size=1, max_size=6),
       st.integers(-2, 2))
def test_host_validation_agrees_with_oracle(cpt, oracle_lib, layout, P, steps, t_off):
    cu = np.concatenate([[0], np.cumsum(steps)]).astype(np.int32)
    T = int(cu[-1]) + t_off
    lay = 0 if layout == 0 else 1
    got = cpt.cpt_validate_layout(lay, P, cu, T)
    if T < 0:
        assert got == cpt.CPT_ERR_INVALID_ARG
        return
    want = oracle_lib.check_layout(lay, P, cu, T) if P >= 1 else 1
    code = {0: cpt.CPT_OK, 1: cpt.CPT_ERR_INVALID_ARG, 2: cpt.CPT_ERR_NOT_DIVISIBLE}[want]
    if P > 8 and want != 1:
        code = cpt.CPT_ERR_INVALID_ARG  # the library caps cp_size at 8
    assert got == code, (lay, P, cu.tolist(), T, cpt.cpt_last_error_string())


@settings(max_examples=200, deadline=None)
@given(raw_batches())
def test_layout_padded_tokens_equals_oracle_pad_cu(cpt, oracle_lib, batch):
    P, lens = batch
    cu = _cu(lens)
    T = int(cu[-1])
    got = cpt.cpt_layout_padded_tokens(cpt.CPT_LAYOUT_DUAL_CHUNK_SWAP_PADDED, P, cu, T)
    assert got == int(oracle_lib.pad_cu(P, cu)[-1])

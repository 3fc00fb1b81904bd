"""Host-side checks of the C ABI that need no GPU.

The library must build, load, and export every function include/cpt.h
declares; the host-only calls (layout validation, workspace sizing) must
agree with the oracle's precondition check on random and edge inputs.
"""
import os

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cpt.h")


def test_library_exports_every_declared_function(cpt):
    declared = cpt.declared_functions(HEADER)
    assert len(declared) >= 18
    missing = sorted(set(declared) - set(cpt.exported_symbols(declared)))
    assert not missing, f"declared but not exported: {missing}"


def test_binding_names_match_header(cpt):
    for name in cpt.declared_functions(HEADER):
        assert hasattr(cpt, name), f"binding lacks {name}"


def test_library_has_no_libcuda_dependency(cpt):
    # the driver API is reached through the runtime's entry-point query
    with open(cpt.library_path(), "rb") as f:
        data = f.read()
    import re

    needed = re.findall(rb"libcuda\.so[.0-9]*", data)
    # the static runtime names libcuda.so.1 as a string it dlopens at run time,
    # but the ELF dynamic section must not list it as NEEDED
    import subprocess

    out = subprocess.run(["readelf", "-d", cpt.library_path()], capture_output=True, text=True)
    if out.returncode == 0:
        assert "libcuda" not in "\n".join(l for l in out.stdout.splitlines() if "NEEDED" in l)
    else:  # no readelf: fall back to the loose check
        assert needed is not None


def test_status_strings(cpt):
    assert cpt.cpt_status_string(0) == "CPT_OK"
    assert cpt.cpt_status_string(7) == "CPT_ERR_TIMEOUT"
    assert cpt.cpt_status_string(10) == "CPT_ERR_NOT_PUBLISHED"


@pytest.mark.parametrize("layout", [0, 1])
def test_validate_layout_agrees_with_oracle(cpt, oracle_lib, layout):
    rng = np.random.default_rng(21 + layout)
    for _ in range(400):
        P = int(rng.integers(1, 9))
        n = int(rng.integers(0, 7))
        lens = rng.integers(0, 5, size=n) * int(rng.choice([1, 2 * P]))
        if rng.random() < 0.3:
            lens = lens + rng.integers(0, 3, size=n)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        T = int(cu[-1])
        if rng.random() < 0.1:
            T += 1  # wrong end
        if n > 1 and rng.random() < 0.1:
            cu[1], cu[2] = cu[2] + 1, cu[1]  # decreasing
        got = cpt.cpt_validate_layout(layout, P, cu, T)
        want = oracle_lib.check_layout(layout, P, cu, T)
        code = {0: cpt.CPT_OK, 1: cpt.CPT_ERR_INVALID_ARG, 2: cpt.CPT_ERR_NOT_DIVISIBLE}[want]
        assert got == code, (layout, P, cu.tolist(), T, cpt.cpt_last_error_string())


def test_validate_layout_rejects_bad_arguments(cpt):
    assert cpt.cpt_validate_layout(0, 0, [0, 8], 8) == cpt.CPT_ERR_INVALID_ARG
    assert cpt.cpt_validate_layout(0, 9, [0, 18], 18) == cpt.CPT_ERR_INVALID_ARG
    assert cpt.cpt_validate_layout(7, 2, [0, 8], 8) == cpt.CPT_ERR_INVALID_ARG
    assert cpt.cpt_validate_layout(0, 2, [0, 6], 6) == cpt.CPT_ERR_NOT_DIVISIBLE
    assert "not a multiple" in cpt.cpt_last_error_string()
    assert cpt.cpt_validate_layout(1, 4, [0, 6], 6) == cpt.CPT_ERR_NOT_DIVISIBLE
    assert cpt.cpt_validate_layout(0, 1, [0], 0) == cpt.CPT_OK  # empty batch
    assert cpt.cpt_validate_layout(1, 8, [0, 0, 0], 0) == cpt.CPT_OK


def test_workspace_bytes(cpt):
    a = cpt.cpt_plan_workspace_bytes(0, 4, 1, 262144)
    assert a >= 2 * 4 * 262144
    assert a % 256 == 0
    assert cpt.cpt_plan_workspace_bytes(0, 4, 100, 262144) > a
    assert cpt.cpt_plan_workspace_bytes(0, 9, 1, 64) == 0
    assert cpt.cpt_plan_workspace_bytes(0, 2, 1, 1 << 31) == 0


def test_retired_packed_super_sequence_selector_is_rejected(cpt):
    """The mirrored packed_super_sequence policy was retired; its selector
    must fail closed, on the host, with a message that says so."""
    code = cpt.CPT_LAYOUT_RETIRED_PACKED_SUPER_SEQUENCE
    assert cpt.cpt_validate_layout(code, 4, [0, 64], 64) == cpt.CPT_ERR_UNSUPPORTED
    assert "retired" in cpt.cpt_last_error_string()
    assert cpt.cpt_plan_workspace_bytes(code, 4, 1, 64) == 0
    assert cpt.cpt_validate_layout(7, 4, [0, 64], 64) == cpt.CPT_ERR_INVALID_ARG


def test_mirrored_map_is_dsc_over_one_sequence(oracle_lib):
    """2P mirrored chunks over the whole buffer = a per-document plan over
    cu_seqlens [0, T]: rank r holds chunks r and 2P-1-r of the buffer."""
    import numpy as np

    o = oracle_lib
    for P in (2, 4, 8):
        T = 2 * P * 7
        l2g, _ = o.index_map(o.LAYOUT_DSC, P, [0, T], T)
        m = T // (2 * P)
        for r in range(P):
            want = list(range(r * m, (r + 1) * m)) + list(range((2 * P - 1 - r) * m, (2 * P - r) * m))
            assert l2g[r * 2 * m:(r + 1) * 2 * m].tolist() == want
        assert np.array_equal(np.sort(l2g), np.arange(T))


def test_padded_layout_validation(cpt):
    """The padded per-document layout takes documents of any length."""
    PAD = cpt.CPT_LAYOUT_DUAL_CHUNK_SWAP_PADDED
    assert cpt.cpt_validate_layout(PAD, 4, [0, 5, 5, 12], 12) == cpt.CPT_OK
    assert cpt.cpt_validate_layout(0, 4, [0, 5, 5, 12], 12) == cpt.CPT_ERR_NOT_DIVISIBLE
    assert cpt.cpt_validate_layout(PAD, 4, [0, 5, 3], 3) == cpt.CPT_ERR_INVALID_ARG
    # workspace sized for the largest padding: n * (2P - 1) extra tokens
    assert cpt.cpt_plan_workspace_bytes(PAD, 4, 3, 12) >= cpt.cpt_plan_workspace_bytes(0, 4, 3, 12)
    big = 2**31 - 8
    assert cpt.cpt_validate_layout(PAD, 8, [0, 1, big], big) == cpt.CPT_ERR_INVALID_ARG


def test_binding_constants_match_header(cpt):
    """Every enumerator and #define of include/cpt.h has the same value in the binding."""
    import re

    with open(HEADER) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    consts = {}
    for body in re.findall(r"typedef enum \w+ \{(.*?)\}", text, flags=re.S):
        nxt = 0
        for item in body.split(","):
            item = item.strip()
            if not item:
                continue
            if "=" in item:
                name, val = (x.strip() for x in item.split("="))
                nxt = int(val, 0)
            else:
                name = item
            consts[name] = nxt
            nxt += 1
    for name, val in re.findall(r"#define (CPT_[A-Z0-9_]+) (\d+)", text):
        consts[name] = int(val)
    assert len(consts) >= 20
    for name, val in consts.items():
        assert getattr(cpt, name) == val, name


def test_kernel_path_choice_validated(cpt):
    """The kernel choice takes the three enumerators and refuses anything else."""
    for bad in (-1, 3, 99):
        with pytest.raises(cpt.CptError):
            cpt.cpt_set_kernel_path(bad)
    for k in (cpt.CPT_KERNEL_LOADS, cpt.CPT_KERNEL_BULK, cpt.CPT_KERNEL_AUTO):
        cpt.cpt_set_kernel_path(k)


def test_layout_padded_tokens_agrees_with_oracle(cpt, oracle_lib):
    """The host-only padded-size query equals the last boundary of the
    oracle's padded cu_seqlens, and the raw total for the other layouts."""
    PAD = cpt.CPT_LAYOUT_DUAL_CHUNK_SWAP_PADDED
    rng = np.random.default_rng(77)
    for _ in range(300):
        P = int(rng.integers(1, 9))
        n = int(rng.integers(0, 9))
        lens = rng.integers(0, 40, size=n)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        T = int(cu[-1])
        assert cpt.cpt_layout_padded_tokens(PAD, P, cu, T) == int(oracle_lib.pad_cu(P, cu)[-1])
        if T % P == 0:
            assert cpt.cpt_layout_padded_tokens(cpt.CPT_LAYOUT_PACKED_CONTIGUOUS, P, cu, T) == T
    assert cpt.cpt_layout_padded_tokens(0, 4, [0, 64, 128], 128) == 128
    assert cpt.cpt_layout_padded_tokens(PAD, 4, [0, 1, 1, 10], 10) == 8 + 0 + 16
    with pytest.raises(cpt.CptError) as ei:
        cpt.cpt_layout_padded_tokens(0, 4, [0, 6], 6)
    assert ei.value.status == cpt.CPT_ERR_NOT_DIVISIBLE
    with pytest.raises(cpt.CptError) as ei:
        cpt.cpt_layout_padded_tokens(PAD, 8, [0, 1, 2**31 - 8], 2**31 - 8)
    assert ei.value.status == cpt.CPT_ERR_INVALID_ARG


def test_both_builds_export_every_declared_function(cpt):
    """The release and the bounds-checked library export the same calls and
    say which build they are."""
    import ctypes

    from context_attention_token_gb300 import build as cpt_build

    declared = cpt.declared_functions(HEADER)
    for variant, flag in (("release", 0), ("checked", 1)):
        lib = ctypes.CDLL(cpt_build.library_path(variant))
        missing = [n for n in declared if not hasattr(lib, n)]
        assert not missing, (variant, missing)
        lib.cpt_bounds_checked.restype = ctypes.c_int32
        assert lib.cpt_bounds_checked() == flag, variant
    if not cpt.cpt_bounds_checked():
        with pytest.raises(cpt.CptError) as ei:
            cpt.cpt_bounds_violations()
        assert ei.value.status == cpt.CPT_ERR_UNSUPPORTED

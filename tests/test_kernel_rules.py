"""The measured kernel rules, as include/cpt.h documents them, checked on the
host through cpt_kernel_path_of (the launchers decide with the same
functions). Each case is a configuration the rules were measured on or an
edge the documentation names."""
import pytest

GATHER, GR, SLOT = 0, 1, 2
F32, BF16 = 0, 1


@pytest.fixture
def path(cpt):
    cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_AUTO)
    yield lambda *a: "bulk" if cpt.cpt_kernel_path_of(*a) == cpt.CPT_KERNEL_BULK else "loads"
    cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_AUTO)


def test_gradient_return_rule(path):
    # the pages' shape: 2 x 262144 owner rows of 5 KB, 13.4 GB per launch
    assert path(GR, 4, BF16, BF16, False, 5120, 2 * 262144) == "bulk"
    # the single-document configuration: 0.67 GB per launch, under 2 GiB at P=4
    assert path(GR, 4, BF16, BF16, False, 2048, 2 * 32768) == "loads"
    # the lognormal configuration: 5.4 GB of 4 KB rows
    assert path(GR, 4, BF16, BF16, False, 4096, 2 * 131072) == "bulk"
    # P <= 2 never; P >= 7 with any launch size
    assert path(GR, 2, BF16, BF16, False, 5120, 2 * 262144) == "loads"
    assert path(GR, 1, F32, F32, False, 8192, 1 << 22) == "loads"
    assert path(GR, 8, BF16, BF16, False, 5120, 2 * 1024) == "bulk"
    # P = 4: bf16 rows from 2 KB, float32 rows up to 2 KB
    assert path(GR, 4, BF16, BF16, False, 1024, 1 << 22) == "loads"
    assert path(GR, 4, F32, F32, False, 2048, 1 << 22) == "bulk"
    assert path(GR, 4, F32, F32, False, 4096, 1 << 22) == "loads"
    # P = 3: bf16 rows from 3 KB only
    assert path(GR, 3, BF16, BF16, False, 3072, 1 << 22) == "bulk"
    assert path(GR, 3, BF16, BF16, False, 2048, 1 << 22) == "loads"
    assert path(GR, 3, F32, F32, False, 4096, 1 << 22) == "loads"
    # shared memory: 2 x (P+1) x row <= 112 KB keeps two CTAs on an SM
    assert path(GR, 8, F32, F32, False, 6368, 1 << 20) == "bulk"
    assert path(GR, 8, F32, F32, False, 6384, 1 << 20) == "loads"
    # mixed types follow the same rule, keyed on the input rows
    assert path(GR, 4, BF16, F32, False, 5120, 2 * 262144) == "bulk"
    assert path(GR, 4, BF16, F32, True, 2048, 2 * 524288) == "bulk"
    assert path(GR, 2, BF16, F32, True, 5120, 2 * 262144) == "loads"
    assert path(GR, 8, BF16, F32, False, 8192, 1 << 20) == "loads"  # 2 x (8 x 8 + 16) KB > 112 KB
    # accumulate mode follows the same rule, its launch counting the owner row
    assert path(GR, 8, BF16, BF16, True, 5120, 1 << 20) == "bulk"
    assert path(GR, 4, BF16, BF16, True, 5120, 2 * 262144) == "bulk"
    assert path(GR, 4, BF16, BF16, True, 2048, 2 * 524288) == "bulk"
    assert path(GR, 4, BF16, BF16, True, 2048, 2 * 32768) == "loads"   # 0.8 GB
    # 2 GiB at P=4 with 5 KB rows: 83887 rows overwrite (5 rows each) is just
    # under it; accumulate (6 rows each) is over it
    assert path(GR, 4, BF16, BF16, False, 5120, 83886) == "loads"
    assert path(GR, 4, BF16, BF16, True, 5120, 83886) == "bulk"


def test_row_gather_rule(path):
    # the pages' partition: 3 x 262144 rows of 5 KB
    assert path(GATHER, 4, BF16, BF16, False, 5120, 3 * 262144) == "bulk"
    # rows of 1 KB lost at every size
    assert path(GATHER, 4, BF16, BF16, False, 1024, 3 * 1 << 22) == "loads"
    # 2 KB rows: 0.2 GB launches lose, 0.8 GB launches win (384 MiB threshold)
    assert path(GATHER, 4, BF16, BF16, False, 2048, 3 * 16384) == "loads"
    assert path(GATHER, 4, BF16, BF16, False, 2048, 3 * 65536) == "bulk"
    # 50 KB rows still fit four one-row stages; 16 bytes more do not
    assert path(GATHER, 4, BF16, BF16, False, 51200, 100000) == "bulk"
    assert path(GATHER, 4, BF16, BF16, False, 51216, 100000) == "loads"


def test_slot_reduce_rule(path):
    assert path(SLOT, 8, BF16, BF16, False, 1 << 30, 0) == "bulk"
    assert path(SLOT, 8, F32, F32, False, 1 << 28, 0) == "loads"
    assert path(SLOT, 8, BF16, F32, False, 1 << 30, 0) == "loads"


def test_forced_paths(cpt, path):
    cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_LOADS)
    assert path(GR, 8, BF16, BF16, False, 5120, 1 << 22) == "loads"
    assert path(GATHER, 4, BF16, BF16, False, 5120, 1 << 22) == "loads"
    assert path(SLOT, 8, BF16, BF16, False, 1 << 30, 0) == "loads"
    cpt.cpt_set_kernel_path(cpt.CPT_KERNEL_BULK)
    # forced bulk runs wherever the bulk kernel can
    assert path(GR, 1, BF16, BF16, False, 16, 10) == "bulk"
    assert path(GATHER, 4, BF16, BF16, False, 16, 10) == "bulk"
    assert path(SLOT, 2, F32, F32, False, 4096, 0) == "bulk"
    # and nowhere else
    assert path(GR, 8, F32, F32, False, 6384, 10) == "loads"
    assert path(GR, 4, BF16, BF16, True, 5120, 10) == "bulk"   # accumulate, when forced
    assert path(GR, 4, BF16, F32, False, 5120, 10) == "bulk"   # mixed types, when forced
    assert path(GR, 4, BF16, F32, True, 5120, 10) == "bulk"
    assert path(GR, 8, BF16, F32, False, 8192, 10) == "loads"  # 2 x (8 x 8 + 16) KB > 112 KB
    assert path(GATHER, 4, BF16, BF16, False, 51216, 10) == "loads"
    assert path(SLOT, 2, F32, F32, False, 4080, 0) == "loads"
    assert path(SLOT, 2, BF16, F32, False, 1 << 30, 0) == "loads"


def test_query_validates_its_arguments(cpt):
    with pytest.raises(cpt.CptError):
        cpt.cpt_kernel_path_of(7, 4, BF16, BF16, False, 5120, 10)
    with pytest.raises(cpt.CptError):
        cpt.cpt_kernel_path_of(GR, 9, BF16, BF16, False, 5120, 10)
    with pytest.raises(cpt.CptError):
        cpt.cpt_kernel_path_of(GR, 4, 5, BF16, False, 5120, 10)
    with pytest.raises(cpt.CptError):
        cpt.cpt_kernel_path_of(GATHER, 4, BF16, BF16, False, -16, 10)

"""The streaming ceiling that the benchmark's roofline divides by
(cpt_stream_ceiling): dst must be a bit copy of the first source whatever
the number of sources, block size, stage count and tail, nothing outside dst
may change, and invalid shapes are refused on the host."""
import pytest
import torch

from gpu_helpers import Guarded

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_src,block,stages,ctas", [
    (1, 32768, 4, 1), (1, 8192, 4, 2), (4, 10240, 4, 1), (4, 5120, 8, 1), (8, 4096, 3, 2), (3, 16, 2, 1),
])
@pytest.mark.parametrize("nbytes", [16, 4096, 10240 * 7 + 48, (1 << 22) + 16])
def test_ceiling_copies_the_first_source(cpt, cuda_device, n_src, block, stages, ctas, nbytes):
    g = torch.Generator(device="cuda")
    g.manual_seed(nbytes + n_src)
    srcs = [torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda", generator=g)
            for _ in range(n_src)]
    keep = [s.clone() for s in srcs]
    dst = Guarded((nbytes,), torch.uint8)
    cpt.cpt_stream_ceiling(srcs, dst.t, block, stages, ctas)
    torch.cuda.synchronize()
    assert torch.equal(dst.t, srcs[0])
    assert dst.bands_intact()
    assert all(torch.equal(a, b) for a, b in zip(srcs, keep))
    assert cpt.cpt_kernel_wait_timeouts() == 0


def test_ceiling_refuses_invalid_shapes(cpt, cuda_device):
    a = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    b = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    for block, stages in ((4096, 1), (4100, 4), (65536, 4), (4096, 9)):
        with pytest.raises(cpt.CptError) as ei:
            cpt.cpt_stream_ceiling([a], b, block, stages, 1)
        assert ei.value.status == cpt.CPT_ERR_INVALID_ARG
    with pytest.raises(cpt.CptError) as ei:
        cpt.cpt_stream_ceiling([a[:4088]], b[:4088], 4096, 4, 1)
    assert ei.value.status == cpt.CPT_ERR_ALIGNMENT
    with pytest.raises(cpt.CptError) as ei:
        cpt.cpt_stream_ceiling([a, b], a, 4096, 4, 1)
    assert ei.value.status == cpt.CPT_ERR_ALIAS

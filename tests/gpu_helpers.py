"""Helpers for the GPU parity tests: host<->device marshalling of raw bf16
bits and guard-banded output buffers."""
import numpy as np
import torch


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    """float32 array or raw-bf16 uint16 array -> device tensor of that type."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    assert a.dtype in (np.float32, np.int32), a.dtype
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return t.detach().cpu().contiguous().numpy()


def bits(a: np.ndarray) -> np.ndarray:
    """Bit view for exact comparison (keeps -0.0 and NaN payloads distinct)."""
    if a.dtype == np.float32:
        return a.view(np.uint32)
    return a


CANARY = 0x5A


class Guarded:
    """A device buffer with canary bands on both sides of the usable region."""

    def __init__(self, shape, dtype, device="cuda", band_bytes=4096):
        elem = torch.tensor([], dtype=dtype).element_size()
        n = int(np.prod(shape)) if len(shape) else 1
        self.band = band_bytes
        self.raw = torch.full((band_bytes * 2 + n * elem,), CANARY, dtype=torch.uint8, device=device)
        self.t = self.raw[band_bytes:band_bytes + n * elem].view(dtype).view(shape)

    def bands_intact(self) -> bool:
        lo = self.raw[: self.band]
        hi = self.raw[self.raw.numel() - self.band:]
        return bool((lo == CANARY).all().item() and (hi == CANARY).all().item())

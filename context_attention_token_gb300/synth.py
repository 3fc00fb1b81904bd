"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the method: it only draws numbers and
document lengths. The same host arrays feed the CPU oracle and, copied to the
device, the CUDA path.

Recipes (workload shapes of the pages: TransformerEngine PRs 3221 and 3235):
  * tiny:     P=2, 3 documents [16, 24, 24] (T=64), H=2, D=8, float32
              uniform[-1, 1].
  * lognormal packed documents: x ~ lognormal(ln 2048, 1.0); raw lengths are
              clip(round(x), 64, 32768); the DualChunkSwap variant rounds to a
              multiple of ``multiple`` first. Documents are appended while the
              running sum stays below T; the last one takes the remainder.
  * bf16 tensors are round-to-nearest-even of float32 draws, converted by
    torch on the CPU (a library routine, shared by neither side's arithmetic).

Seeds: config k uses 1000 + k; tensor t within it uses
``numpy.random.default_rng([1000 + k, t])`` (PCG64).
"""
from __future__ import annotations

import numpy as np
import torch


def rng_for(config: int, tensor: int) -> np.random.Generator:
    return np.random.default_rng([1000 + config, tensor])


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> raw bf16 bits (uint16), round-to-nearest-even by torch."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def uniform_f32(rng: np.random.Generator, shape, lo=-1.0, hi=1.0) -> np.ndarray:
    return rng.uniform(lo, hi, size=shape).astype(np.float32)


def normal_f32(rng: np.random.Generator, shape, sigma=1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if sigma != 1.0:
        x *= np.float32(sigma)
    return x


def normal_bf16(rng: np.random.Generator, shape, sigma=1.0) -> np.ndarray:
    return to_bf16_bits(normal_f32(rng, shape, sigma))


def uniform_bf16(rng: np.random.Generator, shape, lo=-1.0, hi=1.0) -> np.ndarray:
    return to_bf16_bits(uniform_f32(rng, shape, lo, hi))


def lognormal_doc_lengths(total_tokens: int, rng: np.random.Generator, multiple: int = 1,
                          median: float = 2048.0, sigma: float = 1.0,
                          lo: int = 64, hi: int = 32768) -> list[int]:
    """Document lengths summing to ``total_tokens``.

    With ``multiple`` > 1 every length except possibly the last is a multiple
    of it; the last is ``total_tokens - sum`` (a multiple too when
    ``total_tokens`` is).
    """
    lengths: list[int] = []
    s = 0
    while True:
        x = float(rng.lognormal(np.log(median), sigma))
        if multiple > 1:
            L = multiple * int(round(x / multiple))
        else:
            L = int(round(x))
        L = min(max(L, lo), hi)
        if s + L < total_tokens:
            lengths.append(L)
            s += L
        else:
            lengths.append(total_tokens - s)
            return lengths


def cu_from_lengths(lengths) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(lengths, dtype=np.int64))]).astype(np.int32)


def device_normal_bf16(shape, seed: int, sigma: float, device) -> torch.Tensor:
    """Large bf16 N(0, sigma) tensor drawn on the device by torch's seeded RNG.

    Used where a host draw would take minutes (the 10 GB writer gradients);
    sampled rows are copied back to the host for the oracle.
    """
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat_o = out.view(-1)
    n = flat_o.numel()
    step = 1 << 27
    # draw in slices to bound the float32 staging memory
    stage = torch.empty(min(step, max(n, 1)), dtype=torch.float32, device=device)
    for s in range(0, n, step):
        e = min(s + step, n)
        st = stage[: e - s]
        st.normal_(0.0, sigma, generator=g)
        flat_o[s:e].copy_(st)
    del stage
    return out

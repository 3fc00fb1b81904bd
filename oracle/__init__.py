"""CPU oracle for the context-parallel token layout and owner-gradient return.

TEST INFRASTRUCTURE ONLY. The library never imports this package; only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg do.
It shares no code with the CUDA path: the arithmetic lives in ``oracle.c``
(plain loops, binary32 adds in the stated order), and this module only
marshals numpy arrays into it.

Sources, by page title:
  * "[PyTorch] Add experimental packed-contiguous THD all-gather CP"
    (TransformerEngine PR 3221): the two partition policies and the packed
    metadata ("Why", commit messages).
  * "Add stream-ordered CP gradient return primitive" (TransformerEngine
    PR 3235): the owner rule (author's reply on CP-size genericity), the
    scatter / publish / wait / accumulate sequence ("Description", sequence
    diagram).

Parity status: every function is pinned by ``tests/test_oracle_pins.py``,
except the packed metadata *format*, which is a reading of an unspecified
format (its values are pinned, the choice of format is not).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

LAYOUT_DSC = 0
LAYOUT_PACKED = 1
F32 = 0
BF16 = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with IEEE-strict flags.

    -ffp-contract=off keeps every add a separate binary32 rounding; no
    fast-math, so nothing is reassociated and subnormals are kept.
    """
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i32p = ctypes.c_void_p
            lib.oracle_check_layout.argtypes = [ctypes.c_int, ctypes.c_int, i32p, ctypes.c_int, ctypes.c_int64]
            lib.oracle_check_layout.restype = ctypes.c_int
            lib.oracle_index_map.argtypes = [ctypes.c_int, ctypes.c_int, i32p, ctypes.c_int, ctypes.c_int64,
                                             i32p, i32p]
            lib.oracle_index_map.restype = ctypes.c_int
            lib.oracle_thd_metadata.argtypes = [ctypes.c_int, ctypes.c_int, i32p, ctypes.c_int, ctypes.c_int64,
                                                i32p, i32p, i32p, i32p]
            lib.oracle_thd_metadata.restype = ctypes.c_int
            lib.oracle_partition.argtypes = [i32p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
            lib.oracle_partition.restype = None
            lib.oracle_restore.argtypes = [i32p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
            lib.oracle_restore.restype = None
            lib.oracle_pad_cu.argtypes = [ctypes.c_int, i32p, ctypes.c_int, i32p]
            lib.oracle_pad_cu.restype = None
            lib.oracle_partition_padded.argtypes = [i32p, ctypes.c_int64, i32p, i32p, ctypes.c_int,
                                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
            lib.oracle_partition_padded.restype = None
            lib.oracle_restore_padded.argtypes = [i32p, i32p, i32p, ctypes.c_int, ctypes.c_void_p,
                                                  ctypes.c_void_p, ctypes.c_int64]
            lib.oracle_restore_padded.restype = None
            lib.oracle_real_lengths.argtypes = [ctypes.c_int, i32p, ctypes.c_int64, i32p, i32p, ctypes.c_int,
                                                i32p]
            lib.oracle_real_lengths.restype = None
            lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f32.restype = ctypes.c_float
            lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
            lib.oracle_slot_reduce.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_void_p]
            lib.oracle_slot_reduce.restype = None
            lib.oracle_grad_return.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                               ctypes.c_int, i32p, ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_grad_return.restype = None
            lib.oracle_grad_return_accumulate.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                                          ctypes.c_int, ctypes.c_int, i32p, ctypes.c_void_p,
                                                          ctypes.c_void_p]
            lib.oracle_grad_return_accumulate.restype = None
            lib.oracle_grad_scatter.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, i32p,
                                                ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_grad_scatter.restype = None
            _lib = lib
    return _lib


class OracleError(ValueError):
    """The inputs break a layout precondition (malformed or not divisible)."""


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _cu(cu_seqlens) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:  # raw bf16 bits
        return BF16
    raise TypeError(f"oracle takes float32 or raw-bf16 uint16 arrays, got {a.dtype}")


def _np_dtype(code: int):
    return np.float32 if code == F32 else np.uint16


def check_layout(layout: int, cp_size: int, cu_seqlens, total_tokens: int) -> int:
    """0 = valid, 1 = malformed, 2 = a divisibility rule fails."""
    cu = _cu(cu_seqlens)
    return _load().oracle_check_layout(layout, cp_size, _ptr(cu), len(cu) - 1, total_tokens)


def index_map(layout: int, cp_size: int, cu_seqlens, total_tokens: int):
    """Return (l2g, g2l), int32[T] each, local index flattened rank-major."""
    cu = _cu(cu_seqlens)
    T = int(total_tokens)
    l2g = np.empty(T, np.int32)
    g2l = np.empty(T, np.int32)
    rc = _load().oracle_index_map(layout, cp_size, _ptr(cu), len(cu) - 1, T, _ptr(l2g), _ptr(g2l))
    if rc:
        raise OracleError(f"layout precondition failed ({rc})")
    return l2g, g2l


def thd_metadata(layout: int, cp_size: int, cu_seqlens, total_tokens: int):
    """Return (num_segs[P], seg_doc_first[P], cu_local[P][n+1], seg_offsets[P+1])."""
    cu = _cu(cu_seqlens)
    n = len(cu) - 1
    P = cp_size
    num_segs = np.empty(P, np.int32)
    first = np.empty(P, np.int32)
    cu_local = np.empty((P, n + 1), np.int32)
    offs = np.empty(P + 1, np.int32)
    rc = _load().oracle_thd_metadata(layout, P, _ptr(cu), n, int(total_tokens), _ptr(num_segs), _ptr(first),
                                     _ptr(cu_local), _ptr(offs))
    if rc:
        raise OracleError(f"layout precondition failed ({rc})")
    return num_segs, first, cu_local, offs


def partition(l2g: np.ndarray, src: np.ndarray) -> np.ndarray:
    """dst[q] = src[l2g[q]] for a [T, ...] array (any dtype; a byte copy)."""
    src = np.ascontiguousarray(src)
    l2g = np.ascontiguousarray(l2g, dtype=np.int32)
    T = src.shape[0]
    dst = np.empty_like(src)
    row_bytes = src.nbytes // T if T else 0
    _load().oracle_partition(_ptr(l2g), T, _ptr(src), _ptr(dst), row_bytes)
    return dst


def restore(l2g: np.ndarray, local: np.ndarray) -> np.ndarray:
    """global[l2g[q]] = local[q] for a flattened rank-major [T, ...] array."""
    local = np.ascontiguousarray(local)
    l2g = np.ascontiguousarray(l2g, dtype=np.int32)
    T = local.shape[0]
    out = np.empty_like(local)
    row_bytes = local.nbytes // T if T else 0
    _load().oracle_restore(_ptr(l2g), T, _ptr(local), _ptr(out), row_bytes)
    return out


def pad_cu(cp_size: int, cu_seqlens) -> np.ndarray:
    """cu_seqlens with every document padded up to a multiple of 2P."""
    cu = _cu(cu_seqlens)
    out = np.empty_like(cu)
    _load().oracle_pad_cu(cp_size, _ptr(cu), len(cu) - 1, _ptr(out))
    return out


def padded_index_map(cp_size: int, cu_seqlens):
    """(cu_padded, l2g, g2l) of the padded per-document layout (T_pad tokens)."""
    cup = pad_cu(cp_size, cu_seqlens)
    l2g, g2l = index_map(LAYOUT_DSC, cp_size, cup, int(cup[-1]))
    return cup, l2g, g2l


def partition_padded(cp_size: int, cu_seqlens, src: np.ndarray) -> np.ndarray:
    """Rank-local [T_pad, ...] from raw [T, ...], padding rows zero."""
    cu = _cu(cu_seqlens)
    cup, l2g, _ = padded_index_map(cp_size, cu)
    src = np.ascontiguousarray(src)
    Tpad = int(cup[-1])
    dst = np.empty((Tpad,) + src.shape[1:], src.dtype)
    row_bytes = int(np.prod(src.shape[1:], dtype=np.int64)) * src.itemsize
    _load().oracle_partition_padded(_ptr(l2g), Tpad, _ptr(cu), _ptr(cup), len(cu) - 1, _ptr(src),
                                    _ptr(dst), row_bytes)
    return dst


def restore_padded(cp_size: int, cu_seqlens, local: np.ndarray) -> np.ndarray:
    """Raw [T, ...] from the rank-local padded [T_pad, ...] (padding dropped)."""
    cu = _cu(cu_seqlens)
    cup, _, g2l = padded_index_map(cp_size, cu)
    local = np.ascontiguousarray(local)
    T = int(cu[-1])
    out = np.empty((T,) + local.shape[1:], local.dtype)
    row_bytes = int(np.prod(local.shape[1:], dtype=np.int64)) * local.itemsize
    _load().oracle_restore_padded(_ptr(g2l), _ptr(cu), _ptr(cup), len(cu) - 1, _ptr(local), _ptr(out),
                                  row_bytes)
    return out


def real_lengths(layout: int, cp_size: int, cu_seqlens, padded: bool = False) -> np.ndarray:
    """[P][n]: real tokens of document i held by rank r."""
    cu = _cu(cu_seqlens)
    n = len(cu) - 1
    if padded:
        cup, l2g, _ = padded_index_map(cp_size, cu)
    else:
        cup = cu
        l2g, _ = index_map(layout, cp_size, cu, int(cu[-1]))
    out = np.empty((cp_size, n), np.int32)
    _load().oracle_real_lengths(cp_size, _ptr(l2g), int(cup[-1]), _ptr(cu), _ptr(cup), n, _ptr(out))
    return out


def f32_to_bf16(x: float) -> int:
    return int(_load().oracle_f32_to_bf16(float(x)))


def bf16_to_f32(h: int) -> float:
    return float(_load().oracle_bf16_to_f32(int(h)))


def f32_to_bf16_array(x: np.ndarray) -> np.ndarray:
    """Element-wise round-to-nearest-even through the oracle (P=1 slot reduce)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    slots = (ctypes.c_void_p * 1)(_ptr(x))
    _load().oracle_slot_reduce(ctypes.cast(slots, ctypes.c_void_p), 1, x.size, F32, BF16, _ptr(out))
    return out


def slot_reduce(slots, out_dtype: int) -> np.ndarray:
    """Ordered binary32 sum of P equally shaped slot arrays."""
    slots = [np.ascontiguousarray(s) for s in slots]
    P = len(slots)
    in_code = _dtype_code(slots[0])
    for s in slots:
        assert s.shape == slots[0].shape and s.dtype == slots[0].dtype
    out = np.empty(slots[0].shape, _np_dtype(out_dtype))
    arr = (ctypes.c_void_p * P)(*[_ptr(s) for s in slots])
    _load().oracle_slot_reduce(ctypes.cast(arr, ctypes.c_void_p), P, slots[0].size, in_code, out_dtype, _ptr(out))
    return out


def grad_return(l2g: np.ndarray, writers, out_dtype: int):
    """Owner buffers [P][T/P][row...] from P writer arrays [T][row...]."""
    writers = [np.ascontiguousarray(w) for w in writers]
    P = len(writers)
    T = writers[0].shape[0]
    row_elems = writers[0].size // T if T else 0
    in_code = _dtype_code(writers[0])
    owners = [np.empty((T // P,) + writers[0].shape[1:], _np_dtype(out_dtype)) for _ in range(P)]
    l2g = np.ascontiguousarray(l2g, dtype=np.int32)
    warr = (ctypes.c_void_p * P)(*[_ptr(w) for w in writers])
    oarr = (ctypes.c_void_p * P)(*[_ptr(o) for o in owners])
    _load().oracle_grad_return(P, T, row_elems, in_code, out_dtype, _ptr(l2g),
                               ctypes.cast(warr, ctypes.c_void_p), ctypes.cast(oarr, ctypes.c_void_p))
    return owners


def grad_return_accumulate(l2g: np.ndarray, writers, owners):
    """New owner arrays: each owner's current values plus the ordered writer sum."""
    writers = [np.ascontiguousarray(w) for w in writers]
    P = len(writers)
    T = writers[0].shape[0]
    row_elems = writers[0].size // T if T else 0
    out = [np.array(o, copy=True, order="C") for o in owners]
    l2g = np.ascontiguousarray(l2g, dtype=np.int32)
    warr = (ctypes.c_void_p * P)(*[_ptr(w) for w in writers])
    oarr = (ctypes.c_void_p * P)(*[_ptr(o) for o in out])
    _load().oracle_grad_return_accumulate(P, T, row_elems, _dtype_code(writers[0]), _dtype_code(out[0]),
                                          _ptr(l2g), ctypes.cast(warr, ctypes.c_void_p),
                                          ctypes.cast(oarr, ctypes.c_void_p))
    return out


def grad_scatter(l2g: np.ndarray, writer: np.ndarray, cp_size: int):
    """Per-owner slot arrays [T/P][row...] of one writer's global gradient."""
    writer = np.ascontiguousarray(writer)
    T = writer.shape[0]
    P = cp_size
    row_bytes = writer.nbytes // T if T else 0
    slots = [np.empty((T // P,) + writer.shape[1:], writer.dtype) for _ in range(P)]
    l2g = np.ascontiguousarray(l2g, dtype=np.int32)
    sarr = (ctypes.c_void_p * P)(*[_ptr(s) for s in slots])
    _load().oracle_grad_scatter(P, T, row_bytes, _ptr(l2g), _ptr(writer), ctypes.cast(sarr, ctypes.c_void_p))
    return slots

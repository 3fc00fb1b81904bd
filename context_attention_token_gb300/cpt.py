"""Python binding of the C ABI in include/cpt.h (argument marshalling only).

Every function has the name of the C call it wraps. Tensors are torch CUDA
tensors; the binding turns them into device pointers, passes the current
torch stream (or the one given), and raises ``CptError`` on any non-zero
status with the library's message. ctypes releases the GIL for the length of
each call, as the pages' binding does ("Add stream-ordered CP gradient
return primitive", TransformerEngine PR 3235, "Greptile Summary": the
function is registered with a GIL-release guard).

The shared library must have been built (``context_attention_token_gb300.build``);
importing this module without it raises ImportError: there is no fallback.
With CPT_LIBRARY_VARIANT=checked in the environment the binding loads the
bounds-checked build (libcpt_checked.so) instead of libcpt.so.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_VARIANT = os.environ.get("CPT_LIBRARY_VARIANT", "release")
if _VARIANT not in ("release", "checked"):
    raise ImportError(f"CPT_LIBRARY_VARIANT={_VARIANT!r}: expected 'release' or 'checked'")
_LIB_PATH = os.path.join(_PKG, "libcpt.so" if _VARIANT == "release" else "libcpt_checked.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"{_LIB_PATH} is missing: build it with `python -m context_attention_token_gb300.build` "
        "(the CUDA path has no fallback)")

_lib = ctypes.CDLL(_LIB_PATH)

# ------------------------------------------------------------------ constants
CPT_OK = 0
CPT_ERR_INVALID_ARG = 1
CPT_ERR_NOT_DIVISIBLE = 2
CPT_ERR_UNSUPPORTED = 3
CPT_ERR_ALIAS = 4
CPT_ERR_DEVICE = 5
CPT_ERR_ALIGNMENT = 6
CPT_ERR_TIMEOUT = 7
CPT_ERR_CUDA = 8
CPT_ERR_WORKSPACE = 9
CPT_ERR_NOT_PUBLISHED = 10

CPT_LAYOUT_DUAL_CHUNK_SWAP = 0
CPT_LAYOUT_PACKED_CONTIGUOUS = 1
CPT_LAYOUT_RETIRED_PACKED_SUPER_SEQUENCE = 2
CPT_LAYOUT_DUAL_CHUNK_SWAP_PADDED = 3
CPT_F32 = 0
CPT_BF16 = 1
CPT_WAIT_BOUNDED = 0
CPT_WAIT_DRIVER = 1
CPT_MAX_CP_SIZE = 8
CPT_KERNEL_AUTO = 0
CPT_KERNEL_LOADS = 1
CPT_KERNEL_BULK = 2
CPT_CALL_ROW_GATHER = 0
CPT_CALL_GRAD_RETURN = 1
CPT_CALL_SLOT_REDUCE = 2

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64
_sz = ctypes.c_size_t


def _sig(name, res, *args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


_sig("cpt_last_error_string", ctypes.c_char_p)
_sig("cpt_status_string", ctypes.c_char_p, ctypes.c_int)
_sig("cpt_validate_layout", ctypes.c_int, ctypes.c_int, _i32, _vp, _i32, _i64)
_sig("cpt_plan_workspace_bytes", _sz, ctypes.c_int, _i32, _i32, _i64)
_sig("cpt_plan_create", ctypes.c_int, ctypes.c_int, _i32, _vp, _i32, _i64, _vp, _sz, _vp,
     ctypes.POINTER(_vp))
_sig("cpt_plan_destroy", ctypes.c_int, _vp)
_sig("cpt_plan_info", ctypes.c_int, _vp, ctypes.POINTER(_i64), ctypes.POINTER(_i32), ctypes.POINTER(_i32))
_sig("cpt_plan_padded_tokens", ctypes.c_int, _vp, ctypes.POINTER(_i64))
_sig("cpt_layout_padded_tokens", ctypes.c_int, ctypes.c_int, _i32, _vp, _i32, _i64,
     ctypes.POINTER(_i64))
_sig("cpt_thd_real_lengths", ctypes.c_int, _vp, _vp, _vp)
_sig("cpt_index_map", ctypes.c_int, _vp, _vp, _vp, _vp)
_sig("cpt_thd_metadata", ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp)
_sig("cpt_partition", ctypes.c_int, _vp, _i32, _vp, _vp, _i64, ctypes.c_int, _vp)
_sig("cpt_grad_return_accumulate", ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _i64, ctypes.c_int,
     ctypes.c_int, _vp)
_sig("cpt_partition_rows", ctypes.c_int, _vp, _i32, _vp, _vp, _i64, ctypes.c_int, _i64, _i64, _vp)
_sig("cpt_grad_return_rows", ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _i64, ctypes.c_int, ctypes.c_int,
     _i64, _i64, _vp)
_sig("cpt_restore", ctypes.c_int, _vp, _i32, _vp, _vp, _i64, ctypes.c_int, _vp)
_sig("cpt_grad_return", ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _i64, ctypes.c_int, ctypes.c_int, _vp)
_sig("cpt_grad_return_noalloc", ctypes.c_int, ctypes.c_int, _i32, _vp, _i32, _i64, _vp, _vp, _vp, _vp,
     _i64, ctypes.c_int, ctypes.c_int, _vp)
_sig("cpt_grad_scatter", ctypes.c_int, _vp, _i32, _vp, _vp, _vp, _i64, ctypes.c_int, _vp)
_sig("cpt_epoch_create", ctypes.c_int, _i32, _vp, _vp, _vp, ctypes.POINTER(_vp))
_sig("cpt_epoch_destroy", ctypes.c_int, _vp)
_sig("cpt_epoch_advance", ctypes.c_int, _vp, ctypes.POINTER(ctypes.c_uint32))
_sig("cpt_epoch_set", ctypes.c_int, _vp, ctypes.c_uint32)
_sig("cpt_epoch_publish", ctypes.c_int, _vp, _i32, _vp)
_sig("cpt_epoch_wait", ctypes.c_int, _vp, _i32, _u64, ctypes.c_int, _vp)
_sig("cpt_epoch_status", ctypes.c_int, _vp, _i32, _vp, ctypes.POINTER(_i32))
_sig("cpt_kernel_wait_timeouts", ctypes.c_int, ctypes.POINTER(ctypes.c_uint32), _i32)
_sig("cpt_set_kernel_path", ctypes.c_int, _i32)
_sig("cpt_test_stall_bulk_waits", ctypes.c_int, _i32)
_sig("cpt_kernel_path_of", ctypes.c_int, _i32, _i32, _i32, _i32, _i32, _i64, _i64, ctypes.POINTER(_i32))
_sig("cpt_slot_reduce", ctypes.c_int, _vp, _i32, _i64, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp)
_sig("cpt_stream_ceiling", ctypes.c_int, _vp, _i32, _vp, _i64, _i32, _i32, _i32, _vp)
_sig("cpt_bounds_checked", _i32)
_sig("cpt_bounds_violations", ctypes.c_int, ctypes.POINTER(ctypes.c_uint32), _i32)


def library_path() -> str:
    return _LIB_PATH


def exported_symbols(names):
    """Names (of the given ones) the loaded library exports."""
    out = []
    for n in names:
        try:
            getattr(_lib, n)
            out.append(n)
        except AttributeError:
            pass
    return out


class CptError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        name = _lib.cpt_status_string(status).decode()
        super().__init__(f"{name}: {message}")


def _check(status: int):
    if status != CPT_OK:
        raise CptError(status, _lib.cpt_last_error_string().decode())


def cpt_last_error_string() -> str:
    return _lib.cpt_last_error_string().decode()


def cpt_status_string(status: int) -> str:
    return _lib.cpt_status_string(status).decode()


# ------------------------------------------------------------------ marshalling

def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return CPT_F32
    if t.dtype == torch.bfloat16:
        return CPT_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


# ctypes array types of n device pointers, built once per n
_PTR_ARRAYS = {}


def _ptr_array(items):
    """Device pointers of the items as a C array (passed by its address)."""
    n = len(items)
    kind = _PTR_ARRAYS.get(n)
    if kind is None:
        kind = _PTR_ARRAYS.setdefault(n, _vp * n)
    return kind(*[_ptr(x) for x in items])


class _Parts:
    """Device pointers of `parts` equally shaped tensors, given as one
    contiguous [parts, ...] tensor or as a sequence of tensors, with the
    shape and dtype of one part."""

    __slots__ = ("ptrs", "shape", "dtype", "part_bytes")

    def __init__(self, t, parts: int):
        if isinstance(t, torch.Tensor):
            if t.dim() == 0 or t.shape[0] != parts:
                raise ValueError(f"leading dimension of {tuple(t.shape)} != {parts}")
            if not t.is_contiguous():
                raise ValueError("tensors must be contiguous")
            base = t.data_ptr()
            step = t.stride(0) * t.element_size()
            self.ptrs = [base + i * step for i in range(parts)]
            self.shape = tuple(t.shape[1:])
            self.dtype = t.dtype
            self.part_bytes = step
        else:
            t = list(t)
            if len(t) != parts:
                raise ValueError(f"expected {parts} tensors, got {len(t)}")
            first = t[0]
            shape, dtype = first.shape, first.dtype
            ptrs = []
            for x in t:
                if isinstance(x, int):
                    raise TypeError("parts must be tensors")
                if x.shape != shape or x.dtype != dtype:
                    raise ValueError("the parts differ in shape or dtype")
                if not x.is_contiguous():
                    raise ValueError("tensors must be contiguous")
                ptrs.append(x.data_ptr())
            self.ptrs = ptrs
            self.shape = tuple(shape)
            self.dtype = dtype
            self.part_bytes = first.numel() * first.element_size()

    def array(self):
        """The pointers as a C array; ctypes passes an array argument by its
        address, and the call keeps the array alive while it runs."""
        n = len(self.ptrs)
        kind = _PTR_ARRAYS.get(n)
        if kind is None:
            kind = _PTR_ARRAYS.setdefault(n, _vp * n)
        return kind(*self.ptrs)

    def row_elems(self) -> int:
        n = 1
        for d in self.shape[1:]:
            n *= int(d)
        return n

    def code(self) -> int:
        if self.dtype == torch.float32:
            return CPT_F32
        if self.dtype == torch.bfloat16:
            return CPT_BF16
        raise TypeError(f"unsupported dtype {self.dtype} (float32 or bfloat16)")


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


_ELEM_BYTES = {torch.float32: 4, torch.bfloat16: 2, torch.int32: 4}


def _elem_bytes(dtype) -> int:
    n = _ELEM_BYTES.get(dtype)
    return n if n is not None else torch.empty(0, dtype=dtype).element_size()


def _need(t, nbytes: int, what: str, dtype=None):
    """Refuse a buffer smaller than the bytes the call will touch (the C ABI
    sees only its address), or of the wrong element type."""
    if t is None:
        return
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{what} has dtype {t.dtype}, expected {dtype}")
    if _nbytes(t) < nbytes:
        raise ValueError(f"{what} holds {_nbytes(t)} bytes but the call touches {nbytes}")


def _need_parts(parts, rows: int, row_elems: int, what: str):
    """Every part of `parts` must hold `rows` rows of `row_elems` elements."""
    if parts is None:
        return
    if parts.row_elems() != row_elems:
        raise ValueError(f"{what} rows have {parts.row_elems()} elements, expected {row_elems}")
    need = rows * row_elems * _elem_bytes(parts.dtype)
    if parts.part_bytes < need:
        raise ValueError(f"each part of {what} holds {parts.part_bytes} bytes but the call touches {need}")


def _same_kind(ts, what: str):
    """Tensors of one call that must share dtype and row width."""
    for t in ts[1:]:
        if t.dtype != ts[0].dtype or _row_elems(t) != _row_elems(ts[0]):
            raise ValueError(f"the {what} tensors differ in dtype or row width")


def _cu_array(cu_seqlens):
    vals = [int(v) for v in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    return (_i32 * len(vals))(*vals), len(vals) - 1


# ------------------------------------------------------------------ host-only

def cpt_validate_layout(layout: int, cp_size: int, cu_seqlens, total_tokens: int) -> int:
    """Status code of the host-side partition check (0 = valid)."""
    arr, n = _cu_array(cu_seqlens)
    return _lib.cpt_validate_layout(layout, cp_size, ctypes.cast(arr, _vp), n, total_tokens)


def cpt_plan_workspace_bytes(layout: int, cp_size: int, n_docs: int, total_tokens: int) -> int:
    return int(_lib.cpt_plan_workspace_bytes(layout, cp_size, n_docs, total_tokens))


def cpt_layout_padded_tokens(layout: int, cp_size: int, cu_seqlens, total_tokens: int) -> int:
    """Tokens of the buffer the layout partitions (the padded total for the
    padded layout, else total_tokens); raises CptError for a batch the
    layout rejects."""
    arr, n = _cu_array(cu_seqlens)
    v = _i64(0)
    _check(_lib.cpt_layout_padded_tokens(layout, cp_size, ctypes.cast(arr, _vp), n, total_tokens,
                                         ctypes.byref(v)))
    return int(v.value)


# ------------------------------------------------------------------ plan

class Plan:
    """Host handle of a plan plus the workspace tensor it lives in."""

    def __init__(self, handle: int, workspace: torch.Tensor, layout: int, cp_size: int,
                 n_docs: int, total_tokens: int, padded_tokens: int):
        self.handle = handle
        self.workspace = workspace
        self.layout = layout
        self.cp_size = cp_size
        self.n_docs = n_docs
        self.total_tokens = total_tokens
        self.padded_tokens = padded_tokens

    @property
    def local_tokens(self) -> int:
        return self.padded_tokens // self.cp_size

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h:
            _lib.cpt_plan_destroy(h)


def cpt_plan_create(layout: int, cp_size: int, cu_seqlens, total_tokens: int,
                    workspace: torch.Tensor | None = None, stream=None) -> Plan:
    arr, n = _cu_array(cu_seqlens)
    need = cpt_plan_workspace_bytes(layout, cp_size, n, total_tokens)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    h = _vp()
    _check(_lib.cpt_plan_create(layout, cp_size, ctypes.cast(arr, _vp), n, total_tokens,
                                _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _stream(stream), ctypes.byref(h)))
    tp = _i64()
    _check(_lib.cpt_plan_padded_tokens(h.value, ctypes.byref(tp)))
    return Plan(h.value, workspace, layout, cp_size, n, total_tokens, tp.value)


def cpt_plan_destroy(plan: Plan) -> None:
    h, plan.handle = plan.handle, None
    if h:
        _check(_lib.cpt_plan_destroy(h))


def cpt_plan_info(plan: Plan):
    """(total_tokens, cp_size, n_docs) as the library holds them."""
    T, P, n = _i64(), _i32(), _i32()
    _check(_lib.cpt_plan_info(plan.handle, ctypes.byref(T), ctypes.byref(P), ctypes.byref(n)))
    return T.value, P.value, n.value


def cpt_plan_padded_tokens(plan: Plan) -> int:
    v = _i64()
    _check(_lib.cpt_plan_padded_tokens(plan.handle, ctypes.byref(v)))
    return v.value


def cpt_thd_real_lengths(plan: Plan, real_len: torch.Tensor, stream=None):
    """real_len[r][i] ([P, n] int32) = real tokens of document i on rank r."""
    _need(real_len, 4 * plan.cp_size * plan.n_docs, "real_len", torch.int32)
    _check(_lib.cpt_thd_real_lengths(plan.handle, _ptr(real_len), _stream(stream)))


def cpt_index_map(plan: Plan, l2g: torch.Tensor, g2l: torch.Tensor | None = None, stream=None):
    _need(l2g, 4 * plan.padded_tokens, "l2g", torch.int32)
    _need(g2l, 4 * plan.padded_tokens, "g2l", torch.int32)
    _check(_lib.cpt_index_map(plan.handle, _ptr(l2g), _ptr(g2l), _stream(stream)))


def cpt_thd_metadata(plan: Plan, num_segs, seg_doc_first, cu_local, seg_offsets, stream=None):
    P = plan.cp_size
    _need(num_segs, 4 * P, "num_segs", torch.int32)
    _need(seg_doc_first, 4 * P, "seg_doc_first", torch.int32)
    _need(cu_local, 4 * P * (plan.n_docs + 1), "cu_local", torch.int32)
    _need(seg_offsets, 4 * (P + 1), "seg_offsets", torch.int32)
    _check(_lib.cpt_thd_metadata(plan.handle, _ptr(num_segs), _ptr(seg_doc_first), _ptr(cu_local),
                                 _ptr(seg_offsets), _stream(stream)))


def cpt_partition(plan: Plan, srcs, dsts, stream=None):
    """dsts[t] ([P, T/P, ...]) = rank-local reorder of srcs[t] ([T, ...])."""
    srcs, dsts = list(srcs), list(dsts)
    _check_gather(plan, srcs, dsts, plan.total_tokens, plan.padded_tokens, _row_elems(srcs[0]) if srcs else 0)
    _check(_lib.cpt_partition(plan.handle, len(srcs), _ptr_array(srcs),
                              _ptr_array(dsts), _row_elems(srcs[0]), _dtype_code(srcs[0]),
                              _stream(stream)))


def cpt_partition_rows(plan: Plan, srcs, dsts, local_begin: int, local_count: int, stream=None):
    """cpt_partition for flattened local rows [local_begin, local_begin + local_count) only."""
    srcs, dsts = list(srcs), list(dsts)
    _check_gather(plan, srcs, dsts, plan.total_tokens, plan.padded_tokens, _row_elems(srcs[0]) if srcs else 0)
    _check(_lib.cpt_partition_rows(plan.handle, len(srcs), _ptr_array(srcs),
                                   _ptr_array(dsts), _row_elems(srcs[0]),
                                   _dtype_code(srcs[0]), local_begin, local_count, _stream(stream)))


def cpt_restore(plan: Plan, srcs, dsts, stream=None):
    """dsts[t] ([T, ...]) = global-order copy of the rank-local srcs[t] ([P, T/P, ...])."""
    srcs, dsts = list(srcs), list(dsts)
    _check_gather(plan, srcs, dsts, plan.padded_tokens, plan.total_tokens, _row_elems(dsts[0]) if dsts else 0)
    _check(_lib.cpt_restore(plan.handle, len(srcs), _ptr_array(srcs),
                            _ptr_array(dsts), _row_elems(dsts[0]),
                            _dtype_code(srcs[0]), _stream(stream)))


def _check_gather(plan: Plan, srcs, dsts, src_rows: int, dst_rows: int, row: int):
    """Partition, restore: as many sources as destinations, one dtype, every
    buffer large enough for its rows of `row` elements."""
    if len(srcs) != len(dsts):
        raise ValueError("srcs and dsts differ in length")
    if not srcs:
        return
    esz = srcs[0].element_size()
    for i, (a, b) in enumerate(zip(srcs, dsts)):
        if a.dtype != srcs[0].dtype or b.dtype != srcs[0].dtype:
            raise ValueError("srcs and dsts must share one dtype")
        _need(a, src_rows * row * esz, f"srcs[{i}]")
        _need(b, dst_rows * row * esz, f"dsts[{i}]")


def _row_elems(t: torch.Tensor) -> int:
    """Elements of one token row of a [T, ...] tensor."""
    n = 1
    for d in t.shape[1:]:
        n *= int(d)
    return n


def _check_grad_return(Tpad: int, P: int, dkw, dvw, dko, dvo):
    """Writers of Tpad rows, owners of Tpad / P rows, one row width; the dV
    pair like the dK pair."""
    row = dkw.row_elems()
    _need_parts(dkw, Tpad, row, "dk_writers")
    _need_parts(dko, Tpad // P, row, "dk_owners")
    if dvw is not None and dvo is not None:  # one without the other: the library refuses it
        if dvw.dtype != dkw.dtype or dvo.dtype != dko.dtype:
            raise ValueError("the dV pair must have the dtypes of the dK pair")
        _need_parts(dvw, Tpad, row, "dv_writers")
        _need_parts(dvo, Tpad // P, row, "dv_owners")


def _grad_return(fn, plan: Plan, dk_writers, dv_writers, dk_owners, dv_owners, stream):
    P = plan.cp_size
    dkw = _Parts(dk_writers, P)
    dko = _Parts(dk_owners, P)
    dvw = _Parts(dv_writers, P) if dv_writers is not None else None
    dvo = _Parts(dv_owners, P) if dv_owners is not None else None
    _check_grad_return(plan.padded_tokens, P, dkw, dvw, dko, dvo)
    _check(fn(plan.handle, dkw.array(), dvw.array() if dvw is not None else None, dko.array(),
              dvo.array() if dvo is not None else None, dkw.row_elems(), dkw.code(), dko.code(),
              _stream(stream)))


def cpt_grad_return(plan: Plan, dk_writers, dv_writers, dk_owners, dv_owners, stream=None):
    """Owners' local dK (and dV) = ordered sum over writers' global gradients.

    Each of the four arguments is a [P, ...] tensor or a list of P tensors;
    the dV pair may be None.
    """
    _grad_return(_lib.cpt_grad_return, plan, dk_writers, dv_writers, dk_owners, dv_owners, stream)


def cpt_grad_return_rows(plan: Plan, dk_writers, dv_writers, dk_owners, dv_owners,
                         local_begin: int, local_count: int, stream=None):
    """cpt_grad_return for flattened owner-major local rows [local_begin, +local_count) only."""
    P = plan.cp_size
    dkw = _Parts(dk_writers, P)
    dko = _Parts(dk_owners, P)
    dvw = _Parts(dv_writers, P) if dv_writers is not None else None
    dvo = _Parts(dv_owners, P) if dv_owners is not None else None
    _check_grad_return(plan.padded_tokens, P, dkw, dvw, dko, dvo)
    _check(_lib.cpt_grad_return_rows(
        plan.handle, dkw.array(), dvw.array() if dvw is not None else None, dko.array(),
        dvo.array() if dvo is not None else None, dkw.row_elems(), dkw.code(), dko.code(),
        local_begin, local_count, _stream(stream)))


def cpt_grad_return_accumulate(plan: Plan, dk_writers, dv_writers, dk_owners, dv_owners,
                               stream=None):
    """As cpt_grad_return, but the owners' current values start the sums."""
    _grad_return(_lib.cpt_grad_return_accumulate, plan, dk_writers, dv_writers, dk_owners,
                 dv_owners, stream)


CPT_NOALLOC_MAX_TOKENS = 1048576
CPT_NOALLOC_MAX_DOCS = 65536


def cpt_grad_return_noalloc(layout: int, cp_size: int, cu_seqlens, total_tokens: int, dk_writers,
                            dv_writers, dk_owners, dv_owners, stream=None):
    """cpt_grad_return without a plan or workspace, for callers that cannot
    allocate device memory: the map lives in a fixed-size array inside the
    library (at most CPT_NOALLOC_MAX_TOKENS tokens). Calls that overlap on
    the GPU share that array and race."""
    arr, n = _cu_array(cu_seqlens)
    P = cp_size
    dkw = _Parts(dk_writers, P)
    dko = _Parts(dk_owners, P)
    dvw = _Parts(dv_writers, P) if dv_writers is not None else None
    dvo = _Parts(dv_owners, P) if dv_owners is not None else None
    # the library sizes the map; batches it refuses (on layout or size
    # grounds) are left to the call itself to report
    Tmap = _i64(0)
    if _lib.cpt_layout_padded_tokens(layout, P, ctypes.cast(arr, _vp), n, total_tokens,
                                     ctypes.byref(Tmap)) != CPT_OK:
        Tmap.value = 0
    if 0 < Tmap.value <= CPT_NOALLOC_MAX_TOKENS and n <= CPT_NOALLOC_MAX_DOCS:
        _check_grad_return(Tmap.value, P, dkw, dvw, dko, dvo)
    _check(_lib.cpt_grad_return_noalloc(
        layout, P, ctypes.cast(arr, _vp), n, total_tokens, dkw.array(),
        dvw.array() if dvw is not None else None, dko.array(),
        dvo.array() if dvo is not None else None, dkw.row_elems(), dkw.code(), dko.code(),
        _stream(stream)))


def cpt_grad_scatter(plan: Plan, writer: int, src: torch.Tensor, slots, self_slot, stream=None):
    """slots[o] ([T/P, ...]) = writer's rows owned by o; self_slot must be slots[writer]."""
    sl = _Parts(slots, plan.cp_size)
    row = _row_elems(src)
    _need(src, plan.padded_tokens * row * src.element_size(), "src")
    if sl.dtype != src.dtype:
        raise ValueError("slots must have the dtype of src")
    _need_parts(sl, plan.padded_tokens // plan.cp_size, row, "slots")
    _check(_lib.cpt_grad_scatter(plan.handle, writer, _ptr(src), sl.array(), _ptr(self_slot),
                                 _row_elems(src), _dtype_code(src), _stream(stream)))


def cpt_slot_reduce(slots, dst: torch.Tensor, status: torch.Tensor | int | None = None, stream=None):
    n = slots.shape[0] if isinstance(slots, torch.Tensor) else len(slots)
    sl = _Parts(slots, n)
    numel = 1
    for d in sl.shape:
        numel *= int(d)
    _need(dst, numel * dst.element_size(), "dst")
    if isinstance(status, torch.Tensor):
        _need(status, 4, "status", torch.int32)
    _check(_lib.cpt_slot_reduce(sl.array(), n, numel, sl.code(), _dtype_code(dst), _ptr(dst),
                                _ptr(status), _stream(stream)))


# ------------------------------------------------------------------ epochs

class Epoch:
    def __init__(self, handle: int, flags: torch.Tensor, status: torch.Tensor, cp_size: int):
        self.handle = handle
        self.flags = flags
        self.status = status
        self.cp_size = cp_size

    def status_ptr(self, owner: int) -> int:
        return self.status.data_ptr() + 4 * owner

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h:
            _lib.cpt_epoch_destroy(h)


def cpt_epoch_create(cp_size: int, flags: torch.Tensor | None = None, status: torch.Tensor | None = None,
                     stream=None) -> Epoch:
    if flags is None:
        flags = torch.zeros(cp_size * cp_size, dtype=torch.int32, device="cuda")
    if status is None:
        status = torch.zeros(cp_size, dtype=torch.int32, device="cuda")
    h = _vp()
    _check(_lib.cpt_epoch_create(cp_size, _ptr(flags), _ptr(status), _stream(stream), ctypes.byref(h)))
    return Epoch(h.value, flags, status, cp_size)


def cpt_epoch_destroy(ep: Epoch) -> None:
    h, ep.handle = ep.handle, None
    if h:
        _check(_lib.cpt_epoch_destroy(h))


def cpt_epoch_advance(ep: Epoch) -> int:
    e = ctypes.c_uint32()
    _check(_lib.cpt_epoch_advance(ep.handle, ctypes.byref(e)))
    return e.value


def cpt_epoch_set(ep: Epoch, epoch: int) -> None:
    _check(_lib.cpt_epoch_set(ep.handle, epoch))


def cpt_epoch_publish(ep: Epoch, writer: int, stream=None) -> None:
    _check(_lib.cpt_epoch_publish(ep.handle, writer, _stream(stream)))


def cpt_epoch_wait(ep: Epoch, owner: int, timeout_ns: int = 1_000_000_000,
                   mode: int = CPT_WAIT_BOUNDED, stream=None) -> None:
    _check(_lib.cpt_epoch_wait(ep.handle, owner, timeout_ns, mode, _stream(stream)))


def cpt_epoch_status(ep: Epoch, owner: int, stream=None) -> int:
    v = _i32()
    _check(_lib.cpt_epoch_status(ep.handle, owner, _stream(stream), ctypes.byref(v)))
    return v.value


def cpt_set_kernel_path(kernel: int):
    """Process-wide kernel choice of the row gather, the gradient return and
    the slot reduce: CPT_KERNEL_AUTO (measured rule), _LOADS or _BULK."""
    _check(_lib.cpt_set_kernel_path(kernel))


def cpt_kernel_path_of(call: int, cp_size: int, in_dtype: int, out_dtype: int, accumulate: bool,
                       row_bytes: int, rows: int) -> int:
    """CPT_KERNEL_LOADS or CPT_KERNEL_BULK: the kernel the call would run now."""
    v = _i32()
    _check(_lib.cpt_kernel_path_of(call, cp_size, in_dtype, out_dtype, 1 if accumulate else 0,
                                   row_bytes, rows, ctypes.byref(v)))
    return v.value


def cpt_bounds_checked() -> bool:
    """Whether the loaded library is the bounds-checked build."""
    return bool(_lib.cpt_bounds_checked())


def cpt_bounds_violations(reset: bool = False) -> int:
    """Failed device bounds checks so far (bounds-checked build only)."""
    v = ctypes.c_uint32(0)
    _check(_lib.cpt_bounds_violations(ctypes.byref(v), 1 if reset else 0))
    return int(v.value)


def cpt_test_stall_bulk_waits(on: bool):
    """Test switch: make every bulk-copy wait of later launches run out of its
    budget (on) or behave normally (off)."""
    _check(_lib.cpt_test_stall_bulk_waits(1 if on else 0))


def cpt_kernel_wait_timeouts(reset: bool = False) -> int:
    """Bulk-copy waits in the library's kernels that ran out of their budget
    on the current device (blocking; non-zero means an earlier output is not
    valid)."""
    v = ctypes.c_uint32()
    _check(_lib.cpt_kernel_wait_timeouts(ctypes.byref(v), 1 if reset else 0))
    return v.value


def cpt_stream_ceiling(srcs, dst: torch.Tensor, block_bytes: int, stages: int, ctas_per_sm: int = 1,
                       stream=None):
    """dst = copy of srcs[0], every other source read and discarded: the
    read/write mix of an HBM-bound call with no arithmetic (a roofline
    ceiling). All tensors hold the same number of bytes."""
    sl = _Parts(srcs, len(srcs) if not isinstance(srcs, torch.Tensor) else srcs.shape[0])
    nbytes = sl.part_bytes
    _need(dst, nbytes, "dst")
    _check(_lib.cpt_stream_ceiling(sl.array(), len(sl.ptrs), _ptr(dst), nbytes, block_bytes, stages,
                                   ctas_per_sm, _stream(stream)))


def declared_functions(header_path: str) -> list[str]:
    """Function names declared in a C header (for the export check)."""
    with open(header_path) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cpt_[a-z0-9_]+)\s*\(", text)))

"""Thin ctypes binding of libhogwild.so (include/hogwild.h), same names as the C ABI.

Only argument marshalling happens here: torch tensors are passed as raw device pointers and
torch's current CUDA stream as the ``stream`` argument; every step of the computation runs in
the library's kernels.  If the library has not been built this module raises at load time --
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhogwild.so")

HW_OK = 0
HW_ERR_INVALID_ARG = 1
HW_ERR_OUT_OF_PAGES = 2
HW_ERR_CAPACITY = 3
HW_ERR_CUDA = 4
HW_ERR_DEVICE_CHECK = 5
HW_ERR_DEVICE_TIMEOUT = 6
HW_ERR_UNSUPPORTED = 7
HW_OUT_BF16 = 0
HW_OUT_F32 = 1

EXPORTED = (
    "hw_status_string", "hw_last_cuda_error", "hw_pool_size", "hw_workspace_size", "hw_create",
    "hw_destroy", "hw_append_kv", "hw_concurrent_attention", "hw_concurrent_attention_noalloc",
    "hw_concurrent_attention_mq", "hw_concurrent_attention_range", "hw_merge_attention",
    "hw_compact_segments", "hw_compact_auto",
    "hw_step_end", "hw_decode_step_host", "hw_step_scratch_size",
    "hw_check_device_errors", "hw_debug_expire_plans", "hw_profile_enable", "hw_profile_read",
    "hw_get_counts", "hw_get_segment", "hw_get_blocks", "hw_get_view",
)


class hw_config(ctypes.Structure):
    _fields_ = [
        ("num_problems", ctypes.c_int32), ("num_workers", ctypes.c_int32),
        ("num_layers", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("contiguous", ctypes.c_int32),
        ("num_pages", ctypes.c_int32), ("max_position", ctypes.c_int32),
        ("max_segments", ctypes.c_int32), ("max_append_tokens", ctypes.c_int32),
        ("rope_theta", ctypes.c_double), ("layout", ctypes.c_int32), ("reserved", ctypes.c_int32),
    ]


class hw_profile(ctypes.Structure):
    _fields_ = [
        ("launches", ctypes.c_int64), ("attention_launches", ctypes.c_int64),
        ("append_launches", ctypes.c_int64), ("attention_ms", ctypes.c_double),
        ("append_ms", ctypes.c_double), ("timed_attention", ctypes.c_int64),
        ("timed_append", ctypes.c_int64), ("merge_ms", ctypes.c_double),
        ("timed_merge", ctypes.c_int64),
    ]


class HogwildError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {_status_name(status)}{(' ' + detail) if detail else ''}")


_lib: Optional[ctypes.CDLL] = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_PI32 = ctypes.POINTER(ctypes.c_int32)


def load() -> ctypes.CDLL:
    """Load the in-tree library (build it with ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it first (python -c 'import "
                           "__graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    sig = {
        "hw_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "hw_last_cuda_error": (_I32, [ctypes.POINTER(ctypes.c_char_p)]),
        "hw_pool_size": (ctypes.c_int, [ctypes.POINTER(hw_config), ctypes.POINTER(ctypes.c_size_t)]),
        "hw_workspace_size": (ctypes.c_int, [ctypes.POINTER(hw_config), ctypes.POINTER(ctypes.c_size_t)]),
        "hw_create": (ctypes.c_int, [ctypes.POINTER(hw_config), _P, _P, _P, ctypes.c_size_t, _PI32, _P,
                                     ctypes.POINTER(_P)]),
        "hw_destroy": (None, [_P]),
        "hw_append_kv": (ctypes.c_int, [_P, _I32, _P, _P, _P, _P]),
        "hw_concurrent_attention": (ctypes.c_int, [_P, _I32, _P, _P, _I32, _P, _P]),
        "hw_concurrent_attention_noalloc": (ctypes.c_int, [_P, _I32, _P, _P, _I32, _P, _P]),
        "hw_concurrent_attention_mq": (ctypes.c_int, [_P, _I32, _P, _P, _P, _I32, _P, _P]),
        "hw_concurrent_attention_range": (ctypes.c_int, [_P, _I32, _P, _P, _P, _P, _P]),
        "hw_merge_attention": (ctypes.c_int, [_I32, ctypes.c_int64, _I32, _P, _P, _P, _I32, _P,
                                              _P]),
        "hw_compact_segments": (ctypes.c_int, [_P, _I32, _I32, _I32, _P]),
        "hw_compact_auto": (ctypes.c_int, [_P, _I32, _P, _PI32]),
        "hw_step_end": (ctypes.c_int, [_P, _P, _P]),
        "hw_decode_step_host": (ctypes.c_int, [_P, _P, _P, ctypes.c_size_t, _P, _I32, _P, _P,
                                               ctypes.c_size_t, _I32, _P]),
        "hw_step_scratch_size": (ctypes.c_int, [_P, _P, _I32, ctypes.POINTER(ctypes.c_size_t)]),
        "hw_check_device_errors": (ctypes.c_int, [_P, _P, ctypes.POINTER(ctypes.c_uint32)]),
        "hw_debug_expire_plans": (ctypes.c_int, [_P, _I32]),
        "hw_profile_enable": (ctypes.c_int, [_P, _I32]),
        "hw_profile_read": (ctypes.c_int, [_P, ctypes.POINTER(hw_profile)]),
        "hw_get_counts": (ctypes.c_int, [_P, _PI32, _PI32]),
        "hw_get_segment": (ctypes.c_int, [_P, _I32, _PI32, _PI32, _PI32, _PI32, _PI32, _PI32, _I32]),
        "hw_get_blocks": (ctypes.c_int, [_P, _I32, _PI32, _I32, _PI32, _PI32]),
        "hw_get_view": (ctypes.c_int, [_P, _I32, _I32, _PI32, _PI32, _PI32, _I32, _PI32, _PI32]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _status_name(st: int) -> str:
    try:
        return load().hw_status_string(st).decode()
    except Exception:
        return f"status {st}"


def _check(st: int, where: str):
    if st != HW_OK:
        detail = ""
        if st == HW_ERR_CUDA:
            msg = ctypes.c_char_p()
            code = load().hw_last_cuda_error(ctypes.byref(msg))
            detail = f"(cuda error {code}: {msg.value.decode() if msg.value else ''})"
        raise HogwildError(st, where, detail)


def _i32(a) -> np.ndarray:
    if isinstance(a, np.ndarray) and a.dtype == np.int32 and a.flags.c_contiguous:
        return a
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _host_arg(a, dtype):
    """A host array argument as (array to keep alive until the call returns, its address); an
    int is taken as an address already (the caller keeps that array alive), None stays None."""
    if a is None or isinstance(a, int):
        return None, a
    arr = np.ascontiguousarray(np.asarray(a, dtype=dtype))
    return arr, arr.ctypes.data


def _ptr(arr: np.ndarray, ctype):
    return arr.ctypes.data_as(ctypes.POINTER(ctype))


def _dptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


# ---- functions with the C names --------------------------------------------------------


def hw_status_string(st: int) -> str:
    return _status_name(st)


def hw_pool_size(cfg: hw_config) -> int:
    n = ctypes.c_size_t()
    _check(load().hw_pool_size(ctypes.byref(cfg), ctypes.byref(n)), "hw_pool_size")
    return n.value


def hw_workspace_size(cfg: hw_config) -> int:
    n = ctypes.c_size_t()
    _check(load().hw_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "hw_workspace_size")
    return n.value


def hw_create(cfg: hw_config, k_pool, v_pool, workspace, page_order=None, stream=None) -> int:
    ctx = _P()
    po = None if page_order is None else _i32(page_order)
    st = load().hw_create(ctypes.byref(cfg), _dptr(k_pool), _dptr(v_pool), _dptr(workspace),
                          workspace.numel() * workspace.element_size(),
                          None if po is None else _ptr(po, ctypes.c_int32), _stream(stream),
                          ctypes.byref(ctx))
    _check(st, "hw_create")
    return ctx.value


def hw_destroy(ctx: int) -> None:
    load().hw_destroy(ctx)


def hw_append_kv(ctx: int, layer: int, n_new, k_raw, v_raw, stream=None) -> None:
    """n_new: host int32 [P][W + 1] (array-like), or the address (int) of such an array that
    stays alive for the call (saves the per-call conversion in a decode loop)."""
    keep, nptr = _host_arg(n_new, np.int32)
    st = (_lib or load()).hw_append_kv(ctx, layer, nptr, _dptr(k_raw), _dptr(v_raw),
                                       _stream(stream))
    del keep
    if st:
        _check(st, "hw_append_kv")


def hw_concurrent_attention(ctx: int, layer: int, q, out, out_dtype: int, lse=None,
                            stream=None) -> None:
    st = (_lib or load()).hw_concurrent_attention(ctx, layer, q.data_ptr(), out.data_ptr(),
                                                  out_dtype, _dptr(lse), _stream(stream))
    if st:
        _check(st, "hw_concurrent_attention")


def hw_concurrent_attention_mq(ctx: int, layer: int, q, n_q, out, out_dtype: int, lse=None,
                               stream=None) -> None:
    """Several causal query tokens per worker: n_q host int32 [P][W]; q / out [sum n_q][H_q][D]."""
    nq = np.ascontiguousarray(np.asarray(n_q, dtype=np.int32))
    _check(load().hw_concurrent_attention_mq(ctx, layer, _dptr(q), nq.ctypes.data, _dptr(out),
                                             out_dtype, _dptr(lse), _stream(stream)),
           "hw_concurrent_attention_mq")


def hw_concurrent_attention_range(ctx: int, layer: int, q, ranges, out, lse,
                                  stream=None) -> None:
    """Attention over entries [ranges[p][0], ranges[p][1]) of each problem (host int64 [P][2]);
    out fp32 [P][W][H_q][D] normalised over those keys, lse fp32 [P][W][H_q]."""
    rg = np.ascontiguousarray(np.asarray(ranges, dtype=np.int64))
    _check(load().hw_concurrent_attention_range(ctx, layer, _dptr(q), rg.ctypes.data, _dptr(out),
                                                _dptr(lse), _stream(stream)),
           "hw_concurrent_attention_range")


def hw_merge_attention(parts_out, parts_lse, out, out_dtype: int, lse=None, stream=None) -> None:
    """Log-sum-exp merge of partial results: parts_out fp32 [n][..][D], parts_lse fp32 [n][..]
    (the same query rows in every part); out [..][D] bf16 or fp32, lse fp32 [..] or None."""
    n = int(parts_out.shape[0])
    rows = int(parts_lse.numel() // n)
    _check(load().hw_merge_attention(n, rows, int(parts_out.shape[-1]), _dptr(parts_out),
                                     _dptr(parts_lse), _dptr(out), out_dtype, _dptr(lse),
                                     _stream(stream)),
           "hw_merge_attention")


def hw_concurrent_attention_noalloc(ctx: int, layer: int, q, out, out_dtype: int, lse=None,
                                    stream=None) -> None:
    """hw_concurrent_attention with its scratch in the library's fixed device array."""
    _check(load().hw_concurrent_attention_noalloc(ctx, layer, _dptr(q), _dptr(out), out_dtype,
                                                  _dptr(lse), _stream(stream)),
           "hw_concurrent_attention_noalloc")


def hw_compact_segments(ctx: int, problem: int, first: int, count: int, stream=None) -> None:
    _check(load().hw_compact_segments(ctx, problem, first, count, _stream(stream)),
           "hw_compact_segments")


def hw_compact_auto(ctx: int, max_paragraphs: int, stream=None) -> int:
    """The compaction policy; returns the number of merges enqueued."""
    n = ctypes.c_int32()
    _check(load().hw_compact_auto(ctx, int(max_paragraphs), _stream(stream), ctypes.byref(n)),
           "hw_compact_auto")
    return n.value


def hw_step_end(ctx: int, finished=None, stream=None) -> None:
    """finished: host uint8 [P][W] (array-like), None, or the address (int) of such an array."""
    keep, fptr = _host_arg(finished, np.uint8)
    st = (_lib or load()).hw_step_end(ctx, fptr, _stream(stream))
    del keep
    if st:
        _check(st, "hw_step_end")


def hw_step_scratch_size(ctx: int, n_new, out_dtype: int) -> int:
    n = ctypes.c_size_t()
    keep, nptr = _host_arg(n_new, np.int32)
    _check(load().hw_step_scratch_size(ctx, nptr, out_dtype, ctypes.byref(n)),
           "hw_step_scratch_size")
    del keep
    return n.value


def hw_decode_step_host(ctx: int, n_new, in_host: int, in_bytes: int, out_host: int,
                        out_dtype: int, finished, scratch: int, scratch_bytes: int,
                        sync: bool = True, stream=None) -> None:
    """One decode step from host memory.  in_host / out_host: host addresses (ints) of the
    packed [K][V][Q] input and the [L][P][W][H_q][D] output (page-locked for asynchronous
    copies); scratch: device address; n_new and finished as hw_append_kv and hw_step_end
    (array-likes, or addresses of arrays that stay alive for the call)."""
    keep_n, nptr = _host_arg(n_new, np.int32)
    keep_f, fptr = _host_arg(finished, np.uint8)
    st = (_lib or load()).hw_decode_step_host(ctx, nptr, in_host, in_bytes, out_host, out_dtype,
                                              fptr, scratch, scratch_bytes, int(bool(sync)),
                                              _stream(stream))
    del keep_n, keep_f
    if st:
        _check(st, "hw_decode_step_host")


def hw_check_device_errors(ctx: int, stream=None):
    info = (ctypes.c_uint32 * 4)()
    st = load().hw_check_device_errors(ctx, _stream(stream), info)
    return st, list(info)


def hw_debug_expire_plans(ctx: int, count: int) -> None:
    _check(load().hw_debug_expire_plans(ctx, int(count)), "hw_debug_expire_plans")


def hw_profile_enable(ctx: int, enable: bool = True) -> None:
    _check(load().hw_profile_enable(ctx, int(bool(enable))), "hw_profile_enable")


def hw_profile_read(ctx: int) -> dict:
    p = hw_profile()
    _check(load().hw_profile_read(ctx, ctypes.byref(p)), "hw_profile_read")
    return {f: getattr(p, f) for f, _ in hw_profile._fields_}


def hw_get_counts(ctx: int):
    a, b = ctypes.c_int32(), ctypes.c_int32()
    _check(load().hw_get_counts(ctx, ctypes.byref(a), ctypes.byref(b)), "hw_get_counts")
    return a.value, b.value


def hw_get_segment(ctx: int, seg: int, pages_cap: int = 1 << 16):
    vals = [ctypes.c_int32() for _ in range(5)]
    pages = np.zeros(pages_cap, dtype=np.int32)
    _check(load().hw_get_segment(ctx, seg, *[ctypes.byref(v) for v in vals],
                                 _ptr(pages, ctypes.c_int32), pages_cap), "hw_get_segment")
    problem, origin, length, pending, npages = (v.value for v in vals)
    return problem, origin, length, pending, pages[:npages].tolist()


def hw_get_blocks(ctx: int, problem: int, num_workers: int, cap: int = 4096):
    common = np.zeros(cap, dtype=np.int32)
    live = np.zeros(num_workers, dtype=np.int32)
    n = ctypes.c_int32()
    _check(load().hw_get_blocks(ctx, problem, _ptr(common, ctypes.c_int32), cap, ctypes.byref(n),
                                _ptr(live, ctypes.c_int32)), "hw_get_blocks")
    return common[:n.value].tolist(), live.tolist()


def hw_get_view(ctx: int, problem: int, worker: int, cap: int = 4096):
    ids, offs, lens = (np.zeros(cap, dtype=np.int32) for _ in range(3))
    n, iq = ctypes.c_int32(), ctypes.c_int32()
    _check(load().hw_get_view(ctx, problem, worker, _ptr(ids, ctypes.c_int32),
                              _ptr(offs, ctypes.c_int32), _ptr(lens, ctypes.c_int32), cap,
                              ctypes.byref(n), ctypes.byref(iq)), "hw_get_view")
    k = n.value
    return list(zip(ids[:k].tolist(), offs[:k].tolist(), lens[:k].tolist())), iq.value

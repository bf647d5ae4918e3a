"""Thin ctypes binding of ``include/kvd.h``.

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of ``libkvd.so``.  There is no fallback: when the library is missing
or a call returns a non-OK status, these functions raise.

Two layers, same names as the C ABI:

* ``raw`` -- the C functions with integer pointers (``ctypes``), for callers
  that manage their own memory;
* the module-level functions -- take ``torch`` CUDA tensors, check dtype,
  device and contiguity, derive the shape arguments, and pass the current
  stream.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

KVD_OK = 0
KVD_ERR_INVALID_ARG = 1
KVD_ERR_CAPACITY = 2
KVD_ERR_UNSUPPORTED = 3
KVD_ERR_WORKSPACE = 4
KVD_ERR_CUDA = 5

KVD_F32 = 0
KVD_BF16 = 1
KVD_F16 = 2
KVD_E4M3 = 3

KVD_DEVERR_PAST_LEN = 1
KVD_DEVERR_TIMEOUT = 2
KVD_DEVERR_PAGE = 4
KVD_DEVERR_INTERNAL = 8

KVD_STEP_HISTORY_STABLE = 1  # kvd_decode_step_flags: no earlier work writes past_len or the history

_TORCH_DTYPE = {torch.float32: KVD_F32, torch.bfloat16: KVD_BF16, torch.float16: KVD_F16}
_NAME_DTYPE = {"f32": KVD_F32, "bf16": KVD_BF16, "f16": KVD_F16, "e4m3": KVD_E4M3}


class KvdError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {raw.kvd_status_string(status).decode()} ({status})")


class PlanInfo(ctypes.Structure):
    _fields_ = [("tile_keys", ctypes.c_int), ("max_tiles", ctypes.c_int), ("grid", ctypes.c_int),
                ("threads", ctypes.c_int), ("smem_bytes", ctypes.c_int), ("launches", ctypes.c_int),
                ("workspace_bytes", ctypes.c_size_t), ("rows_per_block", ctypes.c_int),
                ("tensor_cores", ctypes.c_int), ("early_start", ctypes.c_int),
                ("cluster", ctypes.c_int)]


class _Lib:
    """The loaded ``libkvd.so`` with typed C signatures."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        vp, sz, ci, cf, u32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
        lib.kvd_append.restype = ci
        lib.kvd_append.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, u32p, vp]
        lib.kvd_decode_workspace_bytes.restype = sz
        lib.kvd_decode_workspace_bytes.argtypes = [ci, ci, ci, ci, ci, ci, ci]
        lib.kvd_decode_attention.restype = ci
        lib.kvd_decode_attention.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cf, ci,
                                             vp, sz, u32p, vp]
        lib.kvd_decode_step.restype = ci
        lib.kvd_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cf, ci,
                                        vp, sz, u32p, vp]
        lib.kvd_decode_step_flags.restype = ci
        lib.kvd_decode_step_flags.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cf, ci,
                                              ctypes.c_uint32, vp, sz, u32p, vp]
        lib.kvd_decode_step_host.restype = ci
        lib.kvd_decode_step_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cf, ci,
                                             vp, sz, vp, sz, u32p, vp]
        lib.kvd_decode_step_host_packed.restype = ci
        lib.kvd_decode_step_host_packed.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cf, ci, vp, sz, vp, sz,
                                                    u32p, vp]
        lib.kvd_host_staging_bytes.restype = sz
        lib.kvd_host_staging_bytes.argtypes = [ci, ci, ci, ci, ci, ci]
        lib.kvd_host_staging_inputs_bytes.restype = sz
        lib.kvd_host_staging_inputs_bytes.argtypes = [ci, ci, ci, ci, ci, ci]
        lib.kvd_paged_append.restype = ci
        lib.kvd_paged_append.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ci, ci, u32p, vp]
        lib.kvd_paged_decode_attention.restype = ci
        lib.kvd_paged_decode_attention.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ci, ci,
                                                   cf, ci, vp, sz, u32p, vp]
        lib.kvd_paged_decode_step.restype = ci
        lib.kvd_paged_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ci,
                                              ci, cf, ci, vp, sz, u32p, vp]
        lib.kvd_append_e4m3.restype = ci
        lib.kvd_append_e4m3.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cf, cf, u32p, vp]
        lib.kvd_decode_attention_e4m3.restype = ci
        lib.kvd_decode_attention_e4m3.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cf, cf, cf,
                                                  vp, sz, u32p, vp]
        lib.kvd_decode_step_e4m3.restype = ci
        lib.kvd_decode_step_e4m3.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cf, cf, cf,
                                             vp, sz, u32p, vp]
        lib.kvd_decode_attention_noalloc.restype = ci
        lib.kvd_decode_attention_noalloc.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cf,
                                                     ci, u32p, vp]
        lib.kvd_decode_plan.restype = ci
        lib.kvd_decode_plan.argtypes = [ci, ci, ci, ci, ci, ci, ci, ctypes.POINTER(PlanInfo)]
        lib.kvd_workspace_init.restype = ci
        lib.kvd_workspace_init.argtypes = [vp, sz, vp]
        lib.kvd_cache_bytes.restype = sz
        lib.kvd_cache_bytes.argtypes = [ci, ci, ci, ci, ci, ci]
        lib.kvd_status_string.restype = ctypes.c_char_p
        lib.kvd_status_string.argtypes = [ci]
        self._lib = lib
        self.path = path

    def __getattr__(self, name):
        return getattr(self._lib, name)


_lock = threading.Lock()
_loaded: Optional[_Lib] = None


def library_path() -> str:
    return _build.LIB_PATH


def load() -> _Lib:
    """Load ``libkvd.so``; raises if it has not been built."""
    global _loaded
    with _lock:
        if _loaded is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            _loaded = _Lib(path)
        return _loaded


class _Raw:
    def __getattr__(self, name):
        return getattr(load(), name)


raw = _Raw()


# ---------------------------------------------------------------------------------
def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


def _need_cuda(name: str, t: torch.Tensor, dtype=None) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _TORCH_DTYPE:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return _TORCH_DTYPE[t.dtype]


def _check(fn: str, status: int) -> None:
    if status != KVD_OK:
        raise KvdError(fn, status)


def kvd_append(k_cache, v_cache, k_new, v_new, past_len, max_past_len: int,
               err_word=None, stream=None) -> None:
    """Write ``k_new``/``v_new`` [B,H_kv,N,D] into slots ``past_len[b] + i`` of the caches."""
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache), ("k_new", k_new), ("v_new", v_new)):
        _need_cuda(n, t, k_cache.dtype)
    _need_cuda("past_len", past_len, torch.int32)
    if err_word is not None:
        _need_cuda("err_word", err_word, torch.int32)
    B, H_kv, T_max, D = k_cache.shape
    N = k_new.shape[2]
    if v_cache.shape != k_cache.shape or tuple(k_new.shape) != (B, H_kv, N, D) or v_new.shape != k_new.shape:
        raise ValueError("shape mismatch between caches and new K/V")
    if past_len.numel() != B:
        raise ValueError("past_len must hold B entries")
    st = raw.kvd_append(k_cache.data_ptr(), v_cache.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                        past_len.data_ptr(), B, H_kv, T_max, D, N, int(max_past_len),
                        _dtype_code(k_cache), _ptr(err_word), _stream_handle(stream))
    _check("kvd_append", st)


def kvd_decode_workspace_bytes(B: int, H_q: int, H_kv: int, D: int, N: int, max_past_len: int,
                               dtype) -> int:
    code = _NAME_DTYPE[dtype] if isinstance(dtype, str) else _TORCH_DTYPE[dtype]
    return int(raw.kvd_decode_workspace_bytes(B, H_q, H_kv, D, N, int(max_past_len), code))


def kvd_decode_plan(B: int, H_q: int, H_kv: int, D: int, N: int, max_past_len: int, dtype) -> dict:
    """The split-T plan kvd_decode_attention uses for these shapes on the current device.

    ``tensor_cores``: 0 the CUDA-core kernel, 1 the mma.sync tensor-core kernel (16-row
    blocks; 8-row blocks for E4M3 caches with at most 8 rows per KV head), 2 the tcgen05 kernel (128-row blocks, for more than 16 query rows per KV
    head); ``launches`` 2 when split heads are merged by the separate merge pass;
    ``early_start`` 1 for small layers (the next kernel on the stream may start early);
    ``cluster`` > 0 when such a layer runs as one thread-block cluster of that many CTAs
    per KV head."""
    code = _NAME_DTYPE[dtype] if isinstance(dtype, str) else _TORCH_DTYPE[dtype]
    info = PlanInfo()
    _check("kvd_decode_plan", raw.kvd_decode_plan(B, H_q, H_kv, D, N, int(max_past_len), code,
                                                  ctypes.byref(info)))
    return {k: getattr(info, k) for k, _ in PlanInfo._fields_}


def alloc_workspace(B, H_q, H_kv, D, N, max_past_len, dtype, device=None) -> Optional[torch.Tensor]:
    """A zero-filled device workspace sized for these shapes (None when none is needed)."""
    n = kvd_decode_workspace_bytes(B, H_q, H_kv, D, N, max_past_len, dtype)
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=device or torch.device("cuda"))


def kvd_workspace_init(workspace: Optional[torch.Tensor], stream=None) -> None:
    if workspace is None:
        return
    _check("kvd_workspace_init", raw.kvd_workspace_init(workspace.data_ptr(), workspace.numel(),
                                                        _stream_handle(stream)))


def kvd_decode_attention(q, k_cache, v_cache, out, past_len, max_past_len: int, scale: float = 0.0,
                         workspace: Optional[torch.Tensor] = None, err_word=None, stream=None) -> None:
    """Attention of the N new rows of ``q`` over the appended caches into ``out`` [B,H_q,N,D]."""
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("out", out)):
        _need_cuda(n, t, q.dtype)
    _need_cuda("past_len", past_len, torch.int32)
    if err_word is not None:
        _need_cuda("err_word", err_word, torch.int32)
    B, H_q, N, D = q.shape
    _, H_kv, T_max, _ = k_cache.shape
    if out.shape != q.shape or v_cache.shape != k_cache.shape or k_cache.shape[0] != B or k_cache.shape[3] != D:
        raise ValueError("shape mismatch between q, out and the caches")
    if past_len.numel() != B:
        raise ValueError("past_len must hold B entries")
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    st = raw.kvd_decode_attention(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(),
                                  past_len.data_ptr(), B, H_q, H_kv, T_max, D, N, int(max_past_len),
                                  float(scale), _dtype_code(q), ws_ptr, ws_bytes, _ptr(err_word),
                                  _stream_handle(stream))
    _check("kvd_decode_attention", st)


def kvd_decode_step(q, k_cache, v_cache, k_new, v_new, out, past_len, max_past_len: int,
                    scale: float = 0.0, workspace: Optional[torch.Tensor] = None, err_word=None,
                    stream=None, flags: Optional[int] = None) -> None:
    """Append ``k_new``/``v_new`` and attend the new rows of ``q`` in one launch.

    ``flags`` (e.g. ``KVD_STEP_HISTORY_STABLE``) calls ``kvd_decode_step_flags``
    with the caller's guarantees instead."""
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("k_new", k_new),
                 ("v_new", v_new), ("out", out)):
        _need_cuda(n, t, q.dtype)
    _need_cuda("past_len", past_len, torch.int32)
    if err_word is not None:
        _need_cuda("err_word", err_word, torch.int32)
    B, H_q, N, D = q.shape
    _, H_kv, T_max, _ = k_cache.shape
    if (out.shape != q.shape or v_cache.shape != k_cache.shape or k_cache.shape[0] != B
            or k_cache.shape[3] != D or tuple(k_new.shape) != (B, H_kv, N, D) or v_new.shape != k_new.shape):
        raise ValueError("shape mismatch between q, out, the caches and the new K/V")
    if past_len.numel() != B:
        raise ValueError("past_len must hold B entries")
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    if flags is not None:
        st = raw.kvd_decode_step_flags(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), k_new.data_ptr(),
                                       v_new.data_ptr(), out.data_ptr(), past_len.data_ptr(), B, H_q, H_kv,
                                       T_max, D, N, int(max_past_len), float(scale), _dtype_code(q), int(flags),
                                       ws_ptr, ws_bytes, _ptr(err_word), _stream_handle(stream))
        _check("kvd_decode_step_flags", st)
        return
    st = raw.kvd_decode_step(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), k_new.data_ptr(),
                             v_new.data_ptr(), out.data_ptr(), past_len.data_ptr(), B, H_q, H_kv, T_max, D,
                             N, int(max_past_len), float(scale), _dtype_code(q), ws_ptr, ws_bytes,
                             _ptr(err_word), _stream_handle(stream))
    _check("kvd_decode_step", st)


def kvd_host_staging_bytes(B, H_q, H_kv, D, N, dtype) -> int:
    return int(raw.kvd_host_staging_bytes(B, H_q, H_kv, D, N, _NAME_DTYPE[dtype] if isinstance(dtype, str)
                                          else _TORCH_DTYPE[dtype]))


def alloc_host_inputs(B, H_q, H_kv, D, N, dtype) -> dict:
    """One page-locked block for ``kvd_decode_step_host_packed`` (key ``block``) and
    views into it: q [B,H_q,N,D], k_new / v_new [B,H_kv,N,D] and past_len [B] (int32),
    laid out as the staging buffer's inputs."""
    tdt = dtype if isinstance(dtype, torch.dtype) else {"f32": torch.float32, "bf16": torch.bfloat16,
                                                         "f16": torch.float16}[dtype]
    code = _TORCH_DTYPE[tdt]
    n = int(raw.kvd_host_staging_inputs_bytes(B, H_q, H_kv, D, N, code))
    if n == 0:
        raise ValueError("no staging layout for these shapes / dtype")
    block = torch.zeros(n, dtype=torch.uint8).pin_memory()
    es = torch.tensor([], dtype=tdt).element_size()
    up = lambda x: (x + 255) // 256 * 256
    qb, nb = B * H_q * N * D * es, B * H_kv * N * D * es
    offs = {"q": 0, "k_new": up(qb), "v_new": up(qb) + up(nb), "past_len": up(qb) + 2 * up(nb)}
    out = {"block": block,
           "q": block[offs["q"]:offs["q"] + qb].view(tdt).view(B, H_q, N, D),
           "k_new": block[offs["k_new"]:offs["k_new"] + nb].view(tdt).view(B, H_kv, N, D),
           "v_new": block[offs["v_new"]:offs["v_new"] + nb].view(tdt).view(B, H_kv, N, D),
           "past_len": block[offs["past_len"]:offs["past_len"] + 4 * B].view(torch.int32)}
    return out


def alloc_host_staging(B, H_q, H_kv, D, N, dtype, device=None) -> torch.Tensor:
    """A device staging buffer for ``kvd_decode_step_host`` with these shapes."""
    n = kvd_host_staging_bytes(B, H_q, H_kv, D, N, dtype)
    if n == 0:
        raise ValueError("no staging layout for these shapes / dtype")
    return torch.empty(n, dtype=torch.uint8, device=device or torch.device("cuda"))


def _need_pinned(name, t, dtype):
    if t.is_cuda or not (t.is_pinned() or (t._base is not None and t._base.is_pinned())) or t.dtype != dtype \
            or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous page-locked host tensor of dtype {dtype}")


def kvd_decode_step_host(q_host, k_cache, v_cache, k_new_host, v_new_host, out_host, past_len_host,
                         max_past_len: int, staging: torch.Tensor, scale: float = 0.0,
                         workspace: Optional[torch.Tensor] = None, err_word=None, stream=None) -> None:
    """``kvd_decode_step`` with q, k_new, v_new, past_len and out in page-locked host memory:
    the library copies them through ``staging`` (device) on the stream."""
    dt = q_host.dtype
    for n, t in (("q_host", q_host), ("k_new_host", k_new_host), ("v_new_host", v_new_host),
                 ("out_host", out_host)):
        _need_pinned(n, t, dt)
    _need_pinned("past_len_host", past_len_host, torch.int32)
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _need_cuda(n, t, dt)
    if staging.device.type != "cuda" or not staging.is_contiguous():
        raise ValueError("staging must be a contiguous CUDA tensor")
    if err_word is not None:
        _need_cuda("err_word", err_word, torch.int32)
    B, H_q, N, D = q_host.shape
    _, H_kv, T_max, _ = k_cache.shape
    if (out_host.shape != q_host.shape or v_cache.shape != k_cache.shape or k_cache.shape[0] != B
            or k_cache.shape[3] != D or tuple(k_new_host.shape) != (B, H_kv, N, D)
            or v_new_host.shape != k_new_host.shape):
        raise ValueError("shape mismatch between q, out, the caches and the new K/V")
    if past_len_host.numel() != B:
        raise ValueError("past_len must hold B entries")
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    st = raw.kvd_decode_step_host(q_host.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), k_new_host.data_ptr(),
                                  v_new_host.data_ptr(), out_host.data_ptr(), past_len_host.data_ptr(), B, H_q,
                                  H_kv, T_max, D, N, int(max_past_len), float(scale), _TORCH_DTYPE[dt],
                                  staging.data_ptr(), staging.numel() * staging.element_size(), ws_ptr, ws_bytes,
                                  _ptr(err_word), _stream_handle(stream))
    _check("kvd_decode_step_host", st)


def kvd_decode_step_host_packed(host_inputs: dict, k_cache, v_cache, out_host, max_past_len: int,
                                staging: torch.Tensor, scale: float = 0.0, workspace: Optional[torch.Tensor] = None,
                                err_word=None, stream=None) -> None:
    """``kvd_decode_step_host`` with the inputs in the one block of ``alloc_host_inputs``
    (copied to the device in one piece)."""
    q = host_inputs["q"]
    dt = q.dtype
    block = host_inputs["block"]
    if block.is_cuda or not block.is_pinned() or block.dtype != torch.uint8:
        raise ValueError("host_inputs must come from alloc_host_inputs")
    _need_pinned("out_host", out_host, dt)
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _need_cuda(n, t, dt)
    if staging.device.type != "cuda" or not staging.is_contiguous():
        raise ValueError("staging must be a contiguous CUDA tensor")
    if err_word is not None:
        _need_cuda("err_word", err_word, torch.int32)
    B, H_q, N, D = q.shape
    _, H_kv, T_max, _ = k_cache.shape
    if out_host.shape != q.shape or v_cache.shape != k_cache.shape or k_cache.shape[0] != B or k_cache.shape[3] != D \
            or tuple(host_inputs["k_new"].shape) != (B, H_kv, N, D):
        raise ValueError("shape mismatch between the inputs, out and the caches")
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    st = raw.kvd_decode_step_host_packed(block.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out_host.data_ptr(),
                                         B, H_q, H_kv, T_max, D, N, int(max_past_len), float(scale), _TORCH_DTYPE[dt],
                                         staging.data_ptr(), staging.numel() * staging.element_size(), ws_ptr,
                                         ws_bytes, _ptr(err_word), _stream_handle(stream))
    _check("kvd_decode_step_host_packed", st)


# ---------------------------------------------------------------------------------
# paged cache: k_pages / v_pages [num_pages, H_kv, page_size, D], block_table int32 [B, max_pages]
def _paged_geometry(k_pages, v_pages, block_table, B: int):
    _need_cuda("block_table", block_table, torch.int32)
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_pages]")
    if v_pages.shape != k_pages.shape or k_pages.dim() != 4:
        raise ValueError("k_pages and v_pages must be the same [num_pages, H_kv, page_size, D]")
    num_pages, H_kv, page_size, D = k_pages.shape
    return num_pages, H_kv, page_size, D, block_table.shape[1]


def kvd_paged_append(k_pages, v_pages, k_new, v_new, block_table, past_len, max_past_len: int,
                     err_word=None, stream=None) -> None:
    """Write ``k_new``/``v_new`` [B,H_kv,N,D] into the page slots of tokens ``past_len[b] + i``."""
    for n, t in (("k_pages", k_pages), ("v_pages", v_pages), ("k_new", k_new), ("v_new", v_new)):
        _need_cuda(n, t, k_pages.dtype)
    _need_cuda("past_len", past_len, torch.int32)
    if err_word is not None:
        _need_cuda("err_word", err_word, torch.int32)
    B, _, N, _ = k_new.shape
    num_pages, H_kv, page_size, D, max_pages = _paged_geometry(k_pages, v_pages, block_table, B)
    if tuple(k_new.shape) != (B, H_kv, N, D) or v_new.shape != k_new.shape:
        raise ValueError("shape mismatch between the pages and the new K/V")
    if past_len.numel() != B:
        raise ValueError("past_len must hold B entries")
    st = raw.kvd_paged_append(k_pages.data_ptr(), v_pages.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                              block_table.data_ptr(), past_len.data_ptr(), B, H_kv, D, N, page_size,
                              max_pages, num_pages, int(max_past_len), _dtype_code(k_pages), _ptr(err_word),
                              _stream_handle(stream))
    _check("kvd_paged_append", st)


def kvd_paged_decode_attention(q, k_pages, v_pages, out, block_table, past_len, max_past_len: int,
                               scale: float = 0.0, workspace: Optional[torch.Tensor] = None,
                               err_word=None, stream=None) -> None:
    """kvd_decode_attention over a paged cache (workspace from alloc_workspace, same shapes)."""
    for n, t in (("q", q), ("k_pages", k_pages), ("v_pages", v_pages), ("out", out)):
        _need_cuda(n, t, q.dtype)
    _need_cuda("past_len", past_len, torch.int32)
    if err_word is not None:
        _need_cuda("err_word", err_word, torch.int32)
    B, H_q, N, D = q.shape
    num_pages, H_kv, page_size, Dp, max_pages = _paged_geometry(k_pages, v_pages, block_table, B)
    if out.shape != q.shape or Dp != D:
        raise ValueError("shape mismatch between q, out and the pages")
    if past_len.numel() != B:
        raise ValueError("past_len must hold B entries")
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    st = raw.kvd_paged_decode_attention(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), out.data_ptr(),
                                        block_table.data_ptr(), past_len.data_ptr(), B, H_q, H_kv, D, N,
                                        page_size, max_pages, num_pages, int(max_past_len), float(scale),
                                        _dtype_code(q), ws_ptr, ws_bytes, _ptr(err_word), _stream_handle(stream))
    _check("kvd_paged_decode_attention", st)


def kvd_paged_decode_step(q, k_pages, v_pages, k_new, v_new, out, block_table, past_len, max_past_len: int,
                          scale: float = 0.0, workspace: Optional[torch.Tensor] = None, err_word=None,
                          stream=None) -> None:
    """kvd_decode_step over a paged cache: append into the page slots and attend, one launch."""
    for n, t in (("q", q), ("k_pages", k_pages), ("v_pages", v_pages), ("k_new", k_new),
                 ("v_new", v_new), ("out", out)):
        _need_cuda(n, t, q.dtype)
    _need_cuda("past_len", past_len, torch.int32)
    if err_word is not None:
        _need_cuda("err_word", err_word, torch.int32)
    B, H_q, N, D = q.shape
    num_pages, H_kv, page_size, Dp, max_pages = _paged_geometry(k_pages, v_pages, block_table, B)
    if out.shape != q.shape or Dp != D or tuple(k_new.shape) != (B, H_kv, N, D) or v_new.shape != k_new.shape:
        raise ValueError("shape mismatch between q, out, the pages and the new K/V")
    if past_len.numel() != B:
        raise ValueError("past_len must hold B entries")
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    st = raw.kvd_paged_decode_step(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), k_new.data_ptr(),
                                   v_new.data_ptr(), out.data_ptr(), block_table.data_ptr(), past_len.data_ptr(),
                                   B, H_q, H_kv, D, N, page_size, max_pages, num_pages, int(max_past_len),
                                   float(scale), _dtype_code(q), ws_ptr, ws_bytes, _ptr(err_word),
                                   _stream_handle(stream))
    _check("kvd_paged_decode_step", st)


# ---------------------------------------------------------------------------------
# E4M3 cache: k_cache / v_cache uint8 [B,H_kv,T_max,D] codes; q, new K/V, out bf16
def _need_e4m3_cache(name: str, t: torch.Tensor) -> None:
    """An E4M3 cache: uint8 codes or torch.float8_e4m3fn (the same bytes)."""
    _need_cuda(name, t)
    if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise ValueError(f"{name} must be uint8 E4M3 codes or float8_e4m3fn, got {t.dtype}")


def kvd_append_e4m3(k_cache, v_cache, k_new, v_new, past_len, max_past_len: int, k_scale: float,
                    v_scale: float, err_word=None, stream=None) -> None:
    """Quantize ``k_new``/``v_new`` [B,H_kv,N,D] (fp32, bf16 or fp16) into E4M3 slots ``past_len[b] + i``."""
    _need_e4m3_cache("k_cache", k_cache)
    _need_e4m3_cache("v_cache", v_cache)
    for n, t in (("k_new", k_new), ("v_new", v_new)):
        _need_cuda(n, t, k_new.dtype)
    _need_cuda("past_len", past_len, torch.int32)
    if err_word is not None:
        _need_cuda("err_word", err_word, torch.int32)
    B, H_kv, T_max, D = k_cache.shape
    N = k_new.shape[2]
    if v_cache.shape != k_cache.shape or tuple(k_new.shape) != (B, H_kv, N, D) or v_new.shape != k_new.shape:
        raise ValueError("shape mismatch between caches and new K/V")
    if past_len.numel() != B:
        raise ValueError("past_len must hold B entries")
    st = raw.kvd_append_e4m3(k_cache.data_ptr(), v_cache.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                             past_len.data_ptr(), B, H_kv, T_max, D, N, int(max_past_len), _dtype_code(k_new),
                             float(k_scale), float(v_scale), _ptr(err_word), _stream_handle(stream))
    _check("kvd_append_e4m3", st)


def kvd_decode_attention_e4m3(q, k_cache, v_cache, out, past_len, max_past_len: int, k_scale: float,
                              v_scale: float, scale: float = 0.0, workspace: Optional[torch.Tensor] = None,
                              err_word=None, stream=None) -> None:
    """Attention of the bf16 rows of ``q`` over E4M3 caches (workspace: alloc_workspace(..., "e4m3"))."""
    for n, t in (("q", q), ("out", out)):
        _need_cuda(n, t, torch.bfloat16)
    _need_e4m3_cache("k_cache", k_cache)
    _need_e4m3_cache("v_cache", v_cache)
    _need_cuda("past_len", past_len, torch.int32)
    if err_word is not None:
        _need_cuda("err_word", err_word, torch.int32)
    B, H_q, N, D = q.shape
    _, H_kv, T_max, _ = k_cache.shape
    if out.shape != q.shape or v_cache.shape != k_cache.shape or k_cache.shape[0] != B or k_cache.shape[3] != D:
        raise ValueError("shape mismatch between q, out and the caches")
    if past_len.numel() != B:
        raise ValueError("past_len must hold B entries")
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    st = raw.kvd_decode_attention_e4m3(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(),
                                       past_len.data_ptr(), B, H_q, H_kv, T_max, D, N, int(max_past_len),
                                       float(scale), float(k_scale), float(v_scale), ws_ptr, ws_bytes,
                                       _ptr(err_word), _stream_handle(stream))
    _check("kvd_decode_attention_e4m3", st)


def kvd_decode_step_e4m3(q, k_cache, v_cache, k_new, v_new, out, past_len, max_past_len: int, k_scale: float,
                         v_scale: float, scale: float = 0.0, workspace: Optional[torch.Tensor] = None,
                         err_word=None, stream=None) -> None:
    """kvd_decode_step over E4M3 caches: quantize the bf16 new rows into their slots and attend, one launch."""
    for n, t in (("q", q), ("k_new", k_new), ("v_new", v_new), ("out", out)):
        _need_cuda(n, t, torch.bfloat16)
    _need_e4m3_cache("k_cache", k_cache)
    _need_e4m3_cache("v_cache", v_cache)
    _need_cuda("past_len", past_len, torch.int32)
    if err_word is not None:
        _need_cuda("err_word", err_word, torch.int32)
    B, H_q, N, D = q.shape
    _, H_kv, T_max, _ = k_cache.shape
    if (out.shape != q.shape or v_cache.shape != k_cache.shape or k_cache.shape[0] != B
            or k_cache.shape[3] != D or tuple(k_new.shape) != (B, H_kv, N, D) or v_new.shape != k_new.shape):
        raise ValueError("shape mismatch between q, out, the caches and the new K/V")
    if past_len.numel() != B:
        raise ValueError("past_len must hold B entries")
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    st = raw.kvd_decode_step_e4m3(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), k_new.data_ptr(),
                                  v_new.data_ptr(), out.data_ptr(), past_len.data_ptr(), B, H_q, H_kv, T_max, D,
                                  N, int(max_past_len), float(scale), float(k_scale), float(v_scale), ws_ptr,
                                  ws_bytes, _ptr(err_word), _stream_handle(stream))
    _check("kvd_decode_step_e4m3", st)


def kvd_decode_attention_noalloc(q, k_cache, v_cache, out, past_len, max_past_len: int,
                                 scale: float = 0.0, err_word=None, stream=None) -> None:
    """kvd_decode_attention with the library's built-in 4 MiB scratch instead of a workspace.

    For callers that cannot allocate device memory where they call; calls whose
    GPU work may overlap must not use it concurrently (they share the scratch).
    """
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("out", out)):
        _need_cuda(n, t, q.dtype)
    _need_cuda("past_len", past_len, torch.int32)
    if err_word is not None:
        _need_cuda("err_word", err_word, torch.int32)
    B, H_q, N, D = q.shape
    _, H_kv, T_max, _ = k_cache.shape
    if out.shape != q.shape or v_cache.shape != k_cache.shape or k_cache.shape[0] != B or k_cache.shape[3] != D:
        raise ValueError("shape mismatch between q, out and the caches")
    if past_len.numel() != B:
        raise ValueError("past_len must hold B entries")
    st = raw.kvd_decode_attention_noalloc(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                          out.data_ptr(), past_len.data_ptr(), B, H_q, H_kv, T_max, D, N,
                                          int(max_past_len), float(scale), _dtype_code(q), _ptr(err_word),
                                          _stream_handle(stream))
    _check("kvd_decode_attention_noalloc", st)


def kvd_cache_bytes(L: int, B: int, H_kv: int, D: int, T: int, dtype) -> int:
    code = _NAME_DTYPE[dtype] if isinstance(dtype, str) else _TORCH_DTYPE[dtype]
    return int(raw.kvd_cache_bytes(L, B, H_kv, D, T, code))


def kvd_status_string(status: int) -> str:
    return raw.kvd_status_string(int(status)).decode()

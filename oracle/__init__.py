"""ctypes wrapper around the plain CPU oracle (``oracle/oracle.c``).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product package
(``kv_cache_decode_append_gb300``) never imports it and shares no code with it.

Arrays are numpy: fp32 data as ``float32``, bf16 and fp16 data as ``uint16``
holding the raw bits.  Outputs of the attention routines are ``float64``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

F32, BF16, F16, E4M3 = 0, 1, 2, 3
_DTYPES = {"f32": F32, "bf16": BF16, "f16": F16, "e4m3": E4M3}

_lock = threading.Lock()
_lib = None


def compile_library(src: str = _SRC, out: str = LIB_PATH, extra_flags=()) -> str:
    """Compile ``src`` with gcc into the shared library ``out`` and return its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", *extra_flags,
           "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build() -> str:
    """Build ``liboracle.so`` if it is missing or older than ``oracle.c``."""
    if (not os.path.exists(LIB_PATH)
            or os.path.getmtime(LIB_PATH) < os.path.getmtime(_SRC)):
        compile_library()
    return LIB_PATH


class Oracle:
    """Typed entry points of one compiled oracle library (the real one or a test mutant)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        vp, i32p, dp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_double)
        ci, cd, cll = ctypes.c_int, ctypes.c_double, ctypes.c_longlong
        lib.oracle_cache_bytes.restype = ctypes.c_ulonglong
        lib.oracle_cache_bytes.argtypes = [cll] * 6
        lib.oracle_max_threads.restype = ci
        lib.oracle_max_threads.argtypes = []
        lib.oracle_set_threads.restype = None
        lib.oracle_set_threads.argtypes = [ci]
        lib.oracle_append.restype = ci
        lib.oracle_append.argtypes = [vp, vp, vp, vp, i32p, ci, ci, ci, ci, ci, ci]
        lib.oracle_decode_attention.restype = ci
        lib.oracle_decode_attention.argtypes = [vp, vp, vp, dp, i32p, ci, ci, ci, ci, ci, ci, cd, ci]
        lib.oracle_paged_append.restype = ci
        lib.oracle_paged_append.argtypes = [vp, vp, vp, vp, i32p, i32p, ci, ci, ci, ci, ci, ci, ci, ci]
        lib.oracle_paged_decode_attention.restype = ci
        lib.oracle_paged_decode_attention.argtypes = [vp, vp, vp, dp, i32p, i32p, ci, ci, ci, ci, ci, ci,
                                                      ci, ci, cd, ci]
        u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.oracle_append_e4m3.restype = ci
        lib.oracle_append_e4m3.argtypes = [u8p, u8p, vp, vp, i32p, ci, ci, ci, ci, ci, ci, ctypes.c_float,
                                           ctypes.c_float]
        lib.oracle_decode_attention_e4m3.restype = ci
        lib.oracle_decode_attention_e4m3.argtypes = [vp, u8p, u8p, dp, i32p, ci, ci, ci, ci, ci, ci, cd, ci,
                                                     cd, cd]
        lib.oracle_quantize_e4m3.restype = ci
        lib.oracle_quantize_e4m3.argtypes = [ctypes.POINTER(ctypes.c_float), u8p, cll]
        lib.oracle_widen.restype = ci
        lib.oracle_widen.argtypes = [vp, dp, cll, ci]
        lib.oracle_full_causal_attention.restype = ci
        lib.oracle_full_causal_attention.argtypes = [dp, dp, dp, dp, ci, ci, cd]
        self.lib = lib
        self.path = path

    # -- helpers ---------------------------------------------------------------
    @staticmethod
    def _check(arr: np.ndarray, dtype: str, name: str) -> None:
        want = {"f32": np.float32, "e4m3": np.uint8}.get(dtype, np.uint16)
        if arr.dtype != want:
            raise TypeError(f"{name}: expected {np.dtype(want)} for {dtype}, got {arr.dtype}")
        if not arr.flags.c_contiguous:
            raise ValueError(f"{name} must be C-contiguous")

    # -- entry points --------------------------------------------------------------
    def widen(self, arr: np.ndarray, dtype: str) -> np.ndarray:
        """The stored values of ``arr`` (oracle representation) as float64."""
        self._check(arr, dtype, "arr")
        out = np.empty(arr.shape, dtype=np.float64)
        if self.lib.oracle_widen(arr.ctypes.data, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                 arr.size, _DTYPES[dtype]) != 0:
            raise ValueError("oracle_widen rejected its arguments")
        return out

    def quantize_e4m3(self, x: np.ndarray) -> np.ndarray:
        """E4M3 codes (uint8) of float32 values: nearest, ties to even, saturating at 448."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty(x.shape, dtype=np.uint8)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        if self.lib.oracle_quantize_e4m3(x.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                         out.ctypes.data_as(u8p), x.size) != 0:
            raise ValueError("oracle_quantize_e4m3 rejected its arguments")
        return out

    def append_e4m3(self, k_cache, v_cache, k_new, v_new, past_len, new_dtype: str, k_scale: float,
                    v_scale: float) -> int:
        """In place on the uint8 E4M3 caches [B,H_kv,T_max,D]; returns the status."""
        self._check(k_cache, "e4m3", "k_cache")
        self._check(v_cache, "e4m3", "v_cache")
        self._check(k_new, new_dtype, "k_new")
        self._check(v_new, new_dtype, "v_new")
        past_len = np.ascontiguousarray(past_len, dtype=np.int32)
        B, H_kv, T_max, D = k_cache.shape
        N = k_new.shape[2]
        if v_cache.shape != k_cache.shape or k_new.shape != (B, H_kv, N, D) or v_new.shape != k_new.shape:
            raise ValueError("shape mismatch")
        u8p = ctypes.POINTER(ctypes.c_uint8)
        return int(self.lib.oracle_append_e4m3(
            k_cache.ctypes.data_as(u8p), v_cache.ctypes.data_as(u8p), k_new.ctypes.data, v_new.ctypes.data,
            past_len.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), B, H_kv, T_max, D, N,
            _DTYPES[new_dtype], float(k_scale), float(v_scale)))

    def decode_attention_e4m3(self, q, k_cache, v_cache, past_len, q_dtype: str, k_scale: float,
                              v_scale: float, scale=None):
        """Returns ``(out float64 [B,H_q,N,D], status)`` over appended E4M3 caches."""
        self._check(q, q_dtype, "q")
        self._check(k_cache, "e4m3", "k_cache")
        self._check(v_cache, "e4m3", "v_cache")
        past_len = np.ascontiguousarray(past_len, dtype=np.int32)
        B, H_q, N, D = q.shape
        _, H_kv, T_max, _ = k_cache.shape
        if scale is None:
            scale = 1.0 / np.sqrt(D)
        out = np.empty((B, H_q, N, D), dtype=np.float64)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        st = self.lib.oracle_decode_attention_e4m3(
            q.ctypes.data, k_cache.ctypes.data_as(u8p), v_cache.ctypes.data_as(u8p),
            out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
            past_len.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            B, H_q, H_kv, T_max, D, N, float(scale), _DTYPES[q_dtype], float(k_scale), float(v_scale))
        return out, int(st)

    def cache_bytes(self, L, B, H_kv, D, T, bytes_per_elem) -> int:
        return int(self.lib.oracle_cache_bytes(L, B, H_kv, D, T, bytes_per_elem))

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def set_threads(self, n: int) -> None:
        self.lib.oracle_set_threads(int(n))

    def append(self, k_cache, v_cache, k_new, v_new, past_len, dtype: str) -> int:
        """In place on ``k_cache``/``v_cache`` ([B,H_kv,T_max,D]); returns the status."""
        for a, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (k_new, "k_new"), (v_new, "v_new")):
            self._check(a, dtype, n)
        past_len = np.ascontiguousarray(past_len, dtype=np.int32)
        B, H_kv, T_max, D = k_cache.shape
        N = k_new.shape[2]
        if v_cache.shape != k_cache.shape or k_new.shape != (B, H_kv, N, D) or v_new.shape != k_new.shape:
            raise ValueError("shape mismatch")
        return int(self.lib.oracle_append(
            k_cache.ctypes.data, v_cache.ctypes.data, k_new.ctypes.data, v_new.ctypes.data,
            past_len.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            B, H_kv, T_max, D, N, _DTYPES[dtype]))

    def decode_attention(self, q, k_cache, v_cache, past_len, dtype: str, scale=None):
        """Returns ``(out float64 [B,H_q,N,D], status)`` for an already-appended cache."""
        for a, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
            self._check(a, dtype, n)
        past_len = np.ascontiguousarray(past_len, dtype=np.int32)
        B, H_q, N, D = q.shape
        _, H_kv, T_max, _ = k_cache.shape
        if scale is None:
            scale = 1.0 / np.sqrt(D)
        out = np.empty((B, H_q, N, D), dtype=np.float64)
        st = self.lib.oracle_decode_attention(
            q.ctypes.data, k_cache.ctypes.data, v_cache.ctypes.data,
            out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
            past_len.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            B, H_q, H_kv, T_max, D, N, float(scale), _DTYPES[dtype])
        return out, int(st)

    def paged_append(self, k_pages, v_pages, k_new, v_new, block_table, past_len, dtype: str) -> int:
        """In place on ``k_pages``/``v_pages`` ([num_pages,H_kv,page_size,D]); returns the status."""
        for a, n in ((k_pages, "k_pages"), (v_pages, "v_pages"), (k_new, "k_new"), (v_new, "v_new")):
            self._check(a, dtype, n)
        past_len = np.ascontiguousarray(past_len, dtype=np.int32)
        block_table = np.ascontiguousarray(block_table, dtype=np.int32)
        num_pages, H_kv, page_size, D = k_pages.shape
        B, max_pages = block_table.shape
        N = k_new.shape[2]
        if v_pages.shape != k_pages.shape or k_new.shape != (B, H_kv, N, D) or v_new.shape != k_new.shape:
            raise ValueError("shape mismatch")
        i32 = ctypes.POINTER(ctypes.c_int32)
        return int(self.lib.oracle_paged_append(
            k_pages.ctypes.data, v_pages.ctypes.data, k_new.ctypes.data, v_new.ctypes.data,
            block_table.ctypes.data_as(i32), past_len.ctypes.data_as(i32),
            B, H_kv, D, N, page_size, max_pages, num_pages, _DTYPES[dtype]))

    def paged_decode_attention(self, q, k_pages, v_pages, block_table, past_len, dtype: str, scale=None):
        """Returns ``(out float64 [B,H_q,N,D], status)`` for an already-appended paged cache."""
        for a, n in ((q, "q"), (k_pages, "k_pages"), (v_pages, "v_pages")):
            self._check(a, dtype, n)
        past_len = np.ascontiguousarray(past_len, dtype=np.int32)
        block_table = np.ascontiguousarray(block_table, dtype=np.int32)
        B, H_q, N, D = q.shape
        num_pages, H_kv, page_size, _ = k_pages.shape
        max_pages = block_table.shape[1]
        if scale is None:
            scale = 1.0 / np.sqrt(D)
        out = np.empty((B, H_q, N, D), dtype=np.float64)
        i32 = ctypes.POINTER(ctypes.c_int32)
        st = self.lib.oracle_paged_decode_attention(
            q.ctypes.data, k_pages.ctypes.data, v_pages.ctypes.data,
            out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
            block_table.ctypes.data_as(i32), past_len.ctypes.data_as(i32),
            B, H_q, H_kv, D, N, page_size, max_pages, num_pages, float(scale), _DTYPES[dtype])
        return out, int(st)

    def full_causal_attention(self, qf, kf, vf, scale):
        """Causal self-attention of one head: float64 [T,D] inputs, float64 [T,D] output."""
        qf, kf, vf = (np.ascontiguousarray(x, dtype=np.float64) for x in (qf, kf, vf))
        T, D = qf.shape
        out = np.empty((T, D), dtype=np.float64)
        dp = ctypes.POINTER(ctypes.c_double)
        st = self.lib.oracle_full_causal_attention(
            qf.ctypes.data_as(dp), kf.ctypes.data_as(dp), vf.ctypes.data_as(dp),
            out.ctypes.data_as(dp), T, D, float(scale))
        if st != 0:
            raise ValueError("oracle_full_causal_attention rejected its arguments")
        return out


def load() -> Oracle:
    """The oracle built from ``oracle.c`` (compiled on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
        return _lib

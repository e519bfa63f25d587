"""ctypes wrapper over the FP64 CPU oracle (TEST INFRASTRUCTURE ONLY).

Only the tests, the smoke check and the benchmark's CPU-baseline leg import this
module.  It loads ``libqsa_oracle.so`` (built from ``qsa_oracle.c``) and shares
nothing with the CUDA path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from . import build_oracle

_P = ctypes.c_void_p
_I = ctypes.c_int32
_lib_cache = {}


def load(path: Optional[str] = None):
    """Load (building first if needed) an oracle library; cached per path."""
    path = path or build_oracle.build()
    if path in _lib_cache:
        return _lib_cache[path]
    lib = ctypes.CDLL(os.path.abspath(path))
    lib.qsa_ref_half_to_double.argtypes = [ctypes.c_uint16]
    lib.qsa_ref_half_to_double.restype = ctypes.c_double
    lib.qsa_ref_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.qsa_ref_bf16_to_double.restype = ctypes.c_double
    lib.qsa_ref_union.argtypes = [_P, _P, _I, _I, _P, _P, _P, _I]
    lib.qsa_ref_union.restype = ctypes.c_int
    lib.qsa_attn_ref.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _I, _I, _P, _I,
                                 ctypes.c_double, _P, _I]
    lib.qsa_attn_ref.restype = ctypes.c_int
    lib.qsa_ref_max_threads.argtypes = []
    lib.qsa_ref_max_threads.restype = ctypes.c_int
    _lib_cache[path] = lib
    return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads(lib=None) -> int:
    return int((lib or load()).qsa_ref_max_threads())


def half_to_double(bits: np.ndarray, lib=None) -> np.ndarray:
    lib = lib or load()
    return np.array([lib.qsa_ref_half_to_double(int(b)) for b in np.asarray(bits).ravel()])


def bf16_to_double(bits: np.ndarray, lib=None) -> np.ndarray:
    lib = lib or load()
    return np.array([lib.qsa_ref_bf16_to_double(int(b)) for b in np.asarray(bits).ravel()])


def union_ref(sel: np.ndarray, sel_count: np.ndarray, ustride: int = 16448, lib=None):
    """Sorted union per group of 8 queries -> (cells [G, ustride], masks, counts [G])."""
    lib = lib or load()
    sel = _c(sel, np.int32)
    cnt = _c(sel_count, np.int32)
    n_q = int(cnt.shape[0])
    n_groups = (n_q + 7) // 8
    ucell = np.full((n_groups, ustride), -1, dtype=np.int32)
    umask = np.zeros((n_groups, ustride), dtype=np.uint8)
    ucount = np.zeros(n_groups, dtype=np.int32)
    rc = lib.qsa_ref_union(_ptr(sel), _ptr(cnt), n_q, int(sel.shape[1]) if sel.ndim == 2 else 1,
                           _ptr(ucell), _ptr(umask), _ptr(ucount), int(ustride))
    if rc != 0:
        raise RuntimeError(f"qsa_ref_union failed with status {rc}")
    return ucell, umask, ucount


def attn_ref(q, k_pool, v_pool, k_scale, v_scale, page_table, sel, sel_count, n_kv,
             sm_scale: float, q_index=None, n_threads: int = 0, lib=None) -> np.ndarray:
    """FP64 per-position selected-cell attention -> out [rows, n_kv*12, 128] float64."""
    lib = lib or load()
    q = _c(q, np.uint16)
    k_pool = _c(k_pool, np.int8)
    v_pool = _c(v_pool, np.int8)
    ks = _c(np.asarray(k_scale).view(np.uint16) if np.asarray(k_scale).dtype == np.float16 else k_scale, np.uint16)
    vs = _c(np.asarray(v_scale).view(np.uint16) if np.asarray(v_scale).dtype == np.float16 else v_scale, np.uint16)
    pt = _c(page_table, np.int32)
    sel = _c(sel, np.int32)
    cnt = _c(sel_count, np.int32)
    n_q = int(cnt.shape[0])
    n_heads = int(n_kv) * 12
    idx = None if q_index is None else _c(q_index, np.int32)
    n_rows = n_q if idx is None else int(idx.shape[0])
    out = np.zeros((n_rows, n_heads, 128), dtype=np.float64)
    n_ppages = int(k_pool.shape[0])
    rc = lib.qsa_attn_ref(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(ks), _ptr(vs), _ptr(pt),
                          int(pt.shape[0]), n_ppages, int(n_kv), _ptr(sel), _ptr(cnt),
                          int(sel.shape[1]), n_q, _ptr(idx), 0 if idx is None else int(idx.shape[0]),
                          float(sm_scale), _ptr(out), int(n_threads))
    if rc != 0:
        raise RuntimeError(f"qsa_attn_ref failed with status {rc}")
    return out


def attn_ref_workload(wl, q_index=None, n_threads: int = 0, lib=None) -> np.ndarray:
    """Convenience: run the oracle on a generator Workload."""
    return attn_ref(wl.q, wl.k_pool, wl.v_pool, wl.k_scale, wl.v_scale, wl.page_table,
                    wl.sel, wl.sel_count, wl.n_kv, wl.sm_scale, q_index=q_index,
                    n_threads=n_threads, lib=lib)

"""Thin ctypes binding over libqsa.so (include/qsa.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  There is no
CPU fallback: when the library is missing the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import gen

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libqsa.so")

QSA_OK, QSA_ERR_ARG, QSA_ERR_UNSUPPORTED, QSA_ERR_CAPACITY, QSA_ERR_CUDA, QSA_ERR_DEVICE_CHECK = range(6)
ATTN_DEFAULT, ATTN_TCGEN05, ATTN_TCGEN05_SM = 0, 1, 2
DEV_BITS = {1: "bad selection count", 2: "union overflow", 4: "bad cell", 8: "bad page-table entry",
            16: "bad union count", 32: "device wait timeout"}

_lib = None
_P, _I, _F, _S = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t


class QsaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status} ({lib().qsa_status_str(status).decode()})")
        self.status = status


def lib():
    """Load libqsa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                               "g.build()'` (no CPU fallback exists)")
        L = ctypes.CDLL(LIB_PATH)
        L.qsa_attn_default_variant.argtypes = []
        L.qsa_attn_default_variant.restype = ctypes.c_int
        L.qsa_status_str.argtypes = [ctypes.c_int]
        L.qsa_status_str.restype = ctypes.c_char_p
        L.qsa_union_workspace_bytes.argtypes = [_I, _I]
        L.qsa_union_workspace_bytes.restype = _S
        L.qsa_union_build.argtypes = [_P, _P, _I, _I, _P, _P, _P, _I, _P, _P]
        L.qsa_union_build.restype = ctypes.c_int
        L.qsa_union_attn.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _I, _I, _F, _P, _I, _P, _P]
        L.qsa_union_attn.restype = ctypes.c_int
        L.qsa_prompt_attn.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _I, _I, _F, _P, _P, _S, _I, _I,
                                      _P, _P]
        L.qsa_prompt_attn.restype = ctypes.c_int
        L.qsa_prompt_attn_static.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _I, _I, _F, _P, _I, _I,
                                             _P, _P]
        L.qsa_prompt_attn_static.restype = ctypes.c_int
        L.qsa_fused_attn.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _I, _I, _F, _P, _P, _P]
        L.qsa_fused_attn.restype = ctypes.c_int
        L.qsa_select_attn.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _I, _I, _F, _P, _P, _P]
        L.qsa_select_attn.restype = ctypes.c_int
        L.qsa_decode_attn.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _I, _F, _P, _P, _P]
        L.qsa_decode_attn.restype = ctypes.c_int
        L.qsa_wait_selftest.argtypes = [_I, _P, _P]
        L.qsa_wait_selftest.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t: torch.Tensor, name: str, dtypes) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


_B16 = (torch.bfloat16, torch.int16, torch.uint16)
_H16 = (torch.float16, torch.int16, torch.uint16)


def _attn_inputs(q, k_pool, v_pool, k_scale, v_scale, page_table, out):
    """Device, dtype and shape checks shared by the attention calls; returns out
    (allocated here when not given: float32 [n_q, n_kv*12, 128])."""
    _dev(q, "q", _B16)
    _dev(k_pool, "k_pool", (torch.int8,))
    _dev(v_pool, "v_pool", (torch.int8,))
    _dev(k_scale, "k_scale", _H16)
    _dev(v_scale, "v_scale", _H16)
    _dev(page_table, "page_table", (torch.int32,))
    if q.dim() != 3 or q.shape[2] != gen.HEAD_DIM or q.shape[1] % gen.HEADS_PER_KV != 0:
        raise ValueError(f"q must be [n_q, n_kv*12, 128], got {tuple(q.shape)}")
    shape = (int(q.shape[0]), int(q.shape[1]), gen.HEAD_DIM)
    if out is None:
        return torch.empty(shape, dtype=torch.float32, device=q.device)
    _dev(out, "out", (torch.float32,))
    if tuple(out.shape) != shape:
        raise ValueError(f"out must have shape {shape}, got {tuple(out.shape)}")
    return out


def _check(fn: str, rc: int):
    if rc != QSA_OK:
        raise QsaError(fn, rc)


def default_variant() -> int:
    """The attention variant QSA_ATTN_DEFAULT resolves to in the loaded library."""
    return int(lib().qsa_attn_default_variant())


def workspace_bytes(n_q: int, union_stride: int = gen.UNION_STRIDE) -> int:
    return int(lib().qsa_union_workspace_bytes(int(n_q), int(union_stride)))


def union_build(sel: torch.Tensor, sel_count: torch.Tensor, union_stride: int = gen.UNION_STRIDE,
                out=None, dev_status: Optional[torch.Tensor] = None, stream=None):
    """-> (union_cells int32 [G, stride], union_mask uint8 [G, stride], union_count int32 [G])."""
    _dev(sel, "sel", (torch.int32,))
    _dev(sel_count, "sel_count", (torch.int32,))
    n_q = int(sel_count.shape[0])
    n_groups = (n_q + 7) // 8
    if out is None:
        out = (torch.empty((n_groups, union_stride), dtype=torch.int32, device=sel.device),
               torch.empty((n_groups, union_stride), dtype=torch.uint8, device=sel.device),
               torch.empty((n_groups,), dtype=torch.int32, device=sel.device))
    ucell, umask, ucount = out
    rc = lib().qsa_union_build(_ptr(sel), _ptr(sel_count), n_q, int(sel.shape[1]), _ptr(ucell), _ptr(umask),
                               _ptr(ucount), int(union_stride), _ptr(dev_status), _stream(stream))
    _check("qsa_union_build", rc)
    return ucell, umask, ucount


def union_attn(q, k_pool, v_pool, k_scale, v_scale, page_table, union_cells, union_mask, union_count,
               sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None, variant: int = ATTN_DEFAULT,
               dev_status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Union attention -> out float32 [n_q, n_kv*12, 128]."""
    out = _attn_inputs(q, k_pool, v_pool, k_scale, v_scale, page_table, out)
    n_q, n_heads = int(q.shape[0]), int(q.shape[1])
    n_kv = n_heads // gen.HEADS_PER_KV
    if sm_scale is None:
        sm_scale = gen.HEAD_DIM ** -0.5
    rc = lib().qsa_union_attn(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale), _ptr(page_table),
                              int(page_table.shape[0]), int(k_pool.shape[0]), n_kv, _ptr(union_cells),
                              _ptr(union_mask), _ptr(union_count), int(union_cells.shape[1]), n_q, float(sm_scale),
                              _ptr(out), int(variant), _ptr(dev_status), _stream(stream))
    _check("qsa_union_attn", rc)
    return out


def prompt_attn(q, k_pool, v_pool, k_scale, v_scale, page_table, sel, sel_count,
                sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                workspace: Optional[torch.Tensor] = None, union_stride: int = gen.UNION_STRIDE,
                variant: int = ATTN_DEFAULT, dev_status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Union build + union attention in one call, over a caller-owned workspace."""
    out = _attn_inputs(q, k_pool, v_pool, k_scale, v_scale, page_table, out)
    _dev(sel, "sel", (torch.int32,))
    _dev(sel_count, "sel_count", (torch.int32,))
    n_q, n_heads = int(q.shape[0]), int(q.shape[1])
    n_kv = n_heads // gen.HEADS_PER_KV
    need = workspace_bytes(n_q, union_stride)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if sm_scale is None:
        sm_scale = gen.HEAD_DIM ** -0.5
    rc = lib().qsa_prompt_attn(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale), _ptr(page_table),
                               int(page_table.shape[0]), int(k_pool.shape[0]), n_kv, _ptr(sel), _ptr(sel_count),
                               int(sel.shape[1]), n_q, float(sm_scale), _ptr(out), _ptr(workspace),
                               int(workspace.numel() * workspace.element_size()), int(union_stride), int(variant),
                               _ptr(dev_status), _stream(stream))
    _check("qsa_prompt_attn", rc)
    return out


def fused_attn(q, k_pool, v_pool, k_scale, v_scale, page_table, sel, sel_count,
               sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
               dev_status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """qsa_fused_attn: the prompt-attention step in one launch, each group's union
    built inside the attention CTA (no workspace) -> out float32 [n_q, n_kv*12, 128]."""
    out = _attn_inputs(q, k_pool, v_pool, k_scale, v_scale, page_table, out)
    _dev(sel, "sel", (torch.int32,))
    _dev(sel_count, "sel_count", (torch.int32,))
    n_q, n_heads = int(q.shape[0]), int(q.shape[1])
    n_kv = n_heads // gen.HEADS_PER_KV
    if sm_scale is None:
        sm_scale = gen.HEAD_DIM ** -0.5
    rc = lib().qsa_fused_attn(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale), _ptr(page_table),
                              int(page_table.shape[0]), int(k_pool.shape[0]), n_kv, _ptr(sel), _ptr(sel_count),
                              int(sel.shape[1]), n_q, float(sm_scale), _ptr(out), _ptr(dev_status), _stream(stream))
    _check("qsa_fused_attn", rc)
    return out


def select_attn(q, k_pool, v_pool, k_scale, v_scale, page_table, sel, sel_count,
                sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                dev_status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Per-position attention without unions (qsa_select_attn) -> out float32 [n_q, n_kv*12, 128]."""
    out = _attn_inputs(q, k_pool, v_pool, k_scale, v_scale, page_table, out)
    _dev(sel, "sel", (torch.int32,))
    _dev(sel_count, "sel_count", (torch.int32,))
    n_q, n_heads = int(q.shape[0]), int(q.shape[1])
    n_kv = n_heads // gen.HEADS_PER_KV
    if sm_scale is None:
        sm_scale = gen.HEAD_DIM ** -0.5
    rc = lib().qsa_select_attn(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale), _ptr(page_table),
                               int(page_table.shape[0]), int(k_pool.shape[0]), n_kv, _ptr(sel), _ptr(sel_count),
                               int(sel.shape[1]), n_q, float(sm_scale), _ptr(out), _ptr(dev_status), _stream(stream))
    _check("qsa_select_attn", rc)
    return out


def decode_attn(q, k_pool, v_pool, k_scale, v_scale, page_tables, sel, sel_count,
                sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                dev_status: Optional[torch.Tensor] = None, stream=None,
                n_lpages: Optional[int] = None) -> torch.Tensor:
    """Decode over a batch of sequences (qsa_decode_attn): page_tables int32 [n_q, width], one table per
    query (the first n_lpages entries of its row; n_lpages defaults to the width, which is the stride)
    -> out float32 [n_q, n_kv*12, 128]."""
    _dev(q, "q", _B16)
    _dev(k_pool, "k_pool", (torch.int8,))
    _dev(v_pool, "v_pool", (torch.int8,))
    _dev(k_scale, "k_scale", _H16)
    _dev(v_scale, "v_scale", _H16)
    _dev(page_tables, "page_tables", (torch.int32,))
    _dev(sel, "sel", (torch.int32,))
    _dev(sel_count, "sel_count", (torch.int32,))
    n_q, n_heads = int(q.shape[0]), int(q.shape[1])
    if page_tables.dim() != 2 or int(page_tables.shape[0]) != n_q or not page_tables.is_contiguous():
        raise ValueError("page_tables must be a contiguous [n_q, width] array")
    n_kv = n_heads // gen.HEADS_PER_KV
    if out is None:
        out = torch.empty((n_q, n_heads, gen.HEAD_DIM), dtype=torch.float32, device=q.device)
    _dev(out, "out", (torch.float32,))
    if sm_scale is None:
        sm_scale = gen.HEAD_DIM ** -0.5
    rc = lib().qsa_decode_attn(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale), _ptr(page_tables),
                               int(page_tables.shape[1]),
                               int(page_tables.shape[1]) if n_lpages is None else int(n_lpages),
                               int(k_pool.shape[0]), n_kv,
                               _ptr(sel), _ptr(sel_count), int(sel.shape[1]), n_q, float(sm_scale), _ptr(out),
                               _ptr(dev_status), _stream(stream))
    _check("qsa_decode_attn", rc)
    return out


def wait_selftest(limit_us: int, dev_status: torch.Tensor, stream=None) -> None:
    """qsa_wait_selftest: one bounded wait that runs out after limit_us and sets QSA_DEV_WAIT_TIMEOUT."""
    _dev(dev_status, "dev_status", (torch.int32,))
    _check("qsa_wait_selftest", lib().qsa_wait_selftest(int(limit_us), _ptr(dev_status), _stream(stream)))


STATIC_SCRATCH_BYTES = 32 << 20   # QSA_STATIC_SCRATCH_BYTES


def prompt_attn_static(q, k_pool, v_pool, k_scale, v_scale, page_table, sel, sel_count,
                       sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                       union_stride: int = gen.UNION_STRIDE, variant: int = ATTN_DEFAULT,
                       dev_status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """qsa_prompt_attn_static: the prompt-attention step over the library's static
    device scratch (no workspace, no allocation inside the call).  Only `out`, when
    not given, is allocated here, by the caller's side of the binding."""
    out = _attn_inputs(q, k_pool, v_pool, k_scale, v_scale, page_table, out)
    _dev(sel, "sel", (torch.int32,))
    _dev(sel_count, "sel_count", (torch.int32,))
    n_q, n_heads = int(q.shape[0]), int(q.shape[1])
    n_kv = n_heads // gen.HEADS_PER_KV
    if sm_scale is None:
        sm_scale = gen.HEAD_DIM ** -0.5
    rc = lib().qsa_prompt_attn_static(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale),
                                      _ptr(page_table), int(page_table.shape[0]), int(k_pool.shape[0]), n_kv,
                                      _ptr(sel), _ptr(sel_count), int(sel.shape[1]), n_q, float(sm_scale), _ptr(out),
                                      int(union_stride), int(variant), _ptr(dev_status), _stream(stream))
    _check("qsa_prompt_attn_static", rc)
    return out


def to_device(wl: "gen.Workload", device="cuda") -> dict:
    """Copy a generator workload's host arrays into device tensors (marshalling only)."""
    t = lambda a, dt=None: torch.from_numpy(a if dt is None else a.view(dt)).to(device)
    import numpy as np
    return dict(q=t(wl.q, np.int16), k_pool=t(wl.k_pool), v_pool=t(wl.v_pool),
                k_scale=t(wl.k_scale.view(np.int16)), v_scale=t(wl.v_scale.view(np.int16)),
                page_table=t(wl.page_table), sel=t(wl.sel), sel_count=t(wl.sel_count))


def decode_status(word: int) -> list:
    return [name for bit, name in DEV_BITS.items() if word & bit]

"""The C ABI of libqsa.so: it loads, exports every declared symbol, and rejects
bad arguments on the host before anything reaches a GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qsa.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qsa_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from sparse_selected_cell_gb300 import build as qbuild
    qbuild.build()
    from sparse_selected_cell_gb300 import qsa
    return qsa.lib()


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert {"qsa_union_build", "qsa_union_attn", "qsa_prompt_attn", "qsa_status_str",
            "qsa_union_workspace_bytes"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"libqsa.so does not export {n}"


def test_status_strings(lib):
    for s in range(6):
        assert lib.qsa_status_str(s)
    assert lib.qsa_status_str(99) == b"unknown status"


def test_workspace_bytes(lib):
    n = lib.qsa_union_workspace_bytes(8192, 16448)
    groups = 1024
    assert n >= groups * 16448 * 5 + groups * 4
    assert n % 256 == 0
    assert lib.qsa_union_workspace_bytes(-1, 16448) == 0
    assert lib.qsa_union_workspace_bytes(8, 0) == 0


def _attn(lib, **kw):
    args = dict(q=None, k=None, v=None, ks=None, vs=None, pt=None, n_lpages=1, n_ppages=1, n_kv=1,
                uc=None, um=None, un=None, ustride=16448, n_q=8, scale=0.088, out=None, variant=0,
                status=None, stream=None)
    args.update(kw)
    return lib.qsa_union_attn(*args.values())


def test_host_argument_checks(lib):
    ERR_ARG = 1
    # n_q == 0: nothing to do, no launch
    assert lib.qsa_union_build(None, None, 0, 2056, None, None, None, 16448, None, None) == 0
    assert _attn(lib, n_q=0) == 0
    # null pointers / bad sizes / bad stride are rejected before any launch
    assert lib.qsa_union_build(None, None, 8, 2056, None, None, None, 16448, None, None) == ERR_ARG
    assert lib.qsa_union_build(None, None, -1, 2056, None, None, None, 16448, None, None) == ERR_ARG
    assert lib.qsa_union_build(None, None, 8, 2056, None, None, None, 100, None, None) == ERR_ARG
    assert _attn(lib) == ERR_ARG
    assert _attn(lib, n_kv=0) == ERR_ARG
    assert _attn(lib, variant=7) == ERR_ARG
    assert _attn(lib, variant=3) == ERR_ARG   # no such variant (QSA_ATTN_TCGEN05_SM is the last)
    # misaligned q / out pointers (never dereferenced: rejected on the host)
    fake = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1008)
    assert _attn(lib, q=odd, k=fake, v=fake, ks=fake, vs=fake, pt=fake, uc=fake, um=fake, un=fake,
                 out=fake) == ERR_ARG


def test_prompt_attn_capacity(lib):
    fake = ctypes.c_void_p(0x100000)
    rc = lib.qsa_prompt_attn(fake, fake, fake, fake, fake, fake, 1, 1, 1, fake, fake, 2056, 8, ctypes.c_float(0.088),
                             fake, fake, ctypes.c_size_t(1024), 16448, 0, None, None)
    assert rc == 3  # QSA_ERR_CAPACITY: workspace smaller than qsa_union_workspace_bytes


def test_decode_host_argument_checks(lib):
    ERR_ARG = 1
    fake = ctypes.c_void_p(0x100000)
    f = ctypes.c_float(0.088)

    def dec(pt_stride, n_lpages=4, n_q=8, sel_stride=2056):
        return lib.qsa_decode_attn(fake, fake, fake, fake, fake, fake, pt_stride, n_lpages, 16, 1, fake, fake,
                                   sel_stride, n_q, f, fake, None, None)
    assert dec(4, n_q=0) == 0                 # nothing to do, no launch
    assert dec(-1) == ERR_ARG                 # negative page-table stride
    assert dec(3) == ERR_ARG                  # tables would overlap: 0 < pt_stride < n_lpages
    assert dec(4, sel_stride=0) == ERR_ARG


def test_fused_host_argument_checks(lib):
    ERR_ARG = 1
    fake = ctypes.c_void_p(0x100000)
    f = ctypes.c_float(0.088)

    def fused(n_q=8, sel_stride=2056, sel=fake, cnt=fake, n_kv=1):
        return lib.qsa_fused_attn(fake, fake, fake, fake, fake, fake, 4, 16, n_kv, sel, cnt, sel_stride, n_q, f, fake,
                                  None, None)
    assert fused(n_q=0) == 0                  # nothing to do, no launch
    assert fused(n_q=-1) == ERR_ARG
    assert fused(sel_stride=0) == ERR_ARG
    assert fused(sel=None) == ERR_ARG
    assert fused(cnt=None) == ERR_ARG
    assert fused(n_kv=0) == ERR_ARG
    # the union of 8 lists of 4,000 entries would not fit a CTA's shared memory
    assert fused(sel_stride=4000) == 2   # QSA_ERR_UNSUPPORTED
    assert fused(n_q=8 * 65536) == 2     # more groups than the grid's y extent holds

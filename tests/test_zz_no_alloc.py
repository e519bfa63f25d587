"""qsa_prompt_attn_static: the prompt-attention step over the library's static
device scratch, called through the C ABI.

The file name sorts last so that the GPU test also runs after every other test
in one session; it passes as well in a fresh process on its own.  Host-side
rejection is checked without a GPU: it happens before any CUDA call.
"""
import ctypes
import warnings

import numpy as np
import pytest

from sparse_selected_cell_gb300 import gen

QSA_OK, QSA_ERR_ARG, QSA_ERR_CAPACITY = 0, 1, 3
SCRATCH = 32 << 20


@pytest.fixture(scope="module")
def lib():
    from sparse_selected_cell_gb300 import build as qbuild
    qbuild.build()
    from sparse_selected_cell_gb300 import qsa
    return qsa.lib()


def _call_null(lib, n_q, union_stride, sel_stride=2056, n_kv=4, variant=0):
    """The static entry point with every pointer NULL (host-side checks only)."""
    return lib.qsa_prompt_attn_static(None, None, None, None, None, None, 640, 640, n_kv, None, None, sel_stride,
                                      n_q, ctypes.c_float(0.088), None, union_stride, variant, None, None)


def test_scratch_limit_matches_workspace_layout(lib):
    assert lib.qsa_union_workspace_bytes(3256, gen.UNION_STRIDE) <= SCRATCH
    assert lib.qsa_union_workspace_bytes(3257, gen.UNION_STRIDE) > SCRATCH


def test_oversize_rejected_before_cuda(lib):
    # one group past the limit, and a single group with a huge stride
    assert _call_null(lib, 3257, gen.UNION_STRIDE) == QSA_ERR_CAPACITY
    assert _call_null(lib, 8192, gen.UNION_STRIDE) == QSA_ERR_CAPACITY
    assert _call_null(lib, 8, 64 * 200000) == QSA_ERR_CAPACITY


def test_bad_arguments_rejected_before_cuda(lib):
    assert _call_null(lib, 3256, gen.UNION_STRIDE) == QSA_ERR_ARG     # fits, but NULL pointers
    assert _call_null(lib, -1, gen.UNION_STRIDE) == QSA_ERR_ARG
    assert _call_null(lib, 8, 100) == QSA_ERR_ARG                     # stride not a multiple of 64
    assert _call_null(lib, 8, 0) == QSA_ERR_ARG
    assert _call_null(lib, 0, gen.UNION_STRIDE) == QSA_OK             # empty: nothing to do


def test_argument_errors_come_before_capacity(lib):
    # an oversized call with a bad variant, n_kv or list stride is an argument error
    assert _call_null(lib, 8192, gen.UNION_STRIDE, variant=3) == QSA_ERR_ARG
    assert _call_null(lib, 8192, gen.UNION_STRIDE, n_kv=0) == QSA_ERR_ARG
    assert _call_null(lib, 8192, gen.UNION_STRIDE, sel_stride=0) == QSA_ERR_ARG


@pytest.mark.gpu
def test_static_matches_workspace_entry_point_two_calls(lib):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required")
    from sparse_selected_cell_gb300 import qsa
    # Call 1 has the larger unions (so call 2 runs over a scratch holding call
    # 1's stale arrays); both fit in the scratch.
    loads = [gen.make(3), gen.make(2, seed=12)]
    for w in loads:
        assert lib.qsa_union_workspace_bytes(w.n_q, gen.UNION_STRIDE) <= SCRATCH
    dev = [qsa.to_device(w) for w in loads]
    refs = []
    for d in dev:      # the existing entry point over a caller-owned workspace
        refs.append(qsa.prompt_attn(d["q"], d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"], d["page_table"],
                                    d["sel"], d["sel_count"]))
    torch.cuda.synchronize()
    outs = [torch.full_like(r, float("nan")) for r in refs]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call(d, out):
        n_q, n_heads = int(d["q"].shape[0]), int(d["q"].shape[1])
        p = lambda t: ctypes.c_void_p(t.data_ptr())
        return lib.qsa_prompt_attn_static(p(d["q"]), p(d["k_pool"]), p(d["v_pool"]), p(d["k_scale"]),
                                          p(d["v_scale"]), p(d["page_table"]), int(d["page_table"].shape[0]),
                                          int(d["k_pool"].shape[0]), n_heads // gen.HEADS_PER_KV, p(d["sel"]),
                                          p(d["sel_count"]), int(d["sel"].shape[1]), n_q, gen.HEAD_DIM ** -0.5,
                                          p(out), gen.UNION_STRIDE, 0, p(status), stream)

    assert call(dev[0], outs[0]) == QSA_OK         # first call on this device: resolves the scratch
    torch.cuda.synchronize()
    alloc0, resv0 = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
    free0 = torch.cuda.mem_get_info()[0]
    for i in range(2):                             # two calls in a row, back to back on one stream
        outs[i].fill_(float("nan"))
        assert call(dev[i], outs[i]) == QSA_OK
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0 and torch.cuda.memory_reserved() == resv0
    # Free device memory is a device-wide figure that other contexts and the driver
    # can move; the allocator checks above are what show this library allocated
    # nothing.  It is only reported, within a 64 MiB band around no change.
    free1 = torch.cuda.mem_get_info()[0]
    if abs(free1 - free0) > (64 << 20):
        warnings.warn(f"device free memory moved by {(free1 - free0) / 2**20:.1f} MiB across the calls")
    assert int(status.item()) == 0, qsa.decode_status(int(status.item()))
    for i in range(2):
        assert torch.equal(outs[i], refs[i]), f"call {i + 1}: differs from qsa_prompt_attn"

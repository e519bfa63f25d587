"""qsa_union_build on the GPU against the oracle's set union: bit-exact."""
import numpy as np
import pytest

from oracle import oracle
from sparse_selected_cell_gb300 import gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qsa():
    from sparse_selected_cell_gb300 import qsa as q
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required")
    q.lib()
    return q


def _gpu_union(qsa, sel, cnt, stride=gen.UNION_STRIDE):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    uc, um, un = qsa.union_build(torch.from_numpy(np.ascontiguousarray(sel)).cuda(),
                                 torch.from_numpy(np.ascontiguousarray(cnt)).cuda(), stride, dev_status=status)
    torch.cuda.synchronize()
    return uc.cpu().numpy(), um.cpu().numpy(), un.cpu().numpy(), int(status.item())


def _compare(gpu, ref):
    uc, um, un, status = gpu
    rc, rm, rn = ref
    assert status == 0
    assert np.array_equal(un, rn)
    for g in range(len(rn)):
        n = rn[g]
        assert np.array_equal(uc[g, :n], rc[g, :n]), f"group {g} cells"
        assert np.array_equal(um[g, :n], rm[g, :n]), f"group {g} masks"


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_union_bit_exact(qsa, workload, cfg):
    w = workload(cfg)
    _compare(_gpu_union(qsa, w.sel, w.sel_count), oracle.union_ref(w.sel, w.sel_count))


def test_union_tiny_closed_form(qsa, workload):
    uc, um, un, st = _gpu_union(qsa, workload(1).sel, workload(1).sel_count)
    assert st == 0 and un[0] == 1536
    assert np.array_equal(uc[0, :1536], np.arange(1536))
    assert (um[0, :1529] == 0xFF).all()
    assert [int(x) for x in um[0, 1529:1536]] == [(0xFF << t) & 0xFF for t in range(1, 8)]


def test_union_edge_cases(qsa):
    rng = np.random.default_rng(7)
    stride = 2056
    # ragged 13 queries: empty lists, a single cell, identical lists, a list spanning > one window
    n_q = 13
    sel = np.full((n_q, stride), -1, dtype=np.int32)
    cnt = np.zeros(n_q, dtype=np.int32)
    sel[1, 0] = 0; cnt[1] = 1
    big = np.sort(rng.choice(300000, size=2000, replace=False)).astype(np.int32)
    for i in (2, 3, 4):
        sel[i, :2000] = big; cnt[i] = 2000
    sel[9, :5] = [5, 70000, 140000, 200001, 299999]; cnt[9] = 5
    sel[12, :3] = [1, 2, 3]; cnt[12] = 3
    _compare(_gpu_union(qsa, sel, cnt), oracle.union_ref(sel, cnt))
    # all lists empty
    z = np.zeros(8, dtype=np.int32)
    uc, um, un, st = _gpu_union(qsa, sel[:8] * 0 - 1, z)
    assert st == 0 and un[0] == 0


def test_union_overflow_reported(qsa, workload):
    w = workload(2)
    sel = np.ascontiguousarray(w.sel[:8])
    uc, um, un, st = _gpu_union(qsa, sel, w.sel_count[:8], stride=2048)
    assert st & 2 and un[0] == 2048           # QSA_DEV_UNION_OVERFLOW, count clamped to the stride
    rc, rm, rn = oracle.union_ref(sel, w.sel_count[:8])
    assert np.array_equal(uc[0], rc[0, :2048]) and np.array_equal(um[0], rm[0, :2048])


def test_union_bad_count_reported(qsa, workload):
    w = workload(2)
    cnt = w.sel_count[:8].copy()
    cnt[3] = 5000                                # > sel_stride: clamped and flagged
    *_, st = _gpu_union(qsa, w.sel[:8], cnt)
    assert st & 1


def test_union_rerun_bitwise(qsa, workload):
    w = workload(5)
    a = _gpu_union(qsa, w.sel, w.sel_count)
    b = _gpu_union(qsa, w.sel, w.sel_count)
    for x, y in zip(a[:3], b[:3]):
        assert np.array_equal(x, y)


def test_union_whole_pages_across_window_edges(qsa):
    """Dense runs of whole 64-cell pages, one crossing the 65,536-cell window edge,
    and a partly filled last page: the compaction walks only the pages that hold a
    marked cell, so every page boundary and window boundary must come out exact."""
    stride = 2056
    n_q = 8
    sel = np.full((n_q, stride), -1, dtype=np.int32)
    cnt = np.zeros(n_q, dtype=np.int32)
    runs = [np.arange(0, 64), np.arange(65472, 65600), np.arange(131008, 131072),
            np.arange(131072, 131105), np.arange(64, 128)[::3]]
    for i in range(n_q):
        cells = np.unique(np.concatenate([runs[(i + k) % len(runs)] for k in range(1 + i % 3)]))
        sel[i, :len(cells)] = cells
        cnt[i] = len(cells)
    _compare(_gpu_union(qsa, sel, cnt), oracle.union_ref(sel, cnt))

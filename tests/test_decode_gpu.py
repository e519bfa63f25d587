"""qsa_decode_attn on the GPU against the FP64 oracle: one query per sequence,
each sequence with its own page table into one shared pool.

The oracle takes one page table per call, so it runs sequence by sequence.
Tolerance as for the other attention paths: max |err| <= 1e-2 * max|ref| and
mean |err| <= 1e-3 * max|ref| over the compared outputs.
"""
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


def check_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    scale = float(np.abs(ref).max())
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert err.max() <= 1e-2 * scale, f"{what}: max err {err.max():.3e} vs scale {scale:.3f}"
    assert err.mean() <= 1e-3 * scale, f"{what}: mean err {err.mean():.3e} vs scale {scale:.3f}"


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def run_decode(qsa, w, page_tables=None, sel=None, sel_count=None, n_lpages=None):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = qsa.decode_attn(_dev(w.q), _dev(w.k_pool), _dev(w.v_pool), _dev(w.k_scale.view(np.int16)),
                          _dev(w.v_scale.view(np.int16)), _dev(w.page_tables if page_tables is None else page_tables),
                          _dev(w.sel if sel is None else sel), _dev(w.sel_count if sel_count is None else sel_count),
                          dev_status=status, n_lpages=n_lpages)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(status.item())


def oracle_decode(w, rows, page_tables=None, sel=None, sel_count=None):
    pts = w.page_tables if page_tables is None else page_tables
    sel = w.sel if sel is None else sel
    cnt = w.sel_count if sel_count is None else sel_count
    out = []
    for i in rows:
        out.append(oracle.attn_ref(w.q[i:i + 1], w.k_pool, w.v_pool, w.k_scale, w.v_scale,
                                   np.ascontiguousarray(pts[i, :w.n_lpages]), sel[i:i + 1], cnt[i:i + 1],
                                   w.n_kv, w.sm_scale)[0])
    return np.stack(out)


def test_decode_vs_oracle(qsa):
    w = gen.make_decode(24, 4096, 2, 160, seed=21, nonresident_frac=0.1)
    got, st = run_decode(qsa, w)
    assert st == 0
    check_close(got, oracle_decode(w, range(w.n_seq)), "decode")


def test_decode_full_size_sampled(qsa):
    """The benchmark's decode workload, sampled sequences against the oracle."""
    w = gen.make_decode(**gen.DECODE_BENCH)
    got, st = run_decode(qsa, w)
    assert st == 0
    rows = np.array(sorted({0, 1, w.n_seq - 1} | set(np.random.default_rng(5).choice(w.n_seq, 13, replace=False).tolist())))
    check_close(got[rows], oracle_decode(w, rows), "decode, benchmark workload")


def test_decode_shared_table_matches_select_attn(qsa):
    """Every sequence on one table: the same per-position computation as
    qsa_select_attn.  Decode splits each list over four warps and merges their
    partial softmax states; each warp rounds its weights P to BF16 relative to
    its own running max, so the two differ by BF16 rounding of the weights
    (relative 2^-9 per term), not by more: both meet the tolerance against the
    oracle and agree with each other within it."""
    w = gen.make_decode(16, 4096, 2, 96, seed=22)
    pts = np.repeat(w.page_tables[:1], w.n_seq, axis=0)
    got, st = run_decode(qsa, w, page_tables=pts)
    assert st == 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = qsa.select_attn(_dev(w.q), _dev(w.k_pool), _dev(w.v_pool), _dev(w.k_scale.view(np.int16)),
                          _dev(w.v_scale.view(np.int16)), _dev(w.page_tables[0]), _dev(w.sel), _dev(w.sel_count),
                          dev_status=status).cpu().numpy()
    assert int(status.item()) == 0
    check_close(got, ref.astype(np.float64), "decode against select_attn")
    check_close(got, oracle_decode(w, range(w.n_seq), page_tables=pts), "decode, shared table")


def test_decode_uneven_splits(qsa):
    """Lists of 1 to 70 cells: most of the four warps of a (query, KV head) get an
    empty or short part of the list, and the merge must weigh them correctly."""
    w = gen.make_decode(12, 2048, 1, 48, seed=25)
    sel, cnt = w.sel.copy(), w.sel_count.copy()
    for i, n in enumerate([1, 2, 15, 16, 17, 31, 33, 47, 48, 49, 64, 70]):
        cnt[i] = min(n, int(w.sel_count[i]))
    got, st = run_decode(qsa, w, sel=sel, sel_count=cnt)
    assert st == 0
    check_close(got, oracle_decode(w, range(w.n_seq), sel=sel, sel_count=cnt), "decode, uneven splits")


def test_decode_edge_cases(qsa):
    """Empty lists, lists whose every page is not resident (both: zero rows), a
    single cell (that cell's V), unsorted lists, and tables with padding past
    n_lpages (pt_stride > n_lpages)."""
    w = gen.make_decode(8, 2048, 1, 64, seed=23)
    sel, cnt, pts = w.sel.copy(), w.sel_count.copy(), w.page_tables.copy()
    cnt[0] = 0                                           # empty
    pts[1, :] = -1                                       # nothing resident
    sel[2, 0] = 100; cnt[2] = 1                          # one cell
    k = int(cnt[3]); sel[3, :k] = sel[3, :k][::-1]       # reversed order
    wide = np.full((w.n_seq, w.n_lpages + 5), 7, dtype=np.int32)
    wide[:, :w.n_lpages] = pts
    got, st = run_decode(qsa, w, page_tables=wide, sel=sel, sel_count=cnt, n_lpages=w.n_lpages)
    assert st == 0
    assert not got[0].any() and not got[1].any()
    page = pts[2, 100 >> 6]
    v = w.v_pool[page, 0, 100 & 63].astype(np.float64) * float(w.v_scale[page, 0, 100 & 63])
    assert np.allclose(got[2], np.broadcast_to(v, got[2].shape), rtol=1e-2, atol=1e-2 * np.abs(v).max())
    check_close(got, oracle_decode(w, range(w.n_seq), page_tables=pts, sel=sel, sel_count=cnt), "decode edges")


def test_decode_bad_page_reported(qsa):
    """A table entry past the pool is masked and flagged (QSA_DEV_BAD_PAGE)."""
    w = gen.make_decode(4, 2048, 1, 48, seed=24)
    pts = w.page_tables.copy()
    pts[2, w.sel[2, 0] >> 6] = w.n_ppages + 3
    got, st = run_decode(qsa, w, page_tables=pts)
    assert st & 8
    assert np.isfinite(got).all()

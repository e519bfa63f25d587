"""qsa_select_attn (per-position attention, no union) on the GPU against the FP64 oracle.

Same tolerance as the union path: max |err| <= 1e-2 * max|ref|, mean |err| <= 1e-3 * max|ref|.
Configs 1-3 in full; configs 4-5 (full size) on sampled positions that cover the first,
last and ragged ones.
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


def run_sel(qsa, w, **over):
    d = qsa.to_device(w)
    d.update({k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in over.items()})
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = qsa.select_attn(d["q"], d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"], d["page_table"],
                          d["sel"], d["sel_count"], dev_status=status)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(status.item())


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_select_full_vs_oracle(qsa, workload, cfg):
    w = workload(cfg)
    got, st = run_sel(qsa, w)
    assert st == 0
    check_close(got, oracle.attn_ref_workload(w), f"config {cfg}")


@pytest.mark.parametrize("cfg", [4, 5])
def test_select_full_size_sampled(qsa, workload, cfg):
    w = workload(cfg)
    got, st = run_sel(qsa, w)
    assert st == 0
    rows = np.array(sorted(set(range(8)) | set(range(w.n_q - 13, w.n_q)) |
                           set(np.random.default_rng(w.seed).choice(w.n_q, 96, replace=False).tolist())),
                    dtype=np.int32)
    ref = oracle.attn_ref_workload(w, q_index=rows)
    check_close(got[rows], ref, f"config {cfg} sampled")


def test_select_matches_union_path(qsa, workload):
    """Both paths compute the same per-position softmax: they agree within the
    union path's tolerance on config 3."""
    w = workload(3)
    got, st = run_sel(qsa, w)
    d = qsa.to_device(w)
    ref = qsa.prompt_attn(d["q"], d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"], d["page_table"],
                          d["sel"], d["sel_count"]).cpu().numpy().astype(np.float64)
    check_close(got, ref, "select vs union")


def test_select_edge_cases(qsa):
    w = gen.make(2, n_q=64, nonresident_frac=0.2, seed=31)
    sel, cnt = w.sel.copy(), w.sel_count.copy()
    cnt[[0, 17, 63]] = 0                                     # empty lists -> zero rows
    cnt[5] = 1                                               # one cell
    cnt[6] = 17                                              # a step and one cell
    rng = np.random.default_rng(3)
    for i in range(8, 16):                                   # order within a list does not matter
        rng.shuffle(sel[i, :cnt[i]])
    got, st = run_sel(qsa, w, sel=sel, sel_count=cnt)
    assert st == 0
    assert (got[[0, 17, 63]] == 0).all()
    ref = oracle.attn_ref(w.q, w.k_pool, w.v_pool, w.k_scale, w.v_scale, w.page_table, sel, cnt, w.n_kv, w.sm_scale)
    check_close(got, ref, "edge cases")


def test_select_bitwise_rerun_and_bad_cells(qsa, workload):
    w = workload(2)
    a, _ = run_sel(qsa, w)
    b, _ = run_sel(qsa, w)
    assert np.array_equal(a, b)
    sel = w.sel.copy()
    sel[3, 0] = 10 ** 7                                      # page beyond n_lpages
    got, st = run_sel(qsa, w, sel=sel)
    assert st & 4 and np.isfinite(got).all()


def test_select_empty_batch(qsa):
    w = gen.make(2, n_q=8)
    d = qsa.to_device(w)
    out = qsa.select_attn(d["q"][:0], d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"], d["page_table"],
                          d["sel"][:0], d["sel_count"][:0])
    assert out.shape == (0, w.n_heads, 128)

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


def run_sel(qsa, w, sm_scale=None, **over):
    d = qsa.to_device(w)
    d.update({k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in over.items()})
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = qsa.select_attn(d["q"], d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"], d["page_table"],
                          d["sel"], d["sel_count"], sm_scale=sm_scale, dev_status=status)
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


def _times_pow2(q_bits, shift):
    """BF16 bits times 2^shift (exact: only the exponent moves)."""
    qf = (q_bits.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** shift)
    return (qf.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("shift", [20, -20])
def test_select_query_magnitudes_far_from_one(qsa, shift):
    """Q times 2^shift with sm_scale times 2^-shift: the same scores.  Rows whose
    largest |q| is 2^14 or more, or below 2^-10, take the exact power-of-two row
    scaling of the FP16 score path; the oracle sees the same scaled inputs."""
    w = gen.make(2, n_q=40, seed=47)
    q = _times_pow2(w.q, shift)
    sm = float(2.0 ** -shift / np.sqrt(128.0))
    got, st = run_sel(qsa, w, sm_scale=sm, q=q)
    assert st == 0
    ref = oracle.attn_ref(q, w.k_pool, w.v_pool, w.k_scale, w.v_scale, w.page_table, w.sel, w.sel_count, w.n_kv, sm)
    check_close(got, ref, f"Q x 2^{shift}")


def test_select_query_rows_scaled_apart(qsa):
    """Some query heads times 2^20, the rest as they are, sm_scale times 2^-20: the
    scaled heads keep their scores and the others get nearly equal weights.  Rows
    of one (position, KV head) then take different power-of-two scalings, rows
    0-7 and 8-11 of the tile among them."""
    w = gen.make(2, n_q=40, seed=53)
    big = np.isin(np.arange(w.n_heads) % 12, [1, 4, 9, 10])
    q = w.q.copy()
    q[:, big] = _times_pow2(w.q[:, big], 20)
    sm = float(2.0 ** -20 / np.sqrt(128.0))
    got, st = run_sel(qsa, w, sm_scale=sm, q=q)
    assert st == 0
    ref = oracle.attn_ref(q, w.k_pool, w.v_pool, w.k_scale, w.v_scale, w.page_table, w.sel, w.sel_count, w.n_kv, sm)
    check_close(got, ref, "rows scaled apart")


def test_select_scale_signs_and_ranges(qsa):
    """K scales of either sign; V scales of either sign and of any FP16 size (zero,
    subnormal, up to 2^15), which the kernel splits into a power of two, carried in
    the softmax's exponent, and a significand in P; a non-default sm_scale."""
    w = gen.make(2, n_q=40, seed=59)
    rng = np.random.default_rng(7)
    ks = (w.k_scale * rng.choice([-1.0, 1.0], size=w.k_scale.shape)).astype(np.float16)
    mag = np.exp2(rng.uniform(-24.0, 15.0, size=w.v_scale.shape))
    vs = (mag * rng.choice([-1.0, 1.0], size=mag.shape)).astype(np.float16)
    vs[rng.random(vs.shape) < 0.05] = 0
    assert (np.abs(vs[vs != 0]) < np.float16(2.0 ** -14)).any()   # FP16 subnormals among them
    got, st = run_sel(qsa, w, sm_scale=0.05, k_scale=ks.view(np.int16), v_scale=vs.view(np.int16))
    assert st == 0
    ref = oracle.attn_ref(w.q, w.k_pool, w.v_pool, ks, vs, w.page_table, w.sel, w.sel_count, w.n_kv, 0.05)
    check_close(got, ref, "scale signs and ranges")


def test_select_zero_scale_is_the_mean_of_v(qsa):
    """sm_scale = 0 makes every selected, resident cell weigh the same: each row is the
    plain mean of its cells' dequantised V (a closed form, computed here in numpy)."""
    w = gen.make(2, n_q=24, nonresident_frac=0.1, seed=41)
    got, st = run_sel(qsa, w, sm_scale=0.0)
    assert st == 0
    v = w.v_pool.astype(np.float64) * w.v_scale.astype(np.float64)[..., None]   # [page][kv][cell][d]
    ref = np.zeros_like(got, dtype=np.float64)
    for i in range(w.n_q):
        cells = w.sel[i, :w.sel_count[i]]
        pages = w.page_table[cells >> 6]
        keep = pages >= 0
        for kh in range(w.n_kv):
            rows = v[pages[keep], kh, cells[keep] & 63]
            if len(rows):
                ref[i, kh * 12:(kh + 1) * 12] = rows.mean(axis=0)
    check_close(got, ref, "sm_scale = 0")

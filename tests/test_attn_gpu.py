"""qsa_union_attn / qsa_prompt_attn on the GPU against the FP64 oracle.

Tolerance (BF16 path): max |err| <= 1e-2 * max|ref| and mean |err| <= 1e-3 * max|ref|,
over the compared outputs.  The oracle never sees the union: it evaluates each
query over its own selection list.  Configs 1-3 are compared in full; configs 4-5
(the full-size workloads, in the launch configuration the benchmark times) on
sampled query positions that cover the first, last and ragged groups.
"""
import numpy as np
import pytest

from oracle import oracle
from sparse_selected_cell_gb300 import gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

VARIANTS = [1, 2]   # QSA_ATTN_TCGEN05 (two CTAs per SM, the default), QSA_ATTN_TCGEN05_SM (one CTA per SM)


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
    return float(err.max() / scale), float(err.mean() / scale)


def run_gpu(qsa, w, variant, **over):
    d = qsa.to_device(w)
    d.update({k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in over.items()})
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = qsa.prompt_attn(d["q"], d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"], d["page_table"],
                          d["sel"], d["sel_count"], variant=variant, dev_status=status)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(status.item())


def sample_rows(w, n=96):
    rows = set(range(min(8, w.n_q))) | set(range(max(0, w.n_q - 13), w.n_q))
    rows |= set(np.random.default_rng(w.seed).choice(w.n_q, size=min(n, w.n_q), replace=False).tolist())
    return np.array(sorted(rows), dtype=np.int32)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_attn_full_vs_oracle(qsa, workload, cfg, variant):
    w = workload(cfg)
    got, st = run_gpu(qsa, w, variant)
    assert st == 0
    ref = oracle.attn_ref_workload(w)
    check_close(got, ref, f"config {cfg} variant {variant}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("cfg", [4, 5])
def test_attn_full_size_sampled(qsa, workload, cfg, variant):
    w = workload(cfg)
    got, st = run_gpu(qsa, w, variant)
    assert st == 0
    assert np.isfinite(got).all()
    rows = sample_rows(w)
    ref = oracle.attn_ref_workload(w, q_index=rows)
    check_close(got[rows], ref, f"config {cfg} variant {variant}")


@pytest.mark.parametrize("variant", VARIANTS)
def test_bitwise_rerun_and_page_permutation(qsa, workload, variant):
    w = workload(5)
    a, _ = run_gpu(qsa, w, variant)
    b, _ = run_gpu(qsa, w, variant)
    assert np.array_equal(a, b), "rerun is not bitwise identical"
    w2 = workload(2)
    base, _ = run_gpu(qsa, w2, variant)
    perm = np.random.default_rng(3).permutation(w2.n_ppages)
    inv = np.argsort(perm)
    moved, _ = run_gpu(qsa, w2, variant, k_pool=w2.k_pool[inv], v_pool=w2.v_pool[inv],
                       k_scale=w2.k_scale[inv].view(np.int16), v_scale=w2.v_scale[inv].view(np.int16),
                       page_table=perm[w2.page_table].astype(np.int32))
    assert np.array_equal(base, moved), "page-table permutation changed the output"


@pytest.mark.parametrize("variant", VARIANTS)
def test_special_cases(qsa, workload, variant):
    w = gen.make(2, n_q=64)
    # one selected cell -> that cell's V (BF16-rounded V times a unit weight)
    sel = np.full_like(w.sel, -1)
    cells = w.q0 + np.arange(w.n_q) - 64 * (np.arange(w.n_q) % 5)
    sel[:, 0] = cells
    cnt = np.ones_like(w.sel_count)
    got, st = run_gpu(qsa, w, variant, sel=sel, sel_count=cnt)
    assert st == 0
    ref = oracle.attn_ref(w.q, w.k_pool, w.v_pool, w.k_scale, w.v_scale, w.page_table, sel, cnt, w.n_kv, w.sm_scale)
    check_close(got, ref, "single cell")
    np.testing.assert_allclose(got, ref, rtol=2 ** -8, atol=0)
    # constant V per KV head -> the constant
    vp = np.empty_like(w.v_pool)
    for kh in range(w.n_kv):
        vp[:, kh] = [5, -9, 33, -100][kh]
    vs = np.full_like(w.v_scale, np.float16(0.03125)).view(np.int16)
    got, st = run_gpu(qsa, w, variant, v_pool=vp, v_scale=vs)
    for h in range(w.n_heads):
        # exact up to the BF16 rounding of the weights that enter P V (relative 2^-9)
        np.testing.assert_allclose(got[:, h], [5, -9, 33, -100][h // 12] * 0.03125, rtol=3e-3)
    # empty selections -> zeros, neighbours unaffected
    cnt = w.sel_count.copy()
    cnt[[0, 9, 63]] = 0
    got, st = run_gpu(qsa, w, variant, sel_count=cnt)
    assert st == 0
    assert (got[[0, 9, 63]] == 0).all()
    ref = oracle.attn_ref(w.q, w.k_pool, w.v_pool, w.k_scale, w.v_scale, w.page_table, w.sel, cnt, w.n_kv, w.sm_scale)
    check_close(got, ref, "empty rows")


@pytest.mark.parametrize("variant", VARIANTS)
def test_nonresident_pages(qsa, variant):
    w = gen.make(3, n_q=256, nonresident_frac=0.3)
    got, st = run_gpu(qsa, w, variant)
    assert st == 0
    ref = oracle.attn_ref_workload(w)
    check_close(got, ref, "non-resident pages")


@pytest.mark.parametrize("variant", VARIANTS)
def test_ragged_small_batches(qsa, variant):
    for n_q in (1, 5, 8, 9, 27):
        w = gen.make(2, n_q=n_q, seed=100 + n_q)
        got, st = run_gpu(qsa, w, variant)
        assert st == 0
        check_close(got, oracle.attn_ref_workload(w), f"n_q={n_q}")


def test_empty_batch(qsa):
    w = gen.make(2, n_q=8)
    d = qsa.to_device(w)
    q = d["q"][:0]
    out = qsa.prompt_attn(q, d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"], d["page_table"],
                          d["sel"][:0], d["sel_count"][:0])
    assert out.shape == (0, w.n_heads, 128)


def test_bad_cells_are_masked_and_reported(qsa):
    w = gen.make(2, n_q=16)
    sel = w.sel.copy()
    sel[3, 0] = 10 ** 7                 # page beyond n_lpages
    sel[3, :w.sel_count[3]] = np.sort(sel[3, :w.sel_count[3]])
    pt = w.page_table.copy()
    pt[0] = w.n_ppages + 3              # page-table entry beyond the pool (page 0 holds the sinks)
    for variant in VARIANTS:
        got, st = run_gpu(qsa, w, variant, sel=sel, page_table=pt)
        assert st & 4 and st & 8
        assert np.isfinite(got).all()


def _lists(w, per_query):
    """A selection array for workload w from per-query lists of cells (sorted, distinct)."""
    sel = np.full_like(w.sel, -1)
    cnt = np.zeros_like(w.sel_count)
    for i, cells in enumerate(per_query):
        cells = np.array(sorted(set(int(c) for c in cells)), dtype=np.int32)
        sel[i, :len(cells)] = cells
        cnt[i] = len(cells)
    return sel, cnt


@pytest.mark.parametrize("variant", VARIANTS)
def test_chunk_placement_edge_cases(qsa, variant):
    """Unions whose loose leading cells wrap into the last chunk: leads of 1, 3 and
    63 entries, unions of 5, 64 and 65 cells, no page-aligned cell at all, and
    partly selected pages inside a chunk."""
    w = gen.make(2, n_q=64)
    rng = np.random.default_rng(7)
    groups = [
        lambda j: [0, 1, 2, 64, 65],                                      # lead 3, U = 5
        lambda j: [0, 1, 2] + list(range(128, 128 + 61)),                 # lead 3, U = 64
        lambda j: [0, 1, 2] + list(range(128, 128 + 62)),                 # lead 3, U = 65
        lambda j: [5] + list(range(64, 64 + 64 + j)),                     # lead 1, a page and a partial one
        lambda j: list(range(1, 64)) + list(range(192, 256)),             # lead 63: 63 loose cells, then a page
        lambda j: list(range(3, 3 + 60, 3)) + list(range(1025, 1025 + 40)),  # no page-aligned cell
        lambda j: [0] + list(range(256 + 8 * j, 320)) + list(range(640, 704)),  # per-query partial pages
        lambda j: sorted(rng.choice(4096, size=int(rng.integers(1, 200)), replace=False).tolist()),
    ]
    per_query = [groups[i // 8](i % 8) for i in range(w.n_q)]
    sel, cnt = _lists(w, per_query)
    got, st = run_gpu(qsa, w, variant, sel=sel, sel_count=cnt)
    assert st == 0
    ref = oracle.attn_ref(w.q, w.k_pool, w.v_pool, w.k_scale, w.v_scale, w.page_table, sel, cnt, w.n_kv, w.sm_scale)
    check_close(got, ref, "chunk placement edge cases")


def _run_scaled(qsa, w, variant, sm_scale, **over):
    d = qsa.to_device(w)
    d.update({k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in over.items()})
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = qsa.prompt_attn(d["q"], d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"], d["page_table"],
                          d["sel"], d["sel_count"], sm_scale=sm_scale, variant=variant, dev_status=status)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(status.item())


@pytest.mark.parametrize("variant", VARIANTS)
def test_zero_scale_is_the_mean_of_v(qsa, variant):
    """sm_scale = 0 makes every selected, resident cell weigh the same: each row is the
    plain mean of its cells' dequantised V (a closed form, computed here in numpy)."""
    w = gen.make(2, n_q=24, nonresident_frac=0.1, seed=41)
    got, st = _run_scaled(qsa, w, variant, 0.0)
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


@pytest.mark.parametrize("variant", VARIANTS)
def test_negative_scales_and_custom_sm_scale(qsa, variant):
    """FP16 scales of either sign and a non-default sm_scale, against the oracle."""
    w = gen.make(2, n_q=40, seed=43)
    rng = np.random.default_rng(5)
    ks = (w.k_scale * rng.choice([-1.0, 1.0], size=w.k_scale.shape)).astype(np.float16)
    vs = (w.v_scale * rng.choice([-1.0, 1.0], size=w.v_scale.shape)).astype(np.float16)
    got, st = _run_scaled(qsa, w, variant, 0.05, k_scale=ks.view(np.int16), v_scale=vs.view(np.int16))
    assert st == 0
    ref = oracle.attn_ref(w.q, w.k_pool, w.v_pool, ks, vs, w.page_table, w.sel, w.sel_count, w.n_kv, 0.05)
    check_close(got, ref, "negative scales")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shift", [20, -20])
def test_query_magnitudes_far_from_one(qsa, variant, shift):
    """Q times 2^shift with sm_scale times 2^-shift: the same scores.  Rows whose
    largest |q| is 2^14 or more, or below 2^-10, take the exact power-of-two row
    scaling of the FP16 score path; the oracle sees the same scaled inputs."""
    w = gen.make(2, n_q=40, seed=47)
    qf = (w.q.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** shift)   # exact
    q = (qf.view(np.uint32) >> 16).astype(np.uint16)
    sm = float(2.0 ** -shift / np.sqrt(128.0))
    got, st = _run_scaled(qsa, w, variant, sm, q=q)
    assert st == 0
    ref = oracle.attn_ref(q, w.k_pool, w.v_pool, w.k_scale, w.v_scale, w.page_table, w.sel, w.sel_count, w.n_kv, sm)
    check_close(got, ref, f"Q x 2^{shift}")


@pytest.mark.parametrize("variant", VARIANTS)
def test_query_rows_scaled_apart(qsa, variant):
    """Some query heads times 2^20, the rest as they are, sm_scale times 2^-20: the
    scaled heads keep their scores and the others get nearly equal weights, so
    rows of one chunk take different power-of-two scalings."""
    w = gen.make(2, n_q=40, seed=53)
    big = np.isin(np.arange(w.n_heads) % 12, [1, 4, 9, 10])
    qf = (w.q.astype(np.uint32) << 16).view(np.float32)
    qf[:, big] *= np.float32(2.0 ** 20)   # exact
    q = (qf.view(np.uint32) >> 16).astype(np.uint16)
    sm = float(2.0 ** -20 / np.sqrt(128.0))
    got, st = _run_scaled(qsa, w, variant, sm, q=q)
    assert st == 0
    ref = oracle.attn_ref(q, w.k_pool, w.v_pool, w.k_scale, w.v_scale, w.page_table, w.sel, w.sel_count, w.n_kv, sm)
    check_close(got, ref, "rows scaled apart")

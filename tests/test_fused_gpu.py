"""qsa_fused_attn (the union built inside the attention CTA, one launch) on the GPU.

Against the launch pair it replaces -- qsa_prompt_attn with the one-CTA-per-SM
attention variant, whose arithmetic it shares -- the output must agree bit for
bit: the in-CTA union build hands the attention pipeline the same chunks in the same
order.  Against the FP64 oracle it must meet the usual tolerance (max |err| <=
1e-2 * max|ref|, mean |err| <= 1e-3 * max|ref|): configs 1-3 in full, configs 4-5
(full size) on sampled positions.  Each CTA builds its group's union in shared
memory with the union kernel's own build before its pipeline starts; config 5's
unions hold ~8,000 cells each.
"""
import numpy as np
import pytest

from oracle import oracle
from sparse_selected_cell_gb300 import gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SM_VARIANT = 2   # QSA_ATTN_TCGEN05_SM


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


def run_both(qsa, w, **over):
    d = qsa.to_device(w)
    d.update({k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in over.items()})
    st_f = torch.zeros(1, dtype=torch.int32, device="cuda")
    st_p = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (d["q"], d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"], d["page_table"], d["sel"], d["sel_count"])
    fused = qsa.fused_attn(*args, dev_status=st_f)
    pair = qsa.prompt_attn(*args, variant=SM_VARIANT, dev_status=st_p)
    torch.cuda.synchronize()
    return fused.cpu().numpy(), pair.cpu().numpy(), int(st_f.item()), int(st_p.item())


def sample_rows(w, n=96):
    rows = set(range(min(8, w.n_q))) | set(range(max(0, w.n_q - 13), w.n_q))
    rows |= set(np.random.default_rng(w.seed).choice(w.n_q, size=min(n, w.n_q), replace=False).tolist())
    return np.array(sorted(rows), dtype=np.int32)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_fused_equals_launch_pair_and_oracle(qsa, workload, cfg):
    w = workload(cfg)
    fused, pair, st_f, st_p = run_both(qsa, w)
    assert st_f == 0 and st_p == 0
    assert np.array_equal(fused, pair), f"config {cfg}: fused output differs from the launch pair"
    if cfg <= 3:
        check_close(fused, oracle.attn_ref_workload(w), f"config {cfg}")
    else:
        rows = sample_rows(w)
        check_close(fused[rows], oracle.attn_ref_workload(w, q_index=rows), f"config {cfg}")


def test_fused_rerun_is_bitwise(qsa, workload):
    w = workload(5)
    a, _, _, _ = run_both(qsa, w)
    b, _, _, _ = run_both(qsa, w)
    assert np.array_equal(a, b)


def test_fused_small_batches_and_nonresident(qsa):
    for n_q in (1, 5, 8, 9, 27):
        w = gen.make(2, n_q=n_q, seed=200 + n_q)
        fused, pair, st_f, _ = run_both(qsa, w)
        assert st_f == 0
        assert np.array_equal(fused, pair)
        check_close(fused, oracle.attn_ref_workload(w), f"n_q={n_q}")
    w = gen.make(3, n_q=256, nonresident_frac=0.3)
    fused, pair, st_f, _ = run_both(qsa, w)
    assert st_f == 0
    assert np.array_equal(fused, pair)
    check_close(fused, oracle.attn_ref_workload(w), "non-resident pages")


def _lists(w, per_query):
    sel = np.full_like(w.sel, -1)
    cnt = np.zeros_like(w.sel_count)
    for i, cells in enumerate(per_query):
        cells = np.array(sorted(set(int(c) for c in cells)), dtype=np.int32)
        sel[i, :len(cells)] = cells
        cnt[i] = len(cells)
    return sel, cnt


def test_fused_chunk_placement_and_empty_lists(qsa):
    """Loose leading cells that wrap into the last chunk (leads of 1, 3, 63), unions
    of 5, 64 and 65 cells, no page-aligned cell, partial pages, a group with no
    cells at all, and single cells."""
    w = gen.make(2, n_q=80)
    rng = np.random.default_rng(9)
    groups = [
        lambda j: [0, 1, 2, 64, 65],
        lambda j: [0, 1, 2] + list(range(128, 128 + 61)),
        lambda j: [0, 1, 2] + list(range(128, 128 + 62)),
        lambda j: [5] + list(range(64, 64 + 64 + j)),
        lambda j: list(range(1, 64)) + list(range(192, 256)),
        lambda j: list(range(3, 3 + 60, 3)) + list(range(1025, 1025 + 40)),
        lambda j: [0] + list(range(256 + 8 * j, 320)) + list(range(640, 704)),
        lambda j: [],
        lambda j: [100 * j + 7] if j % 2 else [],
        lambda j: sorted(rng.choice(4096, size=int(rng.integers(1, 300)), replace=False).tolist()),
    ]
    sel, cnt = _lists(w, [groups[i // 8](i % 8) for i in range(w.n_q)])
    fused, pair, st_f, _ = run_both(qsa, w, sel=sel, sel_count=cnt)
    assert st_f == 0
    assert np.array_equal(fused, pair)
    assert (fused[56:64] == 0).all()   # the group with no cells
    ref = oracle.attn_ref(w.q, w.k_pool, w.v_pool, w.k_scale, w.v_scale, w.page_table, sel, cnt, w.n_kv, w.sm_scale)
    check_close(fused, ref, "chunk placement")


def test_fused_bad_counts_are_clamped_and_reported(qsa):
    w = gen.make(2, n_q=16)
    cnt = w.sel_count.copy()
    cnt[3] = -5
    cnt[12] = w.sel.shape[1] + 7
    fused, _, st_f, _ = run_both(qsa, w, sel_count=cnt)
    assert st_f & 1                      # QSA_DEV_BAD_SEL_COUNT
    assert np.isfinite(fused).all()
    assert (fused[3] == 0).all()         # clamped to an empty list


def test_fused_mixed_whole_and_partial_pages(qsa):
    """Lists that mix whole pages with pages they hold only in part, at every
    density, several lists sharing a page while holding different parts of it, up
    to the 2,051-cell cap (many partly held pages in the in-CTA union build),
    against the launch pair bit for bit and against the oracle."""
    w = gen.make(2, n_q=64)          # 4,096-cell context: pages 0-63
    rng = np.random.default_rng(23)
    shared = sorted(rng.choice(64, size=20, replace=False).tolist())   # pages several lists touch

    def one_list(i):
        cells = []
        for p in range(64):
            if p in shared and rng.random() < 0.7:
                mode = rng.integers(0, 3)
            elif rng.random() < 0.25:
                mode = rng.integers(0, 3)
            else:
                continue
            if mode == 0:                                  # the whole page
                cells += range(64 * p, 64 * p + 64)
            else:                                          # part of it, sparse or dense
                k = int(rng.integers(1, 12)) if mode == 1 else int(rng.integers(40, 64))
                cells += sorted((64 * p + rng.choice(64, size=k, replace=False)).tolist())
        return cells[:2051]

    sel, cnt = _lists(w, [one_list(i) for i in range(w.n_q)])
    fused, pair, st_f, st_p = run_both(qsa, w, sel=sel, sel_count=cnt)
    assert st_f == 0 and st_p == 0
    assert np.array_equal(fused, pair)
    ref = oracle.attn_ref(w.q, w.k_pool, w.v_pool, w.k_scale, w.v_scale, w.page_table, sel, cnt, w.n_kv, w.sm_scale)
    check_close(fused, ref, "mixed pages")

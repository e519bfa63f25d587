"""Seeded generator: the selection layout, page table and value ranges."""
import numpy as np
import pytest

from sparse_selected_cell_gb300 import gen


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_lists_sorted_causal_capped(workload, cfg):
    w = workload(cfg)
    assert w.sel.shape == (w.n_q, gen.SEL_STRIDE)
    assert (w.sel_count <= gen.CAP).all() and (w.sel_count > 0).all()
    for i in range(w.n_q):
        c = w.sel[i, : w.sel_count[i]]
        p = w.q0 + i
        assert (np.diff(c) > 0).all(), "strictly increasing"
        assert c[0] >= 0 and c[-1] == p, "causal, ends at the query's own cell"
        assert (w.sel[i, w.sel_count[i]:] == -1).all()


@pytest.mark.parametrize("cfg", [2, 3])
def test_block_recipe(workload, cfg):
    w = workload(cfg)
    for i in range(0, w.n_q, 37):
        p = w.q0 + i
        b = p >> 6
        c = set(w.sel[i, : w.sel_count[i]].tolist())
        assert {0, 1, 2} <= c, "sinks"
        local = set(range(max(0, (b - 7) * 64), p + 1))
        assert local <= c, "own block and the 7 before it"
        far = sorted(c - local - {0, 1, 2})
        blocks = {x >> 6 for x in far}
        assert len(blocks) <= 24
        for blk in blocks:  # far selections are whole blocks
            assert set(range(blk * 64, blk * 64 + 64)) <= c
        assert w.sel_count[i] == 3 * (0 not in blocks) + 64 * len(blocks) + len(local)


def test_drift_controls_overlap():
    def mean_union_ratio(drift):
        w = gen.make(3, n_q=256, drift=drift)
        r = []
        for g in range(0, w.n_q, 8):
            s = set()
            for i in range(g, g + 8):
                s.update(w.sel[i, : w.sel_count[i]].tolist())
            r.append(len(s) / w.sel_count[g:g + 8].mean())
        return float(np.mean(r))
    r0, r25, r100 = mean_union_ratio(0.0), mean_union_ratio(0.25), mean_union_ratio(1.0)
    assert r0 < r25 < r100
    assert 1.0 < r0 < 1.7 and 2.0 < r25 < 3.2 and r100 > 4.0


def test_page_table_permutation_and_ranges(workload):
    w = workload(2)
    assert sorted(w.page_table.tolist()) == list(range(w.n_lpages))
    assert w.k_pool.dtype == np.int8 and w.k_pool.min() >= -127 and w.k_pool.max() <= 127
    ks = w.k_scale.astype(np.float64)
    assert ks.min() >= 0.0099 and ks.max() <= 0.0301
    q = gen.bf16_bits_to_f32(w.q)
    assert abs(float(q.mean())) < 0.01 and 0.95 < float(q.std()) < 1.05


def test_nonresident_pages():
    w = gen.make(2, n_q=16, nonresident_frac=0.25)
    assert (w.page_table < 0).sum() == 16
    res = w.page_table[w.page_table >= 0]
    assert sorted(res.tolist()) == list(range(w.n_ppages))
    assert w.k_pool.shape[0] == w.n_ppages == 48


def test_same_seed_same_bytes():
    a, b = gen.make(2, n_q=64), gen.make(2, n_q=64)
    for f in ("q", "k_pool", "v_pool", "k_scale", "v_scale", "page_table", "sel", "sel_count"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    c = gen.make(2, n_q=64, seed=99)
    assert not np.array_equal(a.sel, c.sel)


def test_config5_ragged_and_sigma(workload):
    w = workload(5)
    assert w.n_q == 8189 and w.n_q % 8 == 5 and w.q0 + w.n_q == 65536
    q = gen.bf16_bits_to_f32(w.q[:64])
    assert 1.9 < float(q.std()) < 2.1


def test_bf16_rounding_is_nearest_even():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(gen.f32_to_bf16_bits(x), ref)


def test_make_decode_is_seeded_and_well_formed():
    a = gen.make_decode(5, 4096, 2, 100, seed=3, nonresident_frac=0.2)
    b = gen.make_decode(5, 4096, 2, 100, seed=3, nonresident_frac=0.2)
    for x, y in ((a.q, b.q), (a.page_tables, b.page_tables), (a.sel, b.sel), (a.k_pool, b.k_pool)):
        assert np.array_equal(x, y)
    assert a.page_tables.shape == (5, 64) and a.q.shape == (5, 24, 128)
    for i in range(a.n_seq):
        row = a.page_tables[i]
        live = row[row >= 0]
        assert len(set(live.tolist())) == len(live) and (live < a.n_ppages).all()   # no repeats within a sequence
        cells = a.sel[i, :a.sel_count[i]]
        assert (np.diff(cells) > 0).all() and cells[0] == 0 and cells[-1] == a.ctx - 1   # sinks ... last position
        assert a.sel_count[i] <= gen.CAP

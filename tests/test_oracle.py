"""Pins for the FP64 CPU oracle, checked against things other than itself.

Source of the definitions: "sycl: prompt attention over 8-query selection
unions on XMX" (Strata PR #2808), section Summary (each position attends to
exactly its own selected cells; the union of 8 neighbouring positions' lists
marks each cell with the positions that chose it) and section Extra Notes
(non-resident pages are masked; a union cell is an int32 plus a membership byte).

Pins used here:
  * IEEE decoders vs numpy float16 / torch bfloat16 on every bit pattern;
  * library routine: torch scaled_dot_product_attention (FP64) with a boolean
    mask built from the lists, on dense K/V laid out through the page table;
  * closed forms: one selected cell returns its V; equal keys return the mean of
    the values; constant V returns the constant; per-KV-head constants pin the
    query-head -> KV-head grouping;
  * invariants: page-table permutation, non-resident = dropped, empty = 0,
    convex-combination bound;
  * union: closed form on the tiny config, brute-force Python set union,
    identical lists, ragged groups.
A final test plants plausible mistakes in copies of the oracle source and checks
that these pins catch every one of them.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle import build_oracle, oracle
from sparse_selected_cell_gb300 import gen

torch = pytest.importorskip("torch")

SMALL = dict(name="small", ctx=1024, n_q=16, n_kv=2, select="blocks", drift=0.5,
             scale_lo=0.01, scale_hi=0.03, q_sigma=1.0, seed=11)


def _small(**kw):
    cfg = dict(SMALL)
    cfg.update(kw)
    return gen.make(cfg)


def _dense_kv(w):
    """Dequantised K/V [n_kv, ctx, 128] in logical cell order (numpy float16 decoding)."""
    n_cells = w.n_lpages * 64
    k = np.zeros((w.n_kv, n_cells, 128))
    v = np.zeros((w.n_kv, n_cells, 128))
    for lp in range(w.n_lpages):
        pp = w.page_table[lp]
        if pp < 0:
            continue
        ks = w.k_scale[pp].astype(np.float64)[:, :, None]
        vs = w.v_scale[pp].astype(np.float64)[:, :, None]
        k[:, lp * 64:(lp + 1) * 64] = w.k_pool[pp].astype(np.float64) * ks
        v[:, lp * 64:(lp + 1) * 64] = w.v_pool[pp].astype(np.float64) * vs
    return k, v


def _sdpa(w, rows):
    """torch SDPA (FP64, default 1/sqrt(d) scale) over the lists as a boolean mask."""
    k, v = _dense_kv(w)
    n_cells = k.shape[1]
    mask = np.zeros((len(rows), n_cells), dtype=bool)
    for t, i in enumerate(rows):
        c = w.sel[i, : w.sel_count[i]]
        c = c[w.page_table[c >> 6] >= 0]
        mask[t, c] = True
    q = gen.bf16_bits_to_f32(w.q[rows]).astype(np.float64)          # [rows, H, 128]
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]                  # [1, H, rows, 128]
    kt = torch.from_numpy(k).repeat_interleave(12, dim=0)[None]      # [1, H, cells, 128]
    vt = torch.from_numpy(v).repeat_interleave(12, dim=0)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(mask))
    return o[0].permute(1, 0, 2).numpy()


def _run(w, lib, rows=None, **kw):
    sel = kw.pop("sel", w.sel)
    cnt = kw.pop("sel_count", w.sel_count)
    return oracle.attn_ref(kw.pop("q", w.q), kw.pop("k_pool", w.k_pool), kw.pop("v_pool", w.v_pool),
                           kw.pop("k_scale", w.k_scale), kw.pop("v_scale", w.v_scale),
                           kw.pop("page_table", w.page_table), sel, cnt, w.n_kv, w.sm_scale,
                           q_index=None if rows is None else np.asarray(rows), lib=lib)


# ----------------------------------------------------------------------------- pins
def pin_decoders(lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    h = oracle.half_to_double(bits, lib)
    ref = bits.view(np.float16).astype(np.float64)
    ok = ~np.isnan(ref)
    assert np.array_equal(h[ok], ref[ok]) and np.isnan(h[~ok]).all()
    b = oracle.bf16_to_double(bits, lib)
    refb = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    okb = ~np.isnan(refb)
    assert np.array_equal(b[okb], refb[okb]) and np.isnan(b[~okb]).all()


def pin_tiny_vs_sdpa(lib):
    w = gen.make(1)          # every causal cell: textbook causal attention
    rows = list(range(w.n_q))
    np.testing.assert_allclose(_run(w, lib), _sdpa(w, rows), rtol=1e-11, atol=1e-13)


def pin_lists_vs_sdpa(lib):
    w = _small()
    rows = list(range(w.n_q))
    np.testing.assert_allclose(_run(w, lib), _sdpa(w, rows), rtol=1e-11, atol=1e-13)


def pin_lists_vs_sdpa_nonresident(lib):
    w = gen.make(dict(SMALL, seed=12), nonresident_frac=0.3)
    rows = [i for i in range(w.n_q)]
    np.testing.assert_allclose(_run(w, lib), _sdpa(w, rows), rtol=1e-11, atol=1e-13)


def pin_single_cell(lib):
    w = _small()
    sel = np.full_like(w.sel, -1)
    cnt = np.ones_like(w.sel_count)
    cells = (w.q0 + np.arange(w.n_q)) - 5 * np.arange(w.n_q)
    sel[:, 0] = cells
    out = _run(w, lib, sel=sel, sel_count=cnt)
    for i, c in enumerate(cells):
        pp, r = w.page_table[c >> 6], c & 63
        for h in range(w.n_heads):
            kh = h // 12
            vref = w.v_pool[pp, kh, r].astype(np.float64) * float(w.v_scale[pp, kh, r])
            assert np.array_equal(out[i, h], vref)


def pin_equal_keys_mean(lib):
    w = _small()
    kp, ks = w.k_pool.copy(), w.k_scale.copy()
    # cells 64 and 130 get the same key (and scale) in every KV head; values differ
    pa, ra = w.page_table[1], 0
    pb, rb = w.page_table[2], 2
    kp[pb, :, rb] = kp[pa, :, ra]
    ks[pb, :, rb] = ks[pa, :, ra]
    sel = np.full_like(w.sel, -1)
    sel[:, 0], sel[:, 1] = 64, 130
    cnt = np.full_like(w.sel_count, 2)
    out = _run(w, lib, sel=sel, sel_count=cnt, k_pool=kp, k_scale=ks)
    for h in range(w.n_heads):
        kh = h // 12
        va = w.v_pool[pa, kh, ra].astype(np.float64) * float(w.v_scale[pa, kh, ra])
        vb = w.v_pool[pb, kh, rb].astype(np.float64) * float(w.v_scale[pb, kh, rb])
        assert np.array_equal(out[:, h], np.broadcast_to((va + vb) / 2, out[:, h].shape))


def pin_constant_v_per_head(lib):
    w = _small()
    vp = np.empty_like(w.v_pool)
    consts = [77, -31]
    for kh in range(w.n_kv):
        vp[:, kh] = consts[kh]
    vs = np.full_like(w.v_scale, np.float16(0.0234375))
    out = _run(w, lib, v_pool=vp, v_scale=vs)
    for h in range(w.n_heads):
        np.testing.assert_allclose(out[:, h], consts[h // 12] * 0.0234375, rtol=1e-14, atol=0)


def pin_page_permutation(lib):
    w = _small()
    base = _run(w, lib)
    perm = np.random.default_rng(5).permutation(w.n_ppages)      # physical page p moves to perm[p]
    inv = np.argsort(perm)
    out = _run(w, lib, k_pool=w.k_pool[inv], v_pool=w.v_pool[inv], k_scale=w.k_scale[inv],
               v_scale=w.v_scale[inv], page_table=perm[w.page_table].astype(np.int32))
    assert np.array_equal(out, base)


def pin_nonresident_is_dropped(lib):
    w = _small()
    pt = w.page_table.copy()
    drop = [3, 7, 11]
    pt[drop] = -1
    out = _run(w, lib, page_table=pt)
    sel = np.full_like(w.sel, -1)
    cnt = np.zeros_like(w.sel_count)
    for i in range(w.n_q):
        c = w.sel[i, : w.sel_count[i]]
        c = c[~np.isin(c >> 6, drop)]
        sel[i, : c.size] = c
        cnt[i] = c.size
    assert np.array_equal(out, _run(w, lib, sel=sel, sel_count=cnt))
    none = _run(w, lib, page_table=np.full_like(pt, -1))
    assert np.array_equal(none, np.zeros_like(none))


def pin_empty_and_bound(lib):
    w = _small()
    cnt = w.sel_count.copy()
    cnt[3] = 0
    out = _run(w, lib, sel_count=cnt)
    assert np.array_equal(out[3], np.zeros_like(out[3]))
    k, v = _dense_kv(w)
    for i in range(w.n_q):
        if cnt[i] == 0:
            continue
        c = w.sel[i, : cnt[i]]
        for h in range(w.n_heads):
            vv = v[h // 12, c]
            assert (out[i, h] <= vv.max(0) + 1e-12).all() and (out[i, h] >= vv.min(0) - 1e-12).all()


ATTN_PINS = [pin_tiny_vs_sdpa, pin_lists_vs_sdpa, pin_lists_vs_sdpa_nonresident, pin_single_cell,
             pin_equal_keys_mean, pin_constant_v_per_head, pin_page_permutation,
             pin_nonresident_is_dropped, pin_empty_and_bound]


def _py_union(w, g):
    lists = [set(w.sel[i, : w.sel_count[i]].tolist()) for i in range(8 * g, min(8 * g + 8, w.n_q))]
    cells = sorted(set().union(*lists))
    masks = [sum(1 << j for j, s in enumerate(lists) if c in s) for c in cells]
    return cells, masks


def pin_union_tiny_closed_form(lib):
    w = gen.make(1)   # queries 1528..1535, each selecting 0..p
    uc, um, un = oracle.union_ref(w.sel, w.sel_count, lib=lib)
    assert un[0] == 1536
    assert np.array_equal(uc[0, :1536], np.arange(1536))
    expect = np.full(1536, 0xFF, dtype=np.uint8)
    for t in range(1, 8):
        expect[1528 + t] = (0xFF << t) & 0xFF
    assert np.array_equal(um[0, :1536], expect)


def pin_union_bruteforce(lib):
    w = _small(n_q=21, drift=0.7)    # ragged: 2 full groups + 5
    uc, um, un = oracle.union_ref(w.sel, w.sel_count, lib=lib)
    for g in range(3):
        cells, masks = _py_union(w, g)
        assert un[g] == len(cells)
        assert uc[g, : un[g]].tolist() == cells and um[g, : un[g]].tolist() == masks
    assert (um[2, : un[2]] < (1 << 5)).all()            # ragged group: high bits zero
    pop = sum(bin(int(m)).count("1") for g in range(3) for m in um[g, : un[g]])
    assert pop == int(w.sel_count.sum())                 # every selection counted once


def pin_union_identical_lists(lib):
    w = _small()
    sel = np.repeat(w.sel[:1], 8, axis=0)
    cnt = np.repeat(w.sel_count[:1], 8)
    uc, um, un = oracle.union_ref(sel, cnt, lib=lib)
    assert un[0] == cnt[0]
    assert np.array_equal(uc[0, : un[0]], sel[0, : cnt[0]]) and (um[0, : un[0]] == 0xFF).all()


UNION_PINS = [pin_union_tiny_closed_form, pin_union_bruteforce, pin_union_identical_lists]


@pytest.mark.parametrize("pin", [pin_decoders] + ATTN_PINS + UNION_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_union_bruteforce_config2(workload, oracle_lib):
    w = workload(2)
    uc, um, un = oracle.union_ref(w.sel, w.sel_count, lib=oracle_lib)
    for g in range(0, w.n_groups, 7):
        cells, masks = _py_union(w, g)
        assert uc[g, : un[g]].tolist() == cells and um[g, : un[g]].tolist() == masks


def test_union_capacity_error(oracle_lib):
    w = _small()
    with pytest.raises(RuntimeError):
        oracle.union_ref(w.sel, w.sel_count, ustride=100, lib=oracle_lib)


# ------------------------------------------------------------- planted mistakes
MUTANTS = {
    "kv-head-mod": ("int32_t kh = h / HPK;", "int32_t kh = h % n_kv;"),
    "no-sm-scale": ("score[n_sel] = dot * sm_scale;", "score[n_sel] = dot;"),
    "softmax-sign": ("double p = exp(score[s] - m);", "double p = exp(m - score[s]);"),
    "cell-offset": ("(size_t)(c % PAGE);", "(size_t)((c + 1) % PAGE);"),
    "nonresident-as-page0": ("if (pp < 0) continue;", "if (pp < 0) pp = 0;"),
    "v-from-k": ("acc[d] += p * ((double)v_pool[r * D + d] * vs);",
                 "acc[d] += p * ((double)k_pool[r * D + d] * vs);"),
    "k-scale-from-v": ("double ks = qsa_ref_half_to_double(k_scale[r]);",
                       "double ks = qsa_ref_half_to_double(v_scale[r]);"),
    "half-exponent-bias": ("v = ldexp((double)(f + 1024), e - 25);", "v = ldexp((double)(f + 1024), e - 24);"),
    "bf16-no-implicit-one": ("v = ldexp((double)(f + 128), e - 134);", "v = ldexp((double)f, e - 134);"),
    "union-mask-shift": ("m |= (uint8_t)(1u << j);", "m |= (uint8_t)(1u << (nj - 1 - j));"),
    "union-no-dedup": ("if (n_u == 0 || all[t] != all[n_u - 1]) all[n_u++] = all[t];", "all[n_u++] = all[t];"),
    "row-normaliser": ("for (int d = 0; d < D; ++d) o[d] = acc[d] / z;", "for (int d = 0; d < D; ++d) o[d] = acc[d] / (z + 1e-3);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    if shutil.which(os.environ.get("CC", "gcc")) is None:
        pytest.skip("no C compiler")
    old, new = MUTANTS[name]
    src = open(build_oracle.SRC).read()
    assert src.count(old) == 1, "mutation site moved; update the planted mistake"
    msrc = tmp_path / "qsa_oracle.c"
    msrc.write_text(src.replace(old, new))
    lib_path = str(tmp_path / "libmutant.so")
    build_oracle.build(force=True, src=str(msrc), out=lib_path)
    lib = oracle.load(lib_path)
    caught = []
    for pin in [pin_decoders] + ATTN_PINS + UNION_PINS:
        try:
            pin(lib)
        except (AssertionError, RuntimeError):
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name!r} passed every pin"

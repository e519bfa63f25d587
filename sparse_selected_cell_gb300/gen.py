"""Seeded synthetic workloads for selected-cell (QSA union) prompt attention.

This module only *draws inputs*: per-position selection lists, a shuffled page
table, an INT8 K/V pool with FP16 per-cell scales, and BF16 queries.  It holds
none of the method's arithmetic (no union, no softmax, no attention), so both
the CUDA path and the CPU oracle can consume its output without sharing code.

Source: "sycl: prompt attention over 8-query selection unions on XMX" (Strata
PR #2808), sections Summary, Accuracy and Extra Notes: every prompt position
gathers its own sorted list of at most 2,051 selected K/V cells, INT8 K/V sits in
pages behind a shuffled page table, and timing runs use a "drift" knob that sets
how much neighbouring positions' selections differ.  The pages do not print the
selection layout, so the recipe below is this package's reading of it:

  For a query at position p with block b = p >> 6 (64-cell pages/blocks):
    1. the sink cells {0, 1, 2};
    2. the local blocks b-7 .. b (those >= 0), clipped to cells <= p;
    3. per group of 8 queries, a pool of 32 distinct blocks drawn uniformly
       from [0, b_min - 7), b_min = the group's lowest block;
    4. per position, 24 distinct blocks drawn uniformly from that pool;
    5. per position, each of those 24 blocks is replaced, independently with
       probability ``drift``, by a fresh block drawn uniformly from [0, b - 7)
       that is not already chosen.
  The list is the sorted, de-duplicated set of those cells, so
  count <= 3 + 32 * 64 = 2,051.

Random streams: ``numpy.random.default_rng([seed, stream])`` with one stream per
input (selections, page table, K, V, K scales, V scales, Q, residency).
Scales are drawn in FP64 and rounded to FP16; Q is drawn in FP32 and rounded to
BF16 (round to nearest even).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

HEAD_DIM = 128          # d
HEADS_PER_KV = 12       # grouped query heads per KV head
PAGE_CELLS = 64         # cells per page / block
GROUP = 8               # neighbouring positions that share one union
CAP = 2051              # selection cap: 3 sinks + 32 blocks of 64 cells
SEL_STRIDE = 2056       # row stride of the selection array (CAP rounded to 8)
UNION_STRIDE = 16448    # row stride of the union arrays (8 * CAP rounded to 64)

_STREAM_SEL, _STREAM_PT, _STREAM_K, _STREAM_V, _STREAM_KS, _STREAM_VS, _STREAM_Q, _STREAM_RES = range(8)

# The five synthetic workloads (context, queries, heads, drift, value ranges, seed).
CONFIGS = {
    1: dict(name="tiny-1.5k", ctx=1536, n_q=8, n_kv=1, select="causal", drift=0.0,
            scale_lo=0.01, scale_hi=0.03, q_sigma=1.0, seed=1),
    2: dict(name="ctx4k", ctx=4096, n_q=512, n_kv=4, select="blocks", drift=0.1,
            scale_lo=0.01, scale_hi=0.03, q_sigma=1.0, seed=2),
    3: dict(name="ctx16k", ctx=16384, n_q=2048, n_kv=4, select="blocks", drift=0.25,
            scale_lo=0.01, scale_hi=0.03, q_sigma=1.0, seed=3),
    4: dict(name="ctx40k-chunk8k", ctx=40960, n_q=8192, n_kv=4, select="blocks", drift=0.25,
            scale_lo=0.01, scale_hi=0.03, q_sigma=1.0, seed=4),
    5: dict(name="ctx64k-ragged", ctx=65536, n_q=8189, n_kv=8, select="blocks", drift=0.5,
            scale_lo=0.005, scale_hi=0.05, q_sigma=2.0, seed=5),
}


@dataclasses.dataclass
class Workload:
    """One synthetic prompt chunk.  Arrays are host numpy arrays.

    q          uint16 [n_q, n_kv*12, 128]   BF16 bit patterns
    k_pool     int8   [n_ppages, n_kv, 64, 128]
    v_pool     int8   [n_ppages, n_kv, 64, 128]
    k_scale    float16[n_ppages, n_kv, 64]
    v_scale    float16[n_ppages, n_kv, 64]
    page_table int32  [n_lpages]            physical page, or -1 if not resident
    sel        int32  [n_q, sel_stride]     sorted cell ids, -1 past the count
    sel_count  int32  [n_q]
    Query i sits at absolute position q0 + i.
    """
    name: str
    ctx: int
    q0: int
    n_q: int
    n_kv: int
    n_lpages: int
    n_ppages: int
    drift: float
    seed: int
    q: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray
    k_scale: np.ndarray
    v_scale: np.ndarray
    page_table: np.ndarray
    sel: np.ndarray
    sel_count: np.ndarray

    @property
    def n_heads(self) -> int:
        return self.n_kv * HEADS_PER_KV

    @property
    def sel_stride(self) -> int:
        return int(self.sel.shape[1])

    @property
    def n_groups(self) -> int:
        return (self.n_q + GROUP - 1) // GROUP

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(HEAD_DIM)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (nearest even) and return the bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(stream)])


def causal_selection(q0: int, n_q: int, stride: int = SEL_STRIDE):
    """Every causal cell 0..p for each query position p = q0 + i."""
    sel = np.full((n_q, stride), -1, dtype=np.int32)
    cnt = np.zeros(n_q, dtype=np.int32)
    for i in range(n_q):
        p = q0 + i
        if p + 1 > stride:
            raise ValueError("causal selection longer than the stride")
        sel[i, : p + 1] = np.arange(p + 1, dtype=np.int32)
        cnt[i] = p + 1
    return sel, cnt


def block_selection(q0: int, n_q: int, drift: float, rng: np.random.Generator,
                    stride: int = SEL_STRIDE, n_sinks: int = 3, n_local: int = 8,
                    pool_size: int = 32, n_drawn: int = 24):
    """Sinks + local window + drifting per-group block pool (recipe in the module doc)."""
    sel = np.full((n_q, stride), -1, dtype=np.int32)
    cnt = np.zeros(n_q, dtype=np.int32)
    offs = np.arange(PAGE_CELLS, dtype=np.int64)
    for g0 in range(0, n_q, GROUP):
        b_min = (q0 + g0) >> 6
        pool_hi = b_min - (n_local - 1)
        npool = min(pool_size, max(pool_hi, 0))
        pool = rng.choice(pool_hi, size=npool, replace=False) if npool > 0 else np.zeros(0, np.int64)
        for i in range(g0, min(g0 + GROUP, n_q)):
            p = q0 + i
            b = p >> 6
            ndraw = min(n_drawn, npool)
            drawn = [int(x) for x in rng.choice(pool, size=ndraw, replace=False)] if ndraw > 0 else []
            if drift > 0.0 and ndraw > 0:
                fresh_hi = b - (n_local - 1)
                chosen = set(drawn)
                for k in range(ndraw):
                    if rng.random() >= drift:
                        continue
                    free = fresh_hi - sum(1 for x in chosen if 0 <= x < fresh_hi)
                    if fresh_hi <= 0 or free <= 0:
                        continue
                    while True:
                        nb = int(rng.integers(0, fresh_hi))
                        if nb not in chosen:
                            break
                    chosen.discard(drawn[k])
                    drawn[k] = nb
                    chosen.add(nb)
            # drawn blocks lie below b-7 and the local window starts at b-7, so
            # the two block sets are disjoint; only the sinks can repeat (block 0).
            blocks = np.sort(np.asarray(drawn + list(range(max(0, b - n_local + 1), b + 1)),
                                        dtype=np.int64))
            cells = (blocks[:, None] * PAGE_CELLS + offs).ravel()
            cells = cells[cells <= p]
            if blocks.size == 0 or blocks[0] != 0:
                cells = np.concatenate([np.arange(min(n_sinks, p + 1), dtype=np.int64), cells])
            if cells.size > stride:
                raise ValueError("selection longer than the stride")
            sel[i, : cells.size] = cells
            cnt[i] = cells.size
    return sel, cnt


def make_pool(n_ppages: int, n_kv: int, scale_lo: float, scale_hi: float, seed: int):
    """INT8 K/V pages uniform in [-127, 127] and FP16 scales uniform in [lo, hi]."""
    shape = (n_ppages, n_kv, PAGE_CELLS, HEAD_DIM)
    k = _rng(seed, _STREAM_K).integers(-127, 128, size=shape, dtype=np.int8)
    v = _rng(seed, _STREAM_V).integers(-127, 128, size=shape, dtype=np.int8)
    ks = _rng(seed, _STREAM_KS).uniform(scale_lo, scale_hi, size=shape[:3]).astype(np.float16)
    vs = _rng(seed, _STREAM_VS).uniform(scale_lo, scale_hi, size=shape[:3]).astype(np.float16)
    return k, v, ks, vs


def make_page_table(n_lpages: int, seed: int, nonresident_frac: float = 0.0):
    """Seeded shuffled page table; a fraction of logical pages may be non-resident (-1)."""
    nonres = np.zeros(n_lpages, dtype=bool)
    if nonresident_frac > 0.0:
        n_off = int(round(nonresident_frac * n_lpages))
        if n_off > 0:
            off = _rng(seed, _STREAM_RES).choice(n_lpages, size=n_off, replace=False)
            nonres[off] = True
    n_ppages = int((~nonres).sum())
    pt = np.full(n_lpages, -1, dtype=np.int32)
    pt[~nonres] = _rng(seed, _STREAM_PT).permutation(n_ppages).astype(np.int32)
    return pt, n_ppages


def make_q(n_q: int, n_heads: int, sigma: float, seed: int) -> np.ndarray:
    x = _rng(seed, _STREAM_Q).standard_normal(size=(n_q, n_heads, HEAD_DIM), dtype=np.float32)
    if sigma != 1.0:
        x *= np.float32(sigma)
    b = x.view(np.uint32)
    lsb = b >> np.uint32(16)
    lsb &= np.uint32(1)
    b += np.uint32(0x7FFF)
    b += lsb
    b >>= np.uint32(16)
    return b.astype(np.uint16)


def make(config, seed: Optional[int] = None, nonresident_frac: float = 0.0,
         n_q: Optional[int] = None, drift: Optional[float] = None) -> Workload:
    """Build one workload from a config id (1..5) or a config dict.

    ``n_q`` keeps the config's context end but takes fewer queries (the last
    ``n_q`` positions before the chunk end); ``drift`` overrides the config's.
    """
    cfg = dict(CONFIGS[config]) if isinstance(config, int) else dict(config)
    if seed is not None:
        cfg["seed"] = seed
    if drift is not None:
        cfg["drift"] = drift
    ctx, n_kv, s = int(cfg["ctx"]), int(cfg["n_kv"]), int(cfg["seed"])
    nq_full = int(cfg["n_q"])
    q_end = ctx if "q_end" not in cfg else int(cfg["q_end"])
    q0 = q_end - nq_full
    nq = nq_full if n_q is None else int(n_q)
    q0 = q0 + (nq_full - nq)
    n_lpages = (ctx + PAGE_CELLS - 1) // PAGE_CELLS
    if cfg["select"] == "causal":
        sel, cnt = causal_selection(q0, nq)
    else:
        sel, cnt = block_selection(q0, nq, float(cfg["drift"]), _rng(s, _STREAM_SEL))
    pt, n_ppages = make_page_table(n_lpages, s, nonresident_frac)
    k, v, ks, vs = make_pool(n_ppages, n_kv, float(cfg["scale_lo"]), float(cfg["scale_hi"]), s)
    q = make_q(nq, n_kv * HEADS_PER_KV, float(cfg["q_sigma"]), s)
    return Workload(name=str(cfg.get("name", "custom")), ctx=ctx, q0=q0, n_q=nq, n_kv=n_kv,
                    n_lpages=n_lpages, n_ppages=n_ppages, drift=float(cfg["drift"]), seed=s,
                    q=q, k_pool=k, v_pool=v, k_scale=ks, v_scale=vs, page_table=pt,
                    sel=sel, sel_count=cnt)


# The decode workload the benchmark times (`bench.py --decode`): 1,024 sequences
# of 32,768 cells, 4 KV heads, pages drawn from a shared pool of 16,384 pages
# (1 GB of INT8 K and V, far above L2).
DECODE_BENCH = dict(n_seq=1024, ctx=32768, n_kv=4, n_ppages=16384, seed=11)


@dataclasses.dataclass
class DecodeWorkload:
    """One synthetic decode step over a batch of sequences.  Host numpy arrays.

    q           uint16 [n_seq, n_kv*12, 128]   BF16 bit patterns, one query per sequence
    k_pool ...  as in Workload, [n_ppages, n_kv, 64, 128] (shared by all sequences)
    page_tables int32  [n_seq, n_lpages]       sequence i's logical page -> physical page
    sel         int32  [n_seq, sel_stride]     sequence i's selection at its last position
    sel_count   int32  [n_seq]
    Every sequence holds ctx cells; its query sits at position ctx - 1.
    """
    ctx: int
    n_seq: int
    n_kv: int
    n_lpages: int
    n_ppages: int
    seed: int
    q: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray
    k_scale: np.ndarray
    v_scale: np.ndarray
    page_tables: np.ndarray
    sel: np.ndarray
    sel_count: np.ndarray

    @property
    def n_heads(self) -> int:
        return self.n_kv * HEADS_PER_KV

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(HEAD_DIM)


def make_decode(n_seq: int, ctx: int, n_kv: int, n_ppages: int, seed: int, nonresident_frac: float = 0.0,
                scale_lo: float = 0.01, scale_hi: float = 0.03, q_sigma: float = 1.0) -> DecodeWorkload:
    """A decode batch: n_seq sequences of ctx cells whose pages are drawn, each
    sequence without repeats, from one shared pool of n_ppages physical pages (so
    sequences may share pages, as prefix-sharing sequences do); each query selects
    by the block recipe at its position ctx - 1 (sinks, the local window and 24 of
    a 32-block pool; no drift: one position per sequence).  A fraction of every
    table may be marked not resident."""
    n_lpages = (ctx + PAGE_CELLS - 1) // PAGE_CELLS
    if n_lpages > n_ppages:
        raise ValueError("a sequence needs more pages than the pool holds")
    rng_pt = _rng(seed, _STREAM_PT)
    pts = np.empty((n_seq, n_lpages), dtype=np.int32)
    for i in range(n_seq):
        pts[i] = rng_pt.choice(n_ppages, size=n_lpages, replace=False).astype(np.int32)
    if nonresident_frac > 0.0:
        off = _rng(seed, _STREAM_RES).random(size=pts.shape) < nonresident_frac
        pts[off] = -1
    rng_sel = _rng(seed, _STREAM_SEL)
    sel = np.full((n_seq, SEL_STRIDE), -1, dtype=np.int32)
    cnt = np.zeros(n_seq, dtype=np.int32)
    for i in range(n_seq):
        s1, c1 = block_selection(ctx - 1, 1, 0.0, rng_sel)
        sel[i] = s1[0]
        cnt[i] = c1[0]
    k, v, ks, vs = make_pool(n_ppages, n_kv, scale_lo, scale_hi, seed)
    q = make_q(n_seq, n_kv * HEADS_PER_KV, q_sigma, seed)
    return DecodeWorkload(ctx=ctx, n_seq=n_seq, n_kv=n_kv, n_lpages=n_lpages, n_ppages=n_ppages, seed=seed,
                          q=q, k_pool=k, v_pool=v, k_scale=ks, v_scale=vs, page_tables=pts, sel=sel,
                          sel_count=cnt)

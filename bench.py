#!/usr/bin/env python
"""Benchmark: selected-cell (QSA union) prompt attention, query-head rows/s.

One step = the whole hot path over one synthetic prompt chunk resident in HBM:
union build (qsa_union_build) + union attention (qsa_union_attn).  The workload
is the 40,960-cell context with an 8,192-position chunk (positions 32,768-40,959),
4 KV heads x 12 query heads, d = 128, selections capped at 2,051 cells, drift 0.25.

Prints ONE JSON line (rank 0).  `value` = query-head rows/s of the whole job
(every rank processes its own independent chunk: weak scaling, no collective on
the data path).  `roofline` describes the attention kernel (the dominant one).
`e2e` repeats the measurement through the public call with pinned host buffers,
host->device inputs and device->host outputs inside the timed region.
`cpu_baseline` times the FP64 CPU oracle on a bounded sample on the host cores.
On one GPU the default run also nests `decode`: qsa_decode_attn over 1,024
sequences of 32,768 cells, one query each (its own workload, its own roofline;
--no-decode leaves it out, --decode prints it as the only line).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --config N            one of the five workloads (default 4)
  python bench.py --all-configs         one line per workload 1-5
  python bench.py <context> <queries> [reps] [--drift F] [--kv-heads H] [--seed S]
                                        a custom chunk: the last <queries> positions of a
                                        <context>-cell context, timed over [reps] steps
  python bench.py --fused               time qsa_fused_attn (the union built inside the
                                        attention CTA, one launch per step)
"""
import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "query-head rows/sec at 40K ctx, 2,051-cell cap; achieved % of HBM roofline"
UNIT = "query-head rows/s"
CONFIG_ID = 4   # the 40,960-cell context with an 8,192-position chunk: the headline workload


def rank_seed(rank: int, config: int = CONFIG_ID) -> int:
    """Seed of rank `rank`'s chunk: every rank runs its own independent chunk of the
    same shape (weak scaling; the path has no exchange step between ranks)."""
    from sparse_selected_cell_gb300 import gen
    return gen.CONFIGS[config]["seed"] + 1000 * rank


def max_over_ranks(x: float, device) -> float:
    """The slowest rank's figure (timing rule); the identity on a single process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rows_per_s(world: int, rows_per_step: int, steps: int, ms: float) -> float:
    """Whole-job throughput: the rows all ranks processed over the slowest rank's time."""
    return world * rows_per_step * steps / (ms / 1e3)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("context", type=int, nargs="?", default=None, help="custom chunk: context length in cells")
    p.add_argument("queries", type=int, nargs="?", default=None, help="custom chunk: query positions (the last ones)")
    p.add_argument("reps", type=int, nargs="?", default=None, help="custom chunk: timed steps")
    p.add_argument("--drift", type=float, default=None, help="selection drift (custom chunk; default 0.25)")
    p.add_argument("--kv-heads", type=int, default=None, help="KV heads (custom chunk; default 4)")
    p.add_argument("--seed", type=int, default=None, help="workload seed (custom chunk)")
    p.add_argument("--config", type=int, default=CONFIG_ID, choices=[1, 2, 3, 4, 5])
    p.add_argument("--all-configs", action="store_true", help="one line per workload 1-5")
    p.add_argument("--fused", action="store_true", help="time qsa_fused_attn instead of the launch pair")
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--variant", type=int, default=0,
                   help="0 default, 1 tcgen05 (two CTAs per SM), 2 tcgen05 (one CTA per SM)")
    p.add_argument("--e2e-steps", type=int, default=50)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-decode", action="store_true",
                   help="leave out the decode measurement nested in the default line")
    p.add_argument("--decode", action="store_true",
                   help="time decode over a batch of sequences (qsa_decode_attn) instead of the prompt chunk")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    p.add_argument("--drift-sweep", type=str, default=None,
                   help="comma-separated drift values: one line per value with the union ratio, the "
                        "union-build / attention times and the per-position path's time on the benchmark "
                        "workload (not the contract line)")
    p.add_argument("--n-q", type=int, default=None,
                   help="profiling only: take the last N query positions of the chunk (smaller capture)")
    return p.parse_args()


# GB300's nominal HBM3e bandwidth (~8 TB/s): the stricter denominator, reported
# beside the measured copy bandwidth.
NOMINAL_HBM_GBS = 8000.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def workload_desc(w):
    return (f"{w.name}: {w.ctx:,}-cell context, {w.n_q:,} queries (positions {w.q0:,}-{w.q0 + w.n_q - 1:,}), "
            f"{w.n_kv} KV heads x 12 query heads, d=128, 64-cell pages behind a shuffled page table, "
            f"cap 2,051 (3 sinks + 32 blocks), drift {w.drift}")


def algorithmic(w, union_count):
    """Bytes and FLOPs one attention launch must move / do (unpadded, exact unions)."""
    U = union_count.astype(np.int64)
    n_rows = w.n_q * w.n_heads
    kv = int(U.sum()) * w.n_kv * (128 + 128 + 2 + 2)
    q_out = n_rows * 128 * (2 + 4)
    union_reads = int(U.sum()) * w.n_kv * 5
    flops = int(U.sum()) * w.n_kv * 2 * 2 * 96 * 128
    union_build_bytes = int(w.sel_count.astype(np.int64).sum()) * 4 + int(U.sum()) * 5
    return dict(bytes=kv + q_out + union_reads, kv_bytes=kv, flops=flops, union_build_bytes=union_build_bytes,
                mean_union=float(U.mean()), union_ratio=float(U.mean() / w.sel_count.mean()))


def read_traffic(profile: str, kernel: str, sources, pdir: str = None):
    """DRAM bytes per launch from the committed ncu summary profiles/<profile>.txt
    (one kernel on one workload; `pdir` replaces profiles/), if it names `kernel`
    and the kernel's sources still hash to what the capture recorded; else None.
    Returns (bytes, hash)."""
    h = hashlib.sha256()
    for s in sources:
        h.update(open(os.path.join(ROOT, s), "rb").read())
    digest = h.hexdigest()[:16]
    path = os.path.join(pdir or os.path.join(ROOT, "profiles"), profile + ".txt")
    if not os.path.isfile(path):
        return None, digest
    txt = open(path).read()
    m_k = re.search(r"^kernel:\s*(\S+)", txt, re.M)
    m_h = re.search(r"^source_sha256_16:\s*(\S+)", txt, re.M)
    m_t = re.search(r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt, re.M)
    if m_k and m_h and m_t and m_k.group(1) == kernel and m_h.group(1) == digest:
        return float(m_t.group(1)), digest
    return None, digest


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""
    Q = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id):
        self.bus_id = (bus_id or "").lower()
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        rows = []
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 10:
                continue
            if self.bus_id and self.bus_id[-12:] not in f[1].lower():
                continue
            rows.append(f)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v.lower() == "active"})
        pw = [float(r[4]) for r in rows if re.match(r"^[0-9.]+$", r[4])]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


def oracle_sample(w, seconds, threads=0, start=0, fixed_n=None):
    """Time the FP64 oracle on consecutive query positions; returns (rows/s, n_positions, secs, cores)."""
    from oracle import oracle
    n = fixed_n
    if n is None:
        n = 16
        while True:
            idx = (start + np.arange(n)) % w.n_q
            t0 = time.perf_counter()
            oracle.attn_ref_workload(w, q_index=idx.astype(np.int32), n_threads=threads)
            dt = time.perf_counter() - t0
            if dt >= 0.5 or n >= w.n_q:
                break
            n *= 4
        n = int(min(w.n_q, max(n, round(n * seconds / max(dt, 1e-6)))))
    idx = (start + np.arange(n)) % w.n_q
    t0 = time.perf_counter()
    oracle.attn_ref_workload(w, q_index=idx.astype(np.int32), n_threads=threads)
    dt = time.perf_counter() - t0
    return n * w.n_heads / dt, n, dt, oracle.max_threads() if threads <= 0 else threads


def run_reference(args):
    """Reference arm: the FP64 CPU oracle, as it stands, on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from sparse_selected_cell_gb300 import gen
    w = gen.make(args.config)
    n_steps = args.steps + args.warmup
    # size each step's sample so the whole run stays within about two minutes
    rate, n, dt, cores = oracle_sample(w, 0.5)
    per_step = max(1, int(n * min(1.0, 110.0 / n_steps) / max(dt, 1e-3)))
    per_step = min(per_step, w.n_q)
    rows, secs = 0, 0.0
    for s in range(n_steps):
        r, nn, t, cores = oracle_sample(w, 0, start=s * per_step, fixed_n=per_step)
        if s >= args.warmup:
            rows += nn * w.n_heads
            secs += t
    value = rows / secs
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(w), "oracle": "FP64 CPU oracle (OpenMP), per-position lists",
                       "sampled": f"each step times {per_step} of the workload's {w.n_q:,} query positions "
                                  f"(consecutive, all {w.n_heads} heads); value is rows/s over those samples"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{per_step} consecutive query positions (all {w.n_heads} heads) per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def drift_sweep(args):
    """Time of the union path against the union ratio: the benchmark workload with
    the selection drift varied (the union pages' chunk-timing table, Extra Notes)."""
    import torch
    from sparse_selected_cell_gb300 import build as qbuild
    from sparse_selected_cell_gb300 import gen, qsa
    torch.cuda.set_device(0)
    qbuild.build()
    for drift in (float(x) for x in args.drift_sweep.split(",")):
        w = gen.make(CONFIG_ID, drift=drift)
        d = qsa.to_device(w)
        ws = torch.empty(qsa.workspace_bytes(w.n_q), dtype=torch.uint8, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.empty((w.n_q, w.n_heads, 128), dtype=torch.float32, device="cuda")
        G, S = w.n_groups, gen.UNION_STRIDE
        cb = G * S * 4
        mo = (cb + 255) // 256 * 256
        co = mo + (G * S + 255) // 256 * 256
        uc, um, un = ws[:cb].view(torch.int32).view(G, S), ws[mo:mo + G * S].view(G, S), ws[co:co + G * 4].view(torch.int32)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ub, at = [], []
        for k in range(args.warmup + args.steps):
            ev[0].record()
            qsa.union_build(d["sel"], d["sel_count"], S, out=(uc, um, un), dev_status=st)
            ev[1].record()
            qsa.union_attn(d["q"], d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"], d["page_table"], uc, um, un,
                           out=out, variant=args.variant, dev_status=st)
            ev[2].record()
            torch.cuda.synchronize()
            if k >= args.warmup:
                ub.append(ev[0].elapsed_time(ev[1]))
                at.append(ev[1].elapsed_time(ev[2]))
        # the per-position path (no union) on the same inputs: every position gathers its own cells
        sl = []
        for k in range(args.warmup + args.steps):
            ev[0].record()
            qsa.select_attn(d["q"], d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"], d["page_table"],
                            d["sel"], d["sel_count"], out=out, dev_status=st)
            ev[1].record()
            torch.cuda.synchronize()
            if k >= args.warmup:
                sl.append(ev[0].elapsed_time(ev[1]))
        alg = algorithmic(w, un.cpu().numpy())
        attn = sum(at) / len(at)
        sel_ms = sum(sl) / len(sl)
        sel_bytes = int(w.sel_count.astype(np.int64).sum()) * w.n_kv * 260 + w.n_q * w.n_heads * 128 * 6
        print(json.dumps({"sweep": "drift", "drift": drift, "union_ratio": round(alg["union_ratio"], 3),
                          "mean_union_cells": round(alg["mean_union"], 1), "union_build_ms": sum(ub) / len(ub),
                          "attn_ms": attn, "rows_per_s": w.n_q * w.n_heads / ((attn + sum(ub) / len(ub)) / 1e3),
                          "attn_gb_per_s": alg["bytes"] / (attn / 1e3) / 1e9,
                          "ns_per_union_cell_head": attn * 1e6 / (alg["mean_union"] * w.n_groups * w.n_kv),
                          "per_position_ms": sel_ms, "per_position_gb_per_s": sel_bytes / (sel_ms / 1e3) / 1e9,
                          "union_path_speedup": sel_ms / (attn + sum(ub) / len(ub)),
                          "status": int(st.item())}), flush=True)


def decode_bench(args):
    """`--decode`: the decode measurement below as its own JSON line."""
    import torch
    from sparse_selected_cell_gb300 import build as qbuild
    torch.cuda.set_device(0)
    qbuild.build()
    print(json.dumps(decode_measure(args.steps, args.warmup)), flush=True)


def decode_measure(steps: int, warmup: int) -> dict:
    """Decode over a batch of sequences (qsa_decode_attn): one query per sequence,
    each with its own page table into one shared 1 GB pool (far above L2), timed
    with CUDA events over `steps` launches after `warmup` untimed ones."""
    import torch
    from sparse_selected_cell_gb300 import gen, qsa
    w = gen.make_decode(**gen.DECODE_BENCH)

    def dev(x):
        return torch.from_numpy(np.ascontiguousarray(x)).cuda()
    q, kp, vp = dev(w.q), dev(w.k_pool), dev(w.v_pool)
    ks, vs = dev(w.k_scale.view(np.int16)), dev(w.v_scale.view(np.int16))
    pts, sel, cnt = dev(w.page_tables), dev(w.sel), dev(w.sel_count)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((w.n_seq, w.n_heads, 128), dtype=torch.float32, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    for _ in range(max(3, warmup)):
        qsa.decode_attn(q, kp, vp, ks, vs, pts, sel, cnt, out=out, dev_status=st)
    torch.cuda.synchronize()
    ev[0].record()
    for _ in range(steps):
        qsa.decode_attn(q, kp, vp, ks, vs, pts, sel, cnt, out=out, dev_status=st)
    ev[1].record()
    torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[1]) / steps
    hbm, _, _, src = peaks()
    resident = w.page_tables[np.arange(w.n_seq)[:, None], np.where(w.sel >= 0, w.sel >> 6, 0)] >= 0
    cells = int((resident & (np.arange(w.sel.shape[1])[None, :] < w.sel_count[:, None])).sum())
    alg = cells * w.n_kv * 260 + w.n_seq * w.n_heads * 128 * 6
    achieved = alg / (ms / 1e3) / 1e9
    traffic, digest = read_traffic("select_attn_kernel_decode1k-ctx32k", "select_attn_kernel",
                                   ["sparse_selected_cell_gb300/csrc/select_attn.cu",
                                    "sparse_selected_cell_gb300/csrc/qsa_common.cuh"])
    return dict({"mode": "decode", "metric": "decode query-head rows/s", "unit": "query-head rows/s",
                      "value": w.n_seq * w.n_heads / (ms / 1e3), "ms_per_step": ms, "steps": steps,
                      "warmup": max(3, warmup), "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
                      "config": {"workload": f"decode: {w.n_seq:,} sequences x {w.ctx:,} cells, {w.n_kv} KV heads "
                                             f"x 12, one query per sequence, page tables into a shared pool of "
                                             f"{w.n_ppages:,} pages", "l2": "pool of %.2f GB, above L2"
                                             % ((w.k_pool.nbytes + w.v_pool.nbytes) / 1e9)},
                      "roofline": {"bound": "hbm", "kernel": "select_attn_kernel", "achieved": achieved, "peak": hbm,
                                   "unit": "GB/s", "frac": achieved / hbm, "peak_source": src,
                                   "nominal_peak": NOMINAL_HBM_GBS, "frac_nominal": achieved / NOMINAL_HBM_GBS,
                                   "algorithmic_bytes_per_launch": alg, "traffic": traffic,
                                   "traffic_over_algorithmic": (traffic / alg) if traffic else None,
                                   "source_sha256_16": digest},
                      "status": int(st.item())})


def custom_config(args, rank: int):
    """The page's CLI shape: the last <queries> positions of a <context>-cell context
    with the headline workload's value ranges."""
    from sparse_selected_cell_gb300 import gen
    cfg = dict(gen.CONFIGS[CONFIG_ID])
    cfg.update(name=f"custom-ctx{args.context}-q{args.queries}", ctx=int(args.context), n_q=int(args.queries))
    if args.kv_heads is not None:
        cfg["n_kv"] = int(args.kv_heads)
    if args.drift is not None:
        cfg["drift"] = float(args.drift)
    cfg["seed"] = (args.seed if args.seed is not None else cfg["seed"]) + 1000 * rank
    return cfg


def measure(args, w, dev, world: int, rank: int, headline: bool):
    """Times one workload; returns rank 0's JSON line (None on other ranks)."""
    import torch
    from sparse_selected_cell_gb300 import gen, qsa

    d = qsa.to_device(w, dev)
    stream = torch.cuda.current_stream()
    ws = torch.empty(qsa.workspace_bytes(w.n_q), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty((w.n_q, w.n_heads, 128), dtype=torch.float32, device=dev)
    n_groups = w.n_groups
    stride = gen.UNION_STRIDE
    cells_b = n_groups * stride * 4
    mask_off = (cells_b + 255) // 256 * 256
    cnt_off = mask_off + (n_groups * stride + 255) // 256 * 256
    ucell = ws[:cells_b].view(torch.int32).view(n_groups, stride)
    umask = ws[mask_off:mask_off + n_groups * stride].view(n_groups, stride)
    ucount = ws[cnt_off:cnt_off + n_groups * 4].view(torch.int32)
    # the union counts for the algorithmic bytes come from the launch pair's union build
    qsa.union_build(d["sel"], d["sel_count"], stride, out=(ucell, umask, ucount), dev_status=status, stream=stream)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        if args.fused:
            if ev is not None:
                ev[1].record(stream)
            qsa.fused_attn(d["q"], d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"], d["page_table"], d["sel"],
                           d["sel_count"], out=out, dev_status=status, stream=stream)
        else:
            qsa.union_build(d["sel"], d["sel_count"], stride, out=(ucell, umask, ucount), dev_status=status,
                            stream=stream)
            if ev is not None:
                ev[1].record(stream)
            qsa.union_attn(d["q"], d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"], d["page_table"], ucell,
                           umask, ucount, out=out, variant=args.variant, dev_status=status, stream=stream)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {qsa.decode_status(int(status.item()))}")
    alg = algorithmic(w, ucount.cpu().numpy())
    steps = args.steps

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except Exception:
        pass
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(bus) as clk:
        t0.record(stream)
        for k in range(steps):
            step(evs[k])
        t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = t0.elapsed_time(t1)
    attn_ms = [e[1].elapsed_time(e[2]) for e in evs]
    union_ms = [e[0].elapsed_time(e[1]) for e in evs]
    total_ms = max_over_ranks(total_ms, dev)
    rows_per_step = w.n_q * w.n_heads
    value = job_rows_per_s(world, rows_per_step, steps, total_ms)

    # End to end through the public call: every step copies all of its inputs from
    # pinned host memory and reads its output back to pinned host memory.  Steps run
    # as a serving loop would run them: host-to-device copies, compute and
    # device-to-host copies on three streams, over two device buffer sets, so step
    # k+1's inputs travel while step k computes and step k-1's output travels back.
    e2e_steps = args.e2e_steps if headline else 0
    host = {k: v.cpu().pin_memory() for k, v in d.items()}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out.numel() * out.element_size()
    e2e_ms = float("nan")
    if e2e_steps > 0:
        host_outs = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        bufs = [{k: torch.empty_like(v) for k, v in d.items()} for _ in range(2)]
        outs = [out, torch.empty_like(out)]
        wss = [ws, torch.empty_like(ws)]
        s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
        ev_in, ev_cmp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

        def e2e_step(k):
            b = k % 2
            s_in.wait_event(ev_cmp[b])                 # step k-2 is done reading buffer set b
            with torch.cuda.stream(s_in):
                for name, v in host.items():
                    bufs[b][name].copy_(v, non_blocking=True)
            ev_in[b].record(s_in)
            s_cmp.wait_event(ev_in[b])
            s_cmp.wait_event(ev_out[b])                # step k-2's output has been read back
            dd = bufs[b]
            if args.fused:
                qsa.fused_attn(dd["q"], dd["k_pool"], dd["v_pool"], dd["k_scale"], dd["v_scale"], dd["page_table"],
                               dd["sel"], dd["sel_count"], out=outs[b], dev_status=status, stream=s_cmp)
            else:
                qsa.prompt_attn(dd["q"], dd["k_pool"], dd["v_pool"], dd["k_scale"], dd["v_scale"], dd["page_table"],
                                dd["sel"], dd["sel_count"], out=outs[b], workspace=wss[b], variant=args.variant,
                                dev_status=status, stream=s_cmp)
            ev_cmp[b].record(s_cmp)
            s_out.wait_event(ev_cmp[b])
            with torch.cuda.stream(s_out):
                host_outs[b].copy_(outs[b], non_blocking=True)
            ev_out[b].record(s_out)

        for k in range(3):
            e2e_step(k)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for k in range(e2e_steps):
            e2e_step(k)
        e1.record(s_out)                           # after the last read-back, which follows everything
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, dev)
    e2e_value = job_rows_per_s(world, rows_per_step, e2e_steps, e2e_ms) if e2e_steps > 0 else None
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {qsa.decode_status(int(status.item()))}")
    if rank != 0:
        return None

    hbm, bf16, bf16_sus, src = peaks()
    attn_avg = sum(attn_ms) / len(attn_ms)
    abytes = alg["bytes"]
    if args.fused:   # the fused kernel reads each group's lists (once per KV head) instead of the union arrays
        abytes = alg["bytes"] - int(ucount.cpu().numpy().astype(np.int64).sum()) * w.n_kv * 5 \
            + int(w.sel_count.astype(np.int64).sum()) * 4 * w.n_kv
    achieved = abytes / (attn_avg / 1e3) / 1e9
    tflops = alg["flops"] / (attn_avg / 1e3) / 1e12
    t_hbm = abytes / (hbm * 1e9) * 1e3
    t_tc = alg["flops"] / (bf16_sus * 1e12) * 1e3
    resolved = args.variant or qsa.default_variant()
    if args.fused:
        kernel, files, vname = ("attn_sm_kernel", ("attn_sm.cu", "tc_ptx.cuh", "union_core.cuh"),
                                "fused (union built in the CTA)")
    else:
        kernel, files = {qsa.ATTN_TCGEN05: ("attn_tc_kernel", ("attn_tc.cu", "tc_ptx.cuh")),
                         qsa.ATTN_TCGEN05_SM: ("attn_sm_kernel", ("attn_sm.cu", "tc_ptx.cuh"))}[resolved]
        vname = {1: "tcgen05, two CTAs per SM", 2: "tcgen05, one CTA per SM"}[resolved]
    srcs = ["sparse_selected_cell_gb300/csrc/" + f for f in files + ("qsa_common.cuh",)]
    # a capture covers one named workload at its full size and drift
    named = next((c for c in gen.CONFIGS.values() if c["name"] == w.name), None)
    full = named is not None and w.n_q == named["n_q"] and w.drift == named["drift"]
    profile = f"{kernel}{'_fused' if args.fused else ''}_{w.name}"
    traffic, digest = read_traffic(profile, kernel, srcs) if full else (None, None)
    in_bytes = sum(v.numel() * v.element_size() for v in d.values())
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": total_ms / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(w),
                   "l2": "inputs above L2 (%.0f MB read + %.0f MB written per step), so no step starts with "
                         "them in L2; the 42.6 MB KV pool itself is gathered ~2.7x per launch and stays "
                         "L2-resident within a launch (DRAM traffic / algorithmic bytes below)"
                         % (in_bytes / 1e6, out.numel() * 4 / 1e6),
                   "mean_union_cells": round(alg["mean_union"], 1), "union_ratio": round(alg["union_ratio"], 3),
                   "variant": vname, "parallelism": f"dp{world}"},
        "roofline": {"bound": "hbm" if t_hbm >= t_tc else "tensor", "kernel": kernel,
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": traffic,
                     "traffic_over_algorithmic": (traffic / abytes) if traffic else None,
                     "peak_source": src,
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_nominal": achieved / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": abytes, "flops_per_launch": alg["flops"],
                     "attn_ms": attn_avg, "tflops": tflops, "tensor_frac_sustained": tflops / bf16_sus,
                     "roofline_ms": max(t_hbm, t_tc),
                     "union_build_ms": None if args.fused else sum(union_ms) / len(union_ms),
                     "source_sha256_16": digest},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps,
                "pipeline": "copy-in, compute and copy-out streams over two buffer sets"},
        "gpu_launches": (1 if args.fused else 2) * steps,
        "clocks": clk.summary(),
    }
    if world == 1 and not args.no_cpu_baseline:
        rate, n, dt, cores = oracle_sample(w, args.cpu_seconds if headline else min(args.cpu_seconds, 4.0))
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"{n} consecutive query positions x {w.n_heads} heads of the same "
                                          f"chunk ({dt:.1f} s, FP64, OpenMP)"}
    return line


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.drift_sweep:
        return drift_sweep(args)
    if args.decode:
        return decode_bench(args)

    import torch
    from sparse_selected_cell_gb300 import build as qbuild
    from sparse_selected_cell_gb300 import gen, qsa

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    if rank == 0:
        qbuild.build()
    if world > 1:
        torch.distributed.barrier()
    qsa.lib()

    # every rank runs its own independent chunk of the same shape (weak scaling)
    if args.context is not None:
        if args.queries is None:
            raise SystemExit("a custom chunk needs <context> <queries>")
        if args.reps is not None:
            args.steps = int(args.reps)
        jobs = [(gen.make(custom_config(args, rank)), True)]
    elif args.all_configs:
        jobs = [(gen.make(cfg, seed=rank_seed(rank, cfg)), cfg == CONFIG_ID) for cfg in (1, 2, 3, 4, 5)]
    else:
        cfg = args.config
        jobs = [(gen.make(cfg, seed=rank_seed(rank, cfg), n_q=args.n_q), True)]
    for w, headline in jobs:
        line = measure(args, w, dev, world, rank, headline)
        del w
        torch.cuda.empty_cache()
        if line is not None and headline and world == 1 and not (args.no_decode or args.fused) and args.context is None \
                and args.config == CONFIG_ID and args.n_q is None and not args.all_configs:
            # the decode path on its own workload, nested in the same line (one line per run)
            line["decode"] = decode_measure(min(args.steps, 100), args.warmup)
            torch.cuda.empty_cache()
        if line is not None:
            print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

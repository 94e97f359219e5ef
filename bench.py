#!/usr/bin/env python
"""Benchmark: one long-context decoder layer of dynamic sparse prefill attention.

A step is one pass of the whole hot path over one layer's attention: online
estimation of the vertical-slash heads' indices, vertical-slash sparse
attention, block-sparse selection + attention and A-shape attention, all
through the C ABI of libmi.so.  The default workload is the mixed-pattern
layer at 128K tokens (32 q heads / 8 KV heads, d = 128; 24 vertical-slash
heads with 1000 columns / 6096 diagonals, 4 block-sparse heads keeping 100
blocks per row block, 4 A-shape heads with 128 sink tokens and a 4096-token
window) on seeded synthetic inputs.

Prints one JSON line.  `--impl reference` times the CPU oracle instead, on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "ms/layer & dense-equivalent speedup at 128K/1M tokens; % of bf16 tensor peak"

WORKLOADS = {
    "mixed-128k": dict(Hq=32, Hkv=8, N=131072, n_vs=24, n_block=4, n_ashape=4, k_v=1000, k_s=6096,
                       topk=100, n_init=128, window=4096, n_cols=16, n_offsets=8, seed=3),
    "vs-32k": dict(Hq=32, Hkv=8, N=32768, n_vs=32, n_block=0, n_ashape=0, k_v=1000, k_s=6096,
                   topk=100, n_init=128, window=4096, n_cols=16, n_offsets=8, seed=2),
    "vs-1m": dict(Hq=32, Hkv=8, N=1048576, n_vs=32, n_block=0, n_ashape=0, k_v=1000, k_s=6096,
                  topk=100, n_init=128, window=4096, n_cols=16, n_offsets=8, seed=4),
    "vs-4k": dict(Hq=1, Hkv=1, N=4096, n_vs=1, n_block=0, n_ashape=0, k_v=64, k_s=32, topk=100,
                  n_init=128, window=4096, n_cols=8, n_offsets=4, seed=1),
}
KERNELS_PER_STEP = {"vs": 6, "block": 4, "ashape": 1}  # estimate 4 + index 1 + attention 1, ...


def describe(w):
    parts = [f"{w['Hq']}q/{w['Hkv']}kv heads, d=128, N={w['N']}"]
    if w["n_vs"]:
        parts.append(f"{w['n_vs']} vertical-slash heads (top {w['k_v']} columns / {w['k_s']} diagonals)")
    if w["n_block"]:
        parts.append(f"{w['n_block']} block-sparse heads (top {w['topk']} 64x64 blocks)")
    if w["n_ashape"]:
        parts.append(f"{w['n_ashape']} A-shape heads ({w['n_init']} sink + {w['window']} window)")
    return "; ".join(parts)


def head_patterns(w):
    g = torch.Generator().manual_seed(w["seed"])
    perm = torch.randperm(w["Hq"], generator=g).tolist()
    a, b = w["n_vs"], w["n_vs"] + w["n_block"]
    return sorted(perm[:a]), sorted(perm[a:b]), sorted(perm[b:b + w["n_ashape"]])


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), float(p["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


# ------------------------------------------------------------------ clocks ----

class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for ln in f:
                    p = [x.strip() for x in ln.split(",")]
                    if len(p) >= 9:
                        rows.append(p)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        load = [s for s in sm if mx and s > 0.3 * max(mx)] or sm
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------- the layer ----

class Layer:
    """Device tensors, index buffers and workspaces for one layer; step() runs the hot path."""

    def __init__(self, B, w, q, k, v):
        self.B, self.w = B, w
        self.q, self.k, self.v = q, k, v
        dev = q.device
        N, Hkv = w["N"], w["Hkv"]
        self.vs, self.blk, self.ash = head_patterns(w)
        self.out = torch.zeros_like(q)
        nv, nb = len(self.vs), len(self.blk)
        self.v_idx = torch.empty((max(nv, 1), w["k_v"]), dtype=torch.int32, device=dev)
        self.s_idx = torch.empty((max(nv, 1), w["k_s"]), dtype=torch.int32, device=dev)
        self.blk_idx = torch.empty((max(nb, 1), N // 64, w["topk"]), dtype=torch.int32, device=dev)

        def ws(op, n):
            return torch.empty(max(256, B.mi_workspace_bytes(op, max(n, 1), Hkv, N, w["k_v"], w["k_s"], w["topk"])),
                               dtype=torch.uint8, device=dev)
        self.ws_est = ws(B.MI_OP_VS_ESTIMATE, nv)
        self.ws_vs = ws(B.MI_OP_VS_SPARSE_ATTN, nv)
        self.ws_blk = ws(B.MI_OP_BLOCK_SPARSE_ATTN, nb)
        self.ws_ash = ws(B.MI_OP_ASHAPE_ATTN, 1)
        self.ws_dense = ws(B.MI_OP_DENSE_CAUSAL_ATTN, 1)
        self.expanded = False  # vertical-slash heads in the block-expanded slash mode
        self.kernels_per_step = (KERNELS_PER_STEP["vs"] if nv else 0) + (KERNELS_PER_STEP["block"] if nb else 0) \
            + (KERNELS_PER_STEP["ashape"] if self.ash else 0)

    def step(self, ev=None):
        B, w = self.B, self.w
        if ev:
            ev[0].record()
        if self.vs:
            B.mi_vs_estimate(self.q, self.k, heads=self.vs, k_v=w["k_v"], k_s=w["k_s"], v_idx=self.v_idx,
                             s_idx=self.s_idx, workspace=self.ws_est)
            if ev:
                ev[1].record()
            B.mi_vs_sparse_attn(self.q, self.k, self.v, self.v_idx, self.s_idx, heads=self.vs, out=self.out,
                                workspace=self.ws_vs, expanded=self.expanded)
        elif ev:
            ev[1].record()
        if ev:
            ev[2].record()
        if self.blk:
            B.mi_block_sparse_attn(self.q, self.k, self.v, topk=w["topk"], heads=self.blk, blk_idx=self.blk_idx,
                                   out=self.out, workspace=self.ws_blk)
        if ev:
            ev[3].record()
        if self.ash:
            B.mi_ashape_attn(self.q, self.k, self.v, n_init=w["n_init"], window=w["window"], heads=self.ash,
                             out=self.out, workspace=self.ws_ash)
        if ev:
            ev[4].record()

    def step_group(self, hs):
        """The hot path for the q-heads in ``hs`` only (a KV group or several): the same calls as
        step() on a subset of the heads, writing their rows of the index buffers and of out."""
        B, w = self.B, self.w
        vs = [h for h in self.vs if h in hs]
        blk = [h for h in self.blk if h in hs]
        ash = [h for h in self.ash if h in hs]
        if vs:
            i0 = self.vs.index(vs[0])
            vi, si = self.v_idx[i0:i0 + len(vs)], self.s_idx[i0:i0 + len(vs)]
            B.mi_vs_estimate(self.q, self.k, heads=vs, k_v=w["k_v"], k_s=w["k_s"], v_idx=vi, s_idx=si,
                             workspace=self.ws_est)
            B.mi_vs_sparse_attn(self.q, self.k, self.v, vi, si, heads=vs, out=self.out, workspace=self.ws_vs,
                                expanded=self.expanded)
        if blk:
            j0 = self.blk.index(blk[0])
            B.mi_block_sparse_attn(self.q, self.k, self.v, topk=w["topk"], heads=blk,
                                   blk_idx=self.blk_idx[j0:j0 + len(blk)], out=self.out, workspace=self.ws_blk)
        if ash:
            B.mi_ashape_attn(self.q, self.k, self.v, n_init=w["n_init"], window=w["window"], heads=ash,
                             out=self.out, workspace=self.ws_ash)

    def dense(self):
        self.B.mi_dense_causal_attn(self.q, self.k, self.v, out=self.out, workspace=self.ws_dense)

    def layer_cfg(self):
        """The same layer as one mi_layer_attn configuration (one entry per q-head)."""
        B, w = self.B, self.w
        cfg = [B.HeadCfg.skip() for _ in range(w["Hq"])]
        for h in self.vs:
            cfg[h] = B.HeadCfg.vs(w["k_v"], w["k_s"], expanded=self.expanded)
        for h in self.blk:
            cfg[h] = B.HeadCfg.block(w["topk"])
        for h in self.ash:
            cfg[h] = B.HeadCfg.ashape(w["n_init"], w["window"])
        return cfg

    def step_layer(self, ev=None):
        """One layer through the single layer call (estimation, selection, one attention launch)."""
        if not hasattr(self, "_cfg"):
            self._cfg = self.layer_cfg()
            self._ws_layer = torch.empty(self.B.mi_layer_workspace_bytes(self.w["Hq"], self.w["Hkv"], self.w["N"],
                                                                         self._cfg),
                                         dtype=torch.uint8, device=self.q.device)
        self.B.mi_layer_attn(self.q, self.k, self.v, self._cfg, out=self.out, workspace=self._ws_layer)

    def check_status(self):
        used = ([self.ws_est, self.ws_vs] if self.vs else []) + ([self.ws_blk] if self.blk else []) \
            + ([self.ws_ash] if self.ash else [])
        for ws in used:
            st = self.B.mi_read_status(ws)
            if st not in (0,):
                raise RuntimeError(f"device status {st}: {self.B.mi_strerror(st)}")

    def work(self):
        """(algorithmic FLOPs per head group, executed tile FLOPs) of one step, from the indices."""
        from dynamic_sparse_attention_vertical_gb300 import flops as F
        w, N = self.w, self.w["N"]
        dev = self.q.device
        alg = {"vs": 0, "block": 0, "ashape": 0}
        tiles = {"vs": 0, "block": 0, "ashape": 0}
        vi = self.v_idx.cpu().numpy()
        si = self.s_idx.cpu().numpy()
        for n in range(len(self.vs)):
            if self.expanded:
                alg["vs"] += int(F.vs_expanded_kept_per_row(N, vi[n], si[n]).sum())
            else:
                alg["vs"] += int(F.vs_kept_per_row(N, vi[n], si[n], device=dev).sum())
            tiles["vs"] += F.vs_tiles(N, vi[n], si[n], expanded=self.expanded)
        bl = self.blk_idx.cpu().numpy()
        for n in range(len(self.blk)):
            sel = [r[r >= 0] for r in bl[n]]
            alg["block"] += int(F.block_kept_per_row(N, sel).sum())
            tiles["block"] += F.block_tiles(sel)
        if self.ash:
            alg["ashape"] = len(self.ash) * int(F.ashape_kept_per_row(N, w["n_init"], w["window"]).sum())
            tiles["ashape"] = len(self.ash) * F.ashape_tiles(N, w["n_init"], w["window"])
        return ({k2: 4 * F.D * v2 for k2, v2 in alg.items()}, {k2: F.TILE_FLOPS * v2 for k2, v2 in tiles.items()})


# DRAM bytes (read + write) of one vertical-slash attention launch from a one-pass ncu capture,
# with the SHA-256 of the kernel sources it was taken on.  The figure is reported only while
# those sources are unchanged (kernel_sources_sha256() at run time); otherwise traffic is null.
TRAFFIC = {("mixed-128k", "literal"): {"sources_sha256": "4a48c942186e7dd4a07b6a6bbd32d5b44fd4ef43a59d55c570f06686ef2abaf3",
                                      "bytes": 2264800256 + 785736960}}
KERNEL_SOURCES = ("attention.cuh", "ptx.cuh", "common.cuh", "vs_index.cuh", "attn_launch.cuh")


def kernel_sources_sha256():
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "dynamic_sparse_attention_vertical_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_bytes(workload, variant):
    rec = TRAFFIC.get((workload, variant))
    if rec and rec["sources_sha256"] == kernel_sources_sha256():
        return rec["bytes"]
    return None


def e2e_pipelined(B, w, L, K, barrier, kv_per_group=2):
    """K layer steps end to end: Q/K/V from pinned host memory in, O back to pinned host memory,
    every copy inside the CUDA-event-timed region.

    Two device buffer sets let step i+1's input copy and step i's output copy (each on a copy
    stream of its own) overlap step i's compute.  The first step, whose inputs nothing can hide,
    and the last, whose output nothing can hide, run head group by head group (``kv_per_group``
    KV heads and their q-heads): group j computes while group j+1's inputs arrive, and its output
    leaves while group j+1 computes.  Returns (ms per step, host-to-device bytes per step,
    device-to-host bytes per step)."""
    qh, kh, vh = (t.cpu().pin_memory() for t in (L.q, L.k, L.v))
    ohs = [torch.empty(L.out.shape, dtype=L.out.dtype).pin_memory() for _ in range(2)]
    L2 = Layer(B, w, torch.empty_like(L.q), torch.empty_like(L.k), torch.empty_like(L.v))
    bufs = [L, L2]
    main = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event(enable_timing=False)
    Hq, Hkv = w["Hq"], w["Hkv"]
    gq = Hq // Hkv
    groups = [(g0, min(Hkv, g0 + kv_per_group)) for g0 in range(0, Hkv, kv_per_group)]

    def run(n_steps):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(main)
        comp = [None, None]      # compute of the last step that used each buffer set
        out_done = [[], []]      # its output copies
        s_in.wait_event(start)
        s_out.wait_event(start)

        def load(Lb, parts):
            """Input copies of the (KV-head range) parts, one event per part."""
            evs = []
            with torch.cuda.stream(s_in):
                for g0, g1 in parts:
                    Lb.k[g0:g1].copy_(kh[g0:g1], non_blocking=True)
                    Lb.v[g0:g1].copy_(vh[g0:g1], non_blocking=True)
                    Lb.q[g0 * gq:g1 * gq].copy_(qh[g0 * gq:g1 * gq], non_blocking=True)
                    e = ev()
                    e.record(s_in)
                    evs.append(e)
            return evs

        def store(Lb, b, h0, h1, after):
            with torch.cuda.stream(s_out):
                s_out.wait_event(after)
                ohs[b][h0:h1].copy_(Lb.out[h0:h1], non_blocking=True)
                e = ev()
                e.record(s_out)
                out_done[b].append(e)

        loaded = load(bufs[0], groups)
        for i in range(n_steps):
            b = i % 2
            Lb = bufs[b]
            for e in out_done[b]:
                main.wait_event(e)  # the output copies of step i-2 have read this buffer's O
            out_done[b] = []
            grouped = i == 0 or i == n_steps - 1
            if grouped:
                for (g0, g1), e in zip(groups, loaded):
                    main.wait_event(e)
                    Lb.step_group(set(range(g0 * gq, g1 * gq)))
                    if i == n_steps - 1:
                        c = ev()
                        c.record(main)
                        store(Lb, b, g0 * gq, g1 * gq, c)
            else:
                for e in loaded:
                    main.wait_event(e)
                Lb.step()
            comp[b] = ev()
            comp[b].record(main)
            if i + 1 < n_steps:
                nb = 1 - b
                if comp[nb] is not None:
                    s_in.wait_event(comp[nb])  # step i-1 is done with the other buffer's inputs
                loaded = load(bufs[nb], groups if i + 1 == n_steps - 1 else [(0, Hkv)])
            if i != n_steps - 1:
                store(Lb, b, 0, Hq, comp[b])
        for b in (0, 1):
            for e in out_done[b]:
                main.wait_event(e)
        end.record(main)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / n_steps

    run(2)  # warm-up of both buffer sets
    barrier()
    ms = run(K)
    barrier()
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = ohs[0].numel() * ohs[0].element_size()
    del L2, qh, kh, vh, ohs
    torch.cuda.empty_cache()
    return ms, h2d, d2h


def make_inputs(w, variant, device):
    from dynamic_sparse_attention_vertical_gb300 import inputs as I
    kw = dict(n_cols=w["n_cols"], n_offsets=w["n_offsets"], seed=w["seed"], device=device)
    if variant == "local":
        return I.local_inputs(w["Hq"], w["Hkv"], w["N"], **kw)
    return I.literal_inputs(w["Hq"], w["Hkv"], w["N"], **kw)


def timed(fn, K, events_per_step=0):
    """Run fn K times between two events on the current stream; returns (ms per step, per-step events)."""
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(events_per_step)] for _ in range(K)]
    torch.cuda.synchronize()
    start.record()
    for i in range(K):
        fn(evs[i] if events_per_step else None)
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / K, evs


# -------------------------------------------------------------- CPU oracle ----

# attention rows the oracle evaluates per timed sample, in both CPU legs (the product run's
# cpu_baseline and --impl reference)
ORACLE_SAMPLE_ROWS = 128


def oracle_sample(w, x, rows_per_sample, rng):
    """Time the oracle on one vertical-slash head: full estimation + sampled attention rows.

    Returns (extrapolated ms per layer, description).  The per-layer figure scales
    the estimation to every vertical-slash head and the per-row attention cost to
    every row of every head.
    """
    import oracle as O
    vs, _, _ = head_patterns(w)
    h = vs[0] if vs else 0
    g = h // (w["Hq"] // w["Hkv"])
    N = w["N"]
    qh, kh, vh = x.q[h].cpu(), x.k[g].cpu(), x.v[g].cpu()
    t0 = time.perf_counter()
    vi, si, _, _ = O.vs_estimate(qh, kh, 64, w["k_v"], w["k_s"])
    t1 = time.perf_counter()
    rows = np.sort(rng.choice(N, size=min(rows_per_sample, N), replace=False))
    O.attention_rows(qh, kh, vh, rows, lambda r: O.vs_mask_rows(N, r, vi, si), chunk=64)
    t2 = time.perf_counter()
    per_row = (t2 - t1) / len(rows)
    ms = ((t1 - t0) * max(len(vs), 1) + per_row * w["Hq"] * N) * 1e3
    desc = (f"oracle on q-head {h}: full estimation (extrapolated x{max(len(vs), 1)} heads) + "
            f"{len(rows)} sampled attention rows (extrapolated to {w['Hq']} heads x {N} rows)")
    return ms, desc


def _oracle_estimate_task(t):
    """Worker: full estimation of one vertical-slash head -> (v_idx, s_idx)."""
    import oracle as O
    qh, kh, k_v, k_s = t
    vi, si, _, _ = O.vs_estimate(qh, kh, 64, k_v, k_s)
    return vi, si


def _oracle_rows_task(t):
    """Worker: attention of one head over a range of rows under its vertical-slash mask."""
    import oracle as O
    qh, kh, vh, r0, r1, vi, si = t
    N = qh.shape[0]
    o, _ = O.attention_rows(qh, kh, vh, np.arange(r0, r1), lambda r: O.vs_mask_rows(N, r, vi, si), chunk=128)
    return float(np.abs(o).sum())


def oracle_full(w, x, procs):
    """Time the oracle on the WHOLE layer of an all-vertical-slash workload (every head's
    estimation, then every row's attention), on ``procs`` worker processes (a spawn pool;
    procs = 1 runs in this process).  Returns (ms per layer, description)."""
    import multiprocessing as mp
    Hq, Hkv, N = w["Hq"], w["Hkv"], w["N"]
    gq = Hq // Hkv
    q = x.q.float().cpu().numpy()
    k = x.k.float().cpu().numpy()
    v = x.v.float().cpu().numpy()
    est = [(q[h], k[h // gq], w["k_v"], w["k_s"]) for h in range(Hq)]
    rows_per_task = 1024

    def tasks(idx):
        return [(q[h], k[h // gq], v[h // gq], r0, min(N, r0 + rows_per_task), idx[h][0], idx[h][1])
                for h in range(Hq) for r0 in range(0, N, rows_per_task)]
    if procs == 1:
        t0 = time.perf_counter()
        idx = [_oracle_estimate_task(e) for e in est]
        for t in tasks(idx):
            _oracle_rows_task(t)
        dt = time.perf_counter() - t0
    else:
        env = {k2: os.environ.get(k2) for k2 in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k2 in env:
            os.environ[k2] = "1"  # one BLAS thread per worker process
        try:
            with mp.get_context("spawn").Pool(procs) as pool:
                pool.map(abs, range(procs))  # workers started before the clock
                t0 = time.perf_counter()
                idx = pool.map(_oracle_estimate_task, est)
                pool.map(_oracle_rows_task, tasks(idx), chunksize=1)
                dt = time.perf_counter() - t0
        finally:
            for k2, val in env.items():
                if val is None:
                    os.environ.pop(k2, None)
                else:
                    os.environ[k2] = val
    desc = (f"oracle on the whole layer: estimation of all {Hq} heads + attention of all {Hq} x {N} rows "
            f"(nothing extrapolated), {procs} worker process(es) with one BLAS thread each")
    return dt * 1e3, desc


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    from dynamic_sparse_attention_vertical_gb300 import inputs as I
    x = I.literal_inputs(w["Hq"], w["Hkv"], w["N"], n_cols=w["n_cols"], n_offsets=w["n_offsets"],
                         seed=w["seed"], device="cuda" if torch.cuda.is_available() else "cpu")
    rng = np.random.default_rng(0)
    for _ in range(args.warmup):
        oracle_sample(w, x, ORACLE_SAMPLE_ROWS, rng)
    vals, desc = [], ""
    for _ in range(args.steps):
        v, desc = oracle_sample(w, x, ORACLE_SAMPLE_ROWS, rng)
        vals.append(v)
    value = statistics.mean(vals)
    cores = len(os.sched_getaffinity(0))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "ms/layer", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": value, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {describe(w)}", "input": "literal", "seq_len": w["N"]},
        "cpu_baseline": {"value": value, "unit": "ms/layer", "cores": cores, "kind": "oracle", "sample": desc,
                         "extrapolated": True},
        "e2e": {"value": value, "unit": "ms/layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- sweep ----

SWEEP_N = (16384, 65536, 131072, 262144, 524288)
SWEEP_KV = (500, 1000, 2000)
SWEEP_KS = (2048, 6096)


def run_sweep(args, B):
    """All-vertical-slash layers (32 q / 8 KV heads) over N x k_v x k_s, against the
    dense causal kernel on identical inputs.  One JSON line with every point."""
    from dynamic_sparse_attention_vertical_gb300 import flops as F
    from dynamic_sparse_attention_vertical_gb300 import inputs as I
    dev = torch.device("cuda")
    points = []
    Ns = [int(v) for v in args.sweep_n.split(",")] if args.sweep_n else SWEEP_N
    for variant in [v for v in args.variants.split(",") if v]:
        for N in Ns:
            gen = I.local_inputs if variant == "local" else I.literal_inputs
            x = gen(32, 8, N, n_cols=16, n_offsets=8, seed=5, device=dev)
            out = torch.zeros_like(x.q)
            ws_d = torch.empty(256, dtype=torch.uint8, device=dev)
            B.mi_dense_causal_attn(x.q, x.k, x.v, out=out, workspace=ws_d)
            dms, _ = timed(lambda e: B.mi_dense_causal_attn(x.q, x.k, x.v, out=out, workspace=ws_d), 2)
            for k_v in SWEEP_KV:
                for k_s in SWEEP_KS:
                    v_idx = torch.empty((32, k_v), dtype=torch.int32, device=dev)
                    s_idx = torch.empty((32, k_s), dtype=torch.int32, device=dev)
                    ws_e = torch.empty(B.mi_workspace_bytes(B.MI_OP_VS_ESTIMATE, 32, 8, N), dtype=torch.uint8, device=dev)
                    ws_v = torch.empty(B.mi_workspace_bytes(B.MI_OP_VS_SPARSE_ATTN, 32, 8, N), dtype=torch.uint8, device=dev)

                    def step(_):
                        B.mi_vs_estimate(x.q, x.k, k_v=k_v, k_s=k_s, v_idx=v_idx, s_idx=s_idx, workspace=ws_e)
                        B.mi_vs_sparse_attn(x.q, x.k, x.v, v_idx, s_idx, out=out, workspace=ws_v)
                    step(None)
                    ms, _ = timed(step, args.steps)
                    vi, si = v_idx.cpu().numpy(), s_idx.cpu().numpy()
                    alg = sum(int(F.vs_kept_per_row(N, vi[h], si[h], device=dev).sum()) for h in range(32)) * 4 * 128
                    exe = sum(F.vs_tiles(N, vi[h], si[h]) for h in range(32)) * F.TILE_FLOPS
                    points.append({"variant": variant, "N": N, "k_v": k_v, "k_s": k_s, "ms_per_layer": ms,
                                   "dense_ms": dms, "speedup": dms / ms, "alg_tflop": alg / 1e12,
                                   "exec_tflop": exe / 1e12, "exec_tflops": exe / (ms * 1e-3) / 1e12})
            del x, out
            torch.cuda.empty_cache()
    print(json.dumps({"metric": METRIC, "unit": "ms/layer", "sweep": points}), flush=True)


# --------------------------------------------------------- multi-modal heads ----

MM_RUNS = [(0, 8192), (1, 98304), (0, 24576)]  # text, video, text: 131072 tokens


def run_mm(args, B):
    """The multi-modal heads on a 128K layer (32 q / 8 KV heads): grid (estimated lattice), Q-boundary
    and 2D-boundary (two modalities as text / video / text runs), each timed as a whole layer against
    the dense causal kernel on the same inputs.  One JSON line."""
    from dynamic_sparse_attention_vertical_gb300 import inputs as I
    dev = torch.device("cuda")
    N, Hq, Hkv = 131072, 32, 8
    res = {}
    x = I.grid_inputs(Hq, Hkv, N, 256, 37, seed=7, device=dev)
    out = torch.zeros_like(x.q)
    ws_d = torch.empty(256, dtype=torch.uint8, device=dev)
    B.mi_dense_causal_attn(x.q, x.k, x.v, out=out, workspace=ws_d)
    dms, _ = timed(lambda e: B.mi_dense_causal_attn(x.q, x.k, x.v, out=out, workspace=ws_d), 2)
    grid = torch.empty((Hq, 2), dtype=torch.int32, device=dev)
    ws_ge = torch.empty(B.mi_workspace_bytes(B.MI_OP_GRID_ESTIMATE, Hq, Hkv, N), dtype=torch.uint8, device=dev)
    ws_ga = torch.empty(B.mi_workspace_bytes(B.MI_OP_GRID_ATTN, Hq, Hkv, N), dtype=torch.uint8, device=dev)

    def grid_step(_):
        B.mi_grid_estimate(x.q, x.k, 64, 1024, grid=grid, workspace=ws_ge)
        B.mi_grid_attn(x.q, x.k, x.v, grid, 64, out=out, workspace=ws_ga)
    for _ in range(args.warmup):
        grid_step(None)
    ms, _ = timed(grid_step, args.steps)
    res["grid"] = {"ms_per_layer": ms, "dense_ms": dms, "speedup": dms / ms,
                   "lattice": grid[0].tolist(), "inputs": "lattice sigma 256, phi 37 planted; sigma searched in 64..1024"}
    del x, out
    torch.cuda.empty_cache()
    x = I.literal_inputs(Hq, Hkv, N, n_cols=16, n_offsets=8, seed=8, device=dev)
    mod = torch.cat([torch.full((n,), m, dtype=torch.int32) for m, n in MM_RUNS]).to(dev)
    out = torch.zeros_like(x.q)
    B.mi_dense_causal_attn(x.q, x.k, x.v, out=out, workspace=ws_d)
    dms, _ = timed(lambda e: B.mi_dense_causal_attn(x.q, x.k, x.v, out=out, workspace=ws_d), 2)
    vi = torch.empty((2, Hq, 1000), dtype=torch.int32, device=dev)
    si = torch.empty((2, Hq, 6096), dtype=torch.int32, device=dev)
    ws_qe = torch.empty(B.mi_workspace_bytes(B.MI_OP_QBOUNDARY_ESTIMATE, Hq, Hkv, N), dtype=torch.uint8, device=dev)
    ws_qa = torch.empty(B.mi_workspace_bytes(B.MI_OP_QBOUNDARY_ATTN, Hq, Hkv, N), dtype=torch.uint8, device=dev)

    def qb_step(_):
        B.mi_qboundary_estimate(x.q, x.k, mod, 2, k_v=1000, k_s=6096, v_idx=vi, s_idx=si, workspace=ws_qe)
        B.mi_qboundary_attn(x.q, x.k, x.v, mod, 2, vi, si, out=out, workspace=ws_qa)
    for _ in range(args.warmup):
        qb_step(None)
    ms, _ = timed(qb_step, args.steps)
    res["q_boundary"] = {"ms_per_layer": ms, "dense_ms": dms, "speedup": dms / ms, "runs": MM_RUNS,
                         "budgets": "1000 columns / 6096 diagonals per modality"}
    del ws_qe, ws_qa
    torch.cuda.empty_cache()
    ws_2d = torch.empty(B.mi_workspace_bytes(B.MI_OP_BOUNDARY2D_ATTN, Hq, Hkv, N), dtype=torch.uint8, device=dev)

    def b2_step(_):
        B.mi_boundary2d_attn(x.q, x.k, x.v, MM_RUNS, k_v=1000, k_s=6096, v_idx=vi, s_idx=si, out=out,
                             workspace=ws_2d)
    for _ in range(args.warmup):
        b2_step(None)
    ms, _ = timed(b2_step, args.steps)
    res["boundary_2d"] = {"ms_per_layer": ms, "dense_ms": dms, "speedup": dms / ms, "runs": MM_RUNS,
                          "budgets": "1000 columns / 6096 diagonals per modality sub-sequence"}
    print(json.dumps({"metric": "ms/layer of the multi-modal heads at 128K (32 q / 8 KV heads)", "unit": "ms/layer",
                      "steps": args.steps, "warmup": args.warmup, "mm": res}), flush=True)


# -------------------------------------------------------------------- main ----

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixed-128k", choices=sorted(WORKLOADS))
    ap.add_argument("--variants", default="literal,local", help="input variants; the first is the headline")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-layer-call", action="store_true",
                    help="skip the extra timing of the single layer call")
    ap.add_argument("--no-expanded", action="store_true",
                    help="skip the extra timing of the block-expanded slash mode")
    ap.add_argument("--sweep", action="store_true", help="time the N x k_v x k_s sweep instead")
    ap.add_argument("--cpu-full", action="store_true",
                    help="also time the oracle on the whole layer (all-vertical-slash workloads up to 32K tokens; "
                         "single-core and all-core)")
    ap.add_argument("--sweep-n", default="", help="comma-separated N values for --sweep")
    ap.add_argument("--mm", action="store_true", help="time the multi-modal heads (grid, Q-/2D-boundary) instead")
    args = ap.parse_args()
    assert args.warmup >= 3 or args.impl == "reference", "at least 3 warm-up steps"
    w = WORKLOADS[args.workload]
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    def barrier():
        if dist is not None:
            dist.barrier()

    from dynamic_sparse_attention_vertical_gb300.shard import reduce_max

    def max_over_ranks(x):
        return reduce_max(x, dist, device="cuda")

    from dynamic_sparse_attention_vertical_gb300 import binding as B
    B.load()
    if args.sweep:
        run_sweep(args, B)
        return
    if args.mm:
        run_mm(args, B)
        return
    burst, sustained, hbm, peak_src = measured_peaks()
    dev = torch.device("cuda", local_rank)
    variants = [v for v in args.variants.split(",") if v]
    results = {}
    dense_ms = None
    e2e = None
    cpu = None
    cpu_full = None
    clocks = None
    for vi_, variant in enumerate(variants):
        x = make_inputs(w, variant, dev)
        L = Layer(B, w, x.q, x.k, x.v)
        for _ in range(args.warmup):
            L.step()
        torch.cuda.synchronize()
        L.check_status()
        barrier()
        headline = vi_ == 0
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        smi_id = vis.split(",")[local_rank] if vis else str(local_rank)
        sampler = ClockSampler(smi_id) if headline else None
        if sampler:
            sampler.__enter__()
        ms, evs = timed(L.step, args.steps, events_per_step=5)
        if sampler:
            sampler.__exit__(None, None, None)
            clocks = sampler.summary()
        barrier()
        ms_max = max_over_ranks(ms)
        stage = lambda a, b: statistics.mean(e[a].elapsed_time(e[b]) for e in evs)
        st = {"estimate_ms": stage(0, 1), "vs_attention_ms": stage(1, 2), "block_sparse_ms": stage(2, 3),
              "ashape_ms": stage(3, 4)}
        alg, exe = L.work()
        res = {"ms_per_layer": ms_max / world, "ms_per_step": ms_max, "stages": st,
               "alg_tflop_per_layer": sum(alg.values()) / 1e12, "exec_tflop_per_layer": sum(exe.values()) / 1e12,
               "vs_attention_alg_tflops": alg["vs"] / (st["vs_attention_ms"] * 1e-3) / 1e12 if alg["vs"] else None,
               "vs_attention_exec_tflops": exe["vs"] / (st["vs_attention_ms"] * 1e-3) / 1e12 if exe["vs"] else None}
        if not args.no_layer_call:
            # the same layer through mi_layer_attn (one attention launch for every pattern)
            L.step_layer()
            torch.cuda.synchronize()
            if L.B.mi_read_status(L._ws_layer) != 0:
                raise RuntimeError("layer call status " + L.B.mi_strerror(L.B.mi_read_status(L._ws_layer)))
            barrier()
            lms, _ = timed(L.step_layer, args.steps)
            barrier()
            res["layer_call_ms"] = max_over_ranks(lms) / world
        if L.vs and not args.no_expanded:
            # the same layer with the vertical-slash heads in the block-expanded slash mode
            L.expanded = True
            L.step()
            torch.cuda.synchronize()
            L.check_status()
            barrier()
            xms, xevs = timed(L.step, args.steps, events_per_step=5)
            barrier()
            xms = max_over_ranks(xms)
            xst = {"estimate_ms": statistics.mean(e[0].elapsed_time(e[1]) for e in xevs),
                   "vs_attention_ms": statistics.mean(e[1].elapsed_time(e[2]) for e in xevs)}
            xalg, xexe = L.work()
            res["block_expanded"] = {
                "ms_per_layer": xms / world, "stages": xst,
                "alg_tflop_per_layer": sum(xalg.values()) / 1e12,
                "exec_tflop_per_layer": sum(xexe.values()) / 1e12,
                "vs_attention_alg_tflops": xalg["vs"] / (xst["vs_attention_ms"] * 1e-3) / 1e12,
                "vs_attention_exec_tflops": xexe["vs"] / (xst["vs_attention_ms"] * 1e-3) / 1e12}
            L.expanded = False
        if headline:
            if not args.no_dense:
                for _ in range(1):
                    L.dense()
                dms, _ = timed(lambda e: L.dense(), 2)
                dense_ms = max_over_ranks(dms)
            if not args.no_e2e:
                ems, h2d_bytes, d2h_bytes = e2e_pipelined(B, w, L, args.steps, barrier)
                ems = max_over_ranks(ems)
                e2e = {"value": ems / world, "unit": "ms/layer", "h2d_bytes_per_step": h2d_bytes,
                       "d2h_bytes_per_step": d2h_bytes,
                       "overlap": "two device buffer sets: step i+1's host-to-device copy and step i's "
                                  "device-to-host read run on copy streams while step i computes; the first "
                                  "and last steps run by groups of 2 KV heads, so that their copies overlap "
                                  "the other groups' compute"}
            if not args.no_cpu and rank == 0 and world == 1:
                v_ms, desc = oracle_sample(w, x, ORACLE_SAMPLE_ROWS, np.random.default_rng(1))
                cpu = {"value": v_ms, "unit": "ms/layer", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                       "sample": desc, "extrapolated": True}
            if args.cpu_full and rank == 0 and world == 1:
                assert w["n_vs"] == w["Hq"] and w["N"] <= 32768, "--cpu-full is for the 4K and 32K workloads"
                cores = len(os.sched_getaffinity(0))
                full_ms, full_desc = oracle_full(w, x, cores)
                cpu_full = {"value": full_ms, "unit": "ms/layer", "cores": cores, "kind": "oracle",
                            "sample": full_desc, "extrapolated": False}
                if w["N"] <= 4096:
                    one_ms, one_desc = oracle_full(w, x, 1)
                    cpu_full["single_core"] = {"value": one_ms, "unit": "ms/layer", "cores": 1, "sample": one_desc}
            kernels = L.kernels_per_step * args.steps
        results[variant] = res
        del L, x
        torch.cuda.empty_cache()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    head = results[variants[0]]
    Hq, N = w["Hq"], w["N"]
    f_dense = 4 * 128 * Hq * N * (N + 1) / 2
    ach = head["vs_attention_alg_tflops"]
    line = {
        "metric": METRIC, "value": head["ms_per_layer"], "unit": "ms/layer", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{args.workload}: {describe(w)}", "input": variants[0], "seq_len": N,
                   "heads": {"q": Hq, "kv": w["Hkv"]},
                   "parallelism": "replicas" if world > 1 else "single-gpu",
                   "l2": "no flush: the inputs (Q 1 GiB, K and V 256 MiB each at 128K) exceed the 129 MB L2"},
        "dense_equiv_tflops": f_dense / (head["ms_per_layer"] * 1e-3) / 1e12,
        "dense_ms_per_layer": dense_ms,
        "dense_equiv_speedup": (dense_ms / head["ms_per_layer"]) if dense_ms else None,
        "dense_tflops": (f_dense / (dense_ms * 1e-3) / 1e12) if dense_ms else None,
        "stages": head["stages"],
        "roofline": {"bound": "tensor", "kernel": "vertical-slash sparse attention (tcgen05)",
                     "achieved": ach, "peak": sustained, "unit": "TFLOP/s",
                     "frac": (ach / sustained) if ach else None,
                     "traffic": traffic_bytes(args.workload, variants[0]),
                     "flops": "algorithmic: 4*d per kept (q, j) pair; time = the mi_vs_sparse_attn call",
                     "peak_source": f"bf16_tflops_sustained ({peak_src})",
                     "executed_tflops": head["vs_attention_exec_tflops"],
                     "executed_frac": (head["vs_attention_exec_tflops"] / sustained)
                     if head["vs_attention_exec_tflops"] else None},
        "pct_bf16_peak_exec": (head["vs_attention_exec_tflops"] / sustained * 100)
        if head["vs_attention_exec_tflops"] else None,
        "work": {"alg_tflop_per_layer": head["alg_tflop_per_layer"],
                 "exec_tflop_per_layer": head["exec_tflop_per_layer"],
                 "dense_tflop_per_layer": f_dense / 1e12},
        "variants": {k2: {kk: vv for kk, vv in r.items() if kk != "ms_per_step"} for k2, r in results.items()},
        "e2e": e2e,
        "gpu_launches": kernels,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    if cpu_full:
        line["cpu_full_layer"] = cpu_full
    if dense_ms:
        for r in line["variants"].values():
            r["dense_equiv_speedup"] = dense_ms / r["ms_per_layer"]
            if "block_expanded" in r:
                r["block_expanded"]["dense_equiv_speedup"] = dense_ms / r["block_expanded"]["ms_per_layer"]
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

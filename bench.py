#!/usr/bin/env python
"""Benchmark of the sparse-graph attention hot path on GB300.

One step = one pass of the hot path over one batch of the compression-guided 8K
workload (4 sequences x 8192 byte tokens, block 64, 12 heads of 64, 4-block window,
1 global block, top-16 literal blocks): GPU block-CSR build from the per-block ratios,
then the block-sparse attention forward. Inputs (ratios, Q, K, V) are resident in HBM
when the timed region starts; L2 is flushed (256 MB write) between timed steps,
outside the per-step CUDA-event intervals. A step (mask build, then attention) is one replay of
a CUDA graph of its launches, captured once after the warm-up, with an event-record node
between the two segments: the same kernels with the same arguments, without the per-call
host work.

Metric: effective TFLOP/s over mask edges, 4 * edges * d_h / step time, where edges
are the attended (query, key) token pairs after the causal intersection; tokens/s and
the fraction of the measured BF16 tensor peak are reported beside it.

``e2e`` measures the same metric through the C ABI from host buffers: per step, host zlib
ratios of the byte stream, pinned host -> device copies of ratios and Q/K/V, mask build,
attention, device -> host copies of O and LSE, all inside the timed region; consecutive
steps are pipelined over three CUDA streams with two device buffer sets.

``rows`` times the other hot-path rows once each (kernel time, CUDA events, each step's
launches replayed from CUDA graphs as above): BigBird
at N=16384, the 16-layer Fibonacci-offset pass at N=8192 (HBM roofline), the 64K
compression-guided workload (top-64) and the mean-threshold mask split over local,
long-range and hybrid head groups at N=8192.

``--impl reference`` times the CPU oracle (the reference arm) on the
same workload, each step a bounded sample of query blocks.

Multi-GPU (torchrun): rank r processes its own shard of a global batch (sequences
r*B .. r*B+B-1 of the byte stream, its own Q/K/V draw; weak scaling, no collective on
the data path); the timed region is bracketed by barriers and the maximum over ranks
is reported.
"""
from __future__ import annotations

import argparse
import json
import platform
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "bytelm_topk_8k"
METRIC = "effective TFLOP/s over mask edges & tokens/s at N=8K; % of BF16 tensor peak"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 256 << 20


# ------------------------------------------------------------------ ranks

def rank_info() -> tuple[int, int, int]:
    """(rank, world size, local rank) from the torchrun environment (1 process: 0, 1, 0)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard_sequences(rank: int, batch: int) -> range:
    """Global sequence indices of a rank's shard (weak scaling: `batch` per rank)."""
    return range(rank * batch, (rank + 1) * batch)


def make_max_over_ranks(dist, device):
    """A float -> float reduction to the maximum over the ranks of the default process
    group (identity without one)."""
    def max_over_ranks(x: float) -> float:
        if dist is None:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return max_over_ranks


def aggregate_rate(world: int, work_per_rank: float, max_seconds: float) -> float:
    """Whole-job rate: the work of every rank over the slowest rank's time."""
    return world * work_per_rank / max_seconds


def _peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.4)

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts + frac, parts))
            except ValueError:
                continue
        os.unlink(self.path)
        inside = [p for ts, p in rows if t0 - 0.05 <= ts <= t1 + 0.05]
        use = inside if inside else [p for _, p in rows]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(p[2]) for p in use]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in use for i in range(4) if p[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(use[0][3]), "reasons": reasons,
                "samples": len(use), "samples_in_timed_region": len(inside),
                "power_w_max": max(float(p[4]) for p in use if p[4].replace(".", "", 1).isdigit())
                if any(p[4].replace(".", "", 1).isdigit() for p in use) else None}


# ------------------------------------------------------------------ workload set-up (GPU)

def _csr_edges(rp, ci, block, causal, heads) -> int:
    """Attended token pairs of a block CSR (causal diagonal counts b(b+1)/2)."""
    import numpy as np
    nb = rp.shape[1] - 1
    total = 0
    for s in range(rp.shape[0]):
        for I in range(nb):
            row = ci[rp[s, I]:rp[s, I + 1]]
            if causal:
                total += int(np.sum(row < I)) * block * block + int(np.sum(row == I)) * block * (block + 1) // 2
            else:
                total += len(row) * block * block
    return total * heads


def _csr_tile_elements(rp, ci, block, causal, heads) -> int:
    """Score elements the forward kernel computes for a block CSR: each 128-token query tile
    takes the union of its query blocks' rows (key blocks at or before a row's own block under
    causality) and computes 128 rows x 32 keys per 32-key chunk of the union (b / 32 chunks per
    block), masked or not."""
    import numpy as np
    nb = rp.shape[1] - 1
    nq = max(1, 128 // block)
    chunks = 0
    for s in range(rp.shape[0]):
        for t0 in range(0, nb, nq):
            keys = []
            for I in range(t0, min(nb, t0 + nq)):
                row = ci[rp[s, I]:rp[s, I + 1]]
                keys.append(row[row <= I] if causal else row)
            chunks += len(np.unique(np.concatenate(keys))) * max(1, block // 32)
    return chunks * 32 * 128 * heads


class BlockSparseCase:
    """Ratios -> CSR -> attention for one compression-guided / BigBird workload."""

    def __init__(self, name: str, dev, shard: int = 0, **over):
        import numpy as np
        import torch

        import content_adaptive_sparse_gb300 as sa
        from workloads import byte_stream, qkv_bits, workload
        self.sa = sa
        self.cfg = cfg = workload(name, **over)
        self.dev = dev
        b, n, bt = cfg["block"], cfg["n_tokens"], cfg["batch"]
        self.block, self.causal = b, cfg.get("causal", 1)
        self.head_mask = None
        if cfg["kind"] == "topk":
            self.bytes_host = byte_stream(cfg, seq_offset=shard_sequences(shard, bt).start)
            ratios = sa.sa_block_ratios(self.bytes_host, b)
            self.params = sa.mask_params("topk", b, n, bt, 1, cfg["window_blocks"], cfg["global_blocks"], cfg["topk"])
            self.csr_shared = False
        elif cfg["kind"] == "literal_heads":
            # one mean-threshold CSR per mask part; each head reads the part of its group
            self.bytes_host = byte_stream(cfg, seq_offset=shard_sequences(shard, bt).start)
            ratios = sa.sa_block_ratios(self.bytes_host, b, cfg["zlib_level"])
            parts = sorted(set(cfg["head_components"]))
            self.params_list = [sa.mask_params("literal_mean", b, n, bt, cfg["causal"], cfg["window_blocks"],
                                               components=c) for c in parts]
            self.head_mask = [parts.index(c) for c in cfg["head_components"]]
            self.params = self.params_list[0]
            self.csr_shared = False
        elif cfg["kind"] == "bigbird":
            self.bytes_host = None
            ratios = None
            self.params = sa.mask_params("bigbird", b, n, 1, 0, cfg["window_tokens"] // b, cfg["global_tokens"] // b,
                                         0, cfg["random_tokens"] // b, cfg["seed"])
            self.csr_shared = True
        else:
            self.bytes_host = None
            ratios = None
            self.params = sa.mask_params("full", b, n, 1, cfg["causal"])
            self.csr_shared = True
        if self.head_mask is None:
            self.params_list = [self.params]
        self.ratios_host = ratios
        self.ratios = None if ratios is None else torch.from_numpy(ratios).to(dev)
        qb, kb, vb = qkv_bits(cfg, seed_offset=1000 * shard)
        self.qkv_host = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) for x in (qb, kb, vb)]
        self.q, self.k, self.v = (t.to(dev) for t in self.qkv_host)
        self.csrs = []
        for prm in self.params_list:
            cap = sa.sa_mask_nnz_bound(prm)
            self.csrs.append((torch.empty((prm.batch, n // b + 1), dtype=torch.int32, device=dev),
                              torch.empty((cap,), dtype=torch.int32, device=dev)))
        self.row_ptr, self.col_idx = self.csrs[0]
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((bt, cfg["heads"], n), dtype=torch.float32, device=dev)
        # the forward's workspace (work counter, split plan and partial results), allocated once
        self.ws = sa.fwd_workspace(self.q, b, self.csr_shared, len(self.csrs))
        self.step()
        torch.cuda.synchronize()
        heads_of = ([cfg["heads"]] if self.head_mask is None else
                    [self.head_mask.count(m) for m in range(len(self.csrs))])
        per_csr = sum(_csr_edges(rp.cpu().numpy(), ci.cpu().numpy(), b, self.causal, nh)
                      for (rp, ci), nh in zip(self.csrs, heads_of))
        self.edges = per_csr * (bt if self.csr_shared else 1)
        # score elements the kernel computes (whole 32-key chunks of each query tile's union)
        self.computed = sum(_csr_tile_elements(rp.cpu().numpy(), ci.cpu().numpy(), b, self.causal, nh)
                            for (rp, ci), nh in zip(self.csrs, heads_of)) * (bt if self.csr_shared else 1)
        self.flops = 4 * self.edges * cfg["head_dim"]
        self.tokens = bt * n

    def build(self):
        for prm, (rp, ci) in zip(self.params_list, self.csrs):
            self.sa.sa_build_mask(prm, self.ratios, rp, ci)

    def attend(self):
        if self.head_mask is None:
            self.sa.sa_attn_fwd(self.q, self.k, self.v, self.row_ptr, self.col_idx, self.block, self.causal, self.o,
                                self.lse, self.csr_shared, workspace=self.ws)
        else:
            self.sa.sa_attn_fwd_heads(self.q, self.k, self.v, self.csrs, self.head_mask, self.block, self.causal,
                                      self.o, self.lse, self.csr_shared, workspace=self.ws)

    def step(self):
        self.build()
        self.attend()


def _fib_rungs(k: int) -> list[int]:
    out, a, b = [], 1, 2
    for _ in range(k):
        out.append(a)
        a, b = b, a + b
    return out


class OffsetCase:
    """16-layer window + Fibonacci-offset pass (one launch per layer, own Q/K/V each)."""

    def __init__(self, name: str, dev, **over):
        import numpy as np
        import torch

        import content_adaptive_sparse_gb300 as sa
        import workloads
        from workloads import qkv_bits
        self.sa = sa
        self.cfg = cfg = workloads.workload(name, **over)
        L, bt, n, h, hkv, d, W = (cfg[k] for k in ("layers", "batch", "n_tokens", "heads", "kv_heads", "head_dim",
                                                     "window"))
        self.W = W
        self.layers = []
        ladder = sa.sa_pow2_offsets if cfg.get("ladder") == "pow2" else sa.sa_fib_offsets
        self.interp = bool(cfg.get("interp", False))
        self.alphas = []
        self.fracs = []
        self.pow2 = cfg.get("ladder") == "pow2"
        for l in range(L):
            num, den = sa.sa_layer_alpha(l, L, cfg["alpha_lo"], cfg["alpha_hi"], cfg.get("stride", 1))
            self.alphas.append(num / den)
            self.fracs.append((num, den))
            offs = ladder(num, den, cfg["n_rungs"], W, n)
            qb, kb, vb = qkv_bits(cfg, seed_offset=l)
            q, k, v = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev) for x in (qb, kb, vb))
            o = torch.empty_like(q)
            lse = torch.empty((bt, h, n), dtype=torch.float32, device=dev)
            self.layers.append((q, k, v, o, lse, offs))
        # algorithmic bytes: Q, K, V read once, O and LSE written once, per layer
        self.bytes = L * (bt * n * (2 * h * d * 2 + 2 * hkv * d * 2) + bt * h * n * 4)
        keys = 0
        for (*_, offs), alpha in zip(self.layers, self.alphas):
            i = np.arange(n)
            keys += int(np.sum(np.minimum(W, i) + 1))
            if self.interp:   # rung k is one entry for every query i >= alpha f_k (two rows when fractional)
                for f in _fib_rungs(cfg["n_rungs"]):
                    dd = alpha * f
                    if not (float(dd).is_integer() and dd <= W):
                        keys += max(0, n - int(math.ceil(dd)))
            else:
                keys += sum(int(max(0, n - dd)) for dd in offs)
        self.edges = keys * bt * h
        self.flops = 4 * self.edges * d
        self.tokens = bt * n

    def step(self):
        if self.interp:
            for (q, k, v, o, lse, _), alpha in zip(self.layers, self.alphas):
                self.sa.sa_offset_attn_interp_fwd(q, k, v, self.W, alpha, o, lse, self.cfg["n_rungs"])
            return
        if self.pow2:
            for q, k, v, o, lse, offs in self.layers:
                self.sa.sa_offset_attn_fwd_list(q, k, v, self.W, offs, o, lse)
            return
        # the Fibonacci ladder through the entry point that takes the page's parameters
        for (q, k, v, o, lse, _), (num, den) in zip(self.layers, self.fracs):
            self.sa.sa_offset_attn_fwd(q, k, v, self.W, num, den, self.cfg["n_rungs"], o, lse)


def _capture(torch, body):
    """Captures ``body()`` (library launches on the current stream) in a CUDA graph after one
    eager call on the capture's side stream; returns the graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        body()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        body()
    torch.cuda.synchronize()
    return g


def _external_events(torch) -> bool:
    import inspect
    return "external" in inspect.signature(torch.cuda.Event.__new__).parameters


def _time_events(torch, fn_pairs, steps: int, warmup: int, flush, graph: bool = True):
    """Per-step CUDA-event timing on the current stream with an L2 flush between steps
    (outside the events). ``fn_pairs`` is a list of callables (the step's segments). With
    ``graph`` a step is one replay of a CUDA graph of all its launches, the segment boundaries
    being event-record nodes inside the graph (one graph per segment where this torch has no
    external events): the same kernels with the same arguments, without the per-call host work
    (argument checks, tensor maps, ctypes). Returns the mean ms of each segment and of the
    whole step."""
    for _ in range(warmup):
        for fn in fn_pairs:
            fn()
    torch.cuda.synchronize()
    nseg = len(fn_pairs)
    if graph and _external_events(torch):
        inner = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(nseg - 1)]

        def body():
            for j, fn in enumerate(fn_pairs):
                fn()
                if j < nseg - 1:
                    inner[j].record()
        g = _capture(torch, body)
        g.replay()
        torch.cuda.synchronize()
        seg_sum, tot_sum = [0.0] * nseg, 0.0
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(steps):
            flush()
            a.record()
            g.replay()
            b.record()
            b.synchronize()                  # the inner events are re-recorded by the next replay
            marks = [a] + inner + [b]
            for j in range(nseg):
                seg_sum[j] += marks[j].elapsed_time(marks[j + 1])
            tot_sum += a.elapsed_time(b)
        return [x / steps for x in seg_sum], tot_sum / steps
    if graph:
        fn_pairs = [_capture(torch, fn).replay for fn in fn_pairs]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nseg + 1)] for _ in range(steps)]
    for s in range(steps):
        flush()
        evs[s][0].record()
        for j, fn in enumerate(fn_pairs):
            fn()
            evs[s][j + 1].record()
    torch.cuda.synchronize()
    seg = [sum(evs[s][j].elapsed_time(evs[s][j + 1]) for s in range(steps)) / steps for j in range(nseg)]
    total = sum(evs[s][0].elapsed_time(evs[s][nseg]) for s in range(steps)) / steps
    return seg, total


# ------------------------------------------------------------------ CPU oracle legs

def _oracle_sample_child(budget_s: float, units_per_step: int, steps: int) -> dict:
    """Run in a fresh single-threaded process: the oracle on sampled query blocks of the
    8K workload. Returns FLOPs and seconds per step (or the budgeted single run)."""
    import numpy as np

    import oracle
    from oracle import masks as om
    from workloads import bf16_bits_to_f64, byte_stream, qkv_bits, workload
    cfg = workload(WORKLOAD)
    b, n, h, d = cfg["block"], cfg["n_tokens"], cfg["heads"], cfg["head_dim"]
    data = byte_stream(cfg)
    ratios = oracle.block_ratios(data, b)
    p = om.MaskParams("topk", b, n, 1, cfg["window_blocks"], cfg["global_blocks"], cfg["topk"])
    t_mask0 = time.perf_counter()
    rp, ci = om.build_csr(p, ratios, cfg["batch"])
    t_mask = time.perf_counter() - t_mask0
    qb, kb, vb = qkv_bits(cfg)
    nb = n // b
    rng = np.random.default_rng(0)
    units = [(int(rng.integers(cfg["batch"])), int(rng.integers(nb)), int(rng.integers(h))) for _ in range(65536)]

    def run_unit(s, I, hh):
        oracle.attention_csr_block(qb, kb, vb, rp, ci, b, 1, s, I, hh, convert=bf16_bits_to_f64)
        row = ci[rp[s, I]:rp[s, I + 1]]
        edges = int(np.sum(row < I)) * b * b + int(np.sum(row == I)) * b * (b + 1) // 2
        return 4 * edges * d

    out = {"t_mask_s": t_mask, "steps": []}
    if steps <= 0:
        flops, t0, k = 0, time.perf_counter(), 0
        while time.perf_counter() - t0 < budget_s and k < len(units):
            flops += run_unit(*units[k])
            k += 1
        out["single"] = {"flops": flops, "seconds": time.perf_counter() - t0, "units": k}
        return out
    k = 0
    for _ in range(steps):
        t0 = time.perf_counter()
        flops = 0
        for _ in range(units_per_step):
            flops += run_unit(*units[k % len(units)])
            k += 1
        out["steps"].append({"flops": flops, "seconds": time.perf_counter() - t0})
    return out


# The workloads of the oracle timing (the hot path's configurations): name, overrides,
# how the oracle is sampled.
ORACLE_CONFIGS = [
    ("tiny_topk", {}, "full"),
    ("bytelm_topk_8k", {}, "sampled"),
    ("bigbird_4k", {}, "sampled"),
    ("bigbird_16k", {}, "sampled"),
    ("fib_2k", {}, "sampled"),
    ("fib_8k", {}, "sampled"),
    ("long_topk_64k", {"topk": 16}, "sampled"),
    ("long_topk_64k", {"topk": 64}, "sampled"),
    ("long_topk_64k", {"topk": 256}, "extrapolated"),
    ("full_16k", {}, "sampled"),
]


def _oracle_configs_child(budget_s: float) -> dict:
    """Run in a fresh single-threaded process: the oracle, as it stands, on every workload of
    the hot path, each for about ``budget_s`` seconds of work (the tiny one in full; the
    others on random (sequence, query block, head) units, or random queries for the offset
    workloads; top-256 at 64K on a fixed 64-block sample, extrapolated linearly in edges).
    Returns attended edges per second per workload."""
    from fractions import Fraction

    import numpy as np

    import oracle
    from oracle import masks as om
    from workloads import bf16_bits_to_f64, byte_stream, qkv_bits, workload
    out = {}
    data_cache = {}
    for name, over, kind in ORACLE_CONFIGS:
        cfg = workload(name, **over)
        key = name + "".join(f"_{k}{v}" for k, v in over.items())
        rng = np.random.default_rng(0)
        if name not in data_cache:
            data_cache.clear()
            data_cache[name] = qkv_bits(cfg)
        qb, kb, vb = data_cache[name]
        if cfg["kind"] == "fib":
            W = cfg["window"]
            alpha = Fraction(*cfg["alpha_lo"])
            offs = oracle.fib_offsets(alpha, oracle.fib_rungs(cfg["n_rungs"]))
            deltas = sorted(set(range(W + 1)) | set(offs))
            bt, n, h = cfg["batch"], cfg["n_tokens"], cfg["heads"]
            edges, t0, k = 0, time.perf_counter(), 0
            while time.perf_counter() - t0 < budget_s:
                smp = [(int(rng.integers(bt)), int(rng.integers(n)), int(rng.integers(h))) for _ in range(64)]
                oracle.attention_offsets(qb, kb, vb, W, offs, samples=smp, convert=bf16_bits_to_f64)
                edges += sum(sum(1 for dd in deltas if dd <= i) for _, i, _ in smp)
                k += len(smp)
            secs = time.perf_counter() - t0
            out[key] = {"edges_per_s": edges / secs, "tflops": 4 * edges * cfg["head_dim"] / secs / 1e12,
                        "kind": kind, "units": k, "unit": "query (one head)", "seconds": secs}
            continue
        b, n, h, d, bt = cfg["block"], cfg["n_tokens"], cfg["heads"], cfg["head_dim"], cfg["batch"]
        causal = cfg.get("causal", 1)
        if cfg["kind"] == "topk":
            p = om.MaskParams("topk", b, n, 1, cfg["window_blocks"], cfg["global_blocks"], cfg["topk"])
            ratios = oracle.block_ratios(byte_stream(cfg), b)
            rp, ci = om.build_csr(p, ratios, bt)
        elif cfg["kind"] == "bigbird":
            p = om.MaskParams("bigbird", b, n, 0, cfg["window_tokens"] // b, cfg["global_tokens"] // b, 0,
                              cfg["random_tokens"] // b, cfg["seed"])
            rp, ci = om.build_csr(p, None, 1)
        else:
            p = om.MaskParams("full", b, n, causal)
            rp, ci = om.build_csr(p, None, 1)
        nb = n // b

        def unit_edges(s, I):
            cs = s if rp.shape[0] > 1 else 0
            row = ci[rp[cs, I]:rp[cs, I + 1]]
            if causal:
                return int(np.sum(row < I)) * b * b + int(np.sum(row == I)) * b * (b + 1) // 2
            return len(row) * b * b

        if kind == "full":
            t0 = time.perf_counter()
            oracle.attention_csr(bf16_bits_to_f64(qb), bf16_bits_to_f64(kb), bf16_bits_to_f64(vb), rp, ci, b, causal)
            secs = time.perf_counter() - t0
            edges = sum(unit_edges(s, I) for s in range(bt) for I in range(nb)) * h
            out[key] = {"edges_per_s": edges / secs, "tflops": 4 * edges * d / secs / 1e12, "kind": kind,
                        "units": bt * nb * h, "unit": "whole workload", "seconds": secs}
            continue
        units = [(int(rng.integers(bt)), int(rng.integers(nb)), int(rng.integers(h))) for _ in range(4096)]
        if kind == "extrapolated":
            units = units[:64]
        edges, t0, k = 0, time.perf_counter(), 0
        while k < len(units) and (kind == "extrapolated" or time.perf_counter() - t0 < budget_s):
            s_, I, hh = units[k]
            oracle.attention_csr_block(qb, kb, vb, rp, ci, b, causal, s_, I, hh, convert=bf16_bits_to_f64)
            edges += unit_edges(s_, I)
            k += 1
        secs = time.perf_counter() - t0
        rate = edges / secs
        entry = {"edges_per_s": rate, "tflops": 4 * rate * d / 1e12, "kind": kind, "units": k,
                 "unit": "(sequence, query block, head)", "seconds": secs}
        if kind == "extrapolated":
            total_edges = sum(unit_edges(s, I) for s in range(bt) for I in range(nb)) * h
            entry["whole_workload_seconds_extrapolated"] = total_edges / rate
        out[key] = entry
    return out


def _run_oracle_configs_child(budget_s: float) -> dict:
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench._oracle_configs_child(%r)))" % (ROOT, budget_s))
    res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=1800)
    if res.returncode != 0:
        raise RuntimeError("oracle child failed:\n" + res.stderr[-2000:])
    return json.loads(res.stdout.strip().splitlines()[-1])


def _run_oracle_child(budget_s: float, units_per_step: int, steps: int) -> dict:
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench._oracle_sample_child(%r, %r, %r)))" % (ROOT, budget_s, units_per_step, steps))
    res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=1800)
    if res.returncode != 0:
        raise RuntimeError("oracle child failed:\n" + res.stderr[-2000:])
    return json.loads(res.stdout.strip().splitlines()[-1])


ATTN_FWD_SOURCES = ["attn_fwd.cu", "attn_fwd_common.cuh", "attn_fwd_wide.cuh", "csr_union.cuh", "ptx_sm100.cuh",
                    "sa_internal.h", "tma_host.h"]


def source_digest(names) -> str:
    """First 16 hex digits of the SHA-256 of the named kernel sources, concatenated in order."""
    import hashlib
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "content_adaptive_sparse_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(profile: str, names) -> int | None:
    """DRAM bytes (read + write) per launch from a committed ncu summary under profiles/, if the
    summary was taken on the kernel sources as they are now (its ``kernel_source_sha256_16``
    line against source_digest(names)); None otherwise."""
    path = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.split(":", 1)[0] in ("kernel_source_sha256_16", "dram_bytes_per_launch"):
                k, v = line.split(":", 1)
                fields[k] = v.split()[0] if v.split() else ""
    if fields.get("kernel_source_sha256_16") != source_digest(names) or "dram_bytes_per_launch" not in fields:
        return None
    return int(fields["dram_bytes_per_launch"])


def _config_dict(cfg, flush_note: str, world: int) -> dict:
    return {"workload": cfg["name"], "batch": cfg["batch"], "n_tokens": cfg["n_tokens"], "block": cfg["block"],
            "heads": cfg["heads"], "head_dim": cfg["head_dim"], "window_blocks": cfg["window_blocks"],
            "global_blocks": cfg["global_blocks"], "topk": cfg["topk"], "ratio": "zlib level 6 per block",
            "l2": flush_note, "parallelism": f"dp{world}: batch shards of {cfg['batch']} sequences per rank, no collective"}


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on sampled query blocks."""
    rank, world, _ = rank_info()
    if rank != 0:
        return
    from workloads import workload
    cfg = workload(WORKLOAD)
    # calibrate: units per step so that warmup + steps take about a minute
    cal = _run_oracle_child(2.0, 0, 0)["single"]
    per_unit = cal["seconds"] / max(1, cal["units"])
    total_steps = max(1, args.steps + args.warmup)
    units = max(1, min(4096, int(60.0 / total_steps / per_unit)))
    res = _run_oracle_child(0.0, units, total_steps)
    timed = res["steps"][args.warmup:]
    flops = sum(s["flops"] for s in timed)
    secs = sum(s["seconds"] for s in timed)
    value = flops / secs / 1e12
    tok_per_unit = cfg["block"]          # one query block of one head
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * secs / len(timed),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config_dict(cfg, "n/a (CPU)", world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{units} (sequence, query block, head) units per step, random over the "
                                   f"workload, {len(timed)} timed steps; numpy float64, 1 BLAS thread"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "tokens_per_s": units * tok_per_unit * len(timed) / secs / cfg["heads"],
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import numpy as np
    import torch

    import content_adaptive_sparse_gb300 as sa

    rank, world, local = rank_info()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sa.build_library()
    sa.load_library()
    peaks = _peaks()

    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.zero_()

    def barrier():
        if dist is not None:
            dist.barrier()

    max_over_ranks = make_max_over_ranks(dist, dev)

    if args.only_row:
        rows = _measure_rows(torch, sa, dev, flush, peaks, max_over_ranks, only=args.only_row,
                             steps=args.steps, warm=args.warmup)
        if rank == 0:
            print(json.dumps({"only_row": args.only_row, "rows": rows}), flush=True)
        return

    case = BlockSparseCase(WORKLOAD, dev, shard=rank)
    cfg = case.cfg

    # ---------------- main timed region
    for _ in range(args.warmup):
        case.step()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    t0 = time.time()
    seg, step_ms = _time_events(torch, [case.build, case.attend], args.steps, 0, flush)
    torch.cuda.synchronize()
    barrier()
    t1 = time.time()
    clk = clocks.stop(t0, t1)
    step_ms = max_over_ranks(step_ms)
    attn_ms = max_over_ranks(seg[1])
    mask_ms = max_over_ranks(seg[0])
    value = aggregate_rate(world, case.flops, step_ms * 1e-3) / 1e12
    attn_tflops = case.flops / (attn_ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    assert sa.sa_device_status() == 0

    # ---------------- end to end through the C ABI from host buffers
    e2e = _measure_e2e(torch, sa, case, cfg, barrier, max_over_ranks, world)
    # host ratio pass alone, one 8192-byte sequence: the workload's blocks (64 bytes, zlib
    # level 6) and the compression paper's (128 bytes, level 1; "< 1 ms for N = 8192")
    one_seq = case.bytes_host[:1]
    ratio_ms = {}
    for blk, lvl in ((cfg["block"], 6), (128, 1)):
        sa.sa_block_ratios(one_seq, blk, lvl)
        r0 = time.perf_counter()
        for _ in range(20):
            sa.sa_block_ratios(one_seq, blk, lvl)
        ratio_ms[f"b{blk}_level{lvl}"] = (time.perf_counter() - r0) / 20 * 1e3

    # ---------------- other hot-path rows (kernel time only)
    rows = {}
    if not args.no_rows:
        rows = _measure_rows(torch, sa, dev, flush, peaks, max_over_ranks)

    # ---------------- CPU baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        res = _run_oracle_child(args.cpu_seconds, 0, 0)["single"]
        cpu = {"value": res["flops"] / res["seconds"] / 1e12, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{res['units']} random (sequence, query block, head) units of the same workload "
                         f"({res['seconds']:.1f} s, numpy float64, 1 BLAS thread)",
               "host_cpu_count": os.cpu_count(), "blas_threads": 1}
        if not args.no_cpu_configs:
            cpu["per_workload"] = _run_oracle_configs_child(args.cpu_config_seconds)

    # DRAM bytes per launch of the committed ncu capture, while the kernel is unchanged since
    traffic = recorded_traffic("attn_fwd_bytelm_topk_8k.md", ATTN_FWD_SOURCES)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": _config_dict(cfg, "flushed between timed steps (256 MB write, outside events)", world),
        "launch": "each step one CUDA graph replay of its launches (mask build, event node, attention)",
        "tokens_per_s": aggregate_rate(world, case.tokens, step_ms * 1e-3),
        "pct_bf16_peak": 100.0 * value / world / peak,
        "edges_per_step": case.edges,
        "segments_ms": {"sa_build_mask": mask_ms, "sa_attn_fwd": attn_ms},
        "roofline": {"bound": "tensor", "achieved": attn_tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": attn_tflops / peak, "traffic": traffic,
                     "kernel": "attn_fwd_kernel<64> (sa_attn_fwd)",
                     "peak_source": f"{peaks['source']} bf16 burst (kernel timed alone)",
                     "algorithmic_flops_per_launch": case.flops,
                     "tile_fill": case.edges / case.computed,
                     "computed_tflops": 4 * case.computed * cfg["head_dim"] / (attn_ms * 1e-3) / 1e12,
                     "frac_of_sustained": attn_tflops / peaks["bf16_tflops_sustained"]
                     if peaks.get("bf16_tflops_sustained") else None},
        "e2e": dict(e2e, host_ratio_ms_per_8k_sequence=ratio_ms),
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
        "rows": rows,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


E2E_STEPS = 60      # timed end-to-end steps, whatever --steps says (a fixed, long enough sample)
E2E_WARM = 6
E2E_SETS = 2         # device / pinned output buffer sets in flight (measured: 2 sets 0.94 ms, 3 sets 0.97, 4 sets 0.96)


def _measure_e2e(torch, sa, case, cfg, barrier, max_over_ranks, world) -> dict:
    """The headline workload end to end through the C ABI from host buffers.

    Each step uploads its Q, K, V from pinned host memory, runs the mask step from the host
    bytes (sa_build_mask_from_bytes: host zlib ratios on the library's threads, their upload
    and the CSR build), the attention, and reads O and LSE back into pinned host memory.
    Steps are pipelined over three streams (uploads, compute, downloads) with two device
    buffer sets, so the uploads of step i + 1 and the host ratios overlap the kernels of step
    i and the downloads of step i - 1. Reported: the mean time per step over E2E_STEPS steps
    (wall clock, from the first enqueue to the last download), and per stage the median of
    the per-step durations (CUDA events on each stream; host time for the ratio call)."""
    import numpy as np

    nbk = cfg["n_tokens"] // cfg["block"]
    pinned = [t.pin_memory() for t in case.qkv_host]
    # half of the host's cores, shared among the ranks that run on this host
    ratio_threads = max(1, (os.cpu_count() or 2) // (2 * int(os.environ.get("LOCAL_WORLD_SIZE", "1"))))
    ratios_pinned = [torch.empty((cfg["batch"], nbk), dtype=torch.float32).pin_memory() for _ in range(E2E_SETS)]
    o_host = [torch.empty(case.o.shape, dtype=torch.bfloat16).pin_memory() for _ in range(E2E_SETS)]
    lse_host = [torch.empty(case.lse.shape, dtype=torch.float32).pin_memory() for _ in range(E2E_SETS)]
    h2d = sum(t.numel() * t.element_size() for t in pinned) + ratios_pinned[0].numel() * 4
    d2h = o_host[0].numel() * 2 + lse_host[0].numel() * 4
    bufs = []
    for bi in range(E2E_SETS):
        if bi == 0:
            bufs.append((case.q, case.k, case.v, case.ratios, case.row_ptr, case.col_idx, case.o, case.lse, case.ws))
        else:
            bufs.append(tuple(torch.empty_like(x) for x in (case.q, case.k, case.v, case.ratios, case.row_ptr,
                                                             case.col_idx, case.o, case.lse, case.ws)))
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(E2E_SETS)]
    ev_comp = [torch.cuda.Event() for _ in range(E2E_SETS)]
    ev_out = [torch.cuda.Event() for _ in range(E2E_SETS)]
    total = E2E_WARM + E2E_STEPS
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(total)]
    host_ratio_s = []
    started = [False] * E2E_SETS

    def step(i):
        b = i % E2E_SETS
        bq, bk, bv, br, brp, bci, bo, bl, bws = bufs[b]
        m = marks[i]
        with torch.cuda.stream(s_in):
            if started[b]:
                s_in.wait_event(ev_comp[b])   # step i - E2E_SETS has finished reading buffer set b
            m[0].record(s_in)
            bq.copy_(pinned[0], non_blocking=True)
            bk.copy_(pinned[1], non_blocking=True)
            bv.copy_(pinned[2], non_blocking=True)
            m[1].record(s_in)
            ev_in[b].record(s_in)
        if started[b]:
            ev_comp[b].synchronize()          # the ratio upload from ratios_pinned[b] of that step is done
        with torch.cuda.stream(s_comp):
            if started[b]:
                s_comp.wait_event(ev_out[b])  # O / LSE of step i - E2E_SETS have been read back
            m[2].record(s_comp)
            r0 = time.perf_counter()
            sa.sa_build_mask_from_bytes(case.params, case.bytes_host, ratios_pinned[b], br, brp, bci,
                                        n_threads=ratio_threads)
            host_ratio_s.append(time.perf_counter() - r0)
            s_comp.wait_event(ev_in[b])
            sa.sa_attn_fwd(bq, bk, bv, brp, bci, case.block, case.causal, bo, bl, case.csr_shared, workspace=bws)
            m[3].record(s_comp)
            ev_comp[b].record(s_comp)
        with torch.cuda.stream(s_out):
            if started[b]:
                ev_out[b].synchronize()       # the host may reuse o_host[b] / lse_host[b]
            s_out.wait_event(ev_comp[b])
            m[4].record(s_out)
            o_host[b].copy_(bo, non_blocking=True)
            lse_host[b].copy_(bl, non_blocking=True)
            m[5].record(s_out)
            ev_out[b].record(s_out)
        started[b] = True

    for i in range(E2E_WARM):
        step(i)
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for i in range(E2E_WARM, total):
        step(i)
    torch.cuda.synchronize()                  # every step's O and LSE are on the host
    te = max_over_ranks((time.perf_counter() - t0) / E2E_STEPS)
    timed = marks[E2E_WARM:]
    stage = {
        "h2d_qkv_ms": float(np.median([m[0].elapsed_time(m[1]) for m in timed])),
        "mask_and_attention_ms": float(np.median([m[2].elapsed_time(m[3]) for m in timed])),
        "d2h_o_lse_ms": float(np.median([m[4].elapsed_time(m[5]) for m in timed])),
        "host_ratio_call_ms": float(np.median(host_ratio_s[E2E_WARM:]) * 1e3),
    }
    bound = max(stage, key=stage.get)
    return {"value": aggregate_rate(world, case.flops, te) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": te * 1e3, "steps": E2E_STEPS, "warmup": E2E_WARM,
            "stages_median_ms": stage, "slowest_stage": bound,
            "h2d_gbs": h2d / 1e9 / (stage["h2d_qkv_ms"] * 1e-3), "d2h_gbs": d2h / 1e9 / (stage["d2h_o_lse_ms"] * 1e-3),
            "host": {"os_cpu_count": os.cpu_count(), "ratio_threads": ratio_threads,
                     "platform": platform.machine()},
            "includes": "per step: H2D Q+K+V (pinned), host zlib ratios + their H2D + mask build "
                        "(sa_build_mask_from_bytes), attention, D2H O+LSE (pinned); three streams, "
                        f"{E2E_SETS} buffer sets"}


def _measure_rows(torch, sa, dev, flush, peaks, max_over_ranks, only=None, steps=10, warm=3) -> dict:
    rows = {}
    want = (lambda name: only is None or only == name)
    if want("bigbird_16k"):
        rows.update(_row_bigbird(torch, dev, flush, peaks, max_over_ranks, steps, warm))
    if want("long_topk_64k"):
        rows.update(_row_long(torch, dev, flush, peaks, max_over_ranks, steps, warm))
    if want("full_32k_one_head_split"):
        rows.update(_row_split(torch, dev, flush, peaks, max_over_ranks, steps, warm))
    if want("cas_heads_8k"):
        rows.update(_row_block_sparse(torch, dev, flush, peaks, max_over_ranks, steps, warm, "cas_heads_8k"))
    if want("bwd_bytelm_topk_8k"):
        rows.update(_row_bwd(torch, dev, flush, peaks, max_over_ranks, steps, warm))
    if want("fib_8k_16_layers"):
        rows.update(_row_fib(torch, dev, flush, peaks, max_over_ranks, steps, warm))
    if want("fib_8k_coprime_16_layers"):
        rows.update(_row_fib(torch, dev, flush, peaks, max_over_ranks, steps, warm, name="fib_8k_coprime"))
    if want("fib_interp_8k_16_layers"):
        rows.update(_row_fib(torch, dev, flush, peaks, max_over_ranks, steps, warm, name="fib_interp_8k"))
    if want("pow2_8k_16_layers"):
        rows.update(_row_fib(torch, dev, flush, peaks, max_over_ranks, steps, warm, name="pow2_8k"))
    if only == "fib_8k_2_layers":   # same per-layer launch, small device footprint (profiling)
        rows.update(_row_fib(torch, dev, flush, peaks, max_over_ranks, steps, warm, layers=2))
    torch.cuda.empty_cache()
    return rows


def _fill_fields(case, attn_ms: float) -> dict:
    """Tile fill (mask edges / score elements the kernel computes) and the rate over the
    computed elements: the part of a row's distance from peak that its 128 x 128 tiling takes."""
    computed_tflops = 4 * case.computed * case.cfg["head_dim"] / (attn_ms * 1e-3) / 1e12
    return {"tile_fill": case.edges / case.computed, "computed_elements": case.computed,
            "computed_tflops": computed_tflops}


def _row_bigbird(torch, dev, flush, peaks, max_over_ranks, steps, warm):
    rows = {}
    # BigBird 16K: CSR build + attention
    bb = BlockSparseCase("bigbird_16k", dev)
    seg, tot = _time_events(torch, [bb.build, bb.attend], steps, warm, flush)
    a = max_over_ranks(seg[1])
    rows["bigbird_16k"] = {"ms_per_step": max_over_ranks(tot), "attn_ms": a, "mask_ms": seg[0],
                           "effective_tflops": bb.flops / (a * 1e-3) / 1e12,
                           "frac_bf16_peak": bb.flops / (a * 1e-3) / 1e12 / peaks["bf16_tflops"],
                           "tokens_per_s": bb.tokens / (tot * 1e-3), "edges": bb.edges, **_fill_fields(bb, a)}
    return rows


def _row_long(torch, dev, flush, peaks, max_over_ranks, steps, warm):
    rows = {}
    # long context 64K, top-64
    lc = BlockSparseCase("long_topk_64k", dev)
    seg, tot = _time_events(torch, [lc.build, lc.attend], steps, warm, flush)
    a = max_over_ranks(seg[1])
    rows["long_topk_64k"] = {"ms_per_step": max_over_ranks(tot), "attn_ms": a, "mask_ms": seg[0],
                             "effective_tflops": lc.flops / (a * 1e-3) / 1e12,
                             "frac_bf16_peak": lc.flops / (a * 1e-3) / 1e12 / peaks["bf16_tflops"],
                             "tokens_per_s": lc.tokens / (tot * 1e-3), "edges": lc.edges, **_fill_fields(lc, a)}
    return rows


def _row_split(torch, dev, flush, peaks, max_over_ranks, steps, warm):
    """Few work items with long key lists (full causal 32K, one sequence and head): the
    forward with its workspace (the schedule kernel splits long items into parts and merges
    them when the longest item exceeds 1.25x a stream's share) and with a 256-byte workspace
    (no split), at d = 64 (two-pipeline kernel: the items are split) and d = 128 (one-stream
    kernel: the items stay whole)."""
    out = {}
    for d in (64, 128):
        case = BlockSparseCase("full_32k_one_head", dev, head_dim=d, std=1.0 / (d ** 0.5))
        case.ws[64:80].zero_()                       # split header: stays zero unless a launch splits
        seg, _ = _time_events(torch, [case.attend], steps, warm, flush)
        a = max_over_ranks(seg[0])
        full_ws = case.ws
        case.ws = torch.empty((256,), dtype=torch.uint8, device=dev)
        seg2, _ = _time_events(torch, [case.attend], steps, warm, flush)
        case.ws = full_ws
        b = max_over_ranks(seg2[0])
        hdr = full_ws[64:80].cpu().numpy().view("int32")
        out[f"d{d}"] = {"attn_ms": a, "attn_ms_without_split": b,
                        "effective_tflops": case.flops / (a * 1e-3) / 1e12,
                        "frac_bf16_peak": case.flops / (a * 1e-3) / 1e12 / peaks["bf16_tflops"],
                        "effective_tflops_without_split": case.flops / (b * 1e-3) / 1e12,
                        "split_items": int(hdr[3]), "part_tiles": int(hdr[2]), "edges": case.edges,
                        **_fill_fields(case, a)}
        del case
        torch.cuda.empty_cache()
    return {"full_32k_one_head_split": out}


def _row_block_sparse(torch, dev, flush, peaks, max_over_ranks, steps, warm, name):
    case = BlockSparseCase(name, dev)
    seg, tot = _time_events(torch, [case.build, case.attend], steps, warm, flush)
    a = max_over_ranks(seg[1])
    return {name: {"ms_per_step": max_over_ranks(tot), "attn_ms": a, "mask_ms": seg[0],
                   "effective_tflops": case.flops / (a * 1e-3) / 1e12,
                   "frac_bf16_peak": case.flops / (a * 1e-3) / 1e12 / peaks["bf16_tflops"],
                   "tokens_per_s": case.tokens / (tot * 1e-3), "edges": case.edges, **_fill_fields(case, a)}}


def _row_bwd(torch, dev, flush, peaks, max_over_ranks, steps, warm, name="bytelm_topk_8k"):
    """Backward of the compression-guided workload: D = rowsum(dO * O), the transposed
    CSR, dQ and dK / dV (one sa_attn_bwd call). Effective FLOP = 2.5 x the forward's
    4 * edges * d (five products of edges x d instead of two)."""
    import numpy as np

    from workloads import bf16_normal_bits
    case = BlockSparseCase(name, dev)
    torch.cuda.synchronize()
    dob = bf16_normal_bits(np.random.default_rng(77), tuple(case.q.shape), case.cfg["std"])
    d_o = torch.from_numpy(dob.view(np.int16)).view(torch.bfloat16).to(dev)
    dq, dk, dv = torch.empty_like(case.q), torch.empty_like(case.k), torch.empty_like(case.v)
    b, n, h, _ = case.q.shape
    ws_bytes = case.sa.sa_attn_bwd_workspace_size(b, n, h, case.block, case.params.batch, case.col_idx.numel())
    ws = torch.empty((ws_bytes,), dtype=torch.uint8, device=dev)

    def bwd():
        case.sa.sa_attn_bwd(case.q, case.k, case.v, case.o, d_o, case.lse, case.row_ptr, case.col_idx, case.block,
                            case.causal, dq, dk, dv, ws, case.csr_shared)

    seg, tot = _time_events(torch, [bwd], steps, warm, flush)
    t = max_over_ranks(tot)
    flops = 2.5 * case.flops
    return {f"bwd_{name}": {"ms_per_step": t, "effective_tflops": flops / (t * 1e-3) / 1e12,
                            "frac_bf16_peak": flops / (t * 1e-3) / 1e12 / peaks["bf16_tflops"],
                            "tokens_per_s": case.tokens / (t * 1e-3), "edges": case.edges,
                            "launches_per_step": 6}}


def _row_fib(torch, dev, flush, peaks, max_over_ranks, steps, warm, layers=16, name="fib_8k"):
    rows = {}
    # 16-layer Fibonacci pass at 8K (HBM roofline)
    fb = OffsetCase(name, dev, layers=layers)
    seg, tot = _time_events(torch, [fb.step], steps, warm, flush)
    t = max_over_ranks(tot)
    gbs = fb.bytes / (t * 1e-3) / 1e9
    rows[f"{name}_{layers}_layers"] = {"ms_per_step": t, "hbm_gbs": gbs, "frac_hbm": gbs / peaks["hbm_gbs"],
                                "algorithmic_bytes": fb.bytes, "effective_tflops": fb.flops / (t * 1e-3) / 1e12,
                                "tokens_per_s": fb.tokens / (t * 1e-3), "launches_per_step": layers}
    return rows


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-rows", action="store_true", help="skip the other hot-path rows")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-configs", action="store_true", help="skip the oracle timing of the other workloads")
    ap.add_argument("--cpu-config-seconds", type=float, default=1.5,
                    help="oracle seconds per workload in the per-workload CPU timing")
    ap.add_argument("--only-row", choices=["bigbird_16k", "long_topk_64k", "full_32k_one_head_split", "cas_heads_8k",
                                           "bwd_bytelm_topk_8k",
                                           "fib_8k_16_layers",
                                           "fib_8k_coprime_16_layers", "pow2_8k_16_layers", "fib_interp_8k_16_layers",
                                           "fib_8k_2_layers"],
                    default=None,
                    help="time one other hot-path row only (profiling aid; prints that row, not the bench line)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

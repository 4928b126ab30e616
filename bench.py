#!/usr/bin/env python3
"""Benchmark of the INT4 group-quantized paged KV cache decode step on GB300.

A step is one pass of the whole hot path over one batch: quantize-on-append of one
new token per sequence (K and V), then decode attention of every query head over the
packed paged cache (split-KV kernel + combine).  Default workload: Llama-7B-shaped
MHA layer, batch 8, 32 query = 32 KV heads, head_dim 128, context 8192 (+1 appended
token), 16-token pages in a seeded random permutation, K grouped at 64 and V at 128.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kvq|reference] [--workload NAME]

Prints one JSON line (rank 0).  `value` is whole-job HBM throughput: algorithmic bytes
of all ranks' steps / max-over-ranks time, with algorithmic bytes = the packed cache
the decode reads (head_dim + 2*(d/Gk + d/Gv) bytes per token per KV head) plus the
append's fp16 read and packed write.  `--impl reference` times the oracle (plain
single-threaded C, fp64 attention) on the host cores on a bounded sample of the same
workload, in the same metric.
"""
from __future__ import annotations

import argparse
import itertools
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "INT4-KV paged decode attention: HBM GB/s vs peak, tokens/s; quantize GB/s"
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    ap.add_argument("--workload", default="llama7b", help="llama7b (default), gqa8b, ragged, longctx, tiny")
    ap.add_argument("--group", type=int, default=None, help="K and V group size for the longctx sweep")
    ap.add_argument("--graph-steps", type=int, default=200, help="steps captured per CUDA graph")
    ap.add_argument("--eager", action="store_true", help="launch every step from Python instead of graphs")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--compare", action="store_true",
                    help="also time the latency comparison: FP16 cache, INT4 dequantized then attended, INT4 fused")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-quality", action="store_true", help="skip the dequantization quality report")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the other decode workloads and the long-context prefill-quantize pass")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU work budget of the oracle baseline")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


KERNEL_SOURCES = ("int4_group_quantized_kvq_gb300/csrc/decode_impl.cuh",
                  "int4_group_quantized_kvq_gb300/csrc/kvq_device.cuh",
                  "int4_group_quantized_kvq_gb300/csrc/decode_plan.cu")


def measured_traffic(workload: str) -> int | None:
    """DRAM bytes of one decode launch from the committed ncu record, or None when the kernel
    sources changed since the capture or the record is for another workload."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "decode_traffic.txt")
    try:
        rec = {}
        for line in open(path):
            line = line.strip()
            if line and not line.startswith("#") and "=" in line:
                k, v = line.split("=", 1)
                rec[k.strip()] = v.strip()
        h = hashlib.sha256()
        for f in KERNEL_SOURCES:
            with open(os.path.join(ROOT, f), "rb") as fh:
                h.update(fh.read())
        if rec.get("kernel_source_sha256") == h.hexdigest() and rec.get("workload") == workload:
            return int(rec["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        pass
    return None


def make_workload(name: str, group: int | None):
    import workloads as W
    if name == "longctx":
        return W.longctx(group or 64)
    wl = W.ALL[name]()
    return wl.with_groups(group) if group else wl


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu), "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.25)

    def stop(self) -> dict:
        if self.proc is None:
            return {"unavailable": "nvidia-smi could not be started"}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"unavailable": "no samples"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(r[1]) for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median([x for x in sm if x == x] or [float("nan")]),
                "sm_max_mhz": max(num(r[2]) for r in rows), "samples": len(rows),
                "power_w_max": max(num(r[3]) for r in rows), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline / reference arm)
# ---------------------------------------------------------------------------

class OracleSample:
    """A bounded slice of the workload for the oracle: sequence 0, the first `heads` KV
    heads (all their query heads) and the first `tokens` positions; one step appends the
    token at position tokens-1 and attends over `tokens` positions."""

    def __init__(self, wl, heads: int, tokens: int):
        import numpy as np
        import oracle
        import workloads as W
        self.np, self.oracle = np, oracle
        self.wl, self.heads, self.tokens = wl, heads, tokens
        k = W.kv_tensor(W.SEED_K, (1, tokens, wl.Hkv, wl.d), 20.0, W.outlier_channels(wl.Hkv, wl.d))
        v = W.kv_tensor(W.SEED_V, (1, tokens, wl.Hkv, wl.d))
        self.k = np.ascontiguousarray(k[:, :, :heads].numpy())
        self.v = np.ascontiguousarray(v[:, :, :heads].numpy())
        q = W.kv_tensor(W.SEED_Q, (1, 1, wl.Hq, wl.d))[0].numpy()
        self.q = np.ascontiguousarray(q[:, :heads * wl.r])
        npg = (tokens + wl.P - 1) // wl.P
        self.L = oracle.Layout(heads, wl.d, wl.P, wl.Gk, wl.Gv, npg)
        self.bt = np.arange(npg, dtype=np.int32).reshape(1, -1)
        self.pool = np.zeros(self.L.pool_bytes, np.uint8)
        if tokens > 1:
            oracle.quantize_append(self.L, self.pool, self.k[:, :tokens - 1], self.v[:, :tokens - 1], self.bt,
                                   np.zeros(1, np.int32))

    def step(self):
        np = self.np
        t = self.tokens - 1
        self.oracle.quantize_append(self.L, self.pool, self.k[:, t:t + 1], self.v[:, t:t + 1], self.bt,
                                    np.array([t], np.int32))
        return self.oracle.decode_attention(self.L, self.pool, self.q, self.bt, np.array([self.tokens], np.int32),
                                            self.wl.d ** -0.5)

    def bytes(self) -> int:
        wl = self.wl
        per = wl.packed_bytes_per_token_head()
        return self.heads * self.tokens * per + self.heads * (2 * wl.d * 2 + per)

    def describe(self) -> str:
        wl = self.wl
        return (f"{wl.name}: sequence 0, {self.heads} of {wl.Hkv} KV heads ({self.heads * wl.r} query heads), "
                f"{self.tokens} of {wl.seq_lens[0]} positions; append 1 token + fp64 decode attention")


def plan_oracle_sample(wl, seconds_per_step: float) -> "OracleSample":
    """Size a sample so one oracle step takes about seconds_per_step on this host."""
    probe_tokens = min(wl.seq_lens[0], 512)
    probe = OracleSample(wl, 1, probe_tokens)
    t0 = time.perf_counter()
    probe.step()
    per_head_token = max((time.perf_counter() - t0) / probe_tokens, 1e-9)
    budget_ht = max(1.0, seconds_per_step / per_head_token)
    tokens = wl.seq_lens[0]
    heads = int(max(1, min(wl.Hkv, budget_ht // tokens)))
    if heads == 1:
        tokens = int(max(16, min(tokens, budget_ht)))
    return OracleSample(wl, heads, tokens)


def time_oracle(wl, budget_s: float) -> dict:
    """The oracle as it stands, single-threaded, on a sample of about budget_s seconds."""
    smp = plan_oracle_sample(wl, min(budget_s, 4.0))
    reps, t_total = 0, 0.0
    while t_total < budget_s or reps == 0:
        t0 = time.perf_counter()
        smp.step()
        t_total += time.perf_counter() - t0
        reps += 1
    per = t_total / reps
    return {"value": smp.bytes() / per / 1e9, "unit": "GB/s", "cores": 1, "host_cores": os.cpu_count(), "kind": "oracle",
            "sample": smp.describe() + f"; {reps} repetitions, {per * 1e3:.1f} ms each",
            "seconds_per_step": per}


def time_oracle_quantize(wl, budget_s: float) -> dict:
    """The oracle's quantize-append as it stands, single-threaded, on a slice of the workload's history
    (sequence 0, all KV heads, as many tokens as fit about budget_s seconds), over the bytes the GPU
    quantize figure counts: fp16 K and V read, packed codes and scales written."""
    import numpy as np
    import oracle
    import workloads as W
    n_max = wl.seq_lens[0]
    npg = (n_max + wl.P - 1) // wl.P
    L = oracle.Layout(wl.Hkv, wl.d, wl.P, wl.Gk, wl.Gv, npg)
    pool = np.zeros(L.pool_bytes, np.uint8)
    bt = np.arange(npg, dtype=np.int32).reshape(1, -1)
    per_token = wl.Hkv * (2 * wl.d * 2 + wl.packed_bytes_per_token_head())

    def rows(n):  # the first n tokens of sequence 0 (the generator is counter-indexed, so a prefix is exact)
        k = W.kv_tensor(W.SEED_K, (1, n, wl.Hkv, wl.d), 20.0, W.outlier_channels(wl.Hkv, wl.d)).numpy()
        return k, W.kv_tensor(W.SEED_V, (1, n, wl.Hkv, wl.d)).numpy()
    n = min(n_max, 64)
    k, v = rows(n)
    t0 = time.perf_counter()
    oracle.quantize_append(L, pool, k, v, bt, np.zeros(1, np.int32))
    per_tok_s = max((time.perf_counter() - t0) / n, 1e-9)
    n = int(max(16, min(n_max, budget_s / per_tok_s)))
    k, v = rows(n)
    t0 = time.perf_counter()
    oracle.quantize_append(L, pool, k, v, bt, np.zeros(1, np.int32))
    t = time.perf_counter() - t0
    return {"value": n * per_token / t / 1e9, "unit": "GB/s", "cores": 1, "host_cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{wl.name}: sequence 0, {n} of {n_max} tokens x {wl.Hkv} KV heads, K and V; "
                      f"{t * 1e3:.0f} ms"}


# ---------------------------------------------------------------------------
# dequantization quality against the fp16 input
# ---------------------------------------------------------------------------

def quality_report(dev, tokens: int = 4096, heads: int = 32, d: int = 128) -> dict:
    """Per group size G in {32, 64, 128} (K and V both grouped at G): quantize seeded fp16 rows
    through the library, dequantize them back (fp32, exact), and compare with the fp16 input
    row by row (a row = one token of one head, d values).  K carries the x20 outlier channels.
    The group step s is read back from the dequantized values (max |x^| over a nonzero group
    is exactly 7 s)."""
    import torch

    import int4_group_quantized_kvq_gb300 as kvq
    import workloads as W
    k = W.kv_tensor(W.SEED_K, (1, tokens, heads, d), 20.0, W.outlier_channels(heads, d), device=dev)
    v = W.kv_tensor(W.SEED_V, (1, tokens, heads, d), device=dev)
    P = 16
    npg = tokens // P
    bt = torch.arange(npg, dtype=torch.int32, device=dev).view(1, -1)
    rep = {}
    for G in (32, 64, 128):
        cfg = kvq.config(heads, d, P, G, G, npg)
        pool = torch.zeros(kvq.kvq_pool_bytes(cfg), dtype=torch.uint8, device=dev)
        kvq.kvq_quantize_append(cfg, pool, k, v, bt, torch.zeros(1, dtype=torch.int32, device=dev))
        dk = torch.empty((tokens, heads, d), dtype=torch.float32, device=dev)
        dv = torch.empty_like(dk)
        kvq.kvq_dequantize(cfg, pool, bt, 0, 0, tokens, dk, dv)
        out = {}
        for name, x, xh in (("K", k[0].float(), dk), ("V", v[0].float(), dv)):
            cos = torch.nn.functional.cosine_similarity(x.reshape(-1, d), xh.reshape(-1, d), dim=1)
            err = (x - xh).abs()
            step = xh.abs().reshape(tokens, heads, d // G, G).amax(-1, keepdim=True) / 7.0
            ratio = (err.reshape(tokens, heads, d // G, G) / step.clamp_min(1e-30)).amax()
            out[name] = {"cos_mean": float(cos.mean()), "cos_min": float(cos.min()),
                         "max_abs_err": float(err.max()), "max_err_over_scale": float(ratio),
                         "mse": float((err ** 2).mean())}
        rep[f"G{G}"] = out
    # the rotated 4-bit codec (Walsh-Hadamard rotation, Lloyd-Max codebook) on the same rows
    cfg = kvq.config(heads, d, P, 64, 128, npg)
    pool = torch.zeros(kvq.kvq_wht4_pool_bytes(cfg), dtype=torch.uint8, device=dev)
    kvq.kvq_wht4_quantize_append(cfg, pool, k, v, bt, torch.zeros(1, dtype=torch.int32, device=dev))
    dk = torch.empty((tokens, heads, d), dtype=torch.float32, device=dev)
    dv = torch.empty_like(dk)
    kvq.kvq_wht4_dequantize(cfg, pool, bt, 0, 0, tokens, dk, dv)
    out = {}
    for name, x, xh in (("K", k[0].float(), dk), ("V", v[0].float(), dv)):
        cos = torch.nn.functional.cosine_similarity(x.reshape(-1, d), xh.reshape(-1, d), dim=1)
        err = (x - xh).abs()
        out[name] = {"cos_mean": float(cos.mean()), "cos_min": float(cos.min()), "max_abs_err": float(err.max()),
                     "mse": float((err ** 2).mean()), "rel_mse": float((err ** 2).sum() / (x ** 2).sum())}
    rep["rotated_4bit"] = out
    rep["rows"] = f"{tokens} tokens x {heads} heads, d={d}, N(0,1) fp16; K with 4 x20 outlier channels per head"
    return rep


# ---------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------

def run_kvq(args, world, rank, local):
    import torch
    import torch.distributed as dist

    import int4_group_quantized_kvq_gb300 as kvq
    import workloads as W
    from int4_group_quantized_kvq_gb300.cache import PagedKVCache

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = make_workload(args.workload, args.group)
    K, Wm = args.steps, args.warmup
    if Wm < 3:
        raise SystemExit("--warmup must be at least 3")

    # ---- inputs (seeded, synthetic, generated on the GPU) ----
    n_tok = max(wl.seq_lens)
    oidx = W.outlier_channels(wl.Hkv, wl.d)
    k_all = W.kv_tensor(W.SEED_K, (wl.B, n_tok, wl.Hkv, wl.d), 20.0, oidx, device=dev)
    v_all = W.kv_tensor(W.SEED_V, (wl.B, n_tok, wl.Hkv, wl.d), device=dev)
    q = W.kv_tensor(W.SEED_Q, (1, wl.B, wl.Hq, wl.d), device=dev)[0].contiguous()
    cfg = kvq.config(wl.Hkv, wl.d, wl.P, wl.Gk, wl.Gv, wl.num_pages)
    bt = wl.block_table()
    pool_bytes = kvq.kvq_pool_bytes(cfg)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20)
    n_pools = max(2, math.ceil(3 * l2 / pool_bytes))

    caches = [PagedKVCache(cfg, bt, wl.Hq, wl.max_len, device=dev)]
    # prefill the first pool: each sequence's history in one call (timed as the quantize throughput)
    same_ctx = len(set(wl.ctx)) == 1
    zero = torch.zeros(wl.B if same_ctx else 1, dtype=torch.int32, device=dev)
    hist = [(k_all[:, :wl.ctx[0]].contiguous(), v_all[:, :wl.ctx[0]].contiguous())] if same_ctx else \
        [(k_all[b:b + 1, :c].contiguous(), v_all[b:b + 1, :c].contiguous()) for b, c in enumerate(wl.ctx)]
    run_prefill = history_prefill(kvq, cfg, k_all, v_all, wl, dev)

    def prefill(cache):
        run_prefill(cache.pool, cache.block_table, cache.status)

    prefill(caches[0])
    # the comparison's FP16 cache holds the same fp16 history
    pool16 = pool8 = pool4r = None
    if getattr(args, "compare", False):
        pool16 = torch.zeros(kvq.kvq_fp16_pool_bytes(cfg), dtype=torch.uint8, device=dev)
        pool8 = torch.zeros(kvq.kvq_int8_pool_bytes(cfg), dtype=torch.uint8, device=dev)
        pool4r = torch.zeros(kvq.kvq_wht4_pool_bytes(cfg), dtype=torch.uint8, device=dev)
        for fn, pl in ((kvq.kvq_fp16_append, pool16), (kvq.kvq_int8_quantize_append, pool8),
                       (kvq.kvq_wht4_quantize_append, pool4r)):
            if same_ctx:
                fn(cfg, pl, hist[0][0], hist[0][1], caches[0].block_table, zero)
            else:
                for b, (kb, vb) in enumerate(hist):
                    fn(cfg, pl, kb, vb, caches[0].block_table[b:b + 1], zero)
    torch.cuda.synchronize()
    qt = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        prefill(caches[0])
        e1.record()
        torch.cuda.synchronize()
        qt.append(e0.elapsed_time(e1) * 1e-3)
    tok_hist = sum(wl.ctx)
    q_bytes = wl.Hkv * tok_hist * (2 * wl.d * 2 + wl.packed_bytes_per_token_head())
    quantize = {"gbs": q_bytes / min(qt) / 1e9, "tokens": tok_hist, "bytes": q_bytes,
                "what": "prefill quantize of the whole history in one call: fp16 K+V read, packed codes+scales "
                        "written"}
    for _ in range(n_pools - 1):
        caches.append(PagedKVCache(cfg, bt, wl.Hq, wl.max_len, device=dev, pool=caches[0].pool.clone()))

    pos = torch.tensor(wl.ctx, dtype=torch.int32, device=dev)
    idx = pos.long().view(-1, 1, 1, 1).expand(-1, 1, wl.Hkv, wl.d)
    k_new = torch.gather(k_all, 1, idx).contiguous()
    v_new = torch.gather(v_all, 1, idx).contiguous()
    if pool16 is not None:  # the new token, as the INT4 step appends it
        kvq.kvq_fp16_append(cfg, pool16, k_new, v_new, caches[0].block_table, pos)
        kvq.kvq_int8_quantize_append(cfg, pool8, k_new, v_new, caches[0].block_table, pos)
        kvq.kvq_wht4_quantize_append(cfg, pool4r, k_new, v_new, caches[0].block_table, pos)
    del k_all, v_all, hist, run_prefill
    torch.cuda.empty_cache()
    seq_lens = torch.tensor(wl.seq_lens, dtype=torch.int32, device=dev)
    out = torch.empty((wl.B, wl.Hq, wl.d), dtype=torch.float32, device=dev)

    step_bytes = wl.decode_bytes() + wl.append_bytes()
    stream = torch.cuda.Stream(device=dev)

    # ---- warm-up (eager) ----
    with torch.cuda.stream(stream):
        for i in range(Wm):
            caches[i % n_pools].decode_step(q, k_new, v_new, pos, seq_lens, out, stream=stream)
    stream.synchronize()

    # ---- the timed steps: CUDA graphs of G steps (rotating pools).  No event sits between the
    # kernels inside a graph, so each launch keeps its programmatic dependence on the one
    # before (an event node in between would turn it into a full dependence) ----
    use_graph = not args.eager
    G = max(g for g in range(1, min(K, args.graph_steps) + 1) if K % g == 0) if use_graph else K
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(G):
                caches[i % n_pools].decode_step(q, k_new, v_new, pos, seq_lens, out, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(2):
                graph.replay()
        stream.synchronize()

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        if use_graph:
            for _ in range(K // G):
                graph.replay()
        else:
            for i in range(K):
                caches[i % n_pools].decode_step(q, k_new, v_new, pos, seq_lens, out, stream=stream)
        t_end.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    t_local = t_start.elapsed_time(t_end) * 1e-3

    # ---- the decode kernel's own duration: back-to-back decode attention calls over the same
    # rotating pools (a graph of D calls replayed), CUDA events on the launch stream around
    # the replays; the per-call average is what roofline.achieved divides by ----
    D = G if use_graph else min(K, 200)
    n_rep = max(1, min(K // max(D, 1), 20))
    if use_graph:
        dgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(dgraph, stream=stream):
            for i in range(D):
                caches[i % n_pools].attend(q, seq_lens, out, stream=stream)
        with torch.cuda.stream(stream):
            dgraph.replay()
        stream.synchronize()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        d0.record(stream)
        for _ in range(n_rep):
            if use_graph:
                dgraph.replay()
            else:
                for i in range(D):
                    caches[i % n_pools].attend(q, seq_lens, out, stream=stream)
        d1.record(stream)
    stream.synchronize()
    decode_s = d0.elapsed_time(d1) * 1e-3 / (n_rep * D)

    # ---- the latency comparison ("LLM long-context inference: managing the KV cache with an
    # INT4 state machine" section 7.4): FP16 attention; INT4 dequantized to an FP16 pool and
    # then attended; INT4 dequantized inside the operator (decode_s above).  Same workload,
    # same timing (a graph of D back-to-back calls, replayed) ----
    comparison = None
    if pool16 is not None:
        cfg16 = cfg
        ws16 = kvq.new_fp16_workspace(cfg16, wl.B, wl.Hq, wl.max_len, device=dev)
        deq16 = torch.empty_like(pool16)
        out16 = torch.empty_like(out)
        bt0 = caches[0].block_table
        scale = 1.0 / math.sqrt(wl.d)

        def fp16_attend():
            kvq.kvq_fp16_decode_attention(cfg16, pool16, q, bt0, seq_lens, wl.max_len, scale, out16, ws16,
                                          stream=stream)

        def deq_then_attend():
            kvq.kvq_dequantize_to_fp16_pool(cfg16, caches[0].pool, deq16, bt0, seq_lens, wl.max_len, stream=stream)
            kvq.kvq_fp16_decode_attention(cfg16, deq16, q, bt0, seq_lens, wl.max_len, scale, out16, ws16,
                                          stream=stream)

        def per_call(fn, calls=50, reps=4):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                fn()
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(calls):
                    fn()
            with torch.cuda.stream(stream):
                g.replay()
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(reps):
                    g.replay()
                e1.record(stream)
            stream.synchronize()
            return e0.elapsed_time(e1) * 1e-3 / (calls * reps)

        R = 128  # the mixed arm: the last 128 positions in FP16, the older ones in INT4
        wsm = torch.zeros(kvq.kvq_mixed_decode_workspace_bytes(cfg16, wl.B, wl.Hq, wl.max_len, R), dtype=torch.uint8,
                          device=dev)

        def mixed_attend():
            kvq.kvq_mixed_decode_attention(cfg16, caches[0].pool, bt0, pool16, bt0, cfg16.num_pages, q, seq_lens,
                                           wl.max_len, R, scale, out16, wsm, stream=stream)

        ws8 = torch.zeros(kvq.kvq_int8_decode_workspace_bytes(cfg16, wl.B, wl.Hq, wl.max_len), dtype=torch.uint8,
                          device=dev)

        def int8_attend():
            kvq.kvq_int8_decode_attention(cfg16, pool8, q, bt0, seq_lens, wl.max_len, scale, out16, ws8, stream=stream)

        ws4r = torch.zeros(kvq.kvq_wht4_decode_workspace_bytes(cfg16, wl.B, wl.Hq, wl.max_len), dtype=torch.uint8,
                           device=dev)

        def wht4_attend():
            kvq.kvq_wht4_decode_attention(cfg16, pool4r, q, bt0, seq_lens, wl.max_len, scale, out16, ws4r,
                                          stream=stream)

        t4r = per_call(wht4_attend)
        t8 = per_call(int8_attend)
        t16 = per_call(fp16_attend)
        tdq = per_call(deq_then_attend)
        tmx = per_call(mixed_attend)
        fp16_bytes = 4 * wl.d * sum(wl.seq_lens) * wl.Hkv
        comparison = {
            "what": "decode attention latency on the bench workload: FP16 cache; INT4 dequantized to an FP16 pool "
                    "then attended; INT4 dequantized inside the operator (back-to-back calls in CUDA graphs)",
            "fp16_us": t16 * 1e6, "fp16_gbs": fp16_bytes / t16 / 1e9,
            "int4_dequant_then_attend_us": tdq * 1e6,
            "int4_fused_us": decode_s * 1e6,
            "mixed_int4_fp16_last128_us": tmx * 1e6,
            "int8_per_row_us": t8 * 1e6,
            "int8_bytes": (2 * wl.d + 8) * sum(wl.seq_lens) * wl.Hkv,
            "rotated_4bit_us": t4r * 1e6,
            "rotated_4bit_bytes": (wl.d + 8) * sum(wl.seq_lens) * wl.Hkv,
            "fp16_bytes": fp16_bytes, "int4_bytes": wl.decode_bytes(),
            "fused_speedup_vs_fp16": t16 / decode_s, "fused_speedup_vs_dequant_then_attend": tdq / decode_s,
        }
        if rank == 0:
            print(f"[compare] fp16 {t16 * 1e6:.1f} us ({fp16_bytes / t16 / 1e9:.0f} GB/s), dequant+attend "
                  f"{tdq * 1e6:.1f} us, int4 fused {decode_s * 1e6:.1f} us, mixed (last {R} fp16) {tmx * 1e6:.1f} us, "
                  f"int8 {t8 * 1e6:.1f} us ({(2 * wl.d + 8) * sum(wl.seq_lens) * wl.Hkv / t8 / 1e9:.0f} GB/s), "
                  f"rotated 4-bit {t4r * 1e6:.1f} us ({(wl.d + 8) * sum(wl.seq_lens) * wl.Hkv / t4r / 1e9:.0f} GB/s)",
                  file=sys.stderr)
    # the step leaves the output of the last decode step in `out` for e2e and checks
    flags = max(c.flags() for c in caches)
    t_max = max_over_ranks(t_local, world, dev)
    step_s = t_max / K

    # ---- end to end through the public API from pinned host buffers ----
    e2e = None
    if not args.no_e2e:
        from int4_group_quantized_kvq_gb300.cache import HostPipeline
        pipe = HostPipeline(caches[0], compute_stream=stream)
        for st in pipe.slots:
            st.q_host.copy_(q.cpu())
            st.k_host.copy_(k_new.reshape(st.k_host.shape).cpu())
            st.v_host.copy_(v_new.reshape(st.v_host.shape).cpu())
        n_e2e = K

        def timed(run_one, sync):
            for i in range(Wm):
                run_one(i)
            sync()
            if world > 1:
                dist.barrier()
            t0 = time.perf_counter()
            for i in range(n_e2e):
                run_one(i)
            sync()
            return max_over_ranks(time.perf_counter() - t0, world, dev)

        # one kvq_decode_step_host call per step, on one stream; the staging slots alternate so that
        # the host may refill one while the other is in use
        t_e2e = timed(lambda i: caches[i % n_pools].decode_step_host(pipe.slots[i % 2], pos, seq_lens,
                                                                     stream=stream), stream.synchronize)
        # the same steps with the copies on their own streams (kvq_decode_step_host_pipelined)
        t_pipe = timed(lambda i: pipe.step(i, pos, seq_lens, cache=caches[i % n_pools]), pipe.synchronize)
        st0 = pipe.slots[0]
        h2d = st0.host.numel() * 2
        d2h = st0.out_host.numel() * 4
        e2e = {"value": world * n_e2e * step_bytes / t_pipe / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": n_e2e, "ms_per_step": t_pipe / n_e2e * 1e3,
               "how": "one kvq_decode_step_host_pipelined C-ABI call per step (HostPipeline), from pinned host "
                      "buffers: the call copies the step's q/K/V host-to-device (one cudaMemcpyAsync) on an input "
                      "copy stream, runs the step (decode and combine launches) on the compute stream and copies "
                      "its output device-to-host (one cudaMemcpyAsync) on an output copy stream, ordered by "
                      "per-slot events; two staging slots alternate, so step i+1's input copy and step i-1's "
                      "output copy overlap step i's kernels; wall clock over all steps, synchronized at the end",
               "single_call": {"value": world * n_e2e * step_bytes / t_e2e / 1e9, "ms_per_step": t_e2e / n_e2e * 1e3,
                               "how": "one kvq_decode_step_host C-ABI call per step on one stream: a copy kernel "
                                      "reads the inputs from pinned host memory, the step runs, the combine also "
                                      "writes the output to pinned host memory; one chain of programmatic "
                                      "dependent launches"}}

    if rank != 0:
        return None
    peaks = load_peaks()
    achieved = wl.decode_bytes() / decode_s / 1e9
    res = {
        "metric": METRIC,
        "value": world * step_bytes / step_s / 1e9,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": Wm,
        "ms_per_step": step_s * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "dtype_detail": "INT4 codes + fp16 group scales stored; f16 x f16 -> f32 tensor-core MMA; fp32 softmax; "
                        "fp32 output",
        "data": "synthetic",
        "config": {
            "workload": wl.name,
            "description": wl.description,
            "batch": wl.B, "q_heads": wl.Hq, "kv_heads": wl.Hkv, "head_dim": wl.d,
            "context": wl.ctx[0] if len(set(wl.ctx)) == 1 else f"{min(wl.ctx)}..{max(wl.ctx)}",
            "attended_tokens": sum(wl.seq_lens), "page_size": wl.P, "group_k": wl.Gk, "group_v": wl.Gv,
            "step": "quantize-append 1 token per sequence + decode attention, one kvq_decode_step call: "
                    "the split-KV decode grid with the append fused in, then the combine grid",
            "bytes_per_step": step_bytes,
            "l2": f"inputs larger than L2: {n_pools} rotated pool copies of {pool_bytes / 1e6:.1f} MB "
                  f"against a {l2 / 1e6:.0f} MB L2",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "timing": (f"CUDA graphs of {G} steps replayed {K // G} times" if use_graph else "eager launches")
            + ", CUDA events on the launch stream; decode kernel duration from "
            + f"{n_rep} x {D} back-to-back decode calls",
        },
        "tokens_per_s": world * wl.B / step_s,
        "decode_us": decode_s * 1e6,
        "quantize": quantize,
        "roofline": {
            "bound": "hbm",
            "achieved": achieved,
            "peak": peaks["hbm_gbs"],
            "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"],
            "traffic": measured_traffic(wl.name),
            "kernel": "decode_splitkv_kernel (kvq_decode_attention): packed bytes of the cache per call over the "
                      "per-call time of back-to-back calls",
            "peak_source": peaks["source"],
        },
        "e2e": e2e,
        "gpu_launches": 2 * K,  # per step: the decode grid (append fused in) and the combine grid
        "status_flags": flags,
        "clocks": clocks,
    }
    if comparison is not None:
        res["comparison"] = comparison
    if not args.no_quality:
        res["quality"] = quality_report(dev)
    if not args.no_sweep:
        # the other workloads and the prefill-quantize pass, on rank 0's GPU, with their own clocks
        del caches
        torch.cuda.empty_cache()
        sampler = ClockSampler(local)
        sampler.start()
        sweep = {"what": "decode_us: back-to-back kvq_decode_attention calls (split-KV decode) in CUDA graphs "
                         "over rotated pools larger than L2; step_us: the same for kvq_decode_step (append of "
                         "one token per sequence fused in); frac: packed decode bytes / decode_us against the "
                         "measured HBM peak",
                 "decode": decode_sweep(dev, stream, peaks, l2),
                 "prefill_quantize": prefill_quantize_sweep(dev, stream, peaks)}
        sweep["clocks"] = sampler.stop()
        res["workloads"] = sweep
    if world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = time_oracle(wl, args.cpu_seconds)
        res["cpu_baseline"].pop("seconds_per_step", None)
        res["cpu_baseline"]["quantize"] = time_oracle_quantize(wl, 2.0)
        if not args.no_sweep:
            # the oracle on the other configurations too, a short sample each
            per_cfg = {}
            for name, G in (("gqa8b", None), ("ragged", None), ("longctx", 64)):
                w = make_workload(name, G)
                per_cfg[w.name] = time_oracle(w, 1.0)
                per_cfg[w.name].pop("seconds_per_step", None)
            w5 = make_workload("longctx", 64)
            per_cfg["prefill_quantize_" + w5.name] = time_oracle_quantize(w5, 1.0)
            res["cpu_baseline"]["configs"] = per_cfg
    return res


# ---------------------------------------------------------------------------
# the other decode workloads and the long-context prefill-quantize pass, reported beside
# the headline in the same JSON line
# ---------------------------------------------------------------------------

# GQA 8B-shaped, ragged continuous batching, and long context at the three group sizes
SWEEP_DECODE = (("gqa8b", None), ("ragged", None), ("longctx", 32), ("longctx", 64), ("longctx", 128))


def graph_per_call(fn, stream, calls: int = 50, reps: int = 4, warm: int = 3) -> float:
    """Seconds per call of fn(i): `warm` eager calls, then a CUDA graph of `calls` back-to-back
    calls replayed once untimed and `reps` times between two events on the launch stream."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(warm):
            fn(i)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(calls):
            fn(i)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    del g
    return e0.elapsed_time(e1) * 1e-3 / (calls * reps)


def history_prefill(kvq, cfg, k_all, v_all, wl, dev):
    """A callable that quantizes each sequence's history (positions 0 .. ctx[b]-1) into a pool in
    one call: kvq_quantize_append when every sequence has the same history, else the ragged
    kvq_quantize_append_varlen over the histories packed back to back (built here, once)."""
    import torch
    zero = torch.zeros(wl.B, dtype=torch.int32, device=dev)
    if len(set(wl.ctx)) == 1:
        c = wl.ctx[0]
        k_h, v_h = k_all[:, :c].contiguous(), v_all[:, :c].contiguous()

        def run(pool, block_table, status, stream=None):
            kvq.kvq_quantize_append(cfg, pool, k_h, v_h, block_table, zero, status=status, stream=stream)
        return run
    k_rows = torch.cat([k_all[b, :c] for b, c in enumerate(wl.ctx)]).contiguous()
    v_rows = torch.cat([v_all[b, :c] for b, c in enumerate(wl.ctx)]).contiguous()
    cu = torch.tensor([0] + list(itertools.accumulate(wl.ctx)), dtype=torch.int32, device=dev)

    def run(pool, block_table, status, stream=None):
        kvq.kvq_quantize_append_varlen(cfg, pool, k_rows, v_rows, block_table, zero, cu, status=status,
                                       stream=stream)
    return run


def decode_sweep(dev, stream, peaks: dict, l2: int) -> dict:
    """Per workload: the decode attention call and the decode step (append fused in), each timed as
    back-to-back calls over rotated pool copies larger than L2."""
    import torch

    import int4_group_quantized_kvq_gb300 as kvq
    import workloads as W
    from int4_group_quantized_kvq_gb300.cache import PagedKVCache
    res = {}
    for name, G in SWEEP_DECODE:
        wl = make_workload(name, G)
        n_tok = max(wl.seq_lens)
        oidx = W.outlier_channels(wl.Hkv, wl.d)
        k_all = W.kv_tensor(W.SEED_K, (wl.B, n_tok, wl.Hkv, wl.d), 20.0, oidx, device=dev)
        v_all = W.kv_tensor(W.SEED_V, (wl.B, n_tok, wl.Hkv, wl.d), device=dev)
        q = W.kv_tensor(W.SEED_Q, (1, wl.B, wl.Hq, wl.d), device=dev)[0].contiguous()
        cfg = kvq.config(wl.Hkv, wl.d, wl.P, wl.Gk, wl.Gv, wl.num_pages)
        cache0 = PagedKVCache(cfg, wl.block_table(), wl.Hq, wl.max_len, device=dev)
        history_prefill(kvq, cfg, k_all, v_all, wl, dev)(cache0.pool, cache0.block_table, cache0.status)
        pos = torch.tensor(wl.ctx, dtype=torch.int32, device=dev)
        idx = pos.long().view(-1, 1, 1, 1).expand(-1, 1, wl.Hkv, wl.d)
        k_new = torch.gather(k_all, 1, idx).contiguous()
        v_new = torch.gather(v_all, 1, idx).contiguous()
        del k_all, v_all
        pool_bytes = kvq.kvq_pool_bytes(cfg)
        n_pools = max(2, math.ceil(3 * l2 / pool_bytes))
        caches = [cache0] + [PagedKVCache(cfg, cache0.block_table, wl.Hq, wl.max_len, device=dev,
                                          pool=cache0.pool.clone()) for _ in range(n_pools - 1)]
        seq_lens = torch.tensor(wl.seq_lens, dtype=torch.int32, device=dev)
        out = torch.empty((wl.B, wl.Hq, wl.d), dtype=torch.float32, device=dev)
        t_dec = graph_per_call(lambda i: caches[i % n_pools].attend(q, seq_lens, out, stream=stream), stream)
        t_step = graph_per_call(lambda i: caches[i % n_pools].decode_step(q, k_new, v_new, pos, seq_lens, out,
                                                                          stream=stream), stream)
        torch.cuda.synchronize()
        flags = max(c.flags() for c in caches)
        gbs = wl.decode_bytes() / t_dec / 1e9
        res[wl.name] = {
            "batch": wl.B, "q_heads": wl.Hq, "kv_heads": wl.Hkv, "group_k": wl.Gk, "group_v": wl.Gv,
            "attended_tokens": sum(wl.seq_lens), "decode_bytes": wl.decode_bytes(),
            "decode_us": t_dec * 1e6, "decode_gbs": gbs, "frac": gbs / peaks["hbm_gbs"],
            "step_us": t_step * 1e6, "step_gbs": (wl.decode_bytes() + wl.append_bytes()) / t_step / 1e9,
            "tokens_per_s": wl.B / t_step, "status_flags": flags,
            "l2": f"{n_pools} rotated pool copies of {pool_bytes / 1e6:.1f} MB",
        }
        del caches, cache0, q, k_new, v_new, out
        torch.cuda.empty_cache()
    return res


def prefill_quantize_sweep(dev, stream, peaks: dict, reps: int = 5) -> dict:
    """The long-context prefill-quantize pass: 131072 tokens x 8 KV heads x 128, K and V, in one
    kvq_quantize_append call into a permuted page pool, at K = V group sizes 32, 64 and 128.
    Inputs (537 MB of fp16) and the pool exceed L2.  Bytes: fp16 K+V read, codes and scales written."""
    import torch

    import int4_group_quantized_kvq_gb300 as kvq
    import workloads as W
    res = {}
    base = W.longctx(64)
    n = base.ctx[0]
    k = W.kv_tensor(W.SEED_K, (1, n, base.Hkv, base.d), 20.0, W.outlier_channels(base.Hkv, base.d), device=dev)
    v = W.kv_tensor(W.SEED_V, (1, n, base.Hkv, base.d), device=dev)
    zero = torch.zeros(1, dtype=torch.int32, device=dev)
    for G in (32, 64, 128):
        wl = W.longctx(G)
        cfg = kvq.config(wl.Hkv, wl.d, wl.P, wl.Gk, wl.Gv, wl.num_pages)
        bt = wl.block_table().to(dev)
        pool = torch.zeros(kvq.kvq_pool_bytes(cfg), dtype=torch.uint8, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        with torch.cuda.stream(stream):
            for _ in range(3):
                kvq.kvq_quantize_append(cfg, pool, k, v, bt, zero, status=status, stream=stream)
        stream.synchronize()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                kvq.kvq_quantize_append(cfg, pool, k, v, bt, zero, status=status, stream=stream)
                e1.record(stream)
            stream.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e-3)
        nbytes = n * wl.Hkv * (2 * wl.d * 2 + wl.packed_bytes_per_token_head())
        t = statistics.median(ts)
        res[f"G{G}"] = {"tokens": n, "kv_heads": wl.Hkv, "head_dim": wl.d, "bytes": nbytes, "us": t * 1e6,
                        "gbs": nbytes / t / 1e9, "frac": nbytes / t / 1e9 / peaks["hbm_gbs"],
                        "best_us": min(ts) * 1e6, "status_flags": kvq.kvq_read_status(status)}
        del pool
    del k, v
    torch.cuda.empty_cache()
    return res


def max_over_ranks(seconds: float, world: int, device) -> float:
    """The slowest rank's time: every rank contributes its own, all receive the maximum."""
    if world <= 1:
        return seconds
    import torch
    import torch.distributed as dist
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, world, rank):
    """The oracle on the host cores, on a bounded sample per step of the same workload."""
    if rank != 0:
        return None
    wl = make_workload(args.workload, args.group)
    K, Wm = args.steps, args.warmup
    per_step = max(0.002, min(2.0, 150.0 / (K + Wm)))
    smp = plan_oracle_sample(wl, per_step)
    for _ in range(Wm):
        smp.step()
    t0 = time.perf_counter()
    for _ in range(K):
        smp.step()
    t = time.perf_counter() - t0
    value = K * smp.bytes() / t / 1e9
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": Wm,
        "ms_per_step": t / K * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": wl.name, "description": wl.description, "sample": smp.describe()},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "host_cores": os.cpu_count(), "kind": "oracle", "sample": smp.describe()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    world, rank, local = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "kvq" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            res = run_reference(args, world, rank)
        else:
            res = run_kvq(args, world, rank, local)
        if rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()

"""Shared helpers of the GPU parity tests: build inputs, run the oracle beside the
CUDA path on the same bytes, and apply the tolerances.

Tolerance of decode attention (fp32 output against the oracle's fp64 attention over
the dequantized cache), per output row (b, query head):
    max |gpu - ref|                 <= 2e-4
    max |gpu - ref| / max |ref|     <= 1e-3
Packed codes, scales and dequantized values are compared bit for bit.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import workloads as W

ATOL = 2e-4
RTOL_ROW = 1e-3


def assert_attention_close(got: np.ndarray, ref: np.ndarray, what: str = "") -> dict:
    """got fp32 [.., Hq, d] vs ref fp64; per-row absolute and relative infinity-norm gates."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    row_err = err.max(axis=-1)
    row_ref = np.abs(ref).max(axis=-1)
    rel = row_err / np.maximum(row_ref, 1e-30)
    stats = {"max_abs": float(err.max(initial=0.0)), "max_rel_row": float(rel.max(initial=0.0))}
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert stats["max_abs"] <= ATOL, f"{what}: max abs error {stats['max_abs']:.3e} > {ATOL}"
    assert stats["max_rel_row"] <= RTOL_ROW, f"{what}: row relative error {stats['max_rel_row']:.3e} > {RTOL_ROW}"
    return stats


class Case:
    """A decode problem: geometry, lengths, paging and seeded K/V/q (fp16, CPU tensors)."""

    def __init__(self, B, Hq, Hkv, d, lens, P=16, Gk=64, Gv=128, seed=1, permute=True, extra_pages=3,
                 outliers=True, device="cpu"):
        self.B, self.Hq, self.Hkv, self.d, self.P, self.Gk, self.Gv = B, Hq, Hkv, d, P, Gk, Gv
        self.lens = list(lens)
        pages = [(n + P - 1) // P for n in self.lens]
        self.max_blocks = max(1, max(pages))
        self.num_pages = sum(pages) + extra_pages
        order = W.permutation(seed + 100, self.num_pages) if permute else \
            torch.arange(self.num_pages, dtype=torch.int32)
        bt = torch.full((B, self.max_blocks), -1, dtype=torch.int32)
        k = 0
        for b, n in enumerate(pages):
            bt[b, :n] = order[k:k + n]
            k += n
        self.block_table = bt
        n = max(1, max(self.lens))
        oidx = W.outlier_channels(Hkv, d, seed=seed + 5) if outliers else None
        self.k = W.kv_tensor(seed, (B, n, Hkv, d), 20.0 if outliers else 0.0, oidx, device=device).cpu()
        self.v = W.kv_tensor(seed + 1, (B, n, Hkv, d), device=device).cpu()
        self.q = W.kv_tensor(seed + 2, (1, B, Hq, d), device=device).cpu()[0]
        self.scale = 1.0 / math.sqrt(d)

    @property
    def layout(self) -> oracle.Layout:
        return oracle.Layout(self.Hkv, self.d, self.P, self.Gk, self.Gv, self.num_pages)

    def cfg(self, kvq):
        return kvq.config(self.Hkv, self.d, self.P, self.Gk, self.Gv, self.num_pages)

    def oracle_pool(self, fill: int = 0) -> np.ndarray:
        """The pool as the oracle writes it: each sequence's history appended from position 0."""
        L = self.layout
        pool = np.full(L.pool_bytes, fill, np.uint8)
        bt = self.block_table.numpy()
        for b in range(self.B):
            if self.lens[b]:
                oracle.quantize_append(L, pool, self.k[b:b + 1, :self.lens[b]].numpy(),
                                       self.v[b:b + 1, :self.lens[b]].numpy(), bt[b:b + 1],
                                       np.zeros(1, np.int32))
        return pool

    def oracle_attention(self, pool: np.ndarray) -> np.ndarray:
        return oracle.decode_attention(self.layout, pool, self.q.numpy(), self.block_table.numpy(),
                                       np.array(self.lens, np.int32), self.scale)


def gpu_decode(kvq, case: Case, pool_gpu: torch.Tensor, max_len: int | None = None, ws: torch.Tensor | None = None):
    cfg = case.cfg(kvq)
    dev = pool_gpu.device
    q = case.q.to(dev)
    bt = case.block_table.to(dev)
    sl = torch.tensor(case.lens, dtype=torch.int32, device=dev)
    ml = max(case.lens) if max_len is None else max_len
    out = torch.full((case.B, case.Hq, case.d), float("nan"), dtype=torch.float32, device=dev)
    if ws is None:
        ws = kvq.new_workspace(cfg, case.B, case.Hq, ml, device=dev)
    kvq.kvq_decode_attention(cfg, pool_gpu, q, bt, sl, ml, case.scale, out, ws)
    flags = kvq.kvq_read_status(ws)
    return out.cpu().numpy(), flags

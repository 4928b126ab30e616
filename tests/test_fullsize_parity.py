"""Full-size workloads, run through the same decode step the benchmark times
(PagedKVCache.decode_step: quantize-on-append of one token per sequence, then decode
attention with the benchmark's grid), checked against the oracle on sampled sequences:

  - the packed pages of a sampled sequence (every KV head) are compared byte for byte
    with the oracle's quantization of the same history plus the appended token;
  - the sampled sequence's attention output is compared with the oracle's fp64
    attention within the tolerances of kvq_testlib (for long contexts on one query
    head per KV head group at a time, to keep the oracle's CPU time in bounds).

Inputs are generated on the GPU by the seeded generator (workloads), then copied to
the host for the oracle: both sides see the same fp16 bytes.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from conftest import cuda_available
from kvq_testlib import assert_attention_close

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


def run_step(kvq, wl: W.Workload):
    """Build the cache for workload wl on the GPU and run one decode step.  Returns the pieces the checks need."""
    from int4_group_quantized_kvq_gb300.cache import PagedKVCache
    dev = "cuda"
    n_tok = max(wl.seq_lens)
    oidx = W.outlier_channels(wl.Hkv, wl.d)
    k = W.kv_tensor(W.SEED_K, (wl.B, n_tok, wl.Hkv, wl.d), 20.0, oidx, device=dev)
    v = W.kv_tensor(W.SEED_V, (wl.B, n_tok, wl.Hkv, wl.d), device=dev)
    q = W.kv_tensor(W.SEED_Q, (1, wl.B, wl.Hq, wl.d), device=dev)[0].contiguous()
    cfg = kvq.config(wl.Hkv, wl.d, wl.P, wl.Gk, wl.Gv, wl.num_pages)
    bt = wl.block_table()
    cache = PagedKVCache(cfg, bt, wl.Hq, wl.max_len, device=dev)
    # prefill: each sequence's history (positions 0 .. ctx-1)
    for b, ctx in enumerate(wl.ctx):
        kb = k[b:b + 1, :ctx].contiguous()
        vb = v[b:b + 1, :ctx].contiguous()
        kvq.kvq_quantize_append(cfg, cache.pool, kb, vb, cache.block_table[b:b + 1],
                                torch.zeros(1, dtype=torch.int32, device=dev), status=cache.status)
    # the step: append the token at position ctx, attend over ctx + 1
    pos = torch.tensor(wl.ctx, dtype=torch.int32, device=dev)
    idx = pos.long().view(-1, 1, 1, 1).expand(-1, 1, wl.Hkv, wl.d)
    k_new = torch.gather(k, 1, idx).contiguous()
    v_new = torch.gather(v, 1, idx).contiguous()
    seq_lens = torch.tensor(wl.seq_lens, dtype=torch.int32, device=dev)
    out = torch.full((wl.B, wl.Hq, wl.d), float("nan"), dtype=torch.float32, device=dev)
    cache.decode_step(q, k_new, v_new, pos, seq_lens, out)
    torch.cuda.synchronize()
    assert cache.flags() == 0
    return cache, bt.numpy(), k, v, q, out


def check_sequence(kvq, wl, cache, bt, k, v, q, out, b, head_subsample=False):
    L = oracle.Layout(wl.Hkv, wl.d, wl.P, wl.Gk, wl.Gv, wl.num_pages)
    n = wl.seq_lens[b]
    kb = k[b:b + 1, :n].cpu().numpy()
    vb = v[b:b + 1, :n].cpu().numpy()
    ref_pool = np.zeros(L.pool_bytes, np.uint8)
    oracle.quantize_append(L, ref_pool, kb, vb, bt[b:b + 1], np.zeros(1, np.int32))
    # bytes of this sequence's pages, all heads
    gpu_pool = cache.pool.cpu().numpy()
    blk = L.block_bytes
    for pg in bt[b, :wl.pages_per_seq[b]]:
        s0, s1 = int(pg) * wl.Hkv * blk, (int(pg) + 1) * wl.Hkv * blk
        if not np.array_equal(gpu_pool[s0:s1], ref_pool[s0:s1]):
            bad = np.nonzero(gpu_pool[s0:s1] != ref_pool[s0:s1])[0]
            raise AssertionError(f"sequence {b}: page {pg} differs at {bad[:8]} ({bad.size} bytes)")
    got = out[b].cpu().numpy()
    qb = q[b:b + 1].cpu().numpy()
    r = wl.r
    if not head_subsample:
        ref = oracle.decode_attention(L, ref_pool, qb, bt[b:b + 1], np.array([n], np.int32), wl.d ** -0.5)
        return assert_attention_close(got, ref[0], what=f"{wl.name} b={b}")
    stats = []
    for j in sorted({0, r - 1}):
        heads = np.arange(wl.Hkv) * r + j  # one query head of each KV head's group
        ref = oracle.decode_attention(L, ref_pool, np.ascontiguousarray(qb[:, heads]), bt[b:b + 1],
                                      np.array([n], np.int32), wl.d ** -0.5)
        stats.append(assert_attention_close(got[heads], ref[0], what=f"{wl.name} b={b} heads {heads}"))
    return stats


def test_tiny_mha(kvq):
    wl = W.tiny_mha()
    cache, bt, k, v, q, out = run_step(kvq, wl)
    check_sequence(kvq, wl, cache, bt, k, v, q, out, 0)


def test_llama7b_mha_b8_l8192(kvq):
    wl = W.llama7b_mha()
    cache, bt, k, v, q, out = run_step(kvq, wl)
    for b in (0, 5):
        check_sequence(kvq, wl, cache, bt, k, v, q, out, b)


def test_gqa8b_b4_l32768(kvq):
    wl = W.gqa8b()
    cache, bt, k, v, q, out = run_step(kvq, wl)
    check_sequence(kvq, wl, cache, bt, k, v, q, out, 3, head_subsample=True)


def test_ragged_b32(kvq):
    wl = W.ragged()
    cache, bt, k, v, q, out = run_step(kvq, wl)
    shortest = int(np.argmin(wl.seq_lens))
    longest = int(np.argmax(wl.seq_lens))
    for b in (shortest, longest, 17):
        check_sequence(kvq, wl, cache, bt, k, v, q, out, b)


@pytest.mark.parametrize("G", [32, 64, 128])
def test_longctx_b1_l131072(kvq, G):
    wl = W.longctx(G)
    cache, bt, k, v, q, out = run_step(kvq, wl)
    check_sequence(kvq, wl, cache, bt, k, v, q, out, 0, head_subsample=True)


@pytest.mark.parametrize("G", [32, 64, 128])
def test_prefill_quantize_131072x8x128(kvq, G):
    """The separate prefill-quantize pass: 131072 tokens x 8 KV heads x 128, K and V, in one call;
    the whole pool is compared with the oracle's."""
    wl = W.longctx(G)
    n = 131072
    oidx = W.outlier_channels(wl.Hkv, wl.d)
    k = W.kv_tensor(W.SEED_K, (1, n, wl.Hkv, wl.d), 20.0, oidx, device="cuda")
    v = W.kv_tensor(W.SEED_V, (1, n, wl.Hkv, wl.d), device="cuda")
    npg = n // wl.P
    cfg = kvq.config(wl.Hkv, wl.d, wl.P, G, G, npg)
    bt = W.permutation(W.SEED_PERM, npg).view(1, -1)
    pool = torch.full((kvq.kvq_pool_bytes(cfg),), 0xEE, dtype=torch.uint8, device="cuda")
    kvq.kvq_quantize_append(cfg, pool, k, v, bt.cuda(), torch.zeros(1, dtype=torch.int32, device="cuda"))
    L = oracle.Layout(wl.Hkv, wl.d, wl.P, G, G, npg)
    ref = np.full(L.pool_bytes, 0xEE, np.uint8)
    oracle.quantize_append(L, ref, k.cpu().numpy(), v.cpu().numpy(), bt.numpy(), np.zeros(1, np.int32))
    got = pool.cpu().numpy()
    diff = np.nonzero(got != ref)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"

"""The FP16 cache of the latency comparison ("LLM long-context inference: managing the KV
cache with an INT4 state machine" section 7.4) against the oracle:
  - kvq_fp16_append and kvq_dequantize_to_fp16_pool: whole pools bit for bit (both sides
    start from the same fill byte, so a stray or missing write shows up);
  - kvq_fp16_decode_attention: within the tolerances of tests/kvq_testlib.py against the
    oracle's fp64 attention over the same FP16 pool;
  - the dequantize-then-attend arm (INT4 pool -> FP16 pool -> FP16 attention) against the
    oracle's attention over the oracle's FP16 pool."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from conftest import cuda_available
from kvq_testlib import Case, assert_attention_close

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


def _fp16_pool(case: Case, fill=0xA5):
    """Oracle FP16 pool with each sequence's history appended from position 0."""
    L = case.layout
    pool16 = np.full(oracle.fp16_pool_bytes(L), fill, np.uint8)
    bt = case.block_table.numpy()
    for b in range(case.B):
        n = case.lens[b]
        if n:
            oracle.fp16_append(L, pool16, case.k[b:b + 1, :n].numpy(), case.v[b:b + 1, :n].numpy(), bt[b:b + 1],
                               np.zeros(1, np.int32))
    return pool16


def _gpu_fp16_attention(kvq, case: Case, pool16_np, max_len=None):
    cfg = case.cfg(kvq)
    ml = max(case.lens) if max_len is None else max_len
    out = torch.full((case.B, case.Hq, case.d), float("nan"), dtype=torch.float32, device="cuda")
    ws = kvq.new_fp16_workspace(cfg, case.B, case.Hq, ml, device="cuda")
    kvq.kvq_fp16_decode_attention(cfg, torch.from_numpy(pool16_np).cuda(), case.q.cuda(), case.block_table.cuda(),
                                  torch.tensor(case.lens, dtype=torch.int32, device="cuda"), ml, case.scale, out, ws)
    return out.cpu().numpy(), kvq.kvq_read_status(ws)


def test_fp16_pool_bytes(kvq):
    case = Case(1, 8, 4, 128, [5], seed=1)
    assert kvq.kvq_fp16_pool_bytes(case.cfg(kvq)) == oracle.fp16_pool_bytes(case.layout)


@pytest.mark.parametrize("P", [16, 32, 64])
def test_fp16_append_bitexact(kvq, P):
    case = Case(3, 8, 4, 128, [70, 1, 3 * P + 5], P=P, seed=P)
    ref = _fp16_pool(case)
    got = torch.full((oracle.fp16_pool_bytes(case.layout),), 0xA5, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cfg = case.cfg(kvq)
    bt = case.block_table.cuda()
    for b in range(case.B):
        n = case.lens[b]
        kvq.kvq_fp16_append(cfg, got, case.k[b:b + 1, :n].cuda(), case.v[b:b + 1, :n].cuda(), bt[b:b + 1],
                            torch.zeros(1, dtype=torch.int32, device="cuda"), status=status)
    assert kvq.kvq_read_status(status) == 0
    diff = np.nonzero(got.cpu().numpy() != ref)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"


@pytest.mark.parametrize("Gk,Gv,P", [(64, 128, 16), (32, 32, 16), (128, 64, 32), (32, 128, 64)])
def test_dequantize_to_fp16_pool_bitexact(kvq, Gk, Gv, P):
    case = Case(4, 8, 4, 128, [300, 1, 0, 2 * P + 7], P=P, Gk=Gk, Gv=Gv, seed=Gk + Gv + P)
    L = case.layout
    pool = case.oracle_pool()
    ref = np.full(oracle.fp16_pool_bytes(L), 0x3C, np.uint8)
    oracle.dequantize_to_fp16_pool(L, pool, ref, case.block_table.numpy(), np.array(case.lens, np.int32))
    got = torch.full((ref.size,), 0x3C, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_dequantize_to_fp16_pool(case.cfg(kvq), torch.from_numpy(pool).cuda(), got, case.block_table.cuda(),
                                    torch.tensor(case.lens, dtype=torch.int32, device="cuda"), max(case.lens),
                                    status=status)
    assert kvq.kvq_read_status(status) == 0
    diff = np.nonzero(got.cpu().numpy() != ref)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (32, 8), (16, 8), (16, 2), (24, 4), (6, 6), (8, 1)])
def test_fp16_attention_heads(kvq, Hq, Hkv):
    # 1, 4, 2, 8, 6, 1 and 8 query heads per kv head
    case = Case(3, Hq, Hkv, 128, [300, 129, 17], seed=Hq * 3 + Hkv)
    ref_pool = _fp16_pool(case)
    ref = oracle.fp16_decode_attention(case.layout, ref_pool, case.q.numpy(), case.block_table.numpy(),
                                       np.array(case.lens, np.int32), case.scale)
    got, flags = _gpu_fp16_attention(kvq, case, ref_pool)
    assert flags == 0
    assert_attention_close(got, ref, what=f"fp16 Hq{Hq} Hkv{Hkv}")


@pytest.mark.parametrize("P", [16, 32, 64])
def test_fp16_attention_page_sizes_and_edges(kvq, P):
    case = Case(9, 8, 4, 128, [0, 1, 15, 16, 17, P, P + 1, 3 * P - 1, 200], P=P, seed=P + 7)
    ref_pool = _fp16_pool(case)
    ref = oracle.fp16_decode_attention(case.layout, ref_pool, case.q.numpy(), case.block_table.numpy(),
                                       np.array(case.lens, np.int32), case.scale)
    got, flags = _gpu_fp16_attention(kvq, case, ref_pool, max_len=1000)
    assert flags == 0
    assert_attention_close(got, ref, what=f"fp16 P{P}")
    assert np.all(got[0] == 0)


def test_fp16_attention_long_and_ragged(kvq):
    for case in (Case(1, 32, 8, 128, [6000], seed=81), Case(1, 32, 32, 128, [5000], seed=82),
                 Case(33, 8, 2, 128, np.random.default_rng(83).integers(1, 700, size=33).tolist(), seed=83)):
        ref_pool = _fp16_pool(case)
        ref = oracle.fp16_decode_attention(case.layout, ref_pool, case.q.numpy(), case.block_table.numpy(),
                                           np.array(case.lens, np.int32), case.scale)
        got, flags = _gpu_fp16_attention(kvq, case, ref_pool)
        assert flags == 0
        assert_attention_close(got, ref, what=f"fp16 B{case.B}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (32, 8)])
def test_dequantize_then_attend(kvq, Hq, Hkv):
    # the comparison's middle arm: INT4 pool -> FP16 pool (device) -> FP16 attention
    case = Case(3, Hq, Hkv, 128, [513, 64, 200], seed=Hq + 90)
    L = case.layout
    cfg = case.cfg(kvq)
    pool = case.oracle_pool()
    ref16 = np.zeros(oracle.fp16_pool_bytes(L), np.uint8)
    oracle.dequantize_to_fp16_pool(L, pool, ref16, case.block_table.numpy(), np.array(case.lens, np.int32))
    ref = oracle.fp16_decode_attention(L, ref16, case.q.numpy(), case.block_table.numpy(),
                                       np.array(case.lens, np.int32), case.scale)
    pool16 = torch.zeros(ref16.size, dtype=torch.uint8, device="cuda")
    sl = torch.tensor(case.lens, dtype=torch.int32, device="cuda")
    bt = case.block_table.cuda()
    kvq.kvq_dequantize_to_fp16_pool(cfg, torch.from_numpy(pool).cuda(), pool16, bt, sl, max(case.lens))
    out = torch.empty((case.B, Hq, 128), dtype=torch.float32, device="cuda")
    ws = kvq.new_fp16_workspace(cfg, case.B, Hq, max(case.lens), device="cuda")
    kvq.kvq_fp16_decode_attention(cfg, pool16, case.q.cuda(), bt, sl, max(case.lens), case.scale, out, ws)
    assert kvq.kvq_read_status(ws) == 0
    assert_attention_close(out.cpu().numpy(), ref, what="dequantize then attend")


def test_fp16_many_one_page_segments_per_cta(kvq):
    # the FP16 kernel's q barriers: thousands of one-page sequences, most warps without a unit
    # in a given segment (they must not run two segments ahead)
    rng = np.random.default_rng(27)
    case = Case(2100, 32, 16, 128, rng.integers(0, 7, size=2100).tolist(), seed=27, device="cuda")
    pool16 = _fp16_pool(case)
    got, flags = _gpu_fp16_attention(kvq, case, pool16)
    assert flags == 0
    ref = oracle.fp16_decode_attention(case.layout, pool16, case.q.numpy(), case.block_table.numpy(),
                                       np.array(case.lens, np.int32), case.scale)
    assert_attention_close(got, ref, what="fp16 B2100")

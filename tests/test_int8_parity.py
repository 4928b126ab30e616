"""The INT8 per-row cache ("AI inference tuning: KV Cache optimisation and memory management"
section 3.1, KVCacheQuantizer.quantize_int8) against the oracle:
  - kvq_int8_quantize_append: the whole pool bit for bit (codes and fp32 scales), with
    the same fill byte on both sides;
  - kvq_int8_decode_attention: within the tolerances of tests/kvq_testlib.py against the
    oracle's fp64 attention over the same pool."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from conftest import cuda_available
from kvq_testlib import Case, assert_attention_close

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


def _int8_pool(case: Case, fill=0x5C):
    L = case.layout
    pool8 = np.full(oracle.int8_pool_bytes(L), fill, np.uint8)
    bt = case.block_table.numpy()
    for b in range(case.B):
        n = case.lens[b]
        if n:
            oracle.int8_quantize_append(L, pool8, case.k[b:b + 1, :n].numpy(), case.v[b:b + 1, :n].numpy(),
                                        bt[b:b + 1], np.zeros(1, np.int32))
    return pool8


def test_int8_pool_bytes(kvq):
    case = Case(1, 8, 4, 128, [5], seed=1)
    assert kvq.kvq_int8_pool_bytes(case.cfg(kvq)) == oracle.int8_pool_bytes(case.layout)


@pytest.mark.parametrize("P", [16, 32, 64])
@pytest.mark.parametrize("outliers", [True, False])
def test_int8_quantize_append_bitexact(kvq, P, outliers):
    case = Case(3, 8, 4, 128, [70, 1, 3 * P + 5], P=P, seed=P + outliers, outliers=outliers)
    ref = _int8_pool(case)
    got = torch.full((ref.size,), 0x5C, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cfg = case.cfg(kvq)
    bt = case.block_table.cuda()
    for b in range(case.B):
        n = case.lens[b]
        kvq.kvq_int8_quantize_append(cfg, got, case.k[b:b + 1, :n].cuda(), case.v[b:b + 1, :n].cuda(), bt[b:b + 1],
                                     torch.zeros(1, dtype=torch.int32, device="cuda"), status=status)
    assert kvq.kvq_read_status(status) == 0
    diff = np.nonzero(got.cpu().numpy() != ref)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"


def test_int8_quantize_special_rows_bitexact(kvq):
    # all-zero rows (floor scale), rows with amax 127 (scale 1) and exact ties, huge and tiny rows
    L = oracle.Layout(2, 128, 16, 64, 128, 4)
    rows = np.zeros((1, 6, 2, 128), np.float16)
    rows[0, 1, :, :8] = [127, -127, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5]
    rows[0, 2] = 60000.0 * np.sin(np.arange(128))[None, :]
    rows[0, 3] = np.float16(2.0 ** -24) * np.arange(-64, 64)[None, :]
    rows[0, 4, :, 5] = -1e-3
    rows[0, 5] = W.kv_tensor(7, (1, 1, 2, 128)).numpy()[0, 0]
    bt = np.array([[2]], np.int32)
    ref = np.zeros(oracle.int8_pool_bytes(L), np.uint8)
    oracle.int8_quantize_append(L, ref, rows, rows[:, ::-1].copy(), bt, np.zeros(1, np.int32))
    cfg = kvq.config(2, 128, 16, 64, 128, 4)
    got = torch.zeros(ref.size, dtype=torch.uint8, device="cuda")
    kvq.kvq_int8_quantize_append(cfg, got, torch.from_numpy(rows).cuda(), torch.from_numpy(rows[:, ::-1].copy()).cuda(),
                                 torch.from_numpy(bt).cuda(), torch.zeros(1, dtype=torch.int32, device="cuda"))
    assert np.array_equal(got.cpu().numpy(), ref)


def _check_attention(kvq, case: Case, max_len=None):
    pool8 = _int8_pool(case)
    ref = oracle.int8_decode_attention(case.layout, pool8, case.q.numpy(), case.block_table.numpy(),
                                       np.array(case.lens, np.int32), case.scale)
    cfg = case.cfg(kvq)
    ml = max(case.lens) if max_len is None else max_len
    ws = torch.zeros(kvq.kvq_int8_decode_workspace_bytes(cfg, case.B, case.Hq, ml), dtype=torch.uint8, device="cuda")
    out = torch.full((case.B, case.Hq, case.d), float("nan"), dtype=torch.float32, device="cuda")
    kvq.kvq_int8_decode_attention(cfg, torch.from_numpy(pool8).cuda(), case.q.cuda(), case.block_table.cuda(),
                                  torch.tensor(case.lens, dtype=torch.int32, device="cuda"), ml, case.scale, out, ws)
    assert kvq.kvq_read_status(ws) == 0
    assert_attention_close(out.cpu().numpy(), ref, what=f"int8 B{case.B} Hq{case.Hq} Hkv{case.Hkv} P{case.P}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (32, 8), (16, 8), (16, 2), (24, 4), (6, 6)])
def test_int8_attention_heads(kvq, Hq, Hkv):
    _check_attention(kvq, Case(3, Hq, Hkv, 128, [300, 129, 17], seed=Hq * 5 + Hkv))


@pytest.mark.parametrize("P", [16, 32, 64])
def test_int8_attention_page_sizes_and_edges(kvq, P):
    _check_attention(kvq, Case(9, 8, 4, 128, [0, 1, 15, 16, 17, P, P + 1, 3 * P - 1, 200], P=P, seed=P + 9),
                     max_len=1000)


def test_int8_attention_long_and_ragged(kvq):
    _check_attention(kvq, Case(1, 32, 8, 128, [6000], seed=121))
    _check_attention(kvq, Case(33, 8, 2, 128, np.random.default_rng(122).integers(1, 700, size=33).tolist(),
                               seed=122))


@pytest.mark.parametrize("P", [32, 64])
def test_int8_attention_eight_heads_per_kv_head_large_pages(kvq, P):
    # two query-head slots per thread (8 query heads per kv head) on pages taken two 16-token chunks at a time
    _check_attention(kvq, Case(3, 16, 2, 128, [5 * P + 3, 1, 2 * P], P=P, seed=P + 123))


def test_int8_attention_batch_over_the_local_prefix_limit(kvq):
    # more than 256 sequences: the combine reads the pages prefix the decode grid publishes
    lens = np.random.default_rng(124).integers(0, 90, size=300).tolist()
    _check_attention(kvq, Case(300, 8, 8, 128, lens, seed=124), max_len=128)


def test_int8_attention_extreme_codes(kvq):
    # K rows whose first 64 codes are all +-127 (the ends of the score's offset-corrected
    # range, codes + 128 as subnormals), a zero V row (floor scale) and a V row of one
    # large value
    case = Case(2, 8, 4, 128, [70, 33], seed=125)
    case.k[:, :, :, :64] = torch.where(case.k[:, :, :, :64] > 0, 100.0, -100.0).half()
    case.v[:, 5] = 0
    case.v[:, 6, :, 3] = -7.0
    _check_attention(kvq, case)

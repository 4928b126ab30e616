"""Slots past a sequence's end (in its last page) and pages the block table lists but no
position reaches may hold any bytes: a freshly allocated pool is not cleared.  Every
decode kernel must ignore them.  Here every cache starts filled with 0xFF, which reads
as NaN in fp16 and fp32 (scales, sigmas, FP16 rows), and the attention must match the
oracle's, which reads only the attended positions.  Lengths are chosen so that most
sequences end inside a page and inside a 16-token step."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from conftest import cuda_available
from kvq_testlib import Case, assert_attention_close, gpu_decode

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]

FILL = 0xFF
LENS = [37, 5, 16, 1, 100, 63]


def _rows_pool(case: Case, size: int, append) -> np.ndarray:
    pool = np.full(size, FILL, np.uint8)
    bt = case.block_table.numpy()
    for b, n in enumerate(case.lens):
        if n:
            append(case.layout, pool, case.k[b:b + 1, :n].numpy(), case.v[b:b + 1, :n].numpy(), bt[b:b + 1],
                   np.zeros(1, np.int32))
    return pool


def _run_rows(kvq, case, pool, ws_bytes_fn, attend_fn):
    cfg = case.cfg(kvq)
    ml = max(case.lens)
    ws = torch.zeros(ws_bytes_fn(cfg, case.B, case.Hq, ml), dtype=torch.uint8, device="cuda")
    out = torch.full((case.B, case.Hq, case.d), float("nan"), dtype=torch.float32, device="cuda")
    attend_fn(cfg, torch.from_numpy(pool).cuda(), case.q.cuda(), case.block_table.cuda(),
              torch.tensor(case.lens, dtype=torch.int32, device="cuda"), ml, case.scale, out, ws)
    assert kvq.kvq_read_status(ws) == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("P", [16, 32])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 4)])
def test_int4_ignores_unwritten_slots(kvq, P, Hq, Hkv):
    case = Case(len(LENS), Hq, Hkv, 128, LENS, P=P, seed=61 + P + Hq)
    pool = case.oracle_pool(fill=FILL)
    got, flags = gpu_decode(kvq, case, torch.from_numpy(pool).cuda())
    assert flags == 0
    assert_attention_close(got, case.oracle_attention(pool), what=f"int4 0xFF fill P{P}")


@pytest.mark.parametrize("P", [16, 32])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 4)])
def test_fp16_ignores_unwritten_slots(kvq, P, Hq, Hkv):
    case = Case(len(LENS), Hq, Hkv, 128, LENS, P=P, seed=71 + P + Hq)
    pool = _rows_pool(case, oracle.fp16_pool_bytes(case.layout), oracle.fp16_append)
    got = _run_rows(kvq, case, pool, kvq.kvq_fp16_decode_workspace_bytes, kvq.kvq_fp16_decode_attention)
    ref = oracle.fp16_decode_attention(case.layout, pool, case.q.numpy(), case.block_table.numpy(),
                                       np.array(case.lens, np.int32), case.scale)
    assert_attention_close(got, ref, what=f"fp16 0xFF fill P{P}")


@pytest.mark.parametrize("P", [16, 32])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 4)])
def test_int8_ignores_unwritten_slots(kvq, P, Hq, Hkv):
    case = Case(len(LENS), Hq, Hkv, 128, LENS, P=P, seed=81 + P + Hq)
    pool = _rows_pool(case, oracle.int8_pool_bytes(case.layout), oracle.int8_quantize_append)
    got = _run_rows(kvq, case, pool, kvq.kvq_int8_decode_workspace_bytes, kvq.kvq_int8_decode_attention)
    ref = oracle.int8_decode_attention(case.layout, pool, case.q.numpy(), case.block_table.numpy(),
                                       np.array(case.lens, np.int32), case.scale)
    assert_attention_close(got, ref, what=f"int8 0xFF fill P{P}")


@pytest.mark.parametrize("P", [16, 32])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 4)])
def test_wht4_ignores_unwritten_slots(kvq, P, Hq, Hkv):
    case = Case(len(LENS), Hq, Hkv, 128, LENS, P=P, seed=91 + P + Hq)
    pool = _rows_pool(case, oracle.wht4_pool_bytes(case.layout), oracle.wht4_quantize_append)
    got = _run_rows(kvq, case, pool, kvq.kvq_wht4_decode_workspace_bytes, kvq.kvq_wht4_decode_attention)
    ref = oracle.wht4_decode_attention(case.layout, pool, case.q.numpy(), case.block_table.numpy(),
                                       np.array(case.lens, np.int32), case.scale)
    assert_attention_close(got, ref, what=f"wht4 0xFF fill P{P}")

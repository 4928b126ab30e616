"""Mixed-precision decode attention (kvq_mixed_decode_attention): positions older than the
last `residual` from the INT4 pool, the last `residual` from an FP16 pool with its own
block table ("LLM long-context inference: managing the KV cache with an INT4 state
machine" section 8.3), against the oracle's mixed attention, within the tolerances of
tests/kvq_testlib.py."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from conftest import cuda_available
from kvq_testlib import Case, assert_attention_close, gpu_decode

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


def _fp16_side(case: Case, seed: int, only_recent: int | None = None):
    """FP16 pool (own pages, own block table) holding each sequence's rows; with only_recent,
    the table keeps entries only for the pages of the last only_recent positions."""
    P = case.P
    pages = [(n + P - 1) // P for n in case.lens]
    n16 = sum(pages) + 2
    L16 = oracle.Layout(case.Hkv, case.d, P, case.Gk, case.Gv, n16)
    order = W.permutation(seed, n16).numpy()
    bt16 = np.full((case.B, case.block_table.shape[1]), -1, np.int32)
    kk = 0
    for b, n in enumerate(pages):
        bt16[b, :n] = order[kk:kk + n]
        kk += n
    pool16 = np.zeros(oracle.fp16_pool_bytes(L16), np.uint8)
    for b, n in enumerate(case.lens):
        if n:
            oracle.fp16_append(L16, pool16, case.k[b:b + 1, :n].numpy(), case.v[b:b + 1, :n].numpy(), bt16[b:b + 1],
                               np.zeros(1, np.int32))
    if only_recent is not None:
        for b, n in enumerate(case.lens):
            first = max(n - only_recent, 0) // P
            bt16[b, :first] = -1
    return pool16, bt16, n16


def _run(kvq, case: Case, residual: int, seed: int = 5, only_recent: bool = False, max_len=None):
    pool = case.oracle_pool(fill=0xC3)
    pool16, bt16, n16 = _fp16_side(case, seed, residual if only_recent else None)
    sl = np.array(case.lens, np.int32)
    ref = oracle.mixed_decode_attention(case.layout, pool, case.block_table.numpy(), pool16, bt16, n16,
                                        case.q.numpy(), sl, residual, case.scale)
    cfg = case.cfg(kvq)
    ml = max(case.lens) if max_len is None else max_len
    ws = torch.zeros(kvq.kvq_mixed_decode_workspace_bytes(cfg, case.B, case.Hq, ml, residual), dtype=torch.uint8,
                     device="cuda")
    out = torch.full((case.B, case.Hq, case.d), float("nan"), dtype=torch.float32, device="cuda")
    kvq.kvq_mixed_decode_attention(cfg, torch.from_numpy(pool).cuda(), case.block_table.cuda(),
                                   torch.from_numpy(pool16).cuda(), torch.from_numpy(bt16).cuda(), n16, case.q.cuda(),
                                   torch.from_numpy(sl).cuda(), ml, residual, case.scale, out, ws)
    assert kvq.kvq_read_status(ws) == 0
    got = out.cpu().numpy()
    assert_attention_close(got, ref, what=f"mixed residual {residual} B{case.B} Hq{case.Hq} Hkv{case.Hkv} P{case.P}")
    return got, pool


@pytest.mark.parametrize("residual", [1, 16, 17, 100, 300, 1000])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (32, 8), (16, 2), (6, 6)])
def test_mixed_heads_and_residuals(kvq, residual, Hq, Hkv):
    _run(kvq, Case(3, Hq, Hkv, 128, [300, 129, 17], seed=residual + Hq), residual)


@pytest.mark.parametrize("P", [16, 32, 64])
def test_mixed_page_sizes(kvq, P):
    _run(kvq, Case(4, 8, 4, 128, [0, 1, 3 * P + 5, 200], P=P, seed=P + 3), 40)


def test_mixed_fp16_table_holds_only_recent_pages(kvq):
    _run(kvq, Case(3, 16, 4, 128, [500, 64, 33], seed=11), 64, only_recent=True)


def test_mixed_long_and_ragged(kvq):
    _run(kvq, Case(1, 32, 8, 128, [6000], seed=12), 128)
    rng = np.random.default_rng(13)
    _run(kvq, Case(33, 8, 2, 128, rng.integers(0, 700, size=33).tolist(), seed=13), 64, max_len=1000)


def test_mixed_residual_zero_is_plain_int4(kvq):
    case = Case(3, 8, 8, 128, [300, 129, 17], seed=14)
    got, pool = _run(kvq, case, 0)
    plain, _ = gpu_decode(kvq, case, torch.from_numpy(pool).cuda())
    assert np.array_equal(got, plain)

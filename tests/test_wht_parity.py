"""The rotated 4-bit cache ("LARQL KV cache engines", engine three codec/turbo-quant:
Walsh-Hadamard rotation and a Lloyd-Max codebook) against the oracle:
  - kvq_wht4_quantize_append: the whole pool bit for bit (codes and fp32 sigmas), with
    the same fill byte on both sides, over page sizes, outlier channels and special rows
    (zero rows, rows whose rotated values sit exactly on the middle threshold, huge and
    subnormal values);
  - kvq_wht4_dequantize: within fp32 rounding of the oracle's fp64 rotation;
  - kvq_wht4_decode_attention: within the tolerances of tests/kvq_testlib.py against the
    oracle's fp64 attention over the dequantized rows."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from conftest import cuda_available
from kvq_testlib import Case, assert_attention_close

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


def _pool(case: Case, fill=0xA7):
    L = case.layout
    pool = np.full(oracle.wht4_pool_bytes(L), fill, np.uint8)
    bt = case.block_table.numpy()
    for b in range(case.B):
        n = case.lens[b]
        if n:
            oracle.wht4_quantize_append(L, pool, case.k[b:b + 1, :n].numpy(), case.v[b:b + 1, :n].numpy(),
                                        bt[b:b + 1], np.zeros(1, np.int32))
    return pool


def test_wht4_pool_bytes(kvq):
    case = Case(1, 8, 4, 128, [5], seed=1)
    assert kvq.kvq_wht4_pool_bytes(case.cfg(kvq)) == oracle.wht4_pool_bytes(case.layout)


@pytest.mark.parametrize("P", [16, 32, 64])
@pytest.mark.parametrize("outliers", [True, False])
def test_wht4_quantize_append_bitexact(kvq, P, outliers):
    case = Case(3, 8, 4, 128, [70, 1, 3 * P + 5], P=P, seed=P + outliers, outliers=outliers)
    ref = _pool(case)
    got = torch.full((ref.size,), 0xA7, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cfg = case.cfg(kvq)
    bt = case.block_table.cuda()
    for b in range(case.B):
        n = case.lens[b]
        kvq.kvq_wht4_quantize_append(cfg, got, case.k[b:b + 1, :n].cuda(), case.v[b:b + 1, :n].cuda(), bt[b:b + 1],
                                     torch.zeros(1, dtype=torch.int32, device="cuda"), status=status)
    assert kvq.kvq_read_status(status) == 0
    diff = np.nonzero(got.cpu().numpy() != ref)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"


def test_wht4_quantize_special_rows_bitexact(kvq):
    L = oracle.Layout(2, 128, 16, 64, 128, 4)
    rows = np.zeros((1, 8, 2, 128), np.float16)
    rows[0, 1, :, :2] = 1.0                                          # rotated values 2 and exactly 0
    rows[0, 2] = np.float16(60000.0) * np.sin(np.arange(128))[None, :]
    rows[0, 3] = np.float16(2.0 ** -24) * np.arange(-64, 64)[None, :]  # fp16 subnormals
    rows[0, 4, :, ::2] = 3.0                                         # many rotated values exactly 0
    rows[0, 5] = np.arange(128)[None, :] % 7 - 3
    rows[0, 6] = W.kv_tensor(7, (1, 1, 2, 128)).numpy()[0, 0]
    rows[0, 7, :, 5] = -1e-3
    bt = np.array([[2]], np.int32)
    ref = np.zeros(oracle.wht4_pool_bytes(L), np.uint8)
    oracle.wht4_quantize_append(L, ref, rows, rows[:, ::-1].copy(), bt, np.zeros(1, np.int32))
    cfg = kvq.config(2, 128, 16, 64, 128, 4)
    got = torch.zeros(ref.size, dtype=torch.uint8, device="cuda")
    kvq.kvq_wht4_quantize_append(cfg, got, torch.from_numpy(rows).cuda(), torch.from_numpy(rows[:, ::-1].copy()).cuda(),
                                 torch.from_numpy(bt).cuda(), torch.zeros(1, dtype=torch.int32, device="cuda"))
    assert np.array_equal(got.cpu().numpy(), ref)


def test_wht4_dequantize_matches_oracle(kvq):
    case = Case(2, 8, 4, 128, [45, 20], seed=31)
    pool = _pool(case)
    cfg = case.cfg(kvq)
    dp = torch.from_numpy(pool).cuda()
    bt = case.block_table.cuda()
    for b, n in enumerate(case.lens):
        ok = torch.full((n, 4, 128), float("nan"), dtype=torch.float32, device="cuda")
        ov = torch.full((n, 4, 128), float("nan"), dtype=torch.float32, device="cuda")
        kvq.kvq_wht4_dequantize(cfg, dp, bt, b, 0, n, ok, ov)
        rk, rv = oracle.wht4_dequantize(case.layout, pool, case.block_table.numpy(), b, 0, n)
        for got, ref in ((ok.cpu().numpy(), rk), (ov.cpu().numpy(), rv)):
            scale = np.abs(ref).max(axis=-1, keepdims=True) + 1e-30
            assert np.all(np.abs(got - ref) <= 2e-6 * scale), float(np.max(np.abs(got - ref) / scale))


def _check_attention(kvq, case: Case, max_len=None):
    pool = _pool(case)
    ref = oracle.wht4_decode_attention(case.layout, pool, case.q.numpy(), case.block_table.numpy(),
                                       np.array(case.lens, np.int32), case.scale)
    cfg = case.cfg(kvq)
    ml = max(case.lens) if max_len is None else max_len
    ws = torch.zeros(kvq.kvq_wht4_decode_workspace_bytes(cfg, case.B, case.Hq, ml), dtype=torch.uint8, device="cuda")
    out = torch.full((case.B, case.Hq, case.d), float("nan"), dtype=torch.float32, device="cuda")
    kvq.kvq_wht4_decode_attention(cfg, torch.from_numpy(pool).cuda(), case.q.cuda(), case.block_table.cuda(),
                                  torch.tensor(case.lens, dtype=torch.int32, device="cuda"), ml, case.scale, out, ws)
    assert kvq.kvq_read_status(ws) == 0
    assert_attention_close(out.cpu().numpy(), ref, what=f"wht4 B{case.B} Hq{case.Hq} Hkv{case.Hkv} P{case.P}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (32, 8), (16, 8), (16, 2), (24, 4), (6, 6)])
def test_wht4_attention_heads(kvq, Hq, Hkv):
    _check_attention(kvq, Case(3, Hq, Hkv, 128, [300, 129, 17], seed=Hq * 7 + Hkv))


@pytest.mark.parametrize("P", [16, 32, 64])
def test_wht4_attention_page_sizes_and_edges(kvq, P):
    _check_attention(kvq, Case(9, 8, 4, 128, [0, 1, 15, 16, 17, P, P + 1, 3 * P - 1, 200], P=P, seed=P + 19),
                     max_len=1000)


def test_wht4_attention_long_and_ragged(kvq):
    _check_attention(kvq, Case(1, 32, 8, 128, [6000], seed=131))
    _check_attention(kvq, Case(33, 8, 2, 128, np.random.default_rng(132).integers(1, 700, size=33).tolist(),
                               seed=132))

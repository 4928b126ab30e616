"""Decode attention and the decode step at head_dim 64 and 256 (the INT4 cache), against
the oracle on the same pool bytes, with the tolerances of tests/kvq_testlib.py:
  - attention over every unit shape the planner picks at each head_dim (four kv heads per
    unit at 64, one kv head with 1, 2, 4 or 8 query heads), every supported group-size
    pair, page sizes 16/32/64, ragged and edge lengths, one long sequence over many CTAs;
  - the sliding window with sink tokens;
  - the decode step: the pool after the step bit for bit, the output within tolerance and
    bit for bit equal to the two-call path (quantize-append, then attention);
  - the no-allocation entry point at both head_dims.
Head_dim 256 takes up to 4 query heads per kv head and K groups of 64 or 128; other
shapes are rejected on the host (tests/test_abi_cpu.py)."""
from __future__ import annotations

import ctypes as C

import numpy as np
import pytest
import torch

import oracle
import test_decode_step_parity as step
from conftest import cuda_available
from kvq_testlib import Case, assert_attention_close, gpu_decode

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


def _attend(kvq, case: Case, max_len=None):
    pool_np = case.oracle_pool(fill=0xC3)
    ref = case.oracle_attention(pool_np)
    got, flags = gpu_decode(kvq, case, torch.from_numpy(pool_np).cuda(), max_len=max_len)
    assert flags == 0, f"status flags {flags:#x}"
    return assert_attention_close(got, ref, what=f"d{case.d} B{case.B} Hq{case.Hq} Hkv{case.Hkv} P{case.P} "
                                                 f"G{case.Gk}/{case.Gv} lens{case.lens[:6]}")


# ---- head_dim 64 ----

@pytest.mark.parametrize("Gk,Gv", [(32, 32), (32, 64), (64, 32), (64, 64)])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 4), (16, 2)])
def test_d64_groups_and_units(kvq, Gk, Gv, Hq, Hkv):
    # (8, 8): four kv heads per unit; (16, 4): one, 4 query heads; (16, 2): one, 8 query heads
    _attend(kvq, Case(3, Hq, Hkv, 64, [300, 129, 17], Gk=Gk, Gv=Gv, seed=Gk + 3 * Gv + Hq))


@pytest.mark.parametrize("P", [16, 32, 64])
@pytest.mark.parametrize("Hq,Hkv", [(8, 4), (8, 8)])
def test_d64_page_sizes(kvq, P, Hq, Hkv):
    _attend(kvq, Case(3, Hq, Hkv, 64, [1, P + 1, 5 * P - 3], P=P, Gk=32, Gv=64, seed=P + Hkv))


def test_d64_edge_and_ragged(kvq):
    _attend(kvq, Case(9, 4, 2, 64, [0, 1, 15, 16, 17, 31, 32, 33, 2], Gk=32, Gv=32, seed=3))
    rng = np.random.default_rng(64)
    _attend(kvq, Case(33, 8, 8, 64, rng.integers(1, 700, size=33).tolist(), Gk=64, Gv=64, seed=64))


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 16)])
def test_d64_long_single_sequence(kvq, Hq, Hkv):
    _attend(kvq, Case(1, Hq, Hkv, 64, [6000], Gk=32, Gv=64, seed=60 + Hkv))


# ---- head_dim 256 ----

@pytest.mark.parametrize("Gk,Gv", [(64, 128), (128, 128), (64, 32), (128, 64)])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 4), (8, 4)])
def test_d256_groups_and_ratios(kvq, Gk, Gv, Hq, Hkv):
    _attend(kvq, Case(3, Hq, Hkv, 256, [300, 129, 17], Gk=Gk, Gv=Gv, seed=Gk + 5 * Gv + Hq))


@pytest.mark.parametrize("P", [16, 32, 64])
def test_d256_page_sizes(kvq, P):
    _attend(kvq, Case(3, 8, 2, 256, [1, P + 1, 5 * P - 3], P=P, seed=P + 256))


def test_d256_edge_and_ragged(kvq):
    _attend(kvq, Case(9, 4, 2, 256, [0, 1, 15, 16, 17, 31, 32, 33, 2], seed=5))
    rng = np.random.default_rng(256)
    _attend(kvq, Case(33, 4, 4, 256, rng.integers(1, 700, size=33).tolist(), Gk=128, Gv=32, seed=256))


def test_d256_long_single_sequence(kvq):
    _attend(kvq, Case(1, 16, 4, 256, [6000], seed=266))


# ---- sliding window ----

@pytest.mark.parametrize("d,Hq,Hkv,Gk,Gv", [(64, 8, 8, 32, 64), (64, 16, 2, 64, 32), (256, 16, 4, 64, 128),
                                            (256, 8, 8, 128, 32)])
@pytest.mark.parametrize("window,sinks", [(37, 4), (100, 16), (1, 0)])
def test_window(kvq, d, Hq, Hkv, Gk, Gv, window, sinks):
    case = Case(3, Hq, Hkv, d, [300, 129, 17], Gk=Gk, Gv=Gv, seed=window + sinks + d + Hq)
    pool_np = case.oracle_pool(fill=0xC3)
    ref = oracle.decode_attention_window(case.layout, pool_np, case.q.numpy(), case.block_table.numpy(),
                                         np.array(case.lens, np.int32), case.scale, window, sinks)
    cfg = case.cfg(kvq)
    ml = max(case.lens)
    out = torch.full((case.B, case.Hq, case.d), float("nan"), dtype=torch.float32, device="cuda")
    ws = kvq.new_workspace(cfg, case.B, case.Hq, ml, device="cuda")
    kvq.kvq_decode_attention_window(cfg, torch.from_numpy(pool_np).cuda(), case.q.cuda(), case.block_table.cuda(),
                                    torch.tensor(case.lens, dtype=torch.int32, device="cuda"), ml, case.scale,
                                    window, sinks, out, ws)
    assert kvq.kvq_read_status(ws) == 0
    assert_attention_close(out.cpu().numpy(), ref, what=f"d{d} window {window} sinks {sinks}")


# ---- the decode step (append fused) ----

@pytest.mark.parametrize("d,Hq,Hkv,Gk,Gv,P", [(64, 8, 8, 32, 64, 16), (64, 16, 2, 64, 32, 16), (64, 8, 4, 32, 32, 32),
                                              (256, 8, 8, 64, 128, 16), (256, 16, 4, 128, 32, 16),
                                              (256, 8, 2, 64, 64, 64)])
def test_step(kvq, d, Hq, Hkv, Gk, Gv, P):
    step._run(kvq, Case(4, Hq, Hkv, d, [P * 7 + 3, 1, P, 2 * P + 1], P=P, Gk=Gk, Gv=Gv, seed=d + Hq + P))


@pytest.mark.parametrize("d", [64, 256])
def test_step_append_beyond_attended_pages(kvq, d):
    # appends into pages the attention does not stream (handled by the grid's spare warps)
    case = Case(3, 8, 8 if d == 64 else 4, d, [100, 40, 70], Gk=64, Gv=64, seed=d + 1)
    step._run(kvq, case, append_pos=[99, 39, 69], seq_lens=[50, 0, 69])


# ---- the no-allocation entry point ----

@pytest.mark.parametrize("d,Hq,Hkv", [(64, 8, 8), (256, 16, 4)])
def test_noalloc(kvq, d, Hq, Hkv):
    case = Case(3, Hq, Hkv, d, [517, 1200, 40], Gk=64, Gv=64, seed=d + 7)
    cfg = case.cfg(kvq)
    pool_np = case.oracle_pool()
    pool = torch.from_numpy(pool_np).cuda()
    bt = case.block_table.cuda()
    sl = torch.tensor(case.lens, dtype=torch.int32, device="cuda")
    max_len = max(case.lens)
    q = case.q.cuda()
    out = torch.full((case.B, case.Hq, case.d), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.full((1,), 0x7F, dtype=torch.int32, device="cuda")
    rc = kvq.lib().kvq_decode_attention_noalloc(
        C.byref(cfg), C.c_void_p(pool.data_ptr()), C.c_void_p(q.data_ptr()), C.c_void_p(bt.data_ptr()),
        int(bt.shape[1]), C.c_void_p(sl.data_ptr()), case.B, case.Hq, max_len, C.c_float(case.scale),
        C.c_void_p(out.data_ptr()), C.c_void_p(status.data_ptr()), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == kvq.KVQ_OK, kvq.kvq_last_error()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.decode_attention(case.layout, pool_np, case.q.numpy(), case.block_table.numpy(),
                                  np.array(case.lens, np.int32), case.scale)
    assert_attention_close(out.cpu().numpy(), ref, what=f"noalloc d{d}")

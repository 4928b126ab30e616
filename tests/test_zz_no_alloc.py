"""kvq_decode_attention_noalloc: decode attention for callers that cannot allocate
device memory (a plugin whose host engine owns the allocator, a runtime with a fixed
memory budget, code running on an out-of-memory path).  It keeps its scratch in an
array built into the library instead of taking a workspace.

Checked through the C ABI, on two calls in a row each:
  - against the oracle's attention over the same pool, within the attention tolerance
    the other tests use, for a GQA shape (4 query heads per KV head) and an MHA shape
    (the four-KV-head units);
  - bit for bit against kvq_decode_attention with a caller-provided workspace (the same
    kernels over the same cut of the work);
  - its status word: a first call that reads a bad page id reports KVQ_FLAG_BAD_PAGE,
    and the next call, with the table repaired, reports nothing (each call clears the
    flags of the array it shares with the calls before it).
This file is named to be collected last; it needs no state from earlier tests.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import pytest
import torch

from conftest import cuda_available
from kvq_testlib import Case, assert_attention_close

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


def _noalloc(kvq, cfg, pool, q, bt, sl, max_len, scale, out, status):
    stream = torch.cuda.current_stream().cuda_stream
    return kvq.lib().kvq_decode_attention_noalloc(
        C.byref(cfg), C.c_void_p(pool.data_ptr()), C.c_void_p(q.data_ptr()), C.c_void_p(bt.data_ptr()),
        int(bt.shape[1]), C.c_void_p(sl.data_ptr()), int(q.shape[0]), int(q.shape[1]), int(max_len),
        C.c_float(scale), C.c_void_p(out.data_ptr()), C.c_void_p(status.data_ptr()), C.c_void_p(stream))


def _with_workspace(kvq, cfg, pool, q, bt, sl, max_len, scale):
    out = torch.full((q.shape[0], q.shape[1], q.shape[2]), float("nan"), dtype=torch.float32, device="cuda")
    ws = kvq.new_workspace(cfg, int(q.shape[0]), int(q.shape[1]), max_len)
    kvq.kvq_decode_attention(cfg, pool, q, bt, sl, max_len, scale, out, ws)
    return out


@pytest.mark.parametrize("shape", ["gqa_4_per_kv_head", "mha_four_head_units"])
def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls(kvq, shape):
    if shape == "gqa_4_per_kv_head":
        case = Case(5, 16, 4, 128, [900, 1, 333, 0, 2048], seed=31)
    else:
        case = Case(3, 16, 16, 128, [517, 1200, 40], seed=32)
    cfg = case.cfg(kvq)
    pool_np = case.oracle_pool()
    pool = torch.from_numpy(pool_np).cuda()
    bt = case.block_table.cuda()
    sl = torch.tensor(case.lens, dtype=torch.int32, device="cuda")
    max_len = max(case.lens)
    status = torch.full((1,), 0x7F, dtype=torch.int32, device="cuda")
    for call in range(2):
        # a different query on each call, so the second call cannot pass on leftovers of the first
        q_cpu = (case.q.float() * (1.0 if call == 0 else -0.5)).half()
        q = q_cpu.cuda()
        out = torch.full((case.B, case.Hq, case.d), float("nan"), dtype=torch.float32, device="cuda")
        rc = _noalloc(kvq, cfg, pool, q, bt, sl, max_len, case.scale, out, status)
        assert rc == kvq.KVQ_OK, kvq.kvq_last_error()
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: status flags {int(status.item()):#x}"
        import oracle
        ref = oracle.decode_attention(case.layout, pool_np, q_cpu.numpy(), case.block_table.numpy(),
                                      np.array(case.lens, np.int32), case.scale)
        assert_attention_close(out.cpu().numpy(), ref, what=f"{shape} call {call} vs oracle")
        assert torch.equal(out, _with_workspace(kvq, cfg, pool, q, bt, sl, max_len, case.scale)), \
            f"{shape} call {call}: differs from kvq_decode_attention"


def test_noalloc_status_is_this_calls_own(kvq):
    case = Case(3, 16, 4, 128, [700, 64, 333], seed=33)
    cfg = case.cfg(kvq)
    pool_np = case.oracle_pool()
    pool = torch.from_numpy(pool_np).cuda()
    sl = torch.tensor(case.lens, dtype=torch.int32, device="cuda")
    max_len = max(case.lens)
    q = case.q.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((case.B, case.Hq, case.d), dtype=torch.float32, device="cuda")
    # call 0: one block-table entry points past the pool; the kernel reads page 0 instead
    # and flags it
    bad = case.block_table.clone()
    bad[1, 2] = case.num_pages + 5
    assert _noalloc(kvq, cfg, pool, q, bad.cuda(), sl, max_len, case.scale, out, status) == kvq.KVQ_OK
    torch.cuda.synchronize()
    assert int(status.item()) & kvq.KVQ_FLAG_BAD_PAGE
    # call 1: the table repaired; the flags of call 0 are gone, the output is the oracle's
    bt = case.block_table.cuda()
    assert _noalloc(kvq, cfg, pool, q, bt, sl, max_len, case.scale, out, status) == kvq.KVQ_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    import oracle
    ref = oracle.decode_attention(case.layout, pool_np, case.q.numpy(), case.block_table.numpy(),
                                  np.array(case.lens, np.int32), case.scale)
    assert_attention_close(out.cpu().numpy(), ref, what="after a flagged call")


def test_noalloc_rejects_shapes_beyond_its_scratch(kvq):
    # 8 query heads per KV head over many KV heads needs more than the built-in scratch
    cfg = kvq.config(64, 128, 16, 64, 128, 64)
    need = kvq.kvq_decode_workspace_bytes(cfg, 64, 512, 4096)
    assert need > (8 << 20)
    d = torch.zeros(16, dtype=torch.uint8, device="cuda")
    q = torch.zeros((64, 512, 128), dtype=torch.float16, device="cuda")
    bt = torch.zeros((64, 4), dtype=torch.int32, device="cuda")
    sl = torch.zeros(64, dtype=torch.int32, device="cuda")
    out = torch.zeros((64, 512, 128), dtype=torch.float32, device="cuda")
    rc = _noalloc(kvq, cfg, d, q, bt, sl, 4096, 0.1, out, torch.zeros(1, dtype=torch.int32, device="cuda"))
    assert rc == kvq.KVQ_EWORKSPACE
    assert "scratch" in kvq.kvq_last_error()

"""The decode kernel's bounded waits, made to run out on the GPU without any fault.

kvq_test_decode_wait_timeout runs the decode kernel with a short bound on every wait and
each warp's first page copy announced to its mbarrier as 16 bytes larger than it is: every
copy it issues lands, but that phase cannot complete, so the wait for it must run out.  The
kernel must return (no hang), raise KVQ_FLAG_WAIT_TIMEOUT, and leave the context usable: a
normal call right after it gives the oracle's attention with no flag.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from conftest import cuda_available
from kvq_testlib import Case, assert_attention_close, gpu_decode

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


@pytest.mark.parametrize("shape", ["gqa_one_head_units", "mha_four_head_units"])
def test_wait_runs_out_and_is_flagged(kvq, shape):
    case = Case(2, 16, 4, 128, [300, 77], seed=51) if shape == "gqa_one_head_units" else \
        Case(2, 8, 8, 128, [260, 33], seed=52)
    cfg = case.cfg(kvq)
    pool_np = case.oracle_pool()
    pool = torch.from_numpy(pool_np).cuda()
    ml = max(case.lens)
    ws = kvq.new_workspace(cfg, case.B, case.Hq, ml, device="cuda")
    out = torch.empty((case.B, case.Hq, case.d), dtype=torch.float32, device="cuda")
    kvq.kvq_test_decode_wait_timeout(cfg, pool, case.q.cuda(), case.block_table.cuda(),
                                     torch.tensor(case.lens, dtype=torch.int32, device="cuda"), ml, case.scale, out,
                                     ws, 20_000)
    torch.cuda.synchronize()
    assert kvq.kvq_read_status(ws) & kvq.KVQ_FLAG_WAIT_TIMEOUT
    # the context and the pool are intact: the normal call is correct and unflagged
    got, flags = gpu_decode(kvq, case, pool)
    assert flags == 0
    assert_attention_close(got, case.oracle_attention(pool_np), what=f"{shape} after the timeout")
    assert np.array_equal(pool.cpu().numpy(), pool_np)


def test_wait_limit_outside_its_range_is_rejected(kvq):
    case = Case(1, 8, 8, 128, [40], seed=53)
    cfg = case.cfg(kvq)
    ws = kvq.new_workspace(cfg, 1, 8, 40, device="cuda")
    out = torch.empty((1, 8, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(kvq.KvqError):
        kvq.kvq_test_decode_wait_timeout(cfg, torch.zeros(kvq.kvq_pool_bytes(cfg), dtype=torch.uint8, device="cuda"),
                                         case.q.cuda(), case.block_table.cuda(),
                                         torch.tensor([40], dtype=torch.int32, device="cuda"), 40, case.scale, out, ws,
                                         100)

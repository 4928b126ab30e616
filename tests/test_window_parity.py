"""Decode attention with a sliding window and sink tokens (kvq_decode_attention_window,
kvq_decode_step_window) against the oracle: the query at the last position attends to
positions [max(0, L - window), L) and [0, min(sinks, L)) ("AI inference tuning: KV
Cache optimisation and memory management" section 3.2, SlidingWindowAttention).
Tolerances as in tests/kvq_testlib.py; pools bit for bit."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from conftest import cuda_available
from kvq_testlib import Case, assert_attention_close, gpu_decode

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


def _gpu_window(kvq, case: Case, pool_np, window, sinks, max_len=None):
    cfg = case.cfg(kvq)
    ml = max(case.lens) if max_len is None else max_len
    out = torch.full((case.B, case.Hq, case.d), float("nan"), dtype=torch.float32, device="cuda")
    ws = kvq.new_workspace(cfg, case.B, case.Hq, ml, device="cuda")
    kvq.kvq_decode_attention_window(cfg, torch.from_numpy(pool_np).cuda(), case.q.cuda(), case.block_table.cuda(),
                                    torch.tensor(case.lens, dtype=torch.int32, device="cuda"), ml, case.scale,
                                    window, sinks, out, ws)
    return out.cpu().numpy(), kvq.kvq_read_status(ws)


def _check(kvq, case: Case, window, sinks, max_len=None):
    pool_np = case.oracle_pool(fill=0xC3)
    ref = oracle.decode_attention_window(case.layout, pool_np, case.q.numpy(), case.block_table.numpy(),
                                         np.array(case.lens, np.int32), case.scale, window, sinks)
    got, flags = _gpu_window(kvq, case, pool_np, window, sinks, max_len)
    assert flags == 0, f"status flags {flags:#x}"
    assert_attention_close(got, ref, what=f"window {window} sinks {sinks} B{case.B} Hq{case.Hq} Hkv{case.Hkv} P{case.P}")
    return got


WS = [(1, 0), (16, 0), (37, 4), (100, 16), (64, 200), (5, 3), (129, 1)]


@pytest.mark.parametrize("window,sinks", WS)
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (32, 8), (16, 2)])
def test_window_heads(kvq, window, sinks, Hq, Hkv):
    # (8, 8): four kv heads per unit; (32, 8), (16, 2): one kv head per unit, 4 and 8 query heads
    _check(kvq, Case(3, Hq, Hkv, 128, [300, 129, 17], seed=window + 7 * sinks + Hq), window, sinks)


@pytest.mark.parametrize("P", [16, 32, 64])
@pytest.mark.parametrize("window,sinks", [(40, 0), (40, 5), (70, 33), (17, 64)])
def test_window_page_sizes(kvq, P, window, sinks):
    # with 64-token pages a window start of 296 leaves the page's first two 16-token chunks outside
    _check(kvq, Case(3, 8, 4, 128, [336, 1, 5 * P - 3], P=P, seed=P + window + sinks), window, sinks)


@pytest.mark.parametrize("Gk,Gv", [(32, 32), (128, 128), (32, 128)])
def test_window_groups(kvq, Gk, Gv):
    _check(kvq, Case(2, 8, 8, 128, [211, 40], Gk=Gk, Gv=Gv, seed=Gk + Gv), 50, 4)


def test_window_covering_everything_equals_plain_attention(kvq):
    case = Case(4, 16, 4, 128, [700, 1, 333, 0], seed=31)
    pool_np = case.oracle_pool()
    plain, _ = gpu_decode(kvq, case, torch.from_numpy(pool_np).cuda())
    for window, sinks in [(0, 0), (0, 9), (700, 3), (5000, 0)]:
        got, flags = _gpu_window(kvq, case, pool_np, window, sinks)
        assert flags == 0
        assert np.array_equal(got, plain), (window, sinks)


def test_window_long_sequence_many_ctas(kvq):
    _check(kvq, Case(1, 32, 8, 128, [6000], seed=32), 1000, 4)
    _check(kvq, Case(1, 32, 32, 128, [6000], seed=33), 2500, 0)


def test_window_ragged_with_empty_and_short(kvq):
    rng = np.random.default_rng(34)
    lens = rng.integers(0, 500, size=40).tolist()
    lens[:4] = [0, 1, 2, 3]
    _check(kvq, Case(40, 8, 2, 128, lens, seed=34), 64, 4)


def test_window_generous_max_len(kvq):
    _check(kvq, Case(3, 8, 8, 128, [100, 7, 64], seed=35), 20, 2, max_len=4000)


def test_window_bad_arguments_rejected(kvq):
    case = Case(1, 8, 8, 128, [20], seed=36)
    pool_np = case.oracle_pool()
    with pytest.raises(kvq.KvqError):
        _gpu_window(kvq, case, pool_np, -1, 0)
    with pytest.raises(kvq.KvqError):
        _gpu_window(kvq, case, pool_np, 8, -2)


# ---- the decode step with a window: append, then windowed attention ----

@pytest.mark.parametrize("Hq,Hkv,P", [(8, 8, 16), (32, 8, 16), (8, 4, 64)])
@pytest.mark.parametrize("window,sinks", [(33, 4), (1, 0), (256, 16)])
def test_window_step_matches_oracle_and_two_calls(kvq, Hq, Hkv, P, window, sinks):
    case = Case(3, Hq, Hkv, 128, [300, 129, 17], P=P, seed=Hq + P + window)
    L = case.layout
    cfg = case.cfg(kvq)
    bt = case.block_table.numpy()
    ap = [n - 1 for n in case.lens]
    pool = np.full(L.pool_bytes, 0x5A, np.uint8)
    for b in range(case.B):
        if ap[b] > 0:
            oracle.quantize_append(L, pool, case.k[b:b + 1, :ap[b]].numpy(), case.v[b:b + 1, :ap[b]].numpy(),
                                   bt[b:b + 1], np.zeros(1, np.int32))
    k_new = np.stack([case.k[b, ap[b]].numpy() for b in range(case.B)]).astype(np.float16)
    v_new = np.stack([case.v[b, ap[b]].numpy() for b in range(case.B)]).astype(np.float16)
    ref_pool = pool.copy()
    for b in range(case.B):
        oracle.quantize_append(L, ref_pool, k_new[b:b + 1, None], v_new[b:b + 1, None], bt[b:b + 1],
                               np.array([ap[b]], np.int32))
    ref = oracle.decode_attention_window(L, ref_pool, case.q.numpy(), bt, np.array(case.lens, np.int32), case.scale,
                                         window, sinks)
    outs, pools = [], []
    for two_calls in (False, True):
        pool_g = torch.from_numpy(pool.copy()).cuda()
        out = torch.full((case.B, case.Hq, case.d), float("nan"), dtype=torch.float32, device="cuda")
        ws = kvq.new_workspace(cfg, case.B, case.Hq, max(case.lens), device="cuda")
        apg = torch.tensor(ap, dtype=torch.int32, device="cuda")
        sl = torch.tensor(case.lens, dtype=torch.int32, device="cuda")
        kg, vg = torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda()
        if two_calls:
            kvq.kvq_quantize_append(cfg, pool_g, kg[:, None], vg[:, None], case.block_table.cuda(), apg)
            kvq.kvq_decode_attention_window(cfg, pool_g, case.q.cuda(), case.block_table.cuda(), sl, max(case.lens),
                                            case.scale, window, sinks, out, ws)
        else:
            kvq.kvq_decode_step_window(cfg, pool_g, kg, vg, apg, case.q.cuda(), case.block_table.cuda(), sl,
                                       max(case.lens), case.scale, window, sinks, out, ws)
        assert kvq.kvq_read_status(ws) == 0
        outs.append(out.cpu().numpy())
        pools.append(pool_g.cpu().numpy())
    diff = np.nonzero(pools[0] != ref_pool)[0]
    assert diff.size == 0, f"{diff.size} pool bytes differ from the oracle"
    assert_attention_close(outs[0], ref, what=f"window step {window}/{sinks}")
    assert np.array_equal(pools[0], pools[1]) and np.array_equal(outs[0], outs[1])


def test_window_step_through_paged_cache(kvq):
    from int4_group_quantized_kvq_gb300.cache import PagedKVCache
    case = Case(2, 8, 8, 128, [90, 41], seed=37)
    pool_np = case.oracle_pool()
    c = PagedKVCache(case.cfg(kvq), case.block_table, case.Hq, max(case.lens), pool=torch.from_numpy(pool_np).cuda(),
                     window=30, sinks=2)
    out = torch.empty((case.B, case.Hq, case.d), dtype=torch.float32, device="cuda")
    c.attend(case.q.cuda(), torch.tensor(case.lens, dtype=torch.int32, device="cuda"), out)
    ref = oracle.decode_attention_window(case.layout, pool_np, case.q.numpy(), case.block_table.numpy(),
                                         np.array(case.lens, np.int32), case.scale, 30, 2)
    assert_attention_close(out.cpu().numpy(), ref, what="PagedKVCache window")

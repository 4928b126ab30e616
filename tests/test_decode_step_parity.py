"""The decode step in one launch (kvq_decode_step): append one token per sequence, then
attend.  Checked against the oracle on the same bytes:
  - the whole pool after the step is bit-exact with the oracle's quantize-append of the
    new tokens (same fill byte everywhere else, so a stray write shows up);
  - the attention output is within the tolerances of tests/kvq_testlib.py, against the
    oracle's fp64 attention over the updated pool;
  - the step equals the two-call path (kvq_quantize_append, then kvq_decode_attention)
    bit for bit, pool and output.
Cases cover four-head and one-head units, 8 query heads per kv head, page sizes 16/32/64,
every group size pair, ragged batches, one long sequence over many CTAs, appends into a
page the attention does not reach, sequences without an append, bad positions, and a bad
page id in the page taking the new token."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from conftest import cuda_available
from kvq_testlib import Case, assert_attention_close

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


def _setup(case: Case, append_pos, fill):
    """Oracle pool with each sequence's history below its append position (or its whole length
    when it appends nothing), and the new rows k_new / v_new [B, Hkv, d]."""
    L = case.layout
    pool = np.full(L.pool_bytes, fill, np.uint8)
    bt = case.block_table.numpy()
    hist = [ap if ap >= 0 else n for ap, n in zip(append_pos, case.lens)]
    for b in range(case.B):
        n = min(hist[b], case.k.shape[1])
        if n > 0:
            oracle.quantize_append(L, pool, case.k[b:b + 1, :n].numpy(), case.v[b:b + 1, :n].numpy(), bt[b:b + 1],
                                   np.zeros(1, np.int32))
    src = [min(max(ap, 0), case.k.shape[1] - 1) for ap in append_pos]
    k_new = np.stack([case.k[b, src[b]].numpy() for b in range(case.B)]).astype(np.float16)
    v_new = np.stack([case.v[b, src[b]].numpy() for b in range(case.B)]).astype(np.float16)
    return pool, k_new, v_new


def _oracle_step(case: Case, pool, k_new, v_new, append_pos, seq_lens):
    L = case.layout
    ref = pool.copy()
    bt = case.block_table.numpy()
    max_pos = bt.shape[1] * case.P
    for b in range(case.B):
        ap = append_pos[b]
        if 0 <= ap < max_pos and 0 <= bt[b, ap // case.P] < case.num_pages:
            oracle.quantize_append(L, ref, k_new[b:b + 1, None], v_new[b:b + 1, None], bt[b:b + 1],
                                   np.array([ap], np.int32))
    out = oracle.decode_attention(L, ref, case.q.numpy(), bt, np.array(seq_lens, np.int32), case.scale)
    return ref, out


def _gpu_step(kvq, case: Case, pool, k_new, v_new, append_pos, seq_lens, two_calls=False):
    cfg = case.cfg(kvq)
    pool_g = torch.from_numpy(pool.copy()).cuda()
    kg = torch.from_numpy(k_new).cuda()
    vg = torch.from_numpy(v_new).cuda()
    ap = torch.tensor(append_pos, dtype=torch.int32, device="cuda")
    q = case.q.cuda()
    bt = case.block_table.cuda()
    sl = torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    ml = max(max(seq_lens), 1)
    out = torch.full((case.B, case.Hq, case.d), float("nan"), dtype=torch.float32, device="cuda")
    ws = kvq.new_workspace(cfg, case.B, case.Hq, ml, device="cuda")
    if two_calls:
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        kvq.kvq_quantize_append(cfg, pool_g, kg[:, None], vg[:, None], bt, ap, status=status)
        kvq.kvq_decode_attention(cfg, pool_g, q, bt, sl, ml, case.scale, out, ws)
        flags = kvq.kvq_read_status(ws) | kvq.kvq_read_status(status)
    else:
        kvq.kvq_decode_step(cfg, pool_g, kg, vg, ap, q, bt, sl, ml, case.scale, out, ws)
        flags = kvq.kvq_read_status(ws)
    return pool_g.cpu().numpy(), out.cpu().numpy(), flags


def _run(kvq, case: Case, append_pos=None, seq_lens=None, fill=0xC3, expect_flags=0, compare_two_calls=True):
    append_pos = [n - 1 for n in case.lens] if append_pos is None else list(append_pos)
    seq_lens = list(case.lens) if seq_lens is None else list(seq_lens)
    pool, k_new, v_new = _setup(case, append_pos, fill)
    ref_pool, ref_out = _oracle_step(case, pool, k_new, v_new, append_pos, seq_lens)
    got_pool, got_out, flags = _gpu_step(kvq, case, pool, k_new, v_new, append_pos, seq_lens)
    assert flags == expect_flags, f"status flags {flags:#x}, expected {expect_flags:#x}"
    diff = np.nonzero(got_pool != ref_pool)[0]
    assert diff.size == 0, f"{diff.size} pool bytes differ, first at {diff[:8]}"
    stats = assert_attention_close(got_out, ref_out, what=f"B{case.B} Hq{case.Hq} Hkv{case.Hkv} P{case.P}")
    if compare_two_calls:
        pool2, out2, _ = _gpu_step(kvq, case, pool, k_new, v_new, append_pos, seq_lens, two_calls=True)
        assert np.array_equal(pool2, got_pool), "pool differs from the two-call path"
        assert np.array_equal(out2, got_out), "output differs from the two-call path"
    return stats


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (32, 8), (16, 2), (12, 4), (6, 6)])
def test_step_head_ratios(kvq, Hq, Hkv):
    _run(kvq, Case(3, Hq, Hkv, 128, [300, 129, 17], seed=Hq + 3 * Hkv))


@pytest.mark.parametrize("P", [16, 32, 64])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 4)])
def test_step_page_sizes(kvq, P, Hq, Hkv):
    _run(kvq, Case(3, Hq, Hkv, 128, [1, P + 1, 5 * P - 3], P=P, seed=P + Hkv))


@pytest.mark.parametrize("Gk,Gv", [(64, 128), (32, 32), (128, 128), (32, 128), (128, 32)])
def test_step_groups(kvq, Gk, Gv):
    _run(kvq, Case(2, 8, 8, 128, [211, 40], Gk=Gk, Gv=Gv, seed=Gk + Gv))


def test_step_ragged_batch(kvq):
    rng = np.random.default_rng(21)
    lens = rng.integers(1, 700, size=33).tolist()
    _run(kvq, Case(33, 8, 2, 128, lens, seed=21))


def test_step_long_single_sequence(kvq):
    _run(kvq, Case(1, 32, 32, 128, [6000], seed=22))


def test_step_append_beyond_attended_pages(kvq):
    # sequence 0 appends at 99 (page 6) but attends 60 positions (pages 0..3): the append is
    # written by the grid, not by the warp streaming the page; sequence 1 is the usual step
    case = Case(2, 8, 8, 128, [100, 50], seed=23)
    _run(kvq, case, append_pos=[99, 49], seq_lens=[60, 50])


def test_step_without_append_and_empty(kvq):
    # sequence 0 appends nothing; sequence 1 has no history and appends its first token;
    # sequence 2 neither appends nor attends (zeros)
    case = Case(3, 8, 4, 128, [40, 1, 5], seed=24)
    _run(kvq, case, append_pos=[-1, 0, -1], seq_lens=[40, 1, 0])


def test_step_bad_position_flagged(kvq):
    case = Case(2, 8, 8, 128, [64, 33], seed=25)
    max_pos = case.block_table.shape[1] * case.P
    # sequence 0 appends past its block table: skipped and flagged; sequence 1 is normal
    _run(kvq, case, append_pos=[max_pos + 5, 32], seq_lens=[64, 33], expect_flags=kvq.KVQ_FLAG_BAD_POSITION,
         compare_two_calls=False)


@pytest.mark.parametrize("Hkv", [8, 2])
def test_step_bad_page_of_the_append_flagged(kvq, Hkv):
    # the page taking sequence 0's new token has a bad id in the block table: that append is
    # skipped (no byte of the pool changes for it, page 0 included, which the kernel reads in
    # the bad page's place) and flagged; sequence 1 steps as usual.  Hkv = 8: four-head units,
    # Hkv = 2: one-head units with four query heads each.
    case = Case(2, 8, Hkv, 128, [64, 33], seed=26 + Hkv)
    append_pos, seq_lens = [63, 32], [64, 33]
    pool, k_new, v_new = _setup(case, append_pos, 0x5A)
    bt_ok = case.block_table.numpy().copy()
    case.block_table[0, 63 // case.P] = case.num_pages + 5
    L = case.layout
    ref = pool.copy()
    oracle.quantize_append(L, ref, k_new[1:2, None], v_new[1:2, None], bt_ok[1:2], np.array([32], np.int32))
    got_pool, got_out, flags = _gpu_step(kvq, case, pool, k_new, v_new, append_pos, seq_lens)
    assert flags == kvq.KVQ_FLAG_BAD_PAGE, f"status flags {flags:#x}"
    diff = np.nonzero(got_pool != ref)[0]
    assert diff.size == 0, f"{diff.size} pool bytes differ, first at {diff[:8]}"
    out_ref = oracle.decode_attention(L, ref, case.q.numpy(), bt_ok, np.array(seq_lens, np.int32), case.scale)
    assert_attention_close(got_out[1:], out_ref[1:], what=f"sequence 1 beside a bad append page, Hkv {Hkv}")


def test_step_repeated_steps_match_oracle(kvq):
    """Several steps in a row on the same pool, positions advancing across a page boundary."""
    case = Case(2, 16, 4, 128, [40, 70], seed=26)
    L = case.layout
    cfg = case.cfg(kvq)
    bt = case.block_table.numpy()
    hist = [30, 60]
    pool = np.full(L.pool_bytes, 0x11, np.uint8)
    for b in range(2):
        oracle.quantize_append(L, pool, case.k[b:b + 1, :hist[b]].numpy(), case.v[b:b + 1, :hist[b]].numpy(),
                               bt[b:b + 1], np.zeros(1, np.int32))
    pool_g = torch.from_numpy(pool.copy()).cuda()
    btg = case.block_table.cuda()
    ws = kvq.new_workspace(cfg, 2, case.Hq, 70, device="cuda")
    out = torch.empty((2, case.Hq, 128), dtype=torch.float32, device="cuda")
    for step in range(10):
        ap = [hist[0] + step, hist[1] + step]
        sl = [a + 1 for a in ap]
        k_new = np.stack([case.k[b, ap[b]].numpy() for b in range(2)]).astype(np.float16)
        v_new = np.stack([case.v[b, ap[b]].numpy() for b in range(2)]).astype(np.float16)
        pool, ref_out = _oracle_step(case, pool, k_new, v_new, ap, sl)
        kvq.kvq_decode_step(cfg, pool_g, torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda(),
                            torch.tensor(ap, dtype=torch.int32, device="cuda"), case.q.cuda(), btg,
                            torch.tensor(sl, dtype=torch.int32, device="cuda"), 70, case.scale, out, ws)
        assert np.array_equal(pool_g.cpu().numpy(), pool), f"step {step}: pool differs"
        assert_attention_close(out.cpu().numpy(), ref_out, what=f"step {step}")
    assert kvq.kvq_read_status(ws) == 0


def test_step_from_host_staging_matches_device_step(kvq):
    """PagedKVCache.decode_step_host (one pinned H2D copy, the step, one D2H copy) gives the
    device step's pool and output bit for bit."""
    from int4_group_quantized_kvq_gb300.cache import HostStaging, PagedKVCache
    case = Case(3, 16, 4, 128, [90, 33, 200], seed=27)
    append_pos = [n - 1 for n in case.lens]
    pool, k_new, v_new = _setup(case, append_pos, 0x00)
    cfg = case.cfg(kvq)
    ap = torch.tensor(append_pos, dtype=torch.int32, device="cuda")
    sl = torch.tensor(case.lens, dtype=torch.int32, device="cuda")
    c1 = PagedKVCache(cfg, case.block_table, case.Hq, max(case.lens), device="cuda",
                      pool=torch.from_numpy(pool.copy()).cuda())
    c2 = PagedKVCache(cfg, case.block_table, case.Hq, max(case.lens), device="cuda",
                      pool=torch.from_numpy(pool.copy()).cuda())
    out1 = torch.empty((case.B, case.Hq, case.d), dtype=torch.float32, device="cuda")
    c1.decode_step(case.q.cuda(), torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda(), ap, sl, out1)
    st = HostStaging(case.B, case.Hq, case.Hkv, case.d, device="cuda")
    st.q_host.copy_(case.q)
    st.k_host.copy_(torch.from_numpy(k_new))
    st.v_host.copy_(torch.from_numpy(v_new))
    c2.decode_step_host(st, ap, sl)
    torch.cuda.synchronize()
    assert torch.equal(c1.pool, c2.pool)
    assert torch.equal(out1.cpu(), st.out_host)
    assert c1.flags() == 0 and c2.flags() == 0


def test_host_pipeline_matches_sequential_steps(kvq):
    """HostPipeline (double-buffered staging, copies on their own streams) gives every step's
    output and the final pool bit for bit as the same steps run one after another on the
    device; each step writes new rows into the same positions, so the order matters."""
    from int4_group_quantized_kvq_gb300.cache import HostPipeline, PagedKVCache
    case = Case(3, 16, 4, 128, [90, 33, 200], seed=37)
    append_pos = [n - 1 for n in case.lens]
    pool, _, _ = _setup(case, append_pos, 0x00)
    cfg = case.cfg(kvq)
    ap = torch.tensor(append_pos, dtype=torch.int32, device="cuda")
    sl = torch.tensor(case.lens, dtype=torch.int32, device="cuda")
    ref = PagedKVCache(cfg, case.block_table, case.Hq, max(case.lens), device="cuda",
                       pool=torch.from_numpy(pool.copy()).cuda())
    pc = PagedKVCache(cfg, case.block_table, case.Hq, max(case.lens), device="cuda",
                      pool=torch.from_numpy(pool.copy()).cuda())
    pipe = HostPipeline(pc)
    n_steps = 7
    g = torch.Generator().manual_seed(38)
    ins = [(torch.randn(case.B, case.Hq, case.d, generator=g).half(),
            torch.randn(case.B, case.Hkv, case.d, generator=g).half(),
            torch.randn(case.B, case.Hkv, case.d, generator=g).half()) for _ in range(n_steps)]
    want = []
    for q, kn, vn in ins:
        out = torch.empty((case.B, case.Hq, case.d), dtype=torch.float32, device="cuda")
        ref.decode_step(q.cuda(), kn.cuda(), vn.cuda(), ap, sl, out)
        want.append(out.cpu())
    got = [None] * n_steps
    for i, (q, kn, vn) in enumerate(ins):
        if i >= 2:
            pipe.done(i - 2).synchronize()
            got[i - 2] = pipe.slot(i - 2).out_host.clone()
            pipe.inputs_copied(i - 2).synchronize()
        st = pipe.slot(i)
        st.q_host.copy_(q)
        st.k_host.copy_(kn)
        st.v_host.copy_(vn)
        pipe.step(i, ap, sl)
    for i in (n_steps - 2, n_steps - 1):
        pipe.done(i).synchronize()
        got[i] = pipe.slot(i).out_host.clone()
    pipe.synchronize()
    torch.cuda.synchronize()
    for i in range(n_steps):
        assert torch.equal(got[i], want[i]), f"step {i}"
    assert torch.equal(ref.pool, pc.pool)
    assert ref.flags() == 0 and pc.flags() == 0


def test_nonfinite_rows_pack_alike_in_both_quantizers(kvq):
    """Rows holding NaN or +-inf (outside what the pages define) still get the same bytes from
    the quantize-append kernel and from the decode step's fused append: a NaN value codes as 0,
    the group scale comes from the other values, and an infinite value makes the scale infinite."""
    case = Case(4, 8, 4, 128, [40, 17, 64, 3], seed=41)
    append_pos = [n - 1 for n in case.lens]
    pool, k_new, v_new = _setup(case, append_pos, 0x00)
    k_new = k_new.copy()
    v_new = v_new.copy()
    k_new[0, 0, 5] = np.nan
    k_new[1, 2, 70:74] = np.nan
    v_new[2, 1, 3] = np.inf
    v_new[3, 3, 100] = -np.inf
    k_new[2, 3, :] = np.nan
    cfg = case.cfg(kvq)
    ap = torch.tensor(append_pos, dtype=torch.int32, device="cuda")
    sl = torch.tensor(case.lens, dtype=torch.int32, device="cuda")
    bt = case.block_table.cuda()
    pa = torch.from_numpy(pool.copy()).cuda()
    pb = torch.from_numpy(pool.copy()).cuda()
    kn, vn = torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda()
    kvq.kvq_quantize_append(cfg, pa, kn[:, None], vn[:, None], bt, ap)
    ws = kvq.new_workspace(cfg, case.B, case.Hq, max(case.lens), device="cuda")
    out = torch.empty((case.B, case.Hq, case.d), dtype=torch.float32, device="cuda")
    kvq.kvq_decode_step(cfg, pb, kn, vn, ap, case.q.cuda(), bt, sl, max(case.lens), case.scale, out, ws)
    torch.cuda.synchronize()
    assert torch.equal(pa, pb)


def test_decode_step_host_call_matches_device_step(kvq):
    """kvq_decode_step_host (host-to-device copy, the step, device-to-host copy, one C call) gives
    the device step's pool and output bit for bit."""
    from int4_group_quantized_kvq_gb300.cache import HostStaging
    case = Case(3, 16, 4, 128, [90, 33, 200], seed=43)
    append_pos = [n - 1 for n in case.lens]
    pool, k_new, v_new = _setup(case, append_pos, 0x00)
    cfg = case.cfg(kvq)
    ap = torch.tensor(append_pos, dtype=torch.int32, device="cuda")
    sl = torch.tensor(case.lens, dtype=torch.int32, device="cuda")
    bt = case.block_table.cuda()
    p1 = torch.from_numpy(pool.copy()).cuda()
    p2 = torch.from_numpy(pool.copy()).cuda()
    ml = max(case.lens)
    out1 = torch.empty((case.B, case.Hq, case.d), dtype=torch.float32, device="cuda")
    ws1 = kvq.new_workspace(cfg, case.B, case.Hq, ml, device="cuda")
    kvq.kvq_decode_step(cfg, p1, torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda(), ap, case.q.cuda(), bt,
                        sl, ml, case.scale, out1, ws1)
    st = HostStaging(case.B, case.Hq, case.Hkv, case.d, device="cuda")
    st.q_host.copy_(case.q)
    st.k_host.copy_(torch.from_numpy(k_new))
    st.v_host.copy_(torch.from_numpy(v_new))
    ws2 = kvq.new_workspace(cfg, case.B, case.Hq, ml, device="cuda")
    kvq.kvq_decode_step_host(cfg, p2, st.host, st.dev, ap, bt, sl, case.B, case.Hq, ml, case.scale, st.out, st.out_host,
                             ws2)
    torch.cuda.synchronize()
    assert torch.equal(p1, p2)
    assert torch.equal(out1.cpu(), st.out_host)
    assert kvq.kvq_read_status(ws1) == 0 and kvq.kvq_read_status(ws2) == 0


def test_decode_step_host_call_from_pageable_memory(kvq):
    """kvq_decode_step_host with pageable host buffers (the copies then go through cudaMemcpyAsync
    instead of the kernels) gives the same pool and output as with pinned ones."""
    from int4_group_quantized_kvq_gb300.cache import HostStaging
    case = Case(2, 16, 4, 128, [77, 300], seed=44)
    append_pos = [n - 1 for n in case.lens]
    pool, k_new, v_new = _setup(case, append_pos, 0x00)
    cfg = case.cfg(kvq)
    ap = torch.tensor(append_pos, dtype=torch.int32, device="cuda")
    sl = torch.tensor(case.lens, dtype=torch.int32, device="cuda")
    bt = case.block_table.cuda()
    ml = max(case.lens)
    outs, pools = [], []
    for pinned in (True, False):
        st = HostStaging(case.B, case.Hq, case.Hkv, case.d, device="cuda")
        host_in = st.host if pinned else st.host.clone()        # clone(): pageable
        host_out = st.out_host if pinned else st.out_host.clone()
        n = case.B * case.Hq * case.d
        nk = case.B * case.Hkv * case.d
        host_in[:n].copy_(case.q.reshape(-1))
        host_in[n:n + nk].copy_(torch.from_numpy(k_new).reshape(-1))
        host_in[n + nk:].copy_(torch.from_numpy(v_new).reshape(-1))
        p = torch.from_numpy(pool.copy()).cuda()
        ws = kvq.new_workspace(cfg, case.B, case.Hq, ml, device="cuda")
        kvq.kvq_decode_step_host(cfg, p, host_in, st.dev, ap, bt, sl, case.B, case.Hq, ml, case.scale, st.out, host_out,
                                 ws)
        torch.cuda.synchronize()
        assert kvq.kvq_read_status(ws) == 0
        outs.append(host_out.clone())
        pools.append(p)
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(pools[0], pools[1])

"""Decode attention: the CUDA path against the oracle's fp64 attention over the
dequantized cache, on the same pool bytes (written by the oracle), with the
tolerances of tests/kvq_testlib.py.  Cases span several pages and warps, ragged
tails, empty and one-token sequences, every supported group size, page size and
query-heads-per-KV-head ratio."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from conftest import cuda_available
from kvq_testlib import Case, assert_attention_close, gpu_decode

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


def _run(kvq, case: Case, max_len=None):
    pool_np = case.oracle_pool(fill=0xC3)
    ref = case.oracle_attention(pool_np)
    got, flags = gpu_decode(kvq, case, torch.from_numpy(pool_np).cuda(), max_len=max_len)
    assert flags == 0, f"status flags {flags:#x}"
    return assert_attention_close(got, ref, what=f"B{case.B} Hq{case.Hq} Hkv{case.Hkv} lens{case.lens[:6]}")


@pytest.mark.parametrize("Gk,Gv", [(64, 128), (32, 32), (64, 64), (128, 128), (32, 128), (128, 32)])
def test_groups(kvq, Gk, Gv):
    _run(kvq, Case(3, 8, 8, 128, [300, 129, 17], Gk=Gk, Gv=Gv, seed=Gk + Gv))


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 4), (12, 4), (16, 4), (32, 8), (16, 2), (8, 1), (24, 4), (6, 6),
                                     (2, 2), (12, 12)])
def test_gqa_ratios(kvq, Hq, Hkv):
    _run(kvq, Case(2, Hq, Hkv, 128, [211, 64], seed=Hq * 7 + Hkv))


@pytest.mark.parametrize("P", [16, 32, 64])
@pytest.mark.parametrize("Hq,Hkv", [(8, 4), (8, 8)])
def test_page_sizes(kvq, P, Hq, Hkv):
    # (8, 8) takes four kv heads per unit of work, (8, 4) one
    _run(kvq, Case(3, Hq, Hkv, 128, [1, P + 1, 5 * P - 3], P=P, seed=P + Hkv))


def test_edge_lengths(kvq):
    # empty, single token, exactly one page, one past a page, chunk boundaries
    _run(kvq, Case(9, 4, 2, 128, [0, 1, 15, 16, 17, 31, 32, 33, 2], seed=3))


def test_all_empty(kvq):
    case = Case(2, 4, 4, 128, [0, 0], seed=4)
    pool = torch.zeros(case.layout.pool_bytes, dtype=torch.uint8, device="cuda")
    got, flags = gpu_decode(kvq, case, pool, max_len=16)
    assert flags == 0 and np.all(got == 0)


def test_many_sequences_ragged(kvq):
    rng = np.random.default_rng(8)
    lens = rng.integers(1, 700, size=33).tolist()
    _run(kvq, Case(33, 8, 2, 128, lens, seed=8))


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 16), (16, 2)])
def test_long_single_sequence(kvq, Hq, Hkv):
    # one sequence spread over many CTAs: exercises the combine of many partials
    _run(kvq, Case(1, Hq, Hkv, 128, [6000], seed=10 + Hkv))


def test_contiguous_pages_and_no_outliers(kvq):
    _run(kvq, Case(2, 8, 8, 128, [513, 77], permute=False, outliers=False, seed=12))


def test_max_len_larger_than_lengths(kvq):
    # the host bound only sizes the grid: a generous bound must not change results
    _run(kvq, Case(4, 8, 4, 128, [100, 3, 50, 64], seed=14), max_len=5000)


def test_softmax_scale_extremes(kvq):
    case = Case(2, 8, 8, 128, [90, 33], seed=15)
    pool_np = case.oracle_pool()
    for scale in (0.0, 1.0, 1e-3):
        case.scale = scale
        ref = case.oracle_attention(pool_np)
        got, _ = gpu_decode(kvq, case, torch.from_numpy(pool_np).cuda())
        assert_attention_close(got, ref, what=f"scale {scale}")


def test_bad_page_flagged_without_fault(kvq):
    case = Case(2, 8, 8, 128, [40, 40], seed=16)
    pool_np = case.oracle_pool()
    case.block_table[1, 1] = case.num_pages + 5  # out of range
    got, flags = gpu_decode(kvq, case, torch.from_numpy(pool_np).cuda())
    assert flags & kvq.KVQ_FLAG_BAD_PAGE
    # the untouched sequence is still right
    case.block_table[1, 1] = 0
    ref = case.oracle_attention(pool_np)
    assert_attention_close(got[:1], ref[:1], what="sequence without bad pages")


def test_repeated_calls_are_deterministic(kvq):
    case = Case(3, 16, 4, 128, [700, 1, 333], seed=18)
    pool = torch.from_numpy(case.oracle_pool()).cuda()
    a, _ = gpu_decode(kvq, case, pool)
    b, _ = gpu_decode(kvq, case, pool)
    assert np.array_equal(a, b)


def test_large_batch_published_prefix(kvq):
    # more than 256 sequences: the combine reads the pages prefix the decode grid publishes
    # instead of summing seq_lens itself; empty sequences among them get zeros
    rng = np.random.default_rng(19)
    lens = rng.integers(0, 90, size=300).tolist()
    lens[:3] = [0, 1, 17]
    _run(kvq, Case(300, 4, 2, 128, lens, seed=19))


def test_workspace_reused_across_shapes_without_clearing(kvq):
    # nothing in the workspace carries over between calls: one buffer, filled with garbage
    # once, serves calls of three shapes in turn
    cases = [Case(6, 16, 4, 128, [900, 17, 400, 1, 256, 333], seed=20), Case(2, 8, 8, 128, [70, 300], seed=21),
             Case(1, 32, 8, 128, [5000], seed=22)]
    nbytes = max(kvq.kvq_decode_workspace_bytes(c.cfg(kvq), c.B, c.Hq, max(c.lens)) for c in cases)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")
    ws[:256].zero_()  # the status word
    for case in cases:
        pool_np = case.oracle_pool()
        ref = case.oracle_attention(pool_np)
        got, flags = gpu_decode(kvq, case, torch.from_numpy(pool_np).cuda(), ws=ws)
        assert flags == 0
        assert_attention_close(got, ref, what=f"reused workspace B{case.B}")


def test_many_one_page_segments_per_cta(kvq):
    # thousands of sequences of at most one page: a CTA's slice crosses dozens of segments
    # and three of its four warps hold no unit of a given segment.  Those warps must not
    # run two segments ahead on the double-buffered q barriers (a wait that timed out and a
    # flagged, wrong result before the fix)
    rng = np.random.default_rng(25)
    case = Case(2100, 32, 16, 128, rng.integers(0, 7, size=2100).tolist(), seed=25, device="cuda")
    pool_np = case.oracle_pool()
    got, flags = gpu_decode(kvq, case, torch.from_numpy(pool_np).cuda())
    assert flags == 0
    assert_attention_close(got, case.oracle_attention(pool_np), what="B2100")


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 4)])
def test_extreme_k_codes(kvq, Hq, Hkv):
    # K rows whose every code is +-7 (nibbles 1 and 15, the ends of the score's offset
    # correction, 2^24 S - 8 sum q) and q rows of one sign, where the correction is largest
    case = Case(2, Hq, Hkv, 128, [77, 40], seed=Hq + 130)
    case.k = torch.where(case.k >= 0, 3.0, -3.0).half()
    case.q = case.q.abs()
    _run(kvq, case)

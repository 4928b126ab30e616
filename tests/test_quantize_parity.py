"""Quantize-on-append and dequantize: the CUDA path against the oracle, bit for bit.

Pools start from the same fill byte on both sides, so any byte written to the wrong
place (or not written) shows up as a difference anywhere in the pool.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as W

from conftest import cuda_available

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


def _hard_inputs(shape, seed):
    """fp16 rows mixing scales 1e-7 .. 6e4, x20 outlier channels, zero groups, subnormals and ties."""
    rng = np.random.default_rng(seed)
    B, n, H, d = shape
    mag = 10.0 ** rng.uniform(-7, 4.3, size=(B, n, H, 1))
    x = rng.standard_normal(shape) * mag
    x[..., rng.integers(0, d, 4)] *= 20
    x = np.clip(x, -65504, 65504).astype(np.float16)
    x[rng.random(shape) < 0.01] = 0
    x[:, ::7, :, :32] = 0                                   # whole zero groups
    x[:, 1::11] = (rng.integers(-15, 16, size=x[:, 1::11].shape) * 0.5).astype(np.float16)  # exact ties
    return x


def _gpu_pool(kvq, L, fill, k, v, bt, start, status=None):
    cfg = kvq.config(L.Hkv, L.d, L.P, L.Gk, L.Gv, L.num_pages)
    pool = torch.full((kvq.kvq_pool_bytes(cfg),), fill, dtype=torch.uint8, device="cuda")
    kvq.kvq_quantize_append(cfg, pool, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                            torch.from_numpy(bt).cuda(), torch.from_numpy(start).cuda(), status=status)
    return cfg, pool


@pytest.mark.parametrize("d,P,Gk,Gv", [(128, 16, 64, 128), (128, 16, 32, 32), (128, 16, 128, 128),
                                       (128, 32, 64, 64), (64, 16, 32, 64), (64, 64, 64, 32),
                                       (256, 16, 128, 64), (256, 32, 32, 128)])
def test_quantize_append_bitexact(kvq, d, P, Gk, Gv):
    B, n, H = 3, 37, 4
    per = (n + 2 * P) // P  # pages per sequence: positions reach n + P - 2
    npg = B * per + 2
    L = oracle.Layout(H, d, P, Gk, Gv, npg)
    x_k = _hard_inputs((B, n, H, d), seed=d + P + Gk)
    x_v = _hard_inputs((B, n, H, d), seed=d + P + Gv + 1)
    perm = W.permutation(9, npg).numpy()
    bt = np.stack([perm[b * per:(b + 1) * per] for b in range(B)]).astype(np.int32)
    start = np.array([0, 5, P - 1], np.int32)  # ragged starting positions, one crossing a page
    ref = np.full(L.pool_bytes, 0x5A, np.uint8)
    oracle.quantize_append(L, ref, x_k, x_v, bt, start)
    _, pool = _gpu_pool(kvq, L, 0x5A, x_k, x_v, bt, start)
    got = pool.cpu().numpy()
    diff = np.nonzero(got != ref)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"


@pytest.mark.parametrize("B,n,H", [(5, 13, 6), (1, 300, 3), (7, 1, 5)])
def test_quantize_append_odd_shapes(kvq, B, n, H):
    """Row counts, token counts and head counts that are not powers of two."""
    d, P, Gk, Gv = 128, 16, 64, 128
    per = (n + 2 * P) // P
    npg = B * per + 1
    L = oracle.Layout(H, d, P, Gk, Gv, npg)
    x_k = _hard_inputs((B, n, H, d), seed=B * 100 + n + H)
    x_v = _hard_inputs((B, n, H, d), seed=B * 100 + n + H + 1)
    bt = W.permutation(B + n, npg).numpy()[:B * per].reshape(B, per).astype(np.int32)
    start = (np.arange(B, dtype=np.int32) * 3) % P
    ref = np.full(L.pool_bytes, 0x3C, np.uint8)
    oracle.quantize_append(L, ref, x_k, x_v, bt, start)
    _, pool = _gpu_pool(kvq, L, 0x3C, x_k, x_v, bt, start)
    assert np.array_equal(pool.cpu().numpy(), ref)


def _tie_rows(rng):
    """fp16 groups of 64 built around a known scale s: one element 7 s (so the group's scale
    is exactly s), every half-integer multiple (k + 1/2) s for k in -7..6 (exact ties),
    the fp16 neighbours of each tie, and random values in [-7 s, 7 s].  The scales cover
    every 7-bit mantissa over exponents -20..6 and the subnormals m * 2^-24 with 7 m < 1024."""
    scales = [(64 + j) * 2.0 ** e for e in range(-20, 7) for j in range(64)]
    scales += [m * 2.0 ** -24 for m in range(1, 147)]
    groups = []
    for sc in scales:
        s16 = np.float16(sc)
        assert float(s16) == sc and float(np.float16(7 * sc)) == 7 * sc
        ties = np.array([(k + 0.5) * sc for k in range(-7, 7)], np.float16)
        up = np.nextafter(ties, np.float16(np.inf))
        down = np.nextafter(ties, np.float16(-np.inf))
        rnd = (rng.uniform(-7, 7, 21) * sc).astype(np.float16)
        g = np.concatenate([[np.float16(7 * sc)], ties, up, down, rnd]).astype(np.float16)
        assert g.size == 64 and np.max(np.abs(g.astype(np.float64))) == 7 * sc
        groups.append(rng.permutation(g))
    return np.stack(groups)


def test_quantize_rounding_ties_bitexact(kvq):
    """Codes at and next to every half-integer multiple of the scale, for ~1900 scales."""
    rng = np.random.default_rng(77)
    g = _tie_rows(rng)                      # [n_groups, 64]
    H, d, P = 4, 128, 16
    n_rows = -(-g.shape[0] // 2)
    n = -(-n_rows // H)
    pad = np.zeros((n * H * 2 - g.shape[0], 64), np.float16)
    rows = np.concatenate([g, pad]).reshape(1, n, H, d)
    per = -(-n // P)
    L = oracle.Layout(H, d, P, 64, 64, per)
    bt = np.arange(per, dtype=np.int32).reshape(1, per)
    start = np.zeros(1, np.int32)
    ref = np.full(L.pool_bytes, 0xA5, np.uint8)
    oracle.quantize_append(L, ref, rows, rows[:, ::-1].copy(), bt, start)
    _, pool = _gpu_pool(kvq, L, 0xA5, rows, rows[:, ::-1].copy(), bt, start)
    got = pool.cpu().numpy()
    diff = np.nonzero(got != ref)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"


def test_quantize_append_single_token_steps(kvq):
    """The decode step: one token per sequence at a time, positions advancing across pages."""
    B, H, d, P = 4, 8, 128, 16
    L = oracle.Layout(H, d, P, 64, 128, 40)
    bt = W.permutation(3, 40).numpy()[:B * 10].reshape(B, 10).astype(np.int32)
    ref = np.zeros(L.pool_bytes, np.uint8)
    cfg = kvq.config(H, d, P, 64, 128, 40)
    pool = torch.zeros(kvq.kvq_pool_bytes(cfg), dtype=torch.uint8, device="cuda")
    btg = torch.from_numpy(bt).cuda()
    for step in range(40):
        k = W.kv_tensor(11, (B, 1, H, d), token_offset=step).numpy()
        v = W.kv_tensor(12, (B, 1, H, d), token_offset=step).numpy()
        start = np.array([step, step + 3, 2 * step, 100 + step], np.int32)
        oracle.quantize_append(L, ref, k, v, bt, start)
        kvq.kvq_quantize_append(cfg, pool, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), btg,
                                torch.from_numpy(start).cuda())
    assert np.array_equal(pool.cpu().numpy(), ref)


def test_quantize_flags_bad_rows_and_skips_them(kvq):
    H, d, P = 2, 128, 16
    L = oracle.Layout(H, d, P, 64, 128, 4)
    x = _hard_inputs((3, 2, H, d), seed=5)
    bt = np.array([[0, 1], [2, 99], [3, -1]], np.int32)  # page 99 and -1 are out of range
    start = np.array([0, 16, 40], np.int32)               # sequence 2 at 40: beyond 2 pages of 16
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, pool = _gpu_pool(kvq, L, 0x77, x, x, bt, start, status=status)
    flags = kvq.kvq_read_status(status)
    assert flags & kvq.KVQ_FLAG_BAD_PAGE and flags & kvq.KVQ_FLAG_BAD_POSITION
    ref = np.full(L.pool_bytes, 0x77, np.uint8)
    oracle.quantize_append(L, ref, x[:1], x[:1], bt[:1], start[:1])  # only sequence 0 is valid
    assert np.array_equal(pool.cpu().numpy(), ref)


@pytest.mark.parametrize("Gk,Gv,out_fp16", [(64, 128, False), (64, 128, True), (32, 32, True), (128, 64, False)])
def test_dequantize_bitexact(kvq, Gk, Gv, out_fp16):
    H, d, P = 4, 128, 16
    L = oracle.Layout(H, d, P, Gk, Gv, 9)
    x_k = _hard_inputs((1, 50, H, d), seed=Gk)
    x_v = _hard_inputs((1, 50, H, d), seed=Gv + 3)
    bt = np.array([[4, 0, 8, 2]], np.int32)
    ref_pool = np.zeros(L.pool_bytes, np.uint8)
    oracle.quantize_append(L, ref_pool, x_k, x_v, bt, np.array([3], np.int32))
    cfg = kvq.config(H, d, P, Gk, Gv, 9)
    pool = torch.from_numpy(ref_pool).cuda()  # the oracle's bytes: dequantize is checked on its own
    dt = torch.float16 if out_fp16 else torch.float32
    for start, n in [(3, 50), (0, 64), (17, 1), (15, 2)]:
        ok = torch.empty((n, H, d), dtype=dt, device="cuda")
        ov = torch.empty((n, H, d), dtype=dt, device="cuda")
        kvq.kvq_dequantize(cfg, pool, torch.from_numpy(bt).cuda(), 0, start, n, ok, ov)
        rk, rv = oracle.dequantize(L, ref_pool, bt, 0, start, n, out_fp16=out_fp16)
        assert np.array_equal(ok.cpu().numpy().view(np.uint16 if out_fp16 else np.uint32),
                              rk.view(np.uint16 if out_fp16 else np.uint32))
        assert np.array_equal(ov.cpu().numpy().view(np.uint16 if out_fp16 else np.uint32),
                              rv.view(np.uint16 if out_fp16 else np.uint32))


def test_dequantize_arbitrary_bytes(kvq):
    """Any byte pattern decodes like the oracle decodes it (nibble 0 included), for finite scales."""
    H, d, P = 2, 128, 16
    L = oracle.Layout(H, d, P, 64, 128, 3)
    rng = np.random.default_rng(17)
    pool_np = rng.integers(0, 256, L.pool_bytes, dtype=np.uint8)
    # make every scale a finite fp16
    blk = L.block_bytes
    for i in range(L.num_pages * H):
        base = i * blk + P * d
        sc = pool_np[base: base + P * (d // 64 + 1) * 2].view(np.uint16)
        sc &= np.uint16(0x7BFF)
    bt = np.array([[2, 0, 1]], np.int32)
    cfg = kvq.config(H, d, P, 64, 128, 3)
    pool = torch.from_numpy(pool_np).cuda()
    ok = torch.empty((48, H, d), dtype=torch.float32, device="cuda")
    ov = torch.empty_like(ok)
    kvq.kvq_dequantize(cfg, pool, torch.from_numpy(bt).cuda(), 0, 0, 48, ok, ov)
    rk, rv = oracle.dequantize(L, pool_np, bt, 0, 0, 48)
    assert np.array_equal(ok.cpu().numpy().view(np.uint32), rk.view(np.uint32))
    assert np.array_equal(ov.cpu().numpy().view(np.uint32), rv.view(np.uint32))


def _varlen_case(seed, counts, H, d, P, Gk, Gv):
    """Sequences with `counts[b]` new rows each, appended at ragged start positions into a permuted pool."""
    rng = np.random.default_rng(seed)
    B = len(counts)
    start = rng.integers(0, 3 * P, B).astype(np.int32)
    per = (int(max(start)) + max(counts) + P - 1) // P + 1
    npg = B * per + 3
    L = oracle.Layout(H, d, P, Gk, Gv, npg)
    bt = W.permutation(seed, npg).numpy()[:B * per].reshape(B, per).astype(np.int32)
    total = int(sum(counts))
    x_k = _hard_inputs((1, total, H, d), seed=seed + 1)[0]
    x_v = _hard_inputs((1, total, H, d), seed=seed + 2)[0]
    cu = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return L, bt, start, cu, x_k, x_v


@pytest.mark.parametrize("counts,H,d,P,Gk,Gv", [
    ([5, 0, 37, 1, 16, 70], 4, 128, 16, 64, 128),
    ([3, 129, 0, 0, 2], 8, 128, 32, 32, 32),
    ([17, 1, 33], 3, 64, 16, 32, 64),
    ([9, 40], 2, 256, 64, 128, 64),
    ([1] * 40, 8, 128, 16, 64, 128),
])
def test_quantize_append_varlen_bitexact(kvq, counts, H, d, P, Gk, Gv):
    """One ragged call equals the oracle appending each sequence's own rows at its start position."""
    L, bt, start, cu, x_k, x_v = _varlen_case(sum(counts) + H + d, counts, H, d, P, Gk, Gv)
    ref = np.full(L.pool_bytes, 0x6B, np.uint8)
    for b in range(len(counts)):
        if counts[b]:
            oracle.quantize_append(L, ref, x_k[None, cu[b]:cu[b + 1]], x_v[None, cu[b]:cu[b + 1]], bt[b:b + 1],
                                   start[b:b + 1])
    cfg = kvq.config(H, d, P, Gk, Gv, L.num_pages)
    pool = torch.full((kvq.kvq_pool_bytes(cfg),), 0x6B, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_quantize_append_varlen(cfg, pool, torch.from_numpy(x_k).cuda(), torch.from_numpy(x_v).cuda(),
                                   torch.from_numpy(bt).cuda(), torch.from_numpy(start).cuda(),
                                   torch.from_numpy(cu).cuda(), status=status)
    assert kvq.kvq_read_status(status) == 0
    got = pool.cpu().numpy()
    diff = np.nonzero(got != ref)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:8]}"


def test_quantize_append_varlen_equals_fixed_count_call(kvq):
    """With every sequence appending n rows, the ragged call writes what kvq_quantize_append writes."""
    B, n, H, d, P = 4, 45, 8, 128, 16
    L, bt, start, cu, x_k, x_v = _varlen_case(31, [n] * B, H, d, P, 64, 128)
    cfg = kvq.config(H, d, P, 64, 128, L.num_pages)
    pools = []
    for ragged in (False, True):
        pool = torch.full((kvq.kvq_pool_bytes(cfg),), 0x11, dtype=torch.uint8, device="cuda")
        if ragged:
            kvq.kvq_quantize_append_varlen(cfg, pool, torch.from_numpy(x_k).cuda(), torch.from_numpy(x_v).cuda(),
                                           torch.from_numpy(bt).cuda(), torch.from_numpy(start).cuda(),
                                           torch.from_numpy(cu).cuda())
        else:
            kvq.kvq_quantize_append(cfg, pool, torch.from_numpy(x_k.reshape(B, n, H, d)).cuda(),
                                    torch.from_numpy(x_v.reshape(B, n, H, d)).cuda(), torch.from_numpy(bt).cuda(),
                                    torch.from_numpy(start).cuda())
        pools.append(pool.cpu().numpy())
    assert np.array_equal(pools[0], pools[1])


def test_quantize_append_varlen_bad_positions_are_flagged(kvq):
    """A sequence whose positions leave its block table is skipped and flagged; the others are exact."""
    H, d, P = 2, 128, 16
    counts = [10, 12, 10]
    L, bt, _, cu, x_k, x_v = _varlen_case(5, counts, H, d, P, 64, 128)
    start = np.array([0, P + 3, 10 * P], np.int32)  # sequence 2 beyond its block table
    cfg = kvq.config(H, d, P, 64, 128, L.num_pages)
    pool = torch.full((kvq.kvq_pool_bytes(cfg),), 0x22, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_quantize_append_varlen(cfg, pool, torch.from_numpy(x_k).cuda(), torch.from_numpy(x_v).cuda(),
                                   torch.from_numpy(bt).cuda(), torch.from_numpy(start).cuda(),
                                   torch.from_numpy(cu).cuda(), status=status)
    assert kvq.kvq_read_status(status) == kvq.KVQ_FLAG_BAD_POSITION
    ref = np.full(L.pool_bytes, 0x22, np.uint8)
    for b in (0, 1):
        oracle.quantize_append(L, ref, x_k[None, cu[b]:cu[b + 1]], x_v[None, cu[b]:cu[b + 1]], bt[b:b + 1],
                               start[b:b + 1])
    assert np.array_equal(pool.cpu().numpy(), ref)


def test_quantize_append_varlen_decreasing_offsets_stay_in_bounds(kvq):
    """Offsets that decrease move rows to other sequences or positions, but every byte written
    lies in a block of a page the block table names."""
    H, d, P = 2, 128, 16
    counts = [10, 10, 10]
    L, bt, start, _, x_k, x_v = _varlen_case(6, counts, H, d, P, 64, 128)
    cu = np.array([0, 25, 12, 30], np.int32)
    cfg = kvq.config(H, d, P, 64, 128, L.num_pages)
    pool = torch.full((kvq.kvq_pool_bytes(cfg),), 0x33, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_quantize_append_varlen(cfg, pool, torch.from_numpy(x_k).cuda(), torch.from_numpy(x_v).cuda(),
                                   torch.from_numpy(bt).cuda(), torch.from_numpy(start).cuda(),
                                   torch.from_numpy(cu).cuda(), status=status)
    torch.cuda.synchronize()
    changed = np.nonzero(pool.cpu().numpy() != 0x33)[0]
    assert changed.size > 0
    pages = set(bt[bt >= 0].tolist())
    assert set((changed // (L.block_bytes * H)).tolist()) <= pages

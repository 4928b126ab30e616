"""CPU checks of the seeded input recipe in ``workloads/``.

Both sides of every parity test receive the bytes this module makes, so a fault in
it would not show up as a disagreement between them; these tests pin it on its own:
the generator against SplitMix64's published definition, the normals against their
distribution, and the outlier channels, page permutation, ragged lengths and block
tables against what each promises.
"""
from __future__ import annotations

import math

import torch

import workloads as W

_MASK = (1 << 64) - 1


def _splitmix64_int(seed: int, i: int) -> int:
    """SplitMix64 (Steele, Lea and Flood, OOPSLA 2014) written with Python integers."""
    z = ((i + 1) * 0x9E3779B97F4A7C15 + (seed << 32)) & _MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK
    return z ^ (z >> 31)


def test_splitmix64_first_outputs_from_state_zero():
    # stream 0 starts from state 0: its first three outputs are the generator's
    # well-known opening values
    got = [int(x) & _MASK for x in W.splitmix64(0, 0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_splitmix64_matches_integer_definition():
    # int64 wrap-around and the logical shifts in the tensor version must agree with
    # arbitrary-precision arithmetic reduced mod 2^64, for large counters too
    for seed in (0, 1, 6, 0x7FFF):
        for start in (0, 12345, (1 << 40) - 3):
            got = [int(x) & _MASK for x in W.splitmix64(seed, start, 5)]
            assert got == [_splitmix64_int(seed, start + k) for k in range(5)]


def test_uniforms_are_the_top_53_bits():
    u = W.uniform01(3, 100, 64)
    ref = torch.tensor([(_splitmix64_int(3, 100 + k) >> 11) * 2.0 ** -53 for k in range(64)], dtype=torch.float64)
    assert torch.equal(u, ref)
    big = W.uniform01(9, 0, 1 << 16)
    assert float(big.min()) >= 0.0 and float(big.max()) < 1.0


def test_normals_have_standard_moments():
    n = 1 << 20
    x = W.normal(1, n).double()
    assert x.dtype == torch.float64 and torch.isfinite(x).all()
    se = 1.0 / math.sqrt(n)
    assert abs(float(x.mean())) < 5 * se
    assert abs(float(x.var()) - 1.0) < 5 * math.sqrt(2.0) * se
    assert abs(float((x ** 3).mean())) < 5 * math.sqrt(15.0) * se
    assert abs(float((x ** 4).mean()) - 3.0) < 5 * math.sqrt(96.0) * se
    # tail mass beyond 2 sigma: 2 * (1 - Phi(2)) = 0.0455003
    p = 0.04550026
    assert abs(float((x.abs() > 2).double().mean()) - p) < 5 * math.sqrt(p * (1 - p) / n)


def test_normals_come_from_box_muller_of_counter_pairs():
    x = W.normal(5, 4)
    for j in range(4):
        u1 = (_splitmix64_int(5, 2 * j) >> 11) * 2.0 ** -53
        u2 = (_splitmix64_int(5, 2 * j + 1) >> 11) * 2.0 ** -53
        ref = math.sqrt(-2.0 * math.log(1.0 - u1)) * math.cos(2.0 * math.pi * u2)
        assert abs(float(x[j]) - ref) <= 1e-6 * max(1.0, abs(ref))


def test_kv_tensor_is_deterministic_and_counter_indexed():
    a = W.kv_tensor(W.SEED_K, (2, 40, 3, 128))
    b = W.kv_tensor(W.SEED_K, (2, 40, 3, 128))
    assert a.dtype == torch.float16 and torch.equal(a, b)
    # a slice of a sequence regenerates on its own from its token offset
    tail = W.kv_tensor(W.SEED_K, (2, 15, 3, 128), token_offset=25)
    assert torch.equal(tail, a[:, 25:])
    # K and V streams differ
    assert not torch.equal(a, W.kv_tensor(W.SEED_V, (2, 40, 3, 128)))


def test_outlier_channels_and_their_scale():
    H, d = 8, 128
    idx = W.outlier_channels(H, d)
    assert idx.shape == (H, 4) and int(idx.min()) >= 0 and int(idx.max()) < d
    for h in range(H):
        assert len(set(idx[h].tolist())) == 4
    assert torch.equal(idx, W.outlier_channels(H, d))
    plain = W.kv_tensor(W.SEED_K, (1, 512, H, d)).float()
    hot = W.kv_tensor(W.SEED_K, (1, 512, H, d), outlier_scale=20.0, outlier_idx=idx).float()
    mask = torch.zeros(H, d, dtype=torch.bool)
    mask.scatter_(1, idx, True)
    mask = mask.expand_as(hot[0])
    # the other channels are untouched; the chosen ones are the same draws times 20
    assert torch.equal(hot[0][~mask], plain[0][~mask])
    ratio = hot[0][mask] / plain[0][mask]
    big = plain[0][mask].abs() > 0.5
    assert torch.allclose(ratio[big], torch.full_like(ratio[big], 20.0), rtol=2e-3)
    sd = hot[0].std(dim=0)
    assert float(sd[mask[0]].min()) > 15.0 and float(sd[~mask[0]].max()) < 1.3


def test_permutation_and_ragged_lengths():
    for n in (1, 2, 17, 1000):
        p = W.permutation(W.SEED_PERM, n)
        assert p.dtype == torch.int32 and sorted(p.tolist()) == list(range(n))
    assert not torch.equal(W.permutation(W.SEED_PERM, 1000), torch.arange(1000, dtype=torch.int32))
    lens = W.ragged_lengths(32, 512, 4096)
    assert len(lens) == 32 and min(lens) >= 512 and max(lens) <= 4096
    assert lens == W.ragged_lengths(32, 512, 4096) and len(set(lens)) > 16
    r = W.randint_below(11, 1 << 16, 7)
    counts = torch.bincount(r, minlength=7).double()
    assert int(r.min()) == 0 and int(r.max()) == 6
    expect = (1 << 16) / 7
    assert float(((counts - expect) ** 2 / expect).sum()) < 30.0  # chi-square, 6 dof


def test_block_tables_map_every_token_to_one_page():
    for make in W.ALL.values():
        w = make()
        bt = w.block_table()
        assert bt.shape == (w.B, w.max_blocks) and bt.dtype == torch.int32
        used = []
        for b, npg in enumerate(w.pages_per_seq):
            assert npg == -(-w.seq_lens[b] // w.P)
            row = bt[b].tolist()
            assert all(0 <= x < w.num_pages for x in row[:npg]) and all(x == -1 for x in row[npg:])
            used += row[:npg]
        assert len(used) == len(set(used)) == sum(w.pages_per_seq)
        assert w.seq_lens == [c + 1 for c in w.ctx]


def test_workload_shapes_and_byte_counts():
    w = W.llama7b_mha()
    assert (w.B, w.Hq, w.Hkv, w.d, w.r, w.max_len) == (8, 32, 32, 128, 1, 8193)
    # one token of one KV head: 128 bytes of K and V nibbles, 2 K and 1 V fp16 scales
    assert w.packed_bytes_per_token_head() == 128 + 2 * (2 + 1) == 134
    assert w.decode_bytes() == 8 * 32 * 8193 * 134
    assert w.append_bytes() == 8 * 32 * (2 * 128 * 2 + 134)
    g = W.gqa8b()
    assert g.r == 4 and g.decode_bytes() == 140_513_472
    s = W.longctx(32)
    assert (s.Gk, s.Gv) == (32, 32) and s.packed_bytes_per_token_head() == 128 + 2 * 8
    t = W.tiny_mha()
    assert torch.equal(t.block_table()[0], torch.arange(t.num_pages, dtype=torch.int32))

"""Pins for the oracle: checks against what the pages and the mathematics fix,
never against a retyping of the oracle's own formulas.

 - fp16 conversion: exhaustive and randomized agreement with numpy's float16
   (an independent implementation of IEEE-754 binary16 rounding).
 - sizes: the bits-per-element table of "4-bit KV cache compression"
   (lpnh.cn/news/2042373) section 2.2 and the FP16 KV size figures of its
   section 1.2 and of "LLM long-context inference: managing the KV cache with an
   INT4 state machine" (pwwt.cn/news/4219524) sections 2 and 6.2.
 - quantization: hand-worked examples (tests/golden/quantize_examples.txt),
   brute-force nearest-code search, the error bound |x - x^| <= s/2, the
   max-code invariant and sign symmetry.
 - layout: a hand-worked byte map (tests/golden/layout_example.txt).
 - attention: special cases with closed forms (one token, equal keys, one
   dominant logit, zero softmax scale), brute force against numpy/scipy
   softmax attention on tiny inputs, GQA = MHA on repeated KV heads ("AI
   inference tuning: KV Cache optimisation..." section 3.2), page-table
   permutation invariance and exact scaling by powers of two.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import scipy.special

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------------------
# fp16 conversions
# ----------------------------------------------------------------------------

def test_f16_to_f64_exhaustive():
    h = np.arange(65536, dtype=np.uint16)
    ours = oracle.f16_to_f64_array(h)
    ref = h.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_f32_to_f16_midpoints_and_random():
    rng = np.random.default_rng(0)
    # every finite fp16 value, its exact fp32 image, and the midpoints to its neighbours
    h = np.arange(0, 0x7c00, dtype=np.uint16)
    v = h.view(np.float16).astype(np.float64)
    nxt = np.append(v[1:], 65520.0)  # 65520 is the midpoint rounding to infinity
    mids = ((v + nxt) / 2).astype(np.float32)  # exactly representable in fp32
    vals = np.concatenate([v.astype(np.float32), mids, np.nextafter(mids, np.float32(0)),
                           np.nextafter(mids, np.float32(np.inf))])
    rand_bits = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    rand = rand_bits.view(np.float32)
    rand = rand[np.isfinite(rand)]
    small = (rng.standard_normal(500_000) * 10.0 ** rng.uniform(-9, 5, 500_000)).astype(np.float32)
    allv = np.concatenate([vals, -vals, rand, small, np.array([65519.996, 65520.0, 1e-8, 2.0 ** -25,
                                                               2.0 ** -25 * 1.0000001], dtype=np.float32)])
    ours = oracle.f32_to_f16_array(allv)
    with np.errstate(over="ignore"):
        ref = allv.astype(np.float16).view(np.uint16)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first {allv[bad[:5]]}: {ours[bad[:5]]} vs {ref[bad[:5]]}"


def test_f32_to_f16_infinities_and_nans():
    # IEEE 754 conversion: an infinity stays that infinity and a NaN stays a NaN (all-ones
    # exponent, nonzero fraction) of the same sign; the NaN payload is not fixed by the
    # standard, so only NaN-ness and sign are compared with numpy's cast
    inf = np.array([np.inf, -np.inf, 3.4e38, -3.4e38], dtype=np.float32)
    with np.errstate(over="ignore"):
        assert np.array_equal(oracle.f32_to_f16_array(inf), inf.astype(np.float16).view(np.uint16))
    nan_bits = np.array([0x7FC00000, 0x7F800001, 0x7FFFFFFF, 0xFFC00000, 0xFF800001, 0x7FA00000], dtype=np.uint32)
    ours = oracle.f32_to_f16_array(nan_bits.view(np.float32))
    assert np.all((ours & 0x7C00) == 0x7C00) and np.all((ours & 0x03FF) != 0)
    assert np.array_equal(ours >> 15, (nan_bits >> 31).astype(ours.dtype))


# ----------------------------------------------------------------------------
# sizes
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("G,bits,ratio", [(32, 4.5, 3.56), (64, 4.25, 3.76), (128, 4.125, 3.88)])
def test_bits_per_element_table(G, bits, ratio):
    """Section 2.2 of the 4-bit compression page: 4 + 16/G bits per element."""
    d, P = 128, 16
    blk = oracle.block_bytes(d, P, G, G)
    got_bits = 8.0 * blk / (2 * P * d)  # K and V elements of one page and head
    assert got_bits == bits
    assert round(16.0 / got_bits, 2) == ratio


def test_block_bytes_default_k64_v128():
    # K at 64 and V at 128: 2048 code bytes + 16*(2+1)*2 scale bytes; a 16-byte multiple
    assert oracle.block_bytes(128, 16, 64, 128) == 2144
    assert oracle.block_bytes(128, 16, 64, 128) % 16 == 0


def test_fp16_kv_size_figures():
    GiB = 1024 ** 3
    # 32 layers x 32 heads x 128: 512 KB per token; 10k tokens about 5 GB, 100k about 50 GB
    assert oracle.fp16_kv_bytes(32, 32, 128, 1) == 512 * 1024
    assert 4.5e9 < oracle.fp16_kv_bytes(32, 32, 128, 10_000) < 5.5e9
    assert 45e9 < oracle.fp16_kv_bytes(32, 32, 128, 100_000) < 55e9
    # the 7B MHA table: 2048x1 -> 1 GB, 4096x4 -> 8 GB, 8192x8 -> 32 GB
    assert oracle.fp16_kv_bytes(32, 32, 128, 2048 * 1) == 1 * GiB
    assert oracle.fp16_kv_bytes(32, 32, 128, 4096 * 4) == 8 * GiB
    assert oracle.fp16_kv_bytes(32, 32, 128, 8192 * 8) == 32 * GiB
    # GQA 8B with 8 KV heads: 128 KB per token, 32K x batch 4 -> 16 GB
    assert oracle.fp16_kv_bytes(32, 8, 128, 1) == 128 * 1024
    assert oracle.fp16_kv_bytes(32, 8, 128, 32768 * 4) == 16 * GiB
    # the cache_memory estimator of section 6.2: FP16 2/4/8/16 GiB, 4 bits 0.5/1/2/4 GiB at 4K..32K
    for seq, gib in [(4096, 2.0), (8192, 4.0), (16384, 8.0), (32768, 16.0)]:
        assert oracle.fp16_kv_bytes(32, 32, 128, seq) / GiB == gib
        assert oracle.fp16_kv_bytes(32, 32, 128, seq) / 4 / GiB == gib / 4
    # "LARQL KV cache engines", engines one and two: at 4096 positions of a 34-layer model with 4 KV heads of
    # 256 kept as f32 rows (twice the fp16 bytes: 8 KiB per layer and position), the full cache holds
    # 34 x 4096 rows and the window engine 29 sliding layers x 1024 rows plus 5 global layers x 4096:
    # 1.06 GiB against 0.38 GiB
    row_f32 = 2 * oracle.fp16_kv_bytes(1, 4, 256, 1)
    assert row_f32 == 8 * 1024
    full = 34 * 4096 * row_f32
    window = (29 * 1024 + 5 * 4096) * row_f32
    assert 34 * 4096 == 139264 and 29 * 1024 + 5 * 4096 == 50176
    assert full / GiB == 1.0625 and round(window / GiB, 2) == 0.38
    assert round(1 - window / full, 2) == 0.64  # the page's "-64%"


# ----------------------------------------------------------------------------
# quantization: golden worked examples
# ----------------------------------------------------------------------------

def _parse_value(tok: str) -> np.float16:
    if tok.startswith("h0x"):
        return np.array([int(tok[1:], 16)], dtype=np.uint16).view(np.float16)[0]
    return np.float16(float(tok))


def load_quantize_cases():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "quantize_examples.txt")) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest, "x": {}, "codes": {}, "bytes": None}
                cases.append(cur)
            elif key == "G":
                cur["G"] = int(rest)
            elif key == "x":
                for tok in rest.split():
                    i, v = tok.split(":")
                    cur["x"][int(i)] = _parse_value(v)
            elif key == "scale":
                cur["scale"] = int(rest, 16)
            elif key == "codes":
                for tok in rest.split():
                    i, c = tok.split(":")
                    cur["codes"][int(i)] = int(c)
            elif key == "bytes":
                cur["bytes"] = [int(t, 16) for t in rest.split()]
    return cases


QCASES = load_quantize_cases()


@pytest.mark.parametrize("case", QCASES, ids=[c["name"] for c in QCASES])
def test_quantize_golden(case):
    G = case["G"]
    x = np.zeros(G, dtype=np.float16)
    for i, v in case["x"].items():
        x[i] = v
    codes, scale = oracle.quantize_group(x)
    assert scale == case["scale"], f"scale {scale:#06x} != {case['scale']:#06x}"
    want = np.zeros(G, dtype=np.int8)
    for i, c in case["codes"].items():
        want[i] = c
    assert np.array_equal(codes, want), f"codes {codes} != {want}"
    if case["bytes"] is not None:
        # pack through the pool writer: one token, one head, d = G, K and V groups = G
        L = oracle.Layout(1, G, 16, G, G, 1)
        pool = np.zeros(L.pool_bytes, dtype=np.uint8)
        k = x.reshape(1, 1, 1, G)
        oracle.quantize_append(L, pool, k, k, np.zeros((1, 1), np.int32), np.zeros(1, np.int32))
        nb = len(case["bytes"])
        assert list(pool[:nb]) == case["bytes"]


def test_quantize_golden_covers_cases():
    assert len(QCASES) >= 12


# ----------------------------------------------------------------------------
# quantization: brute force and invariants on random groups
# ----------------------------------------------------------------------------

def _random_groups(n, G, seed):
    """fp16 groups with magnitudes from 1e-7 to 6e4, some with x20 outliers, a few exact zeros."""
    rng = np.random.default_rng(seed)
    mag = 10.0 ** rng.uniform(-7, 4.5, size=(n, 1))
    x = rng.standard_normal((n, G)) * mag
    out = rng.random((n, G)) < 0.05
    x = np.where(out, x * 20, x)
    x = np.clip(x, -65504, 65504).astype(np.float16)
    x[rng.random((n, G)) < 0.02] = 0
    x[: max(1, n // 50)] = 0  # some all-zero groups
    return x


@pytest.mark.parametrize("G", [32, 64, 128])
def test_quantize_brute_force_nearest_code(G):
    """The code is the integer in [-7, 7] nearest to fp32(x / s), ties to even: found by exhaustive search."""
    groups = _random_groups(400, G, seed=G)
    ks = np.arange(-7, 8, dtype=np.float64)
    for x in groups:
        codes, sbits = oracle.quantize_group(x)
        s = np.float32(np.array([sbits], np.uint16).view(np.float16)[0])
        qf = (x.astype(np.float32) / s).astype(np.float64)  # IEEE fp32 quotient
        dist = np.abs(qf[:, None] - ks[None, :])
        best = dist.min(axis=1, keepdims=True)
        cand = np.where(dist == best, ks[None, :], np.nan)
        # tie: prefer the even integer
        even = np.where(np.isnan(cand), np.nan, np.where(cand % 2 == 0, cand, np.nan))
        even_max = np.max(np.where(np.isnan(even), -np.inf, even), axis=1)
        cand_max = np.max(np.where(np.isnan(cand), -np.inf, cand), axis=1)
        pick = np.where(np.isfinite(even_max), even_max, cand_max)
        assert np.array_equal(codes.astype(np.float64), pick)


@pytest.mark.parametrize("G", [32, 64, 128])
def test_quantize_scale_is_fp16_of_fp32_amax_over_7(G):
    groups = _random_groups(400, G, seed=100 + G)
    for x in groups:
        _, sbits = oracle.quantize_group(x)
        amax = np.float32(np.max(np.abs(x.astype(np.float32))))
        s_ref = np.float16(amax / np.float32(7.0))  # numpy: IEEE fp32 division, fp16 RNE
        if s_ref == 0:
            s_ref = np.float16(1.0)
        assert sbits == int(np.array([s_ref]).view(np.uint16)[0])


@pytest.mark.parametrize("G", [32, 64, 128])
def test_quantize_invariants(G):
    groups = _random_groups(600, G, seed=200 + G)
    for x in groups:
        codes, sbits = oracle.quantize_group(x)
        s = float(np.array([sbits], np.uint16).view(np.float16)[0])
        assert codes.min() >= -7 and codes.max() <= 7
        xf = x.astype(np.float64)
        xhat = codes.astype(np.float64) * s
        nonzero = np.any(xf != 0)
        if s >= 2.0 ** -14 and nonzero:  # a normal fp16 scale
            assert np.all(np.abs(xf - xhat) <= s / 2 * (1 + 2.0 ** -20))
            # amax / s lies within 7 * (1 +- 2^-11), so the largest |code| is exactly 7
            assert np.abs(codes).max() == 7
        if not nonzero:
            assert sbits == 0x3C00 and np.all(codes == 0)
        # sign symmetry: quantize(-x) = -quantize(x), same scale
        c2, s2 = oracle.quantize_group(-x)
        assert s2 == sbits and np.array_equal(c2, -codes)


def test_dequantize_roundtrip_exact_on_grid():
    """Values that are exact multiples k*s with max |k| = 7 come back exactly (closed form)."""
    rng = np.random.default_rng(7)
    L = oracle.Layout(2, 64, 16, 32, 64, 4)
    for s in [1.0, 0.5, 0.25, 2.0 ** -6, 3.0, 96.0]:
        ks = rng.integers(-7, 8, size=(1, 5, 2, 64))
        ks[..., 0] = 7
        ks[..., 32] = -7
        x = (ks * s).astype(np.float16)
        assert np.array_equal(x.astype(np.float64), ks * s)
        pool = np.zeros(L.pool_bytes, np.uint8)
        bt = np.array([[3, 1, 0, 2]], np.int32)
        oracle.quantize_append(L, pool, x, x, bt, np.array([9], np.int32))
        dk, dv = oracle.dequantize(L, pool, bt, 0, 9, 5)
        assert np.array_equal(dk, x[0].astype(np.float32))
        assert np.array_equal(dv, x[0].astype(np.float32))
        hk, hv = oracle.dequantize(L, pool, bt, 0, 9, 5, out_fp16=True)
        assert np.array_equal(hk, x[0]) and np.array_equal(hv, x[0])



def test_quantize_store_read_roundtrip_mse_at_g32():
    # "LLM long-context inference: managing the KV cache with an INT4 state machine", section 7.1: quantize at
    # group size 32, write, read back, dequantize, and the MSE must stay under a threshold.  Here the write and
    # the read go through the paged pool; the thresholds are the hard bound (|x - x^| <= s/2 gives MSE <= s^2/4)
    # and, for Gaussian rows, the uniform rounding-error model s^2/12 to within 10%.
    L = oracle.Layout(8, 128, 16, 32, 32, 64)
    n = 1000
    bt = np.arange(64, dtype=np.int32).reshape(1, -1)
    for outl in (0.0, 20.0):
        x = W.kv_tensor(301, (1, n, 8, 128), outl, W.outlier_channels(8, 128, seed=302) if outl else None).numpy()
        pool = np.zeros(L.pool_bytes, np.uint8)
        oracle.quantize_append(L, pool, x, x, bt, np.zeros(1, np.int32))
        dk, dv = oracle.dequantize(L, pool, bt, 0, 0, n)
        assert np.array_equal(dk, dv)
        xd = x[0].astype(np.float64)
        mse = ((dk.astype(np.float64) - xd) ** 2).mean()
        step = np.abs(dk.astype(np.float64)).reshape(n, 8, 4, 32).max(-1) / 7.0
        s2 = np.repeat(step ** 2, 32, axis=-1).reshape(n, 8, 128)
        assert mse <= (s2 / 4).mean()
        if outl == 0.0:
            assert 0.9 <= mse / (s2 / 12).mean() <= 1.05
            assert mse < 0.012  # under 1.2% of the rows' unit power

@pytest.mark.parametrize("Gk,Gv", [(32, 64), (64, 128), (32, 32)])
def test_dequantize_error_bound_per_group(Gk, Gv):
    """Each element comes back within half its own group's step amax_g / 7 (computed here from
    the input), with groups of very different magnitude side by side."""
    d = 128
    L = oracle.Layout(2, d, 16, Gk, Gv, 6)
    rng = np.random.default_rng(Gk + Gv)
    n = 23
    mags = 10.0 ** rng.uniform(-3, 3, size=(1, n, 2, d // 16)).repeat(16, axis=3)
    x = (rng.standard_normal((1, n, 2, d)) * mags).astype(np.float16)
    bt = np.array([[5, 0, 3]], np.int32)
    pool = np.zeros(L.pool_bytes, np.uint8)
    oracle.quantize_append(L, pool, x, x, bt, np.array([3], np.int32))
    dk, dv = oracle.dequantize(L, pool, bt, 0, 3, n)
    xf = x[0].astype(np.float64)
    for deq, G in [(dk, Gk), (dv, Gv)]:
        amax = np.abs(xf).reshape(n, 2, d // G, G).max(axis=3, keepdims=True)
        step = (amax / 7.0) * (1 + 2.0 ** -10)  # the fp16 scale is within 2^-11 of amax/7
        err = np.abs(xf - deq.astype(np.float64)).reshape(n, 2, d // G, G)
        assert np.all(err <= step / 2 * (1 + 2.0 ** -20) + 1e-30)


# ----------------------------------------------------------------------------
# layout
# ----------------------------------------------------------------------------

def _parse_expect(toks):
    out = []
    for t in toks:
        if "*" in t:
            b, n = t.split("*")
            out += [int(b, 16)] * int(n)
        else:
            out.append(int(t, 16))
    return out


def test_layout_golden():
    spec = {"expect": []}
    with open(os.path.join(GOLDEN, "layout_example.txt")) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            key, *toks = line.split()
            if key == "expect":
                spec["expect"].append((int(toks[0]), _parse_expect(toks[1:])))
            else:
                spec[key] = toks
    Hkv, d, P, Gk, Gv, npg = map(int, spec["geometry"])
    L = oracle.Layout(Hkv, d, P, Gk, Gv, npg)
    assert L.block_bytes == int(spec["block_bytes"][0])
    k = np.zeros((1, 1, Hkv, d), np.float16)
    v = np.zeros((1, 1, Hkv, d), np.float16)
    for arr, key in [(k, "k"), (v, "v")]:
        for t in spec[key]:
            h, i, val = t.split(":")
            arr[0, 0, int(h), int(i)] = float(val)
    pool = np.full(L.pool_bytes, 0xA5, np.uint8)
    bt = np.array([list(map(int, spec["block_table"]))], np.int32)
    oracle.quantize_append(L, pool, k, v, bt, np.array([int(spec["start_pos"][0])], np.int32))
    touched = np.zeros(pool.size, bool)
    for off, bs in spec["expect"]:
        assert list(pool[off:off + len(bs)]) == bs, f"bytes at {off}"
        touched[off:off + len(bs)] = True
    assert np.all(pool[~touched] == 0xA5)


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------

def _build_cache(L, B, lens, seed, permute=True, outliers=True, extra_pages=0):
    """Quantize seeded K/V histories of the given lengths into a pool; return (pool, bt, k, v)."""
    P = L.P
    pages = [(n + P - 1) // P for n in lens]
    maxb = max(pages)
    total = sum(pages)
    assert total + extra_pages <= L.num_pages
    order = W.permutation(seed + 11, L.num_pages).numpy() if permute else np.arange(L.num_pages, dtype=np.int32)
    bt = np.full((B, maxb), -1, np.int32)
    kk = 0
    for b in range(B):
        bt[b, :pages[b]] = order[kk:kk + pages[b]]
        kk += pages[b]
    n = max(lens)
    oidx = W.outlier_channels(L.Hkv, L.d, seed=seed + 13) if outliers else None
    k = W.kv_tensor(seed, (B, n, L.Hkv, L.d), 20.0 if outliers else 0.0, oidx).numpy()
    v = W.kv_tensor(seed + 1, (B, n, L.Hkv, L.d)).numpy()
    pool = np.zeros(L.pool_bytes, np.uint8)
    for b in range(B):
        if lens[b]:
            oracle.quantize_append(L, pool, k[b:b + 1, :lens[b]], v[b:b + 1, :lens[b]], bt[b:b + 1],
                                   np.array([0], np.int32))
    return pool, bt, k, v


def _reference_attention(L, pool, bt, q, lens, scale):
    """numpy/scipy softmax attention over the oracle's dequantized cache (GQA by repetition)."""
    B, Hq, d = q.shape
    r = Hq // L.Hkv
    out = np.zeros((B, Hq, d))
    for b in range(B):
        if lens[b] == 0:
            continue
        dk, dv = oracle.dequantize(L, pool, bt, b, 0, lens[b])
        for hq in range(Hq):
            kh = dk[:, hq // r, :].astype(np.float64)
            vh = dv[:, hq // r, :].astype(np.float64)
            s = (kh @ q[b, hq].astype(np.float64)) * scale
            out[b, hq] = scipy.special.softmax(s) @ vh
    return out


@pytest.mark.parametrize("lens,Hq,Hkv", [([1, 15], 4, 2), ([16, 17], 4, 4), ([40, 33], 8, 2), ([5, 0], 2, 2)])
def test_attention_brute_force(lens, Hq, Hkv):
    L = oracle.Layout(Hkv, 64, 16, 32, 64, 16)
    pool, bt, _, _ = _build_cache(L, len(lens), lens, seed=21)
    q = W.kv_tensor(W.SEED_Q, (1, len(lens), Hq, 64)).numpy()[0]
    scale = 64 ** -0.5
    got = oracle.decode_attention(L, pool, q, bt, np.array(lens, np.int32), scale)
    ref = _reference_attention(L, pool, bt, q, lens, scale)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    for b, n in enumerate(lens):
        if n == 0:
            assert np.all(got[b] == 0)


def test_attention_single_token_returns_its_value():
    L = oracle.Layout(2, 64, 16, 32, 64, 4)
    pool, bt, _, _ = _build_cache(L, 1, [1], seed=31)
    q = W.kv_tensor(W.SEED_Q, (1, 1, 4, 64)).numpy()[0]
    got = oracle.decode_attention(L, pool, q, bt, np.array([1], np.int32), 0.125)
    _, dv = oracle.dequantize(L, pool, bt, 0, 0, 1)
    for hq in range(4):
        assert np.array_equal(got[0, hq], dv[0, hq // 2].astype(np.float64))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_split_combine_rule_reproduces_attention(seed):
    # the split-KV merge: a segment of positions keeps its running maximum m, its sum
    # l = sum exp(z - m) and its unnormalised output o = sum exp(z - m) v; segments merge
    # as M = max m_i, out = sum exp(m_i - M) o_i / sum exp(m_i - M) l_i, an empty segment
    # (m = -inf, l = 0) contributing nothing.  Over the oracle's dequantized cache this must
    # give the oracle's attention, for any cut of the positions into segments.
    L = oracle.Layout(2, 64, 16, 32, 64, 16)
    lens = [150, 37]
    pool, bt, _, _ = _build_cache(L, 2, lens, seed=41 + seed)
    q = W.kv_tensor(W.SEED_Q + seed, (1, 2, 4, 64)).numpy()[0] * np.float16(4)  # sharp softmax
    scale = 0.125
    want = oracle.decode_attention(L, pool, q, bt, np.array(lens, np.int32), scale)
    rng = np.random.default_rng(seed)
    for b, n in enumerate(lens):
        dk, dv = oracle.dequantize(L, pool, bt, b, 0, n)
        cuts = np.sort(np.concatenate([[0, 0, n, n], rng.integers(0, n + 1, 6)]))  # repeats give empty segments
        for hq in range(4):
            k = dk[:, hq // 2].astype(np.float64)
            v = dv[:, hq // 2].astype(np.float64)
            z = (k @ q[b, hq].astype(np.float64)) * scale
            parts = []
            for a, e in zip(cuts[:-1], cuts[1:]):
                if e == a:
                    parts.append((-np.inf, 0.0, np.zeros(64)))
                    continue
                m = z[a:e].max()
                w = np.exp(z[a:e] - m)
                parts.append((m, w.sum(), w @ v[a:e]))
            M = max(m for m, _, _ in parts)
            num = sum(np.exp(m - M) * o for m, l, o in parts if l > 0)
            den = sum(np.exp(m - M) * l for m, l, o in parts if l > 0)
            got = num / den
            assert np.abs(got - want[b, hq]).max() <= 1e-12 * max(1.0, np.abs(want[b, hq]).max())


def test_attention_equal_keys_gives_mean_value():
    L = oracle.Layout(1, 64, 16, 32, 64, 4)
    n = 37
    k = np.repeat(W.kv_tensor(1, (1, 1, 1, 64)).numpy(), n, axis=1)
    v = W.kv_tensor(2, (1, n, 1, 64)).numpy()
    pool = np.zeros(L.pool_bytes, np.uint8)
    bt = np.array([[2, 0, 3]], np.int32)
    oracle.quantize_append(L, pool, k, v, bt, np.array([0], np.int32))
    q = W.kv_tensor(3, (1, 1, 1, 64)).numpy()[0]
    got = oracle.decode_attention(L, pool, q, bt, np.array([n], np.int32), 0.3)
    _, dv = oracle.dequantize(L, pool, bt, 0, 0, n)
    np.testing.assert_allclose(got[0, 0], dv[:, 0].astype(np.float64).mean(axis=0), rtol=1e-13, atol=1e-13)
    # zero softmax scale makes any keys uniform too
    pool2, bt2, _, _ = _build_cache(L, 1, [n], seed=41)
    got0 = oracle.decode_attention(L, pool2, q, bt2, np.array([n], np.int32), 0.0)
    _, dv2 = oracle.dequantize(L, pool2, bt2, 0, 0, n)
    np.testing.assert_allclose(got0[0, 0], dv2[:, 0].astype(np.float64).mean(axis=0), rtol=1e-13, atol=1e-13)


def test_attention_dominant_logit_selects_value():
    L = oracle.Layout(1, 64, 16, 32, 64, 4)
    n = 20
    k = np.zeros((1, n, 1, 64), np.float16)
    k[0, :, 0, 0] = 0.0
    k[0, 13, 0, 0] = 7.0     # one key aligned with q
    v = W.kv_tensor(2, (1, n, 1, 64)).numpy()
    pool = np.zeros(L.pool_bytes, np.uint8)
    bt = np.array([[1, 3]], np.int32)
    oracle.quantize_append(L, pool, k, v, bt, np.array([0], np.int32))
    q = np.zeros((1, 1, 64), np.float16)
    q[0, 0, 0] = 1000.0
    # logit 7000 against 0: exp(7000) overflows fp64, so the maximum must be subtracted first
    got = oracle.decode_attention(L, pool, q, bt, np.array([n], np.int32), 1.0)
    _, dv = oracle.dequantize(L, pool, bt, 0, 0, n)
    np.testing.assert_allclose(got[0, 0], dv[13, 0].astype(np.float64), rtol=0, atol=1e-300)


def test_attention_gqa_equals_mha_on_repeated_heads():
    """Query head h reads KV head h // r: the same as MHA over KV heads repeated r times (section 3.2)."""
    r, Hkv, d = 4, 2, 64
    Lg = oracle.Layout(Hkv, d, 16, 32, 64, 8)
    Lm = oracle.Layout(Hkv * r, d, 16, 32, 64, 8)
    n = 45
    k = W.kv_tensor(1, (1, n, Hkv, d), 20.0, W.outlier_channels(Hkv, d)).numpy()
    v = W.kv_tensor(2, (1, n, Hkv, d)).numpy()
    bt = np.array([[4, 0, 6]], np.int32)
    pg, pm = np.zeros(Lg.pool_bytes, np.uint8), np.zeros(Lm.pool_bytes, np.uint8)
    oracle.quantize_append(Lg, pg, k, v, bt, np.array([0], np.int32))
    oracle.quantize_append(Lm, pm, np.repeat(k, r, axis=2), np.repeat(v, r, axis=2), bt, np.array([0], np.int32))
    q = W.kv_tensor(3, (1, 1, Hkv * r, d)).numpy()[0]
    og = oracle.decode_attention(Lg, pg, q, bt, np.array([n], np.int32), d ** -0.5)
    om = oracle.decode_attention(Lm, pm, q, bt, np.array([n], np.int32), d ** -0.5)
    assert np.array_equal(og, om)


def test_attention_page_permutation_invariance_and_pow2_scaling():
    L = oracle.Layout(2, 64, 16, 32, 64, 12)
    n = 70
    k = W.kv_tensor(1, (1, n, 2, 64), 20.0, W.outlier_channels(2, 64)).numpy()
    v = W.kv_tensor(2, (1, n, 2, 64)).numpy()
    q = W.kv_tensor(3, (1, 1, 4, 64)).numpy()[0]
    outs = []
    for bt in (np.array([[0, 1, 2, 3, 4]], np.int32), np.array([[11, 3, 7, 0, 5]], np.int32)):
        pool = np.zeros(L.pool_bytes, np.uint8)
        oracle.quantize_append(L, pool, k, v, bt, np.array([0], np.int32))
        outs.append(oracle.decode_attention(L, pool, q, bt, np.array([n], np.int32), 0.125))
    assert np.array_equal(outs[0], outs[1])
    # V x 2 doubles every V scale and keeps the codes, so the output doubles exactly
    pool = np.zeros(L.pool_bytes, np.uint8)
    bt = np.array([[11, 3, 7, 0, 5]], np.int32)
    oracle.quantize_append(L, pool, k, (v.astype(np.float32) * 2).astype(np.float16), bt, np.array([0], np.int32))
    out2 = oracle.decode_attention(L, pool, q, bt, np.array([n], np.int32), 0.125)
    assert np.array_equal(out2, 2 * outs[1])


# ----------------------------------------------------------------------------
# sliding window with sink tokens ("AI inference tuning: KV Cache optimisation and
# memory management" section 3.2): the decode query at position L-1 sees keys
# [max(0, L - W), L) and the first S positions
# ----------------------------------------------------------------------------

def _window_visible(n, window, sinks):
    """Visible key positions of query row i = n - 1, from the page's mask construction."""
    i = n - 1
    mask = np.zeros(n, bool)
    mask[max(0, i - window + 1):i + 1] = True
    if sinks > 0:
        mask[:sinks] = True
    return np.nonzero(mask)[0]


@pytest.mark.parametrize("window,sinks", [(1, 0), (5, 0), (5, 3), (17, 4), (16, 16), (3, 40), (40, 0), (100, 2)])
def test_window_equals_full_attention_on_compacted_cache(window, sinks):
    # the windowed result equals plain decode attention over a cache that holds only the
    # visible rows (re-quantized row by row: the codes are the same), in the same order
    L = oracle.Layout(2, 64, 16, 32, 64, 32)
    lens = [40, 23, 7]
    pool, bt, k, v = _build_cache(L, len(lens), lens, seed=51)
    q = W.kv_tensor(W.SEED_Q + 50, (1, len(lens), 8, 64)).numpy()[0]
    scale = 0.3
    got = oracle.decode_attention_window(L, pool, q, bt, np.array(lens, np.int32), scale, window, sinks)
    for b, n in enumerate(lens):
        vis = _window_visible(n, window, sinks)
        pages = (len(vis) + L.P - 1) // L.P
        bt1 = np.arange(pages, dtype=np.int32)[None, :]
        pool1 = np.zeros(L.pool_bytes, np.uint8)
        oracle.quantize_append(L, pool1, k[b:b + 1, vis], v[b:b + 1, vis], bt1, np.array([0], np.int32))
        ref = oracle.decode_attention(L, pool1, q[b:b + 1], bt1, np.array([len(vis)], np.int32), scale)
        assert np.array_equal(got[b], ref[0]), (b, window, sinks)


def test_window_covering_everything_is_plain_attention():
    L = oracle.Layout(2, 64, 16, 32, 64, 16)
    lens = [1, 33, 17, 0]
    pool, bt, _, _ = _build_cache(L, len(lens), lens, seed=52)
    q = W.kv_tensor(W.SEED_Q + 51, (1, len(lens), 4, 64)).numpy()[0]
    full = oracle.decode_attention(L, pool, q, bt, np.array(lens, np.int32), 0.125)
    for window, sinks in [(0, 0), (0, 5), (33, 0), (1000, 4), (-1, 2)]:
        got = oracle.decode_attention_window(L, pool, q, bt, np.array(lens, np.int32), 0.125, window, sinks)
        assert np.array_equal(got, full), (window, sinks)


def test_window_of_one_returns_the_last_value_row():
    L = oracle.Layout(2, 64, 16, 32, 64, 16)
    lens = [29, 1, 16]
    pool, bt, _, _ = _build_cache(L, len(lens), lens, seed=53)
    q = W.kv_tensor(W.SEED_Q + 52, (1, len(lens), 4, 64)).numpy()[0]
    got = oracle.decode_attention_window(L, pool, q, bt, np.array(lens, np.int32), 0.125, 1, 0)
    for b, n in enumerate(lens):
        _, dv = oracle.dequantize(L, pool, bt, b, n - 1, 1)
        for hq in range(4):
            assert np.array_equal(got[b, hq], dv[0, hq // 2].astype(np.float64))


@pytest.mark.parametrize("window,sinks", [(4, 2), (9, 0), (2, 6), (30, 30)])
def test_window_brute_force(window, sinks):
    # numpy softmax over the page's mask, against the oracle, on tiny inputs with large logits
    L = oracle.Layout(2, 64, 16, 32, 64, 16)
    lens = [26, 11]
    pool, bt, _, _ = _build_cache(L, len(lens), lens, seed=54)
    q = W.kv_tensor(W.SEED_Q + 53, (1, len(lens), 4, 64)).numpy()[0]
    scale = 40.0  # logits far past exp's range: the maximum has to be subtracted
    got = oracle.decode_attention_window(L, pool, q, bt, np.array(lens, np.int32), scale, window, sinks)
    for b, n in enumerate(lens):
        dk, dv = oracle.dequantize(L, pool, bt, b, 0, n)
        vis = _window_visible(n, window, sinks)
        for hq in range(4):
            s = (dk[vis, hq // 2, :].astype(np.float64) @ q[b, hq].astype(np.float64)) * scale
            ref = scipy.special.softmax(s) @ dv[vis, hq // 2, :].astype(np.float64)
            np.testing.assert_allclose(got[b, hq], ref, rtol=1e-10, atol=1e-10)


# ----------------------------------------------------------------------------
# the FP16 cache of the latency comparison ("LLM long-context inference: managing
# the KV cache with an INT4 state machine" section 7.4)
# ----------------------------------------------------------------------------

def _fp16_blocks(L, pool16):
    """The FP16 pool as [page, kv head, K|V, slot, d] fp16 (the layout of the oracle's header)."""
    return pool16.view(np.float16).reshape(L.num_pages, L.Hkv, 2, L.P, L.d)


def test_fp16_append_places_rows_by_page_table():
    L = oracle.Layout(3, 64, 16, 32, 64, 12)
    lens = [37, 5]
    pages = [(n + 15) // 16 for n in lens]
    order = W.permutation(61, L.num_pages).numpy()
    bt = np.full((2, max(pages)), -1, np.int32)
    bt[0, :pages[0]] = order[:pages[0]]
    bt[1, :pages[1]] = order[pages[0]:pages[0] + pages[1]]
    k = W.kv_tensor(61, (2, 37, 3, 64)).numpy()
    v = W.kv_tensor(62, (2, 37, 3, 64)).numpy()
    pool16 = np.zeros(oracle.fp16_pool_bytes(L), np.uint8)
    assert oracle.fp16_block_bytes(64, 16) == 4 * 16 * 64
    for b in range(2):
        oracle.fp16_append(L, pool16, k[b:b + 1, :lens[b]], v[b:b + 1, :lens[b]], bt[b:b + 1], np.array([0], np.int32))
    blocks = _fp16_blocks(L, pool16)
    for b in range(2):
        for t in range(lens[b]):
            pg, sl = bt[b, t // 16], t % 16
            assert np.array_equal(blocks[pg, :, 0, sl], k[b, t])
            assert np.array_equal(blocks[pg, :, 1, sl], v[b, t])


def test_fp16_decode_attention_brute_force():
    L = oracle.Layout(2, 64, 16, 32, 64, 16)
    lens = [40, 1, 17]
    pool16 = np.zeros(oracle.fp16_pool_bytes(L), np.uint8)
    bt = np.arange(9, dtype=np.int32).reshape(3, 3)[:, :3]
    bt = np.array([[4, 0, 8], [2, -1, -1], [7, 5, -1]], np.int32)
    k = W.kv_tensor(63, (3, 40, 2, 64), 20.0, W.outlier_channels(2, 64, seed=3)).numpy()
    v = W.kv_tensor(64, (3, 40, 2, 64)).numpy()
    for b in range(3):
        oracle.fp16_append(L, pool16, k[b:b + 1, :lens[b]], v[b:b + 1, :lens[b]], bt[b:b + 1], np.array([0], np.int32))
    q = W.kv_tensor(65, (1, 3, 8, 64)).numpy()[0]
    got = oracle.fp16_decode_attention(L, pool16, q, bt, np.array(lens, np.int32), 0.2)
    for b in range(3):
        for hq in range(8):
            kh = k[b, :lens[b], hq // 4].astype(np.float64)
            s_ = (kh @ q[b, hq].astype(np.float64)) * 0.2
            ref = scipy.special.softmax(s_) @ v[b, :lens[b], hq // 4].astype(np.float64)
            np.testing.assert_allclose(got[b, hq], ref, rtol=1e-12, atol=1e-12)


def test_dequantize_to_fp16_pool_matches_dequantize():
    L = oracle.Layout(2, 64, 16, 32, 64, 16)
    lens = [33, 16, 7]
    pool, bt, _, _ = _build_cache(L, len(lens), lens, seed=66)
    pool16 = np.zeros(oracle.fp16_pool_bytes(L), np.uint8)
    oracle.dequantize_to_fp16_pool(L, pool, pool16, bt, np.array(lens, np.int32))
    blocks = _fp16_blocks(L, pool16)
    for b, n in enumerate(lens):
        dk, dv = oracle.dequantize(L, pool, bt, b, 0, n, out_fp16=True)
        for t in range(n):
            assert np.array_equal(blocks[bt[b, t // 16], :, 0, t % 16], dk[t])
            assert np.array_equal(blocks[bt[b, t // 16], :, 1, t % 16], dv[t])


def test_fp16_attention_equals_int4_attention_when_dequant_is_exact():
    # every group's amax is 7 * 2^k, so every scale is a power of two and every
    # dequantized value is exact in fp16: attention over the FP16 pool built by
    # dequantize_to_fp16_pool must equal the INT4 attention bit for bit
    L = oracle.Layout(2, 64, 16, 32, 64, 12)
    lens = [45, 19]
    rng = np.random.default_rng(67)
    n = max(lens)
    k = rng.standard_normal((2, n, 2, 64)).astype(np.float16)
    v = rng.standard_normal((2, n, 2, 64)).astype(np.float16)
    for x, G in ((k, 32), (v, 64)):
        g = x.reshape(2, n, 2, 64 // G, G)
        e = rng.integers(-2, 3, size=g.shape[:-1])
        g[...] = np.clip(g, -0.9, 0.9) * (7.0 * 2.0 ** e)[..., None] / 0.9 * 0.5
        g[..., 0] = (7.0 * 2.0 ** e).astype(np.float16)
    pool = np.zeros(L.pool_bytes, np.uint8)
    bt = np.array([[3, 9, 0], [5, 1, -1]], np.int32)
    for b in range(2):
        oracle.quantize_append(L, pool, k[b:b + 1, :lens[b]], v[b:b + 1, :lens[b]], bt[b:b + 1], np.array([0], np.int32))
    pool16 = np.zeros(oracle.fp16_pool_bytes(L), np.uint8)
    oracle.dequantize_to_fp16_pool(L, pool, pool16, bt, np.array(lens, np.int32))
    q = W.kv_tensor(68, (1, 2, 4, 64)).numpy()[0]
    a = oracle.decode_attention(L, pool, q, bt, np.array(lens, np.int32), 0.125)
    b_ = oracle.fp16_decode_attention(L, pool16, q, bt, np.array(lens, np.int32), 0.125)
    assert np.array_equal(a, b_)


def test_fp16_single_token_returns_its_value():
    L = oracle.Layout(1, 64, 16, 32, 64, 2)
    pool16 = np.zeros(oracle.fp16_pool_bytes(L), np.uint8)
    k = W.kv_tensor(69, (1, 1, 1, 64)).numpy()
    v = W.kv_tensor(70, (1, 1, 1, 64)).numpy()
    bt = np.array([[1]], np.int32)
    oracle.fp16_append(L, pool16, k, v, bt, np.array([0], np.int32))
    q = W.kv_tensor(71, (1, 1, 2, 64)).numpy()[0]
    got = oracle.fp16_decode_attention(L, pool16, q, bt, np.array([1], np.int32), 0.125)
    assert np.array_equal(got[0, 0], v[0, 0, 0].astype(np.float64))
    assert np.array_equal(got[0, 1], v[0, 0, 0].astype(np.float64))


# ----------------------------------------------------------------------------
# mixed precision ("LLM long-context inference: managing the KV cache with an INT4
# state machine" section 8.3): positions before len - residual from the INT4 pool,
# the last `residual` from the FP16 pool
# ----------------------------------------------------------------------------

def _mixed_setup(seed, lens, Hkv=2, d=64, P=16):
    L = oracle.Layout(Hkv, d, P, 32, 64, 24)
    pool, bt, k, v = _build_cache(L, len(lens), lens, seed=seed)
    # the FP16 pool: its own pages and block table, holding every position
    n16 = 20
    pool16 = np.zeros(n16 * Hkv * oracle.fp16_block_bytes(d, P), np.uint8)
    L16 = oracle.Layout(Hkv, d, P, 32, 64, n16)
    pages = [(n + P - 1) // P for n in lens]
    order = W.permutation(seed + 77, n16).numpy()
    bt16 = np.full((len(lens), max(pages)), -1, np.int32)
    kk = 0
    for b, n in enumerate(pages):
        bt16[b, :n] = order[kk:kk + n]
        kk += n
    for b, n in enumerate(lens):
        if n:
            oracle.fp16_append(L16, pool16, k[b:b + 1, :n], v[b:b + 1, :n], bt16[b:b + 1], np.array([0], np.int32))
    q = W.kv_tensor(seed + 5, (1, len(lens), 2 * Hkv, d)).numpy()[0]
    return L, L16, pool, bt, pool16, bt16, n16, k, v, q


def test_mixed_residual_zero_is_int4_attention_and_large_residual_is_fp16():
    lens = [37, 16, 1, 0]
    L, L16, pool, bt, pool16, bt16, n16, _, _, q = _mixed_setup(91, lens)
    sl = np.array(lens, np.int32)
    int4 = oracle.decode_attention(L, pool, q, bt, sl, 0.2)
    fp16 = oracle.fp16_decode_attention(L16, pool16, q, bt16, sl, 0.2)
    assert np.array_equal(oracle.mixed_decode_attention(L, pool, bt, pool16, bt16, n16, q, sl, 0, 0.2), int4)
    for r in (37, 100):
        assert np.array_equal(oracle.mixed_decode_attention(L, pool, bt, pool16, bt16, n16, q, sl, r, 0.2), fp16)


@pytest.mark.parametrize("residual", [1, 5, 16, 20, 36])
def test_mixed_brute_force(residual):
    lens = [37, 23]
    L, L16, pool, bt, pool16, bt16, n16, k, v, q = _mixed_setup(92 + residual, lens)
    scale = 25.0  # large logits: the maximum must be subtracted
    got = oracle.mixed_decode_attention(L, pool, bt, pool16, bt16, n16, q, np.array(lens, np.int32), residual, scale)
    for b, n in enumerate(lens):
        split = max(n - residual, 0)
        dk, dv = oracle.dequantize(L, pool, bt, b, 0, n)
        kk = np.concatenate([dk[:split].astype(np.float64), k[b, split:n].astype(np.float64)])
        vv = np.concatenate([dv[:split].astype(np.float64), v[b, split:n].astype(np.float64)])
        for hq in range(4):
            s_ = (kk[:, hq // 2] @ q[b, hq].astype(np.float64)) * scale
            ref = scipy.special.softmax(s_) @ vv[:, hq // 2]
            np.testing.assert_allclose(got[b, hq], ref, rtol=1e-10, atol=1e-10)


# ----------------------------------------------------------------------------
# INT8 per-row codec ("AI inference tuning: KV Cache optimisation and memory
# management" section 3.1, KVCacheQuantizer.quantize_int8)
# ----------------------------------------------------------------------------

def test_int8_worked_examples():
    # amax 127: the scale is exactly 1 and the codes are the values rounded, ties to even
    x = np.zeros(64, np.float16)
    x[:6] = [127.0, -127.0, 2.5, 3.5, -2.5, 0.49]
    codes, s = oracle.int8_quantize_row(x)
    assert s == 1.0
    assert codes[:6].tolist() == [127, -127, 2, 4, -2, 0]
    # an all-zero row takes the floor scale 1e-8 and zero codes
    codes, s = oracle.int8_quantize_row(np.zeros(64, np.float16))
    assert s == float(np.float32(1e-8)) and not codes.any()
    # a single nonzero value maps to +-127
    x = np.zeros(64, np.float16)
    x[7] = -0.3
    codes, s = oracle.int8_quantize_row(x)
    assert codes[7] == -127 and np.count_nonzero(codes) == 1


def test_int8_codes_are_nearest_within_range():
    rng = np.random.default_rng(101)
    for _ in range(200):
        x = (rng.standard_normal(128) * rng.uniform(0.01, 50)).astype(np.float16)
        codes, s = oracle.int8_quantize_row(x)
        amax = float(np.abs(x.astype(np.float64)).max())
        assert abs(s - amax / 127) <= 2 ** -23 * s  # the fp32 quotient
        assert codes.min() >= -128 and codes.max() <= 127
        assert np.abs(codes).max() == 127
        # brute force: every code is the integer nearest to x / s (f64), except where the
        # quotient lies within fp32 rounding (the definition divides in fp32) of a tie
        y = x.astype(np.float64) / s
        cand = np.arange(-128, 128)
        best = cand[np.argmin(np.abs(y[:, None] - cand[None, :]), axis=1)]
        tie = np.abs(np.abs(y - np.floor(y)) - 0.5) < 2.0 ** -22 * np.maximum(np.abs(y), 1.0)
        assert np.array_equal(codes[~tie], best[~tie])
        # half a step, plus the fp32 rounding of a quotient up to 127
        assert np.all(np.abs(x.astype(np.float64) - codes * np.float64(s)) <= s * (0.5 + 127 * 2.0 ** -23))


def test_int8_layout_and_dequantize():
    L = oracle.Layout(2, 64, 16, 32, 64, 6)
    assert oracle.int8_block_bytes(64, 16) == 2 * 16 * 64 + 8 * 16
    k = W.kv_tensor(111, (1, 20, 2, 64)).numpy()
    v = W.kv_tensor(112, (1, 20, 2, 64)).numpy()
    bt = np.array([[4, 1]], np.int32)
    pool8 = np.zeros(oracle.int8_pool_bytes(L), np.uint8)
    oracle.int8_quantize_append(L, pool8, k, v, bt, np.array([0], np.int32))
    blocks = pool8.reshape(L.num_pages, L.Hkv, -1)
    dk, dv = oracle.int8_dequantize(L, pool8, bt, 0, 0, 20)
    for t in range(20):
        for h in range(2):
            blk = blocks[bt[0, t // 16], h]
            ck, sk = oracle.int8_quantize_row(k[0, t, h])
            cv, sv = oracle.int8_quantize_row(v[0, t, h])
            assert np.array_equal(blk[(t % 16) * 64:(t % 16 + 1) * 64].view(np.int8), ck)
            assert np.array_equal(blk[(16 + t % 16) * 64:(17 + t % 16) * 64].view(np.int8), cv)
            assert blk[2048 + 4 * (t % 16):2052 + 4 * (t % 16)].view(np.float32)[0] == np.float32(sk)
            assert blk[2048 + 64 + 4 * (t % 16):2052 + 64 + 4 * (t % 16)].view(np.float32)[0] == np.float32(sv)
            assert np.array_equal(dk[t, h], ck.astype(np.float32) * np.float32(sk))
            assert np.array_equal(dv[t, h], cv.astype(np.float32) * np.float32(sv))


def test_int8_attention_brute_force_and_exact_case():
    L = oracle.Layout(2, 64, 16, 32, 64, 8)
    lens = [30, 9]
    bt = np.array([[3, 0], [6, -1]], np.int32)
    k = W.kv_tensor(113, (2, 30, 2, 64), 20.0, W.outlier_channels(2, 64, seed=9)).numpy()
    v = W.kv_tensor(114, (2, 30, 2, 64)).numpy()
    pool8 = np.zeros(oracle.int8_pool_bytes(L), np.uint8)
    for b in range(2):
        oracle.int8_quantize_append(L, pool8, k[b:b + 1, :lens[b]], v[b:b + 1, :lens[b]], bt[b:b + 1],
                                    np.array([0], np.int32))
    q = W.kv_tensor(115, (1, 2, 4, 64)).numpy()[0]
    got = oracle.int8_decode_attention(L, pool8, q, bt, np.array(lens, np.int32), 30.0)
    for b in range(2):
        dk, dv = oracle.int8_dequantize(L, pool8, bt, b, 0, lens[b])
        for hq in range(4):
            s_ = (dk[:, hq // 2].astype(np.float64) @ q[b, hq].astype(np.float64)) * 30.0
            ref = scipy.special.softmax(s_) @ dv[:, hq // 2].astype(np.float64)
            np.testing.assert_allclose(got[b, hq], ref, rtol=1e-10, atol=1e-10)
    # integer rows holding +-127: scale 1, codes equal the values, so the INT8 attention
    # equals the FP16 attention over the same rows bit for bit
    rng = np.random.default_rng(116)
    ki = rng.integers(-127, 128, size=(2, 30, 2, 64)).astype(np.float16)
    vi = rng.integers(-127, 128, size=(2, 30, 2, 64)).astype(np.float16)
    ki[..., 0] = 127
    vi[..., 1] = -127
    pool8 = np.zeros(oracle.int8_pool_bytes(L), np.uint8)
    pool16 = np.zeros(oracle.fp16_pool_bytes(L), np.uint8)
    for b in range(2):
        oracle.int8_quantize_append(L, pool8, ki[b:b + 1, :lens[b]], vi[b:b + 1, :lens[b]], bt[b:b + 1],
                                    np.array([0], np.int32))
        oracle.fp16_append(L, pool16, ki[b:b + 1, :lens[b]], vi[b:b + 1, :lens[b]], bt[b:b + 1],
                           np.array([0], np.int32))
    a = oracle.int8_decode_attention(L, pool8, q, bt, np.array(lens, np.int32), 0.01)
    f = oracle.fp16_decode_attention(L, pool16, q, bt, np.array(lens, np.int32), 0.01)
    assert np.array_equal(a, f)


# ----------------------------------------------------------------------------
# The rotated 4-bit codec ("LARQL KV cache engines", engine three codec/turbo-quant:
# Walsh-Hadamard rotation, Lloyd-Max quantization, per-row cosine about 0.9954 at
# 4 bits)
# ----------------------------------------------------------------------------

# J. Max, "Quantizing for minimum distortion", IRE Trans. Information Theory IT-6
# (1960), table for the normal law: the positive output levels of the minimum mean
# square error quantizer with 8 and 16 levels (four decimals) and its distortion.
MAX_1960 = {
    3: ([0.2451, 0.7560, 1.3440, 2.1520], 0.03455),
    4: ([0.1284, 0.3881, 0.6568, 0.9424, 1.2562, 1.6180, 2.0690, 2.7326], 0.009497),
}


def _cell_stats(levels, thresholds):
    """Mass, mean and distortion of N(0,1) per cell, by quadrature (independent of the oracle)."""
    import scipy.integrate
    import scipy.stats
    edges = np.concatenate([[-np.inf], thresholds, [np.inf]])
    pdf = scipy.stats.norm.pdf
    mass, mean, dist = [], [], 0.0
    for j, lv in enumerate(levels):
        a, b = edges[j], edges[j + 1]
        m = scipy.integrate.quad(pdf, a, b, epsabs=1e-14, epsrel=1e-13)[0]
        mu = scipy.integrate.quad(lambda t: t * pdf(t), a, b, epsabs=1e-14, epsrel=1e-13)[0] / m
        dist += scipy.integrate.quad(lambda t: (t - lv) ** 2 * pdf(t), a, b, epsabs=1e-14, epsrel=1e-13)[0]
        mass.append(m)
        mean.append(mu)
    return np.array(mass), np.array(mean), dist


@pytest.mark.parametrize("bits", [3, 4])
def test_lloyd_max_matches_the_published_table(bits):
    lv, tb = oracle.lloyd_max_normal(bits)
    pos, mse = MAX_1960[bits]
    n = 1 << bits
    assert np.all(np.diff(lv) > 0)
    np.testing.assert_allclose(lv[n // 2:], pos, atol=1.5e-4)
    np.testing.assert_allclose(lv[:n // 2], -np.array(pos[::-1]), atol=1.5e-4)
    _, _, dist = _cell_stats(lv, tb)
    assert abs(dist - mse) <= 2e-3 * mse


@pytest.mark.parametrize("bits", [3, 4])
def test_lloyd_max_optimality_conditions(bits):
    lv, tb = oracle.lloyd_max_normal(bits)
    # nearest-neighbour condition: thresholds are the midpoints of adjacent levels
    np.testing.assert_allclose(tb, 0.5 * (lv[:-1] + lv[1:]), rtol=0, atol=1e-15)
    # centroid condition: every level is the mean of the normal law on its cell
    _, mean, _ = _cell_stats(lv, tb)
    np.testing.assert_allclose(lv, mean, rtol=1e-10, atol=1e-12)
    # symmetric law, antisymmetric quantizer, the middle threshold exactly at 0
    assert np.array_equal(lv, -lv[::-1]) and tb[len(tb) // 2] == 0.0


def test_wht4_tables_are_the_codebook_in_fp32():
    c, t = oracle.wht4_tables()
    lv, tb = oracle.lloyd_max_normal(4)
    assert np.array_equal(c, lv.astype(np.float32)) and np.array_equal(t, tb.astype(np.float32))
    # every fp64 value lies well inside its fp32 rounding interval, so any implementation
    # that reaches the fixed point to 1e-12 rounds it to the same fp32 value
    for arr in (lv, tb[tb != 0]):
        f = arr.astype(np.float32)
        up = np.nextafter(f, np.float32(np.inf)).astype(np.float64)
        dn = np.nextafter(f, np.float32(-np.inf)).astype(np.float64)
        f = f.astype(np.float64)
        margin = np.minimum(np.abs(arr - (f + up) / 2), np.abs(arr - (f + dn) / 2)) / np.abs(arr)
        assert margin.min() > 1e-10


def test_wht_is_the_hadamard_matrix():
    import scipy.linalg
    H = scipy.linalg.hadamard(128).astype(np.float64)  # Sylvester order
    rng = np.random.default_rng(201)
    # integer rows: every partial sum is exact in fp32, so the fast transform equals H x exactly
    for _ in range(20):
        x = rng.integers(-1000, 1001, size=128).astype(np.float32)
        assert np.array_equal(oracle.wht_f32(x).astype(np.float64), H @ x.astype(np.float64))
    x = rng.standard_normal(128).astype(np.float32)
    y = oracle.wht_f32(x).astype(np.float64)
    np.testing.assert_allclose(y, H @ x.astype(np.float64), rtol=0, atol=1e-5 * np.linalg.norm(x))
    # H H = d I
    np.testing.assert_allclose(oracle.wht_f32(oracle.wht_f32(x)), 128 * x, rtol=0, atol=1e-4)


def test_wht4_worked_example():
    # x = e_0 + e_1: (Hx)_i = 1 + H[i][1] = 2 (i even) or 0 (i odd); sigma = |x| = sqrt 2, so
    # u = sqrt 2 = 1.41421 on even i and 0 on odd i.  The thresholds at or below sqrt 2 are the
    # twelve up to (L_11 + L_12) / 2 = 1.0993 (the next one, (L_12 + L_13) / 2 = 1.4371, is above):
    # code 12; u = 0 meets the middle threshold 0 itself: code 8.  Bytes: 12 | 8 << 4 = 0x8C.
    x = np.zeros(128, np.float16)
    x[:2] = 1.0
    codes, s = oracle.wht4_quantize_row(x)
    assert s == np.float32(np.sqrt(np.float32(2.0)))
    assert np.all(codes == 0x8C)
    # an all-zero row: sigma 0 and codes 0, which dequantize to zeros
    codes, s = oracle.wht4_quantize_row(np.zeros(128, np.float16))
    assert s == 0.0 and not codes.any()


def test_wht4_codes_are_nearest_levels():
    import scipy.linalg
    H = scipy.linalg.hadamard(128).astype(np.float64)
    lv, tb = oracle.lloyd_max_normal(4)
    rng = np.random.default_rng(202)
    for i in range(100):
        x = (rng.standard_normal(128) * rng.uniform(0.01, 30)).astype(np.float16)
        if i % 3 == 0:
            x[rng.integers(0, 128, 3)] *= 20  # outlier channels
        codes, s = oracle.wht4_quantize_row(x)
        xd = x.astype(np.float64)
        assert abs(s - np.linalg.norm(xd)) <= 2e-6 * np.linalg.norm(xd)
        nib = np.stack([codes & 15, codes >> 4], axis=1).reshape(-1)  # element 2j in the low nibble
        u = (H @ xd) / np.linalg.norm(xd)
        best = np.argmin(np.abs(u[:, None] - lv[None, :]), axis=1)
        near = np.min(np.abs(u[:, None] - tb[None, :]), axis=1) < 1e-5
        assert np.array_equal(nib[~near], best[~near])


def _wht4_case(seed, lens, Hkv=2, P=16, pages=10):
    L = oracle.Layout(Hkv, 128, P, 64, 128, pages)
    n = max(lens)
    k = W.kv_tensor(seed, (len(lens), n, Hkv, 128), 20.0, W.outlier_channels(Hkv, 128, seed=seed + 1)).numpy()
    v = W.kv_tensor(seed + 2, (len(lens), n, Hkv, 128)).numpy()
    perm = np.random.default_rng(seed + 3).permutation(pages).astype(np.int32)
    mb = (n + P - 1) // P
    bt = np.full((len(lens), mb), -1, np.int32)
    used = 0
    for b, m in enumerate(lens):
        np_ = (m + P - 1) // P
        bt[b, :np_] = perm[used:used + np_]
        used += np_
    pool = np.zeros(oracle.wht4_pool_bytes(L), np.uint8)
    for b, m in enumerate(lens):
        oracle.wht4_quantize_append(L, pool, k[b:b + 1, :m], v[b:b + 1, :m], bt[b:b + 1], np.array([0], np.int32))
    return L, pool, bt, k, v


def test_wht4_layout_and_dequantize():
    import scipy.linalg
    H = scipy.linalg.hadamard(128).astype(np.float64)
    c, _ = oracle.wht4_tables()
    assert oracle.wht4_block_bytes(128, 16) == 16 * (128 + 8)
    L, pool, bt, k, v = _wht4_case(211, [20])
    blocks = pool.reshape(L.num_pages, L.Hkv, -1)
    dk, dv = oracle.wht4_dequantize(L, pool, bt, 0, 0, 20)
    for t in range(20):
        for h in range(2):
            blk = blocks[bt[0, t // 16], h]
            s = t % 16
            ck, sk = oracle.wht4_quantize_row(k[0, t, h])
            cv, sv = oracle.wht4_quantize_row(v[0, t, h])
            assert np.array_equal(blk[s * 64:(s + 1) * 64], ck)
            assert np.array_equal(blk[(16 + s) * 64:(17 + s) * 64], cv)
            assert blk[2048 + 4 * s:2052 + 4 * s].view(np.float32)[0] == np.float32(sk)
            assert blk[2112 + 4 * s:2116 + 4 * s].view(np.float32)[0] == np.float32(sv)
            for codes, sg, got in ((ck, sk, dk[t, h]), (cv, sv, dv[t, h])):
                nib = np.stack([codes & 15, codes >> 4], axis=1).reshape(-1)
                ref = H @ (np.float32(sg) * c[nib]).astype(np.float64) / 128
                np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-7 * max(sg, 1e-30))


def test_wht4_round_trip_cosine():
    # rows of N(0, 1) values: after the rotation the coordinates over the row RMS are close to
    # N(0, 1), so the per-row cosine is near sqrt(1 - D16), D16 = 0.009497 the Lloyd-Max
    # distortion (0.99524); the page reports about 0.9954 at 4 bits
    L, pool, bt, k, v = _wht4_case(212, [1000], Hkv=4, pages=63)
    dk, dv = oracle.wht4_dequantize(L, pool, bt, 0, 0, 1000)
    x = v[0, :1000].astype(np.float64)
    xh = dv.astype(np.float64)
    cos = (x * xh).sum(-1) / np.linalg.norm(x, axis=-1) / np.linalg.norm(xh, axis=-1)
    assert 0.9945 <= cos.mean() <= 0.9960, cos.mean()
    assert cos.min() > 0.985
    rel_mse = ((x - xh) ** 2).sum() / (x ** 2).sum()
    assert 0.0085 <= rel_mse <= 0.0105, rel_mse


def test_wht4_attention_brute_force_and_exact_case():
    lens = [37, 5]
    L, pool, bt, k, v = _wht4_case(213, lens)
    q = W.kv_tensor(214, (1, 2, 4, 128)).numpy()[0]
    got = oracle.wht4_decode_attention(L, pool, q, bt, np.array(lens, np.int32), 0.3)
    for b, n in enumerate(lens):
        dk, dv = oracle.wht4_dequantize(L, pool, bt, b, 0, n)
        for hq in range(4):
            s_ = (dk[:, hq // 2].astype(np.float64) @ q[b, hq].astype(np.float64)) * 0.3
            ref = scipy.special.softmax(s_) @ dv[:, hq // 2].astype(np.float64)
            np.testing.assert_allclose(got[b, hq], ref, rtol=2e-6, atol=2e-7)
    # one position: the output is that position's dequantized V row
    got1 = oracle.wht4_decode_attention(L, pool, q, bt, np.array([1, 1], np.int32), 5.0)
    for b in range(2):
        _, dv = oracle.wht4_dequantize(L, pool, bt, b, 0, 1)
        for hq in range(4):
            np.testing.assert_allclose(got1[b, hq], dv[0, hq // 2].astype(np.float64), rtol=1e-6, atol=1e-7)


def test_wht4_attention_in_the_rotated_domain():
    # the decode kernel never forms a dequantized row: with x = H (sigma c) / d and H
    # symmetric, q . x = (H q / d) . (sigma c), and sum_t p_t x_t = H (sum_t p_t sigma_t c_t) / d.
    # Taken that way from the stored codes and norms, with each sigma * c rounded to fp32 as
    # the dequantized row defines it, the scores and weighted sum give the oracle's attention
    # to fp64 rounding; with sigma applied after the reduction, as the kernel does, they agree
    # to the fp32 rounding of those products.
    import scipy.linalg
    H = scipy.linalg.hadamard(128).astype(np.float64)
    levels, _ = oracle.wht4_tables()
    lens = [45, 16]
    L, pool, bt, _, _ = _wht4_case(215, lens)
    q = W.kv_tensor(216, (1, 2, 4, 128)).numpy()[0]
    scale = 0.2
    want = oracle.wht4_decode_attention(L, pool, q, bt, np.array(lens, np.int32), scale)
    blocks = pool.reshape(L.num_pages, L.Hkv, -1)
    for b, n in enumerate(lens):
        for hq in range(4):
            h = hq // 2
            qr = H @ q[b, hq].astype(np.float64) / 128
            ck, cv, sk, sv = [], [], [], []
            for t in range(n):
                blk, s_ = blocks[bt[b, t // 16], h], t % 16
                for base, out in ((s_ * 64, ck), ((16 + s_) * 64, cv)):
                    by = blk[base:base + 64]
                    out.append(levels[np.stack([by & 15, by >> 4], axis=1).reshape(-1)].astype(np.float64))
                sk.append(float(blk[2048 + 4 * s_:2052 + 4 * s_].view(np.float32)[0]))
                sv.append(float(blk[2112 + 4 * s_:2116 + 4 * s_].view(np.float32)[0]))
            ck, cv = np.array(ck), np.array(cv)
            sk, sv = np.array(sk)[:, None], np.array(sv)[:, None]
            xk = (sk.astype(np.float32) * ck.astype(np.float32)).astype(np.float64)  # fp32 products
            xv = (sv.astype(np.float32) * cv.astype(np.float32)).astype(np.float64)
            p = scipy.special.softmax((xk @ qr) * scale)
            np.testing.assert_allclose(H @ (p @ xv) / 128, want[b, hq], rtol=1e-9, atol=1e-12)
            p = scipy.special.softmax(sk[:, 0] * (ck @ qr) * scale)
            got = H @ ((p * sv[:, 0]) @ cv) / 128
            # bound: each fp32 product is off by at most 2^-24 of itself, which moves an
            # output element by at most 2^-24 mean|sigma c| through the transform, and a
            # score by at most scale 2^-24 sum|H q / d| |sigma c|, which moves the
            # softmax-weighted mean by at most 2 max|dz| max|x|
            u = 2.0 ** -24
            dz = scale * u * (np.abs(xk) @ np.abs(qr)).max()
            bound = u * np.abs(xv).mean(1).max() + 2 * dz * np.abs(xv @ H / 128).max()
            assert np.abs(got - want[b, hq]).max() <= bound

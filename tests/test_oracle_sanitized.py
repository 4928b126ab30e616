"""The oracle under AddressSanitizer and UndefinedBehaviorSanitizer (no GPU needed).

An out-of-bounds read or an undefined operation in the C oracle could still give
plausible numbers, so its pins and the edge cases below are re-run against a build of
the same source with both sanitizers, which stop at the first fault.
"""
from __future__ import annotations

import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _layout_and_table(Hkv, d, P, Gk, Gv, lens):
    import oracle
    B = len(lens)
    mb = max(1, -(-max(lens) // P)) + 1
    npg = B * mb + 2
    L = oracle.Layout(Hkv, d, P, Gk, Gv, npg)
    bt = np.full((B, mb), -1, np.int32)
    k = 0
    for b, n in enumerate(lens):
        m = -(-n // P)
        bt[b, :m] = np.arange(k, k + m)
        k += m
    return L, bt, npg


@pytest.mark.parametrize("Hkv,d,P,Gk,Gv,r", [(2, 128, 16, 64, 128, 4), (1, 64, 32, 32, 64, 1), (2, 256, 64, 128, 32, 2)])
def test_every_oracle_call_on_edge_cases(Hkv, d, P, Gk, Gv, r):
    # empty and one-token sequences, a page boundary either side, windows and sinks longer
    # than the sequence, residuals beyond it, and zero / subnormal / largest-fp16 groups
    import oracle
    rng = np.random.default_rng(d + P)
    lens = [0, 1, P, P + 1, 3 * P - 1]
    L, bt, npg = _layout_and_table(Hkv, d, P, Gk, Gv, lens)
    sl = np.array(lens, np.int32)
    B, n_max = len(lens), max(lens)
    K = rng.standard_normal((B, n_max, Hkv, d)).astype(np.float16)
    V = rng.standard_normal((B, n_max, Hkv, d)).astype(np.float16)
    q = rng.standard_normal((B, Hkv * r, d)).astype(np.float16)
    s = 1.0 / np.sqrt(d)
    pool = np.zeros(L.pool_bytes, np.uint8)
    for b, n in enumerate(lens):
        for t in range(n):
            oracle.quantize_append(L, pool, K[b:b + 1, t:t + 1], V[b:b + 1, t:t + 1], bt[b:b + 1],
                                   np.array([t], np.int32))
    out = oracle.decode_attention(L, pool, q, bt, sl, s)
    assert not out[0].any() and np.isfinite(out).all()  # an empty sequence gives zeros
    for w, sk in [(0, 0), (1, 0), (5, 2), (1000, 1000), (3, 100)]:
        assert np.isfinite(oracle.decode_attention_window(L, pool, q, bt, sl, s, w, sk)).all()
    for b, n in enumerate(lens):
        oracle.dequantize(L, pool, bt, b, 0, n)
        oracle.dequantize(L, pool, bt, b, 0, n, True)
    p16 = np.zeros(oracle.fp16_pool_bytes(L), np.uint8)
    oracle.dequantize_to_fp16_pool(L, pool, p16, bt, sl)
    oracle.fp16_decode_attention(L, p16, q, bt, sl, s)
    for res in (0, 1, P, 10 * P):
        oracle.mixed_decode_attention(L, pool, bt, p16, bt, npg, q, sl, res, s)
    p8 = np.zeros(oracle.int8_pool_bytes(L), np.uint8)
    for b, n in enumerate(lens):
        if n:
            oracle.int8_quantize_append(L, p8, K[b:b + 1, :n], V[b:b + 1, :n], bt[b:b + 1], np.zeros(1, np.int32))
            oracle.int8_dequantize(L, p8, bt, b, 0, n)
    oracle.int8_decode_attention(L, p8, q, bt, sl, s)
    if d == 128:
        p4 = np.zeros(oracle.wht4_pool_bytes(L), np.uint8)
        for b, n in enumerate(lens):
            if n:
                oracle.wht4_quantize_append(L, p4, K[b:b + 1, :n], V[b:b + 1, :n], bt[b:b + 1], np.zeros(1, np.int32))
                oracle.wht4_dequantize(L, p4, bt, b, 0, n)
        oracle.wht4_decode_attention(L, p4, q, bt, sl, s)
    z = np.zeros((1, 1, Hkv, d), np.float16)
    z[..., :3] = np.float16(6e-8)
    z[..., -1] = np.float16(65504)
    oracle.quantize_append(L, pool, z, -z, bt[1:2], np.zeros(1, np.int32))
    for bits in (1, 2, 3, 4):
        oracle.lloyd_max_normal(bits)


def test_oracle_under_address_and_undefined_behaviour_sanitizers(tmp_path):
    if os.environ.get("KVQ_ORACLE_SANITIZED"):
        pytest.skip("already running under the sanitizers")
    asan = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True, text=True).stdout.strip()
    if not os.path.isabs(asan) or not os.path.exists(asan):
        pytest.skip("gcc has no AddressSanitizer runtime here")
    sys.path.insert(0, ROOT)
    from oracle import build as ob
    lib = ob.build(out=str(tmp_path / "libkvq_oracle_san.so"), force=True,
                   extra_flags=["-g", "-fsanitize=address,undefined", "-fno-sanitize-recover=undefined",
                                "-fno-omit-frame-pointer"])
    env = dict(os.environ, KVQ_ORACLE_LIB=lib, KVQ_ORACLE_SANITIZED="1", LD_PRELOAD=asan,
               ASAN_OPTIONS="detect_leaks=0:abort_on_error=1", UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1",
               PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"), os.path.abspath(__file__)],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    assert " passed" in r.stdout and "runtime error" not in r.stderr and "AddressSanitizer" not in r.stderr

"""The oracle: a plain, slow, single-threaded CPU statement of the INT4
group-quantized paged KV cache (quantize-on-append, dequantize, decode
attention in fp64).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
never does, and this package imports nothing from the product.

The arithmetic lives in ``kvq_oracle.c`` (see its header for the cited
passages and the layout it restates).  This module only marshals numpy arrays
into that library through ctypes.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(worked examples, closed forms, invariants and brute force); none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None


def lib() -> C.CDLL:
    """The oracle library.  KVQ_ORACLE_LIB may name another build of the same source
    (the planted-mistake tests use it to load deliberately broken copies)."""
    global _lib
    if _lib is None:
        path = os.environ.get("KVQ_ORACLE_LIB") or _build.build()
        L = C.CDLL(path)
        L.kvq_oracle_f32_to_f16.argtypes = [C.c_float]
        L.kvq_oracle_f32_to_f16.restype = C.c_uint16
        L.kvq_oracle_f16_to_f64.argtypes = [C.c_uint16]
        L.kvq_oracle_f16_to_f64.restype = C.c_double
        L.kvq_oracle_f32_to_f16_array.argtypes = [C.c_void_p, C.c_void_p, C.c_size_t]
        L.kvq_oracle_f32_to_f16_array.restype = None
        L.kvq_oracle_f16_to_f64_array.argtypes = [C.c_void_p, C.c_void_p, C.c_size_t]
        L.kvq_oracle_f16_to_f64_array.restype = None
        L.kvq_oracle_block_bytes.argtypes = [C.c_int] * 4
        L.kvq_oracle_block_bytes.restype = C.c_size_t
        L.kvq_oracle_fp16_kv_bytes.argtypes = [C.c_int, C.c_int, C.c_int, C.c_double]
        L.kvq_oracle_fp16_kv_bytes.restype = C.c_double
        L.kvq_oracle_quantize_group.argtypes = [C.c_void_p, C.c_int, C.c_void_p, C.c_void_p]
        L.kvq_oracle_quantize_group.restype = None
        L.kvq_oracle_quantize_append.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int,
                                                 C.c_void_p] + [C.c_int] * 8
        L.kvq_oracle_quantize_append.restype = C.c_int
        L.kvq_oracle_dequantize.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int,
                                            C.c_void_p, C.c_void_p, C.c_int] + [C.c_int] * 6
        L.kvq_oracle_dequantize.restype = C.c_int
        L.kvq_oracle_decode_attention.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_void_p,
                                                  C.c_int, C.c_int, C.c_double, C.c_void_p] + [C.c_int] * 6
        L.kvq_oracle_decode_attention.restype = C.c_int
        L.kvq_oracle_decode_attention_window.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_void_p,
                                                         C.c_int, C.c_int, C.c_double, C.c_int, C.c_int,
                                                         C.c_void_p] + [C.c_int] * 6
        L.kvq_oracle_decode_attention_window.restype = C.c_int
        L.kvq_oracle_fp16_block_bytes.argtypes = [C.c_int, C.c_int]
        L.kvq_oracle_fp16_block_bytes.restype = C.c_size_t
        L.kvq_oracle_fp16_append.argtypes = [C.c_void_p] * 4 + [C.c_int, C.c_void_p] + [C.c_int] * 6
        L.kvq_oracle_fp16_append.restype = C.c_int
        L.kvq_oracle_dequantize_to_fp16_pool.argtypes = [C.c_void_p] * 3 + [C.c_int, C.c_void_p] + [C.c_int] * 7
        L.kvq_oracle_dequantize_to_fp16_pool.restype = C.c_int
        L.kvq_oracle_fp16_decode_attention.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_void_p,
                                                       C.c_int, C.c_int, C.c_double, C.c_void_p] + [C.c_int] * 4
        L.kvq_oracle_fp16_decode_attention.restype = C.c_int
        L.kvq_oracle_mixed_decode_attention.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_void_p, C.c_void_p,
                                                        C.c_int, C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int,
                                                        C.c_double, C.c_void_p] + [C.c_int] * 7
        L.kvq_oracle_mixed_decode_attention.restype = C.c_int
        L.kvq_oracle_int8_block_bytes.argtypes = [C.c_int, C.c_int]
        L.kvq_oracle_int8_block_bytes.restype = C.c_size_t
        L.kvq_oracle_int8_quantize_row.argtypes = [C.c_void_p, C.c_int, C.c_void_p, C.c_void_p]
        L.kvq_oracle_int8_quantize_row.restype = None
        L.kvq_oracle_int8_quantize_append.argtypes = [C.c_void_p] * 4 + [C.c_int, C.c_void_p] + [C.c_int] * 6
        L.kvq_oracle_int8_quantize_append.restype = C.c_int
        L.kvq_oracle_int8_dequantize.argtypes = [C.c_void_p, C.c_void_p] + [C.c_int] * 4 + [C.c_void_p] * 2 + \
            [C.c_int] * 4
        L.kvq_oracle_int8_dequantize.restype = C.c_int
        L.kvq_oracle_int8_decode_attention.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_void_p,
                                                       C.c_int, C.c_int, C.c_double, C.c_void_p] + [C.c_int] * 4
        L.kvq_oracle_int8_decode_attention.restype = C.c_int
        L.kvq_oracle_lloyd_max_normal.argtypes = [C.c_int, C.c_void_p, C.c_void_p]
        L.kvq_oracle_lloyd_max_normal.restype = C.c_int
        L.kvq_oracle_wht_f32.argtypes = [C.c_void_p, C.c_int]
        L.kvq_oracle_wht_f32.restype = None
        L.kvq_oracle_wht4_block_bytes.argtypes = [C.c_int, C.c_int]
        L.kvq_oracle_wht4_block_bytes.restype = C.c_size_t
        L.kvq_oracle_wht4_tables.argtypes = [C.c_void_p, C.c_void_p]
        L.kvq_oracle_wht4_tables.restype = None
        L.kvq_oracle_wht4_quantize_row.argtypes = [C.c_void_p, C.c_int, C.c_void_p, C.c_void_p]
        L.kvq_oracle_wht4_quantize_row.restype = C.c_int
        L.kvq_oracle_wht4_quantize_append.argtypes = [C.c_void_p] * 4 + [C.c_int, C.c_void_p] + [C.c_int] * 6
        L.kvq_oracle_wht4_quantize_append.restype = C.c_int
        L.kvq_oracle_wht4_dequantize.argtypes = [C.c_void_p, C.c_void_p] + [C.c_int] * 4 + [C.c_void_p] * 2 + \
            [C.c_int] * 4
        L.kvq_oracle_wht4_dequantize.restype = C.c_int
        L.kvq_oracle_wht4_decode_attention.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_void_p,
                                                       C.c_int, C.c_int, C.c_double, C.c_void_p] + [C.c_int] * 4
        L.kvq_oracle_wht4_decode_attention.restype = C.c_int
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle buffers must be C-contiguous"
    return a.ctypes.data


def f32_to_f16_bits(x: float) -> int:
    return int(lib().kvq_oracle_f32_to_f16(float(x)))


def f16_bits_to_f64(h: int) -> float:
    return float(lib().kvq_oracle_f16_to_f64(int(h)))


def f32_to_f16_array(x: np.ndarray) -> np.ndarray:
    """fp32 array -> fp16 bit patterns (uint16), round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().kvq_oracle_f32_to_f16_array(_ptr(x), _ptr(out), x.size)
    return out


def f16_to_f64_array(h: np.ndarray) -> np.ndarray:
    """fp16 bit patterns (uint16) -> float64 values."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float64)
    lib().kvq_oracle_f16_to_f64_array(_ptr(h), _ptr(out), h.size)
    return out


def block_bytes(head_dim: int, page_size: int, group_k: int, group_v: int) -> int:
    return int(lib().kvq_oracle_block_bytes(head_dim, page_size, group_k, group_v))


def fp16_kv_bytes(layers: int, kv_heads: int, head_dim: int, tokens: float) -> float:
    return float(lib().kvq_oracle_fp16_kv_bytes(layers, kv_heads, head_dim, float(tokens)))


def quantize_group(x_f16: np.ndarray) -> tuple[np.ndarray, int]:
    """One group of fp16 values -> (int8 codes in [-7, 7], fp16 scale bits)."""
    x = np.ascontiguousarray(x_f16, dtype=np.float16)
    codes = np.zeros(x.size, dtype=np.int8)
    s = np.zeros(1, dtype=np.uint16)
    lib().kvq_oracle_quantize_group(_ptr(x), int(x.size), _ptr(codes), _ptr(s))
    return codes, int(s[0])


class Layout:
    """Cache geometry (kv heads, head_dim, page size, K/V group sizes, pages)."""

    def __init__(self, num_kv_heads: int, head_dim: int, page_size: int, group_k: int, group_v: int,
                 num_pages: int):
        self.Hkv, self.d, self.P = num_kv_heads, head_dim, page_size
        self.Gk, self.Gv, self.num_pages = group_k, group_v, num_pages

    @property
    def geom(self) -> list[int]:
        return [self.Hkv, self.d, self.P, self.Gk, self.Gv, self.num_pages]

    @property
    def block_bytes(self) -> int:
        return block_bytes(self.d, self.P, self.Gk, self.Gv)

    @property
    def pool_bytes(self) -> int:
        return self.num_pages * self.Hkv * self.block_bytes


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def quantize_append(L: Layout, pool: np.ndarray, k: np.ndarray, v: np.ndarray, block_table: np.ndarray,
                    start_pos: np.ndarray) -> None:
    """In-place quantize-on-append into the uint8 pool.  k, v: fp16 [B, n_new, Hkv, d]."""
    k = np.ascontiguousarray(k, dtype=np.float16)
    v = np.ascontiguousarray(v, dtype=np.float16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sp = np.ascontiguousarray(start_pos, dtype=np.int32)
    B, n_new = k.shape[0], k.shape[1]
    assert pool.dtype == np.uint8 and pool.size >= L.pool_bytes
    rc = lib().kvq_oracle_quantize_append(_ptr(pool), _ptr(k), _ptr(v), _ptr(bt), int(bt.shape[1]), _ptr(sp),
                                          B, n_new, *L.geom)
    _check(rc, "quantize_append")


def dequantize(L: Layout, pool: np.ndarray, block_table: np.ndarray, b: int, start: int, n: int,
               out_fp16: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """Positions [start, start+n) of sequence b -> (K, V) each [n, Hkv, d] (fp32, or fp16)."""
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    dt = np.float16 if out_fp16 else np.float32
    ok = np.zeros((n, L.Hkv, L.d), dtype=dt)
    ov = np.zeros((n, L.Hkv, L.d), dtype=dt)
    rc = lib().kvq_oracle_dequantize(_ptr(pool), _ptr(bt), int(bt.shape[1]), b, start, n, _ptr(ok), _ptr(ov),
                                     1 if out_fp16 else 0, *L.geom)
    _check(rc, "dequantize")
    return ok, ov


def decode_attention(L: Layout, pool: np.ndarray, q: np.ndarray, block_table: np.ndarray, seq_lens: np.ndarray,
                     softmax_scale: float) -> np.ndarray:
    """fp64 decode attention over the quantized cache.  q: fp16 [B, Hq, d] -> fp64 [B, Hq, d]."""
    q = np.ascontiguousarray(q, dtype=np.float16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, _ = q.shape
    out = np.zeros((B, Hq, L.d), dtype=np.float64)
    rc = lib().kvq_oracle_decode_attention(_ptr(pool), _ptr(q), _ptr(bt), int(bt.shape[1]), _ptr(sl), B, Hq,
                                           float(softmax_scale), _ptr(out), *L.geom)
    _check(rc, "decode_attention")
    return out


def decode_attention_window(L: Layout, pool: np.ndarray, q: np.ndarray, block_table: np.ndarray,
                            seq_lens: np.ndarray, softmax_scale: float, window: int, sinks: int) -> np.ndarray:
    """fp64 decode attention over the quantized cache, restricted to the last `window` positions and
    the first `sinks` ("AI inference tuning: KV Cache optimisation and memory management" section 3.2,
    SlidingWindowAttention).  window <= 0: no window.  q: fp16 [B, Hq, d] -> fp64 [B, Hq, d]."""
    q = np.ascontiguousarray(q, dtype=np.float16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, _ = q.shape
    out = np.zeros((B, Hq, L.d), dtype=np.float64)
    rc = lib().kvq_oracle_decode_attention_window(_ptr(pool), _ptr(q), _ptr(bt), int(bt.shape[1]), _ptr(sl), B, Hq,
                                                  float(softmax_scale), int(window), int(sinks), _ptr(out), *L.geom)
    _check(rc, "decode_attention_window")
    return out


# ---------------------------------------------------------------------------
# The FP16 cache of the latency comparison ("LLM long-context inference: managing the KV
# cache with an INT4 state machine" section 7.4): same pages, K then V rows in fp16.
# ---------------------------------------------------------------------------

def fp16_block_bytes(head_dim: int, page_size: int) -> int:
    return int(lib().kvq_oracle_fp16_block_bytes(head_dim, page_size))


def fp16_pool_bytes(L: Layout) -> int:
    return L.num_pages * L.Hkv * fp16_block_bytes(L.d, L.P)


def fp16_append(L: Layout, pool16: np.ndarray, k: np.ndarray, v: np.ndarray, block_table: np.ndarray,
                start_pos: np.ndarray) -> None:
    """fp16 rows k, v [B, n_new, Hkv, d] into the FP16 pool at start_pos[b] + t."""
    k = np.ascontiguousarray(k, dtype=np.float16)
    v = np.ascontiguousarray(v, dtype=np.float16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sp = np.ascontiguousarray(start_pos, dtype=np.int32)
    B, n = k.shape[0], k.shape[1]
    rc = lib().kvq_oracle_fp16_append(_ptr(pool16), _ptr(k), _ptr(v), _ptr(bt), int(bt.shape[1]), _ptr(sp), B, n,
                                      L.Hkv, L.d, L.P, L.num_pages)
    _check(rc, "fp16_append")


def dequantize_to_fp16_pool(L: Layout, pool: np.ndarray, pool16: np.ndarray, block_table: np.ndarray,
                            seq_lens: np.ndarray) -> None:
    """Every attended position of the INT4 pool, dequantized (fp16 RNE) into the FP16 pool."""
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    rc = lib().kvq_oracle_dequantize_to_fp16_pool(_ptr(pool), _ptr(pool16), _ptr(bt), int(bt.shape[1]), _ptr(sl),
                                                  int(sl.shape[0]), *L.geom)
    _check(rc, "dequantize_to_fp16_pool")


def fp16_decode_attention(L: Layout, pool16: np.ndarray, q: np.ndarray, block_table: np.ndarray,
                          seq_lens: np.ndarray, softmax_scale: float) -> np.ndarray:
    """fp64 decode attention over the FP16 cache.  q: fp16 [B, Hq, d] -> fp64 [B, Hq, d]."""
    q = np.ascontiguousarray(q, dtype=np.float16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, _ = q.shape
    out = np.zeros((B, Hq, L.d), dtype=np.float64)
    rc = lib().kvq_oracle_fp16_decode_attention(_ptr(pool16), _ptr(q), _ptr(bt), int(bt.shape[1]), _ptr(sl), B, Hq,
                                                float(softmax_scale), _ptr(out), L.Hkv, L.d, L.P, L.num_pages)
    _check(rc, "fp16_decode_attention")
    return out


def mixed_decode_attention(L: Layout, pool: np.ndarray, block_table: np.ndarray, pool16: np.ndarray,
                           block_table16: np.ndarray, num_pages16: int, q: np.ndarray, seq_lens: np.ndarray,
                           residual: int, softmax_scale: float) -> np.ndarray:
    """fp64 decode attention with the last `residual` positions read from the FP16 pool and the
    older ones from the INT4 pool ("LLM long-context inference: managing the KV cache with an
    INT4 state machine" section 8.3).  q: fp16 [B, Hq, d] -> fp64 [B, Hq, d]."""
    q = np.ascontiguousarray(q, dtype=np.float16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    bt16 = np.ascontiguousarray(block_table16, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, _ = q.shape
    out = np.zeros((B, Hq, L.d), dtype=np.float64)
    rc = lib().kvq_oracle_mixed_decode_attention(_ptr(pool), _ptr(bt), int(bt.shape[1]), _ptr(pool16), _ptr(bt16),
                                                 int(bt16.shape[1]), _ptr(q), _ptr(sl), B, Hq, int(residual),
                                                 float(softmax_scale), _ptr(out), *L.geom, int(num_pages16))
    _check(rc, "mixed_decode_attention")
    return out


# ---------------------------------------------------------------------------
# INT8 per-row codec ("AI inference tuning: KV Cache optimisation and memory management"
# section 3.1, KVCacheQuantizer): one fp32 scale per (token, kv head) row.
# ---------------------------------------------------------------------------

def int8_block_bytes(head_dim: int, page_size: int) -> int:
    return int(lib().kvq_oracle_int8_block_bytes(head_dim, page_size))


def int8_pool_bytes(L: Layout) -> int:
    return L.num_pages * L.Hkv * int8_block_bytes(L.d, L.P)


def int8_quantize_row(x_f16: np.ndarray) -> tuple[np.ndarray, float]:
    """One fp16 row -> (int8 codes, fp32 scale)."""
    x = np.ascontiguousarray(x_f16, dtype=np.float16)
    codes = np.zeros(x.size, np.int8)
    s = np.zeros(1, np.float32)
    lib().kvq_oracle_int8_quantize_row(_ptr(x), int(x.size), _ptr(codes), _ptr(s))
    return codes, float(s[0])


def int8_quantize_append(L: Layout, pool8: np.ndarray, k: np.ndarray, v: np.ndarray, block_table: np.ndarray,
                         start_pos: np.ndarray) -> None:
    k = np.ascontiguousarray(k, dtype=np.float16)
    v = np.ascontiguousarray(v, dtype=np.float16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sp = np.ascontiguousarray(start_pos, dtype=np.int32)
    rc = lib().kvq_oracle_int8_quantize_append(_ptr(pool8), _ptr(k), _ptr(v), _ptr(bt), int(bt.shape[1]), _ptr(sp),
                                               int(k.shape[0]), int(k.shape[1]), L.Hkv, L.d, L.P, L.num_pages)
    _check(rc, "int8_quantize_append")


def int8_dequantize(L: Layout, pool8: np.ndarray, block_table: np.ndarray, b: int, start: int,
                    n: int) -> tuple[np.ndarray, np.ndarray]:
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    ok = np.zeros((n, L.Hkv, L.d), np.float32)
    ov = np.zeros((n, L.Hkv, L.d), np.float32)
    rc = lib().kvq_oracle_int8_dequantize(_ptr(pool8), _ptr(bt), int(bt.shape[1]), b, start, n, _ptr(ok), _ptr(ov),
                                          L.Hkv, L.d, L.P, L.num_pages)
    _check(rc, "int8_dequantize")
    return ok, ov


def int8_decode_attention(L: Layout, pool8: np.ndarray, q: np.ndarray, block_table: np.ndarray,
                          seq_lens: np.ndarray, softmax_scale: float) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, _ = q.shape
    out = np.zeros((B, Hq, L.d), dtype=np.float64)
    rc = lib().kvq_oracle_int8_decode_attention(_ptr(pool8), _ptr(q), _ptr(bt), int(bt.shape[1]), _ptr(sl), B, Hq,
                                                float(softmax_scale), _ptr(out), L.Hkv, L.d, L.P, L.num_pages)
    _check(rc, "int8_decode_attention")
    return out


# ---------------------------------------------------------------------------
# The rotated 4-bit codec ("LARQL KV cache engines", engine three: Walsh-Hadamard
# rotation, Lloyd-Max codebook; the reading is written out in kvq_oracle.c).
# ---------------------------------------------------------------------------
def lloyd_max_normal(bits: int) -> tuple[np.ndarray, np.ndarray]:
    """Lloyd-Max levels (2^bits, ascending) and thresholds (2^bits - 1) of N(0, 1), fp64."""
    n = 1 << bits
    lv = np.zeros(n, np.float64)
    tb = np.zeros(n - 1, np.float64)
    it = lib().kvq_oracle_lloyd_max_normal(bits, _ptr(lv), _ptr(tb))
    if it < 0:
        raise ValueError("bits out of range")
    return lv, tb


def wht_f32(y: np.ndarray) -> np.ndarray:
    """The fast Walsh-Hadamard transform (unnormalised, stage order h = 1, 2, ..) in fp32."""
    out = np.ascontiguousarray(y, dtype=np.float32).copy()
    lib().kvq_oracle_wht_f32(_ptr(out), int(out.size))
    return out


def wht4_tables() -> tuple[np.ndarray, np.ndarray]:
    """fp32 levels (16) and thresholds (15) of the 4-bit codec."""
    c = np.zeros(16, np.float32)
    t = np.zeros(15, np.float32)
    lib().kvq_oracle_wht4_tables(_ptr(c), _ptr(t))
    return c, t


def wht4_block_bytes(head_dim: int, page_size: int) -> int:
    return int(lib().kvq_oracle_wht4_block_bytes(head_dim, page_size))


def wht4_pool_bytes(L: Layout) -> int:
    return L.num_pages * L.Hkv * wht4_block_bytes(L.d, L.P)


def wht4_quantize_row(x_f16: np.ndarray) -> tuple[np.ndarray, float]:
    """One fp16 row of 128 -> (64 code bytes, fp32 sigma)."""
    x = np.ascontiguousarray(x_f16, dtype=np.float16)
    codes = np.zeros(x.size // 2, np.uint8)
    s = np.zeros(1, np.float32)
    _check(lib().kvq_oracle_wht4_quantize_row(_ptr(x), int(x.size), _ptr(codes), _ptr(s)), "wht4_quantize_row")
    return codes, float(s[0])


def wht4_quantize_append(L: Layout, pool: np.ndarray, k: np.ndarray, v: np.ndarray, block_table: np.ndarray,
                         start_pos: np.ndarray) -> None:
    k = np.ascontiguousarray(k, dtype=np.float16)
    v = np.ascontiguousarray(v, dtype=np.float16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sp = np.ascontiguousarray(start_pos, dtype=np.int32)
    rc = lib().kvq_oracle_wht4_quantize_append(_ptr(pool), _ptr(k), _ptr(v), _ptr(bt), int(bt.shape[1]), _ptr(sp),
                                               int(k.shape[0]), int(k.shape[1]), L.Hkv, L.d, L.P, L.num_pages)
    _check(rc, "wht4_quantize_append")


def wht4_dequantize(L: Layout, pool: np.ndarray, block_table: np.ndarray, b: int, start: int,
                    n: int) -> tuple[np.ndarray, np.ndarray]:
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    ok = np.zeros((n, L.Hkv, L.d), np.float32)
    ov = np.zeros((n, L.Hkv, L.d), np.float32)
    rc = lib().kvq_oracle_wht4_dequantize(_ptr(pool), _ptr(bt), int(bt.shape[1]), b, start, n, _ptr(ok), _ptr(ov),
                                          L.Hkv, L.d, L.P, L.num_pages)
    _check(rc, "wht4_dequantize")
    return ok, ov


def wht4_decode_attention(L: Layout, pool: np.ndarray, q: np.ndarray, block_table: np.ndarray,
                          seq_lens: np.ndarray, softmax_scale: float) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq = int(q.shape[0]), int(q.shape[1])
    out = np.zeros((B, Hq, L.d), np.float64)
    rc = lib().kvq_oracle_wht4_decode_attention(_ptr(pool), _ptr(q), _ptr(bt), int(bt.shape[1]), _ptr(sl), B, Hq,
                                                float(softmax_scale), _ptr(out), L.Hkv, L.d, L.P, L.num_pages)
    _check(rc, "wht4_decode_attention")
    return out

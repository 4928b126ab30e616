"""Host-side checks of the C ABI library (no GPU needed): it builds, loads, exports
every function include/kvq.h declares, sizes blocks like the oracle, and rejects bad
arguments on the host before touching the device."""
from __future__ import annotations

import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")


@pytest.fixture(scope="module")
def built():
    from int4_group_quantized_kvq_gb300 import _build
    return _build.build()


def header_functions() -> set[str]:
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", text))


def test_header_declares_the_abi():
    names = header_functions()
    assert {"kvq_quantize_append", "kvq_decode_attention", "kvq_dequantize", "kvq_block_bytes",
            "kvq_decode_workspace_bytes", "kvq_read_status", "kvq_last_error"} <= names


def test_library_exports_every_declared_symbol(built):
    out = subprocess.run(["nm", "-D", "--defined-only", built], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (kvq_[a-z0-9_]+)\b", out))
    missing = header_functions() - exported
    assert not missing, f"declared but not exported: {missing}"
    lib = C.CDLL(built)
    for name in header_functions():
        assert hasattr(lib, name)


def test_binding_names_match_header(built):
    import int4_group_quantized_kvq_gb300 as kvq
    assert set(kvq.ABI_SYMBOLS) == header_functions()
    for name in kvq.ABI_SYMBOLS:
        assert callable(getattr(kvq, name))


@pytest.mark.parametrize("d,P,Gk,Gv", [(128, 16, 64, 128), (128, 16, 32, 32), (128, 16, 128, 128),
                                       (64, 16, 32, 64), (256, 64, 128, 32), (128, 32, 64, 64)])
def test_block_bytes_agree_with_oracle(built, d, P, Gk, Gv):
    import int4_group_quantized_kvq_gb300 as kvq
    import oracle
    cfg = kvq.config(8, d, P, Gk, Gv, 10)
    assert kvq.kvq_block_bytes(cfg) == oracle.block_bytes(d, P, Gk, Gv)
    assert kvq.kvq_pool_bytes(cfg) == 10 * 8 * oracle.block_bytes(d, P, Gk, Gv)


@pytest.mark.parametrize("field,value,code", [("head_dim", 96, 2), ("page_size", 24, 2), ("group_k", 16, 2),
                                              ("group_v", 256, 2), ("num_kv_heads", 0, 1), ("num_pages", 0, 1)])
def test_bad_geometry_rejected_on_host(built, field, value, code):
    import int4_group_quantized_kvq_gb300 as kvq
    cfg = kvq.config(8, 128, 16, 64, 128, 10)
    setattr(cfg, field, value)
    assert kvq.lib().kvq_block_bytes(C.byref(cfg)) == 0
    rc = kvq.lib().kvq_quantize_append(C.byref(cfg), None, None, None, None, 1, None, 1, 1, None, None)
    assert rc == code
    assert kvq.kvq_last_error()


def test_null_and_misaligned_pointers_rejected_on_host(built):
    import int4_group_quantized_kvq_gb300 as kvq
    L = kvq.lib()
    cfg = kvq.config(8, 128, 16, 64, 128, 10)
    assert L.kvq_quantize_append(C.byref(cfg), None, None, None, None, 4, None, 2, 1, None, None) == kvq.KVQ_EINVAL
    assert L.kvq_quantize_append(C.byref(cfg), 0x1008, 0x2000, 0x3000, 0x4000, 4, 0x5000, 2, 1, None,
                                 None) == kvq.KVQ_EINVAL  # pool not 16-byte aligned
    assert "aligned" in kvq.kvq_last_error()
    # nothing to do is not an error
    assert L.kvq_quantize_append(C.byref(cfg), None, None, None, None, 4, None, 0, 1, None, None) == kvq.KVQ_OK
    # decode: ratio > 8; head_dim 256 with more than 4 query heads per kv head or K groups of
    # 32; misaligned workspace
    assert L.kvq_decode_attention(C.byref(cfg), 0x1000, 0x2000, 0x3000, 4, 0x4000, 1, 72, 10, 1.0, 0x5000,
                                  0x6000, 1 << 20, None) == kvq.KVQ_EUNSUPPORTED
    cfg256 = kvq.config(8, 256, 16, 64, 128, 10)
    assert L.kvq_decode_attention(C.byref(cfg256), 0x1000, 0x2000, 0x3000, 4, 0x4000, 1, 64, 10, 1.0, 0x5000,
                                  0x6000, 1 << 20, None) == kvq.KVQ_EUNSUPPORTED
    assert "query heads" in kvq.kvq_last_error()
    cfg256.group_k = 32
    assert L.kvq_decode_step(C.byref(cfg256), 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 4, 0x7000, 1, 8,
                             10, 1.0, 0x8000, 0x9000, 1 << 20, None) == kvq.KVQ_EUNSUPPORTED
    assert "group_k" in kvq.kvq_last_error()
    assert L.kvq_decode_attention(C.byref(cfg), 0x1000, 0x2000, 0x3000, 4, 0x4000, 1, 8, 10, 1.0, 0x5000,
                                  0x6010, 1 << 20, None) == kvq.KVQ_EINVAL
    assert L.kvq_decode_attention(C.byref(cfg), 0x1000, 0x2000, 0x3000, 4, 0x4000, 1, 12, 10, 1.0, 0x5000,
                                  0x6000, 1 << 20, None) == kvq.KVQ_EINVAL  # 12 % 8 != 0
    assert L.kvq_dequantize(C.byref(cfg), 0x1000, 0x2000, 4, 0, 0, 4, 0x3000, 0x4000, 2, None,
                            None) == kvq.KVQ_EINVAL  # out_dtype
    assert L.kvq_read_status(None, None, None) == kvq.KVQ_EINVAL


def test_version_string(built):
    import int4_group_quantized_kvq_gb300 as kvq
    assert "sm_103a" in kvq.kvq_version()


def test_wht4_codebook_is_the_oracles():
    # host code only: the library computes the rotated codec's Lloyd-Max codebook with its
    # own routine; its fp32 levels and thresholds must equal the oracle's bit for bit
    import numpy as np
    import oracle
    import int4_group_quantized_kvq_gb300 as kvq
    lv, tb = kvq.kvq_wht4_codebook()
    c, t = oracle.wht4_tables()
    assert np.array_equal(np.array(lv, np.float32), c) and np.array_equal(np.array(tb, np.float32), t)


def test_codec_and_host_step_calls_reject_bad_arguments_on_host(built):
    # the rotated 4-bit, INT8 and host-buffer calls check their arguments before touching the device
    import int4_group_quantized_kvq_gb300 as kvq
    L = kvq.lib()
    cfg = kvq.config(8, 128, 16, 64, 128, 10)
    cfg64 = kvq.config(8, 64, 16, 32, 64, 10)
    bad = kvq.config(8, 128, 16, 64, 128, 10)
    bad.page_size = 24
    assert L.kvq_wht4_pool_bytes(C.byref(bad)) == 0 and L.kvq_int8_pool_bytes(C.byref(bad)) == 0
    assert L.kvq_wht4_pool_bytes(C.byref(cfg)) == 10 * 8 * 16 * (128 + 8)
    # quantize-append: NULL, misaligned, head_dim other than 128, nothing to do
    assert L.kvq_wht4_quantize_append(C.byref(cfg), None, None, None, None, 4, None, 2, 1, None, None) == kvq.KVQ_EINVAL
    assert L.kvq_wht4_quantize_append(C.byref(cfg), 0x1008, 0x2000, 0x3000, 0x4000, 4, 0x5000, 2, 1, None,
                                      None) == kvq.KVQ_EINVAL
    assert L.kvq_wht4_quantize_append(C.byref(cfg64), 0x1000, 0x2000, 0x3000, 0x4000, 4, 0x5000, 2, 1, None,
                                      None) == kvq.KVQ_EUNSUPPORTED
    assert L.kvq_wht4_quantize_append(C.byref(cfg), None, None, None, None, 4, None, 0, 1, None, None) == kvq.KVQ_OK
    assert L.kvq_int8_quantize_append(C.byref(cfg), None, None, None, None, 4, None, 2, 1, None, None) == kvq.KVQ_EINVAL
    # dequantize: head_dim, negative sequence, NULL, misaligned output, nothing to do
    assert L.kvq_wht4_dequantize(C.byref(cfg64), 0x1000, 0x2000, 4, 0, 0, 4, 0x3000, 0x4000, None,
                                 None) == kvq.KVQ_EUNSUPPORTED
    assert L.kvq_wht4_dequantize(C.byref(cfg), 0x1000, 0x2000, 4, -1, 0, 4, 0x3000, 0x4000, None,
                                 None) == kvq.KVQ_EINVAL
    assert L.kvq_wht4_dequantize(C.byref(cfg), None, 0x2000, 4, 0, 0, 4, 0x3000, 0x4000, None, None) == kvq.KVQ_EINVAL
    assert L.kvq_wht4_dequantize(C.byref(cfg), 0x1000, 0x2000, 4, 0, 0, 4, 0x3004, 0x4000, None,
                                 None) == kvq.KVQ_EINVAL
    assert L.kvq_wht4_dequantize(C.byref(cfg), None, None, 4, 0, 0, 0, None, None, None, None) == kvq.KVQ_OK
    # decode attention over the codecs: more than 8 query heads per kv head, head_dim 64
    for fn in (L.kvq_wht4_decode_attention, L.kvq_int8_decode_attention, L.kvq_fp16_decode_attention):
        assert fn(C.byref(cfg), 0x1000, 0x2000, 0x3000, 4, 0x4000, 1, 72, 10, 1.0, 0x5000, 0x6000, 1 << 20,
                  None) == kvq.KVQ_EUNSUPPORTED
        assert fn(C.byref(cfg64), 0x1000, 0x2000, 0x3000, 4, 0x4000, 1, 8, 10, 1.0, 0x5000, 0x6000, 1 << 20,
                  None) == kvq.KVQ_EUNSUPPORTED
    # the host-buffer step: NULL buffers, a misaligned device copy, nothing to do
    assert L.kvq_decode_step_host(C.byref(cfg), 0x1000, None, 0x2000, 0x3000, 0x4000, 4, 0x5000, 2, 8, 10, 1.0,
                                  0x6000, 0x7000, 0x8000, 1 << 20, None) == kvq.KVQ_EINVAL
    assert L.kvq_decode_step_host(C.byref(cfg), 0x1000, 0x9000, 0x2008, 0x3000, 0x4000, 4, 0x5000, 2, 8, 10, 1.0,
                                  0x6000, 0x7000, 0x8000, 1 << 20, None) == kvq.KVQ_EINVAL
    assert "aligned" in kvq.kvq_last_error()
    assert L.kvq_decode_step_host(C.byref(cfg), None, None, None, None, None, 4, None, 0, 8, 10, 1.0, None, None,
                                  None, 0, None) == kvq.KVQ_OK
    # the pipelined host-buffer step: missing events, streams that are not three distinct ones
    ev = (C.c_void_p * 3)(0xA000, 0xB000, 0xC000)
    no_ev = (C.c_void_p * 3)(0xA000, None, 0xC000)
    args = (C.byref(cfg), 0x1000, 0x9000, 0x2000, 0x3000, 0x4000, 4, 0x5000, 2, 8, 10, 1.0, 0x6000, 0x7000, 0x8000,
            1 << 20)
    assert L.kvq_decode_step_host_pipelined(*args, 0x11, 0x22, 0x33, no_ev) == kvq.KVQ_EINVAL
    assert L.kvq_decode_step_host_pipelined(*args, 0x11, 0x22, 0x22, ev) == kvq.KVQ_EINVAL
    assert L.kvq_decode_step_host_pipelined(*args, 0x11, 0x11, 0x33, ev) == kvq.KVQ_EINVAL
    assert "distinct" in kvq.kvq_last_error()
    assert L.kvq_decode_step_host_pipelined(C.byref(cfg), None, None, None, None, None, 4, None, 0, 8, 10, 1.0, None,
                                            None, None, 0, None, None, None, None) == kvq.KVQ_OK

"""ctypes binding of libkvq.so: the C ABI of include/kvq.h under the same names.

Argument marshalling only: every function checks that the torch tensors it is
handed have the dtype, device and layout the C ABI expects, passes raw pointers
and the current CUDA stream, and turns a non-zero status into an exception.  All
computation happens in the library's CUDA kernels; there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvq.so")

KVQ_OK, KVQ_EINVAL, KVQ_EUNSUPPORTED, KVQ_EWORKSPACE, KVQ_ECUDA = 0, 1, 2, 3, 4
KVQ_FLAG_BAD_PAGE, KVQ_FLAG_BAD_POSITION, KVQ_FLAG_WAIT_TIMEOUT, KVQ_FLAG_STALE_WORKSPACE = 0x1, 0x2, 0x4, 0x8

ABI_SYMBOLS = ("kvq_block_bytes", "kvq_pool_bytes", "kvq_quantize_append", "kvq_quantize_append_varlen",
               "kvq_decode_workspace_bytes",
               "kvq_decode_attention", "kvq_dequantize", "kvq_read_status", "kvq_last_error", "kvq_version",
               "kvq_decode_attention_noalloc", "kvq_decode_step", "kvq_decode_attention_window",
               "kvq_decode_step_window", "kvq_fp16_pool_bytes", "kvq_fp16_append", "kvq_dequantize_to_fp16_pool",
               "kvq_fp16_decode_workspace_bytes", "kvq_fp16_decode_attention", "kvq_mixed_decode_workspace_bytes",
               "kvq_mixed_decode_attention", "kvq_int8_pool_bytes", "kvq_int8_quantize_append",
               "kvq_int8_decode_workspace_bytes", "kvq_int8_decode_attention", "kvq_wht4_codebook",
               "kvq_wht4_pool_bytes", "kvq_wht4_quantize_append", "kvq_wht4_dequantize",
               "kvq_wht4_decode_workspace_bytes", "kvq_wht4_decode_attention", "kvq_decode_step_host",
               "kvq_decode_step_host_pipelined", "kvq_test_decode_wait_timeout")


class KvqError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"kvq error {code}: {msg}")
        self.code = code


class CacheConfig(C.Structure):
    """kvq_cache_config: num_kv_heads, head_dim, page_size, group_k, group_v, num_pages."""

    _fields_ = [("num_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("page_size", C.c_int32),
                ("group_k", C.c_int32), ("group_v", C.c_int32), ("num_pages", C.c_int32)]

    def __repr__(self) -> str:
        return (f"CacheConfig(Hkv={self.num_kv_heads}, d={self.head_dim}, P={self.page_size}, "
                f"Gk={self.group_k}, Gv={self.group_v}, pages={self.num_pages})")


_lib: C.CDLL | None = None


def lib() -> C.CDLL:
    """Load libkvq.so.  Raises if it has not been built: there is no other implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                              f"g.build()'` (nvcc, sm_103a)")
        L = C.CDLL(LIB_PATH)
        P, I32, SZ = C.c_void_p, C.c_int32, C.c_size_t
        cfgp = C.POINTER(CacheConfig)
        L.kvq_block_bytes.argtypes = [cfgp]
        L.kvq_block_bytes.restype = SZ
        L.kvq_pool_bytes.argtypes = [cfgp]
        L.kvq_pool_bytes.restype = SZ
        L.kvq_quantize_append.argtypes = [cfgp, P, P, P, P, I32, P, I32, I32, P, P]
        L.kvq_quantize_append.restype = C.c_int
        L.kvq_quantize_append_varlen.argtypes = [cfgp, P, P, P, P, I32, P, P, I32, I32, P, P]
        L.kvq_quantize_append_varlen.restype = C.c_int
        L.kvq_decode_workspace_bytes.argtypes = [cfgp, I32, I32, I32]
        L.kvq_decode_workspace_bytes.restype = SZ
        L.kvq_decode_attention.argtypes = [cfgp, P, P, P, I32, P, I32, I32, I32, C.c_float, P, P, SZ, P]
        L.kvq_decode_attention.restype = C.c_int
        L.kvq_decode_attention_noalloc.argtypes = [cfgp, P, P, P, I32, P, I32, I32, I32, C.c_float, P, P, P]
        L.kvq_decode_attention_noalloc.restype = C.c_int
        L.kvq_decode_step.argtypes = [cfgp, P, P, P, P, P, P, I32, P, I32, I32, I32, C.c_float, P, P, SZ, P]
        L.kvq_decode_step.restype = C.c_int
        L.kvq_decode_attention_window.argtypes = [cfgp, P, P, P, I32, P, I32, I32, I32, C.c_float, I32, I32, P, P,
                                                  SZ, P]
        L.kvq_decode_attention_window.restype = C.c_int
        L.kvq_decode_step_window.argtypes = [cfgp, P, P, P, P, P, P, I32, P, I32, I32, I32, C.c_float, I32, I32, P,
                                             P, SZ, P]
        L.kvq_decode_step_window.restype = C.c_int
        L.kvq_fp16_pool_bytes.argtypes = [cfgp]
        L.kvq_fp16_pool_bytes.restype = SZ
        L.kvq_fp16_append.argtypes = [cfgp, P, P, P, P, I32, P, I32, I32, P, P]
        L.kvq_fp16_append.restype = C.c_int
        L.kvq_dequantize_to_fp16_pool.argtypes = [cfgp, P, P, P, I32, P, I32, I32, P, P]
        L.kvq_dequantize_to_fp16_pool.restype = C.c_int
        L.kvq_fp16_decode_workspace_bytes.argtypes = [cfgp, I32, I32, I32]
        L.kvq_fp16_decode_workspace_bytes.restype = SZ
        L.kvq_fp16_decode_attention.argtypes = [cfgp, P, P, P, I32, P, I32, I32, I32, C.c_float, P, P, SZ, P]
        L.kvq_fp16_decode_attention.restype = C.c_int
        L.kvq_mixed_decode_workspace_bytes.argtypes = [cfgp, I32, I32, I32, I32]
        L.kvq_mixed_decode_workspace_bytes.restype = SZ
        L.kvq_mixed_decode_attention.argtypes = [cfgp, P, P, I32, P, P, I32, I32, P, P, I32, I32, I32, I32, C.c_float,
                                                 P, P, SZ, P]
        L.kvq_mixed_decode_attention.restype = C.c_int
        L.kvq_int8_pool_bytes.argtypes = [cfgp]
        L.kvq_int8_pool_bytes.restype = SZ
        L.kvq_int8_quantize_append.argtypes = [cfgp, P, P, P, P, I32, P, I32, I32, P, P]
        L.kvq_int8_quantize_append.restype = C.c_int
        L.kvq_int8_decode_workspace_bytes.argtypes = [cfgp, I32, I32, I32]
        L.kvq_int8_decode_workspace_bytes.restype = SZ
        L.kvq_int8_decode_attention.argtypes = [cfgp, P, P, P, I32, P, I32, I32, I32, C.c_float, P, P, SZ, P]
        L.kvq_int8_decode_attention.restype = C.c_int
        L.kvq_decode_step_host.argtypes = [cfgp, P, P, P, P, P, I32, P, I32, I32, I32, C.c_float, P, P, P, SZ, P]
        L.kvq_decode_step_host.restype = C.c_int
        L.kvq_decode_step_host_pipelined.argtypes = [cfgp, P, P, P, P, P, I32, P, I32, I32, I32, C.c_float, P, P, P,
                                                     SZ, P, P, P, C.POINTER(C.c_void_p)]
        L.kvq_decode_step_host_pipelined.restype = C.c_int
        L.kvq_test_decode_wait_timeout.argtypes = [cfgp, P, P, P, I32, P, I32, I32, I32, C.c_float, P, P, SZ,
                                                   C.c_uint64, P]
        L.kvq_test_decode_wait_timeout.restype = C.c_int
        L.kvq_wht4_codebook.argtypes = [P, P]
        L.kvq_wht4_codebook.restype = None
        L.kvq_wht4_pool_bytes.argtypes = [cfgp]
        L.kvq_wht4_pool_bytes.restype = SZ
        L.kvq_wht4_quantize_append.argtypes = [cfgp, P, P, P, P, I32, P, I32, I32, P, P]
        L.kvq_wht4_quantize_append.restype = C.c_int
        L.kvq_wht4_dequantize.argtypes = [cfgp, P, P, I32, I32, I32, I32, P, P, P, P]
        L.kvq_wht4_dequantize.restype = C.c_int
        L.kvq_wht4_decode_workspace_bytes.argtypes = [cfgp, I32, I32, I32]
        L.kvq_wht4_decode_workspace_bytes.restype = SZ
        L.kvq_wht4_decode_attention.argtypes = [cfgp, P, P, P, I32, P, I32, I32, I32, C.c_float, P, P, SZ, P]
        L.kvq_wht4_decode_attention.restype = C.c_int
        L.kvq_dequantize.argtypes = [cfgp, P, P, I32, I32, I32, I32, P, P, I32, P, P]
        L.kvq_dequantize.restype = C.c_int
        L.kvq_read_status.argtypes = [P, C.POINTER(C.c_uint32), P]
        L.kvq_read_status.restype = C.c_int
        L.kvq_last_error.argtypes = []
        L.kvq_last_error.restype = C.c_char_p
        L.kvq_version.argtypes = []
        L.kvq_version.restype = C.c_char_p
        _lib = L
    return _lib


def kvq_last_error() -> str:
    return lib().kvq_last_error().decode()


def kvq_version() -> str:
    return lib().kvq_version().decode()


def _check(rc: int) -> None:
    if rc != KVQ_OK:
        raise KvqError(rc, kvq_last_error())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, name: str, dtype: torch.dtype | None = None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _status(t: torch.Tensor) -> int:
    """A device status word: the library writes or ORs 4 bytes into it."""
    if not isinstance(t, torch.Tensor) or t.dtype not in (torch.int32, getattr(torch, "uint32", torch.int32)):
        raise ValueError("status must be an int32 (or uint32) CUDA tensor")
    if t.numel() < 1:
        raise ValueError("status must hold at least one element")
    return _dev(t, "status")


def config(num_kv_heads: int, head_dim: int, page_size: int = 16, group_k: int = 64, group_v: int = 128,
           num_pages: int = 1) -> CacheConfig:
    return CacheConfig(num_kv_heads, head_dim, page_size, group_k, group_v, num_pages)


def kvq_block_bytes(cfg: CacheConfig) -> int:
    n = lib().kvq_block_bytes(C.byref(cfg))
    if n == 0:
        raise KvqError(KVQ_EINVAL, kvq_last_error())
    return int(n)


def kvq_pool_bytes(cfg: CacheConfig) -> int:
    n = lib().kvq_pool_bytes(C.byref(cfg))
    if n == 0:
        raise KvqError(KVQ_EINVAL, kvq_last_error())
    return int(n)


def kvq_quantize_append(cfg: CacheConfig, pool: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                        block_table: torch.Tensor, start_pos: torch.Tensor, status: torch.Tensor | None = None,
                        stream=None) -> None:
    """k, v: fp16 [B, n_new, Hkv, d]; block_table int32 [B, max_blocks]; start_pos int32 [B]."""
    if k.shape != v.shape or k.dim() != 4:
        raise ValueError("k and v must both be [B, n_new, Hkv, d]")
    B, n_new = int(k.shape[0]), int(k.shape[1])
    rc = lib().kvq_quantize_append(
        C.byref(cfg), _dev(pool, "pool", torch.uint8), _dev(k, "k", torch.float16), _dev(v, "v", torch.float16),
        _dev(block_table, "block_table", torch.int32), int(block_table.shape[1]),
        _dev(start_pos, "start_pos", torch.int32), B, n_new,
        None if status is None else _status(status), _stream(stream))
    _check(rc)


def kvq_quantize_append_varlen(cfg: CacheConfig, pool: torch.Tensor, k_rows: torch.Tensor, v_rows: torch.Tensor,
                               block_table: torch.Tensor, start_pos: torch.Tensor, cu_rows: torch.Tensor,
                               status: torch.Tensor | None = None, stream=None) -> None:
    """k_rows, v_rows: fp16 [total_rows, Hkv, d], the sequences' new rows back to back; cu_rows int32 [B + 1]:
    sequence b owns rows cu_rows[b] .. cu_rows[b + 1] - 1; start_pos int32 [B]."""
    if k_rows.shape != v_rows.shape or k_rows.dim() != 3:
        raise ValueError("k_rows and v_rows must both be [total_rows, Hkv, d]")
    B = int(block_table.shape[0])
    if cu_rows.dim() != 1 or int(cu_rows.shape[0]) != B + 1 or int(start_pos.shape[0]) != B:
        raise ValueError("cu_rows must be [B + 1] and start_pos [B] for a block table of B rows")
    rc = lib().kvq_quantize_append_varlen(
        C.byref(cfg), _dev(pool, "pool", torch.uint8), _dev(k_rows, "k_rows", torch.float16),
        _dev(v_rows, "v_rows", torch.float16), _dev(block_table, "block_table", torch.int32),
        int(block_table.shape[1]), _dev(start_pos, "start_pos", torch.int32), _dev(cu_rows, "cu_rows", torch.int32),
        B, int(k_rows.shape[0]), None if status is None else _status(status), _stream(stream))
    _check(rc)


def kvq_decode_workspace_bytes(cfg: CacheConfig, batch: int, num_q_heads: int, max_len: int) -> int:
    n = lib().kvq_decode_workspace_bytes(C.byref(cfg), batch, num_q_heads, max_len)
    if n == 0:
        raise KvqError(KVQ_EUNSUPPORTED, kvq_last_error())
    return int(n)


def kvq_decode_attention(cfg: CacheConfig, pool: torch.Tensor, q: torch.Tensor, block_table: torch.Tensor,
                         seq_lens: torch.Tensor, max_len: int, softmax_scale: float, out: torch.Tensor,
                         workspace: torch.Tensor, stream=None) -> None:
    """q: fp16 [B, Hq, d]; out: fp32 [B, Hq, d]; seq_lens int32 [B]; workspace uint8 (first 4 bytes: status)."""
    B, Hq = int(q.shape[0]), int(q.shape[1])
    rc = lib().kvq_decode_attention(
        C.byref(cfg), _dev(pool, "pool", torch.uint8), _dev(q, "q", torch.float16),
        _dev(block_table, "block_table", torch.int32), int(block_table.shape[1]),
        _dev(seq_lens, "seq_lens", torch.int32), B, Hq, int(max_len), float(softmax_scale),
        _dev(out, "out", torch.float32), _dev(workspace, "workspace", torch.uint8), workspace.numel(),
        _stream(stream))
    _check(rc)


def kvq_decode_step(cfg: CacheConfig, pool: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                    append_pos: torch.Tensor, q: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                    max_len: int, softmax_scale: float, out: torch.Tensor, workspace: torch.Tensor,
                    stream=None) -> None:
    """One decode step in one call (the append fused into the decode grid): append k_new, v_new (fp16 [B, Hkv, d], or [B, 1, Hkv, d]) at
    append_pos (int32 [B], negative: none), then attend q (fp16 [B, Hq, d]) over seq_lens into out
    (fp32 [B, Hq, d])."""
    B, Hq = int(q.shape[0]), int(q.shape[1])
    rc = lib().kvq_decode_step(
        C.byref(cfg), _dev(pool, "pool", torch.uint8), _dev(k_new, "k_new", torch.float16),
        _dev(v_new, "v_new", torch.float16), _dev(append_pos, "append_pos", torch.int32),
        _dev(q, "q", torch.float16), _dev(block_table, "block_table", torch.int32), int(block_table.shape[1]),
        _dev(seq_lens, "seq_lens", torch.int32), B, Hq, int(max_len), float(softmax_scale),
        _dev(out, "out", torch.float32), _dev(workspace, "workspace", torch.uint8), workspace.numel(),
        _stream(stream))
    _check(rc)


def kvq_decode_attention_window(cfg: CacheConfig, pool: torch.Tensor, q: torch.Tensor, block_table: torch.Tensor,
                                seq_lens: torch.Tensor, max_len: int, softmax_scale: float, window: int, sinks: int,
                                out: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """kvq_decode_attention over the last `window` positions (0: all) and the first `sinks`."""
    B, Hq = int(q.shape[0]), int(q.shape[1])
    rc = lib().kvq_decode_attention_window(
        C.byref(cfg), _dev(pool, "pool", torch.uint8), _dev(q, "q", torch.float16),
        _dev(block_table, "block_table", torch.int32), int(block_table.shape[1]),
        _dev(seq_lens, "seq_lens", torch.int32), B, Hq, int(max_len), float(softmax_scale), int(window), int(sinks),
        _dev(out, "out", torch.float32), _dev(workspace, "workspace", torch.uint8), workspace.numel(),
        _stream(stream))
    _check(rc)


def kvq_decode_step_window(cfg: CacheConfig, pool: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                           append_pos: torch.Tensor, q: torch.Tensor, block_table: torch.Tensor,
                           seq_lens: torch.Tensor, max_len: int, softmax_scale: float, window: int, sinks: int,
                           out: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """kvq_decode_step attending to the last `window` positions (0: all) and the first `sinks`."""
    B, Hq = int(q.shape[0]), int(q.shape[1])
    rc = lib().kvq_decode_step_window(
        C.byref(cfg), _dev(pool, "pool", torch.uint8), _dev(k_new, "k_new", torch.float16),
        _dev(v_new, "v_new", torch.float16), _dev(append_pos, "append_pos", torch.int32),
        _dev(q, "q", torch.float16), _dev(block_table, "block_table", torch.int32), int(block_table.shape[1]),
        _dev(seq_lens, "seq_lens", torch.int32), B, Hq, int(max_len), float(softmax_scale), int(window), int(sinks),
        _dev(out, "out", torch.float32), _dev(workspace, "workspace", torch.uint8), workspace.numel(),
        _stream(stream))
    _check(rc)


def kvq_decode_attention_noalloc(cfg: CacheConfig, pool: torch.Tensor, q: torch.Tensor, block_table: torch.Tensor,
                                 seq_lens: torch.Tensor, max_len: int, softmax_scale: float, out: torch.Tensor,
                                 status: torch.Tensor | None = None, stream=None) -> None:
    """kvq_decode_attention for callers that cannot allocate: no workspace argument; the
    library's built-in scratch (8 MiB) is used.  Calls that overlap on the GPU race on it."""
    B, Hq = int(q.shape[0]), int(q.shape[1])
    rc = lib().kvq_decode_attention_noalloc(
        C.byref(cfg), _dev(pool, "pool", torch.uint8), _dev(q, "q", torch.float16),
        _dev(block_table, "block_table", torch.int32), int(block_table.shape[1]),
        _dev(seq_lens, "seq_lens", torch.int32), B, Hq, int(max_len), float(softmax_scale),
        _dev(out, "out", torch.float32), None if status is None else _status(status), _stream(stream))
    _check(rc)


def kvq_dequantize(cfg: CacheConfig, pool: torch.Tensor, block_table: torch.Tensor, b: int, start: int, n: int,
                   out_k: torch.Tensor, out_v: torch.Tensor, status: torch.Tensor | None = None,
                   stream=None) -> None:
    """out_k, out_v: [n, Hkv, d] fp16 or fp32 (both the same dtype)."""
    if out_k.dtype != out_v.dtype or out_k.dtype not in (torch.float16, torch.float32):
        raise ValueError("out_k and out_v must both be fp16 or both fp32")
    out_dtype = 1 if out_k.dtype == torch.float32 else 0
    rc = lib().kvq_dequantize(
        C.byref(cfg), _dev(pool, "pool", torch.uint8), _dev(block_table, "block_table", torch.int32),
        int(block_table.shape[1]), b, start, n, _dev(out_k, "out_k"), _dev(out_v, "out_v"), out_dtype,
        None if status is None else _status(status), _stream(stream))
    _check(rc)


def kvq_read_status(status_word: torch.Tensor, stream=None) -> int:
    """Flags of a status word (a uint32 status tensor or a decode workspace); synchronizes the stream."""
    flags = C.c_uint32(0)
    _check(lib().kvq_read_status(_dev(status_word, "status_word"), C.byref(flags), _stream(stream)))
    return int(flags.value)


def new_workspace(cfg: CacheConfig, batch: int, num_q_heads: int, max_len: int, device="cuda") -> torch.Tensor:
    """A zeroed decode workspace of the size the library asks for (allocated by torch, not the library)."""
    n = kvq_decode_workspace_bytes(cfg, batch, num_q_heads, max_len)
    return torch.zeros(n, dtype=torch.uint8, device=device)


# ---------------------------------------------------------------------------
# The FP16 cache of the latency comparison (same pages; K then V rows in fp16).
# ---------------------------------------------------------------------------

def kvq_fp16_pool_bytes(cfg: CacheConfig) -> int:
    return int(lib().kvq_fp16_pool_bytes(C.byref(cfg)))


def kvq_fp16_append(cfg: CacheConfig, pool16: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                    block_table: torch.Tensor, start_pos: torch.Tensor, status: torch.Tensor | None = None,
                    stream=None) -> None:
    """fp16 rows k, v [B, n_new, Hkv, d] into the FP16 pool at start_pos[b] + t."""
    B, n = int(k.shape[0]), int(k.shape[1])
    rc = lib().kvq_fp16_append(
        C.byref(cfg), _dev(pool16, "pool16", torch.uint8), _dev(k, "k", torch.float16), _dev(v, "v", torch.float16),
        _dev(block_table, "block_table", torch.int32), int(block_table.shape[1]),
        _dev(start_pos, "start_pos", torch.int32), B, n, None if status is None else _status(status),
        _stream(stream))
    _check(rc)


def kvq_dequantize_to_fp16_pool(cfg: CacheConfig, pool: torch.Tensor, pool16: torch.Tensor,
                                block_table: torch.Tensor, seq_lens: torch.Tensor, max_len: int,
                                status: torch.Tensor | None = None, stream=None) -> None:
    """Every attended position of the INT4 pool, dequantized to fp16, into the FP16 pool."""
    rc = lib().kvq_dequantize_to_fp16_pool(
        C.byref(cfg), _dev(pool, "pool", torch.uint8), _dev(pool16, "pool16", torch.uint8),
        _dev(block_table, "block_table", torch.int32), int(block_table.shape[1]),
        _dev(seq_lens, "seq_lens", torch.int32), int(seq_lens.shape[0]), int(max_len),
        None if status is None else _status(status), _stream(stream))
    _check(rc)


def kvq_fp16_decode_workspace_bytes(cfg: CacheConfig, batch: int, num_q_heads: int, max_len: int) -> int:
    n = int(lib().kvq_fp16_decode_workspace_bytes(C.byref(cfg), batch, num_q_heads, max_len))
    if n == 0:
        raise KvqError(KVQ_EINVAL, kvq_last_error())
    return n


def new_fp16_workspace(cfg: CacheConfig, batch: int, num_q_heads: int, max_len: int, device="cuda") -> torch.Tensor:
    return torch.zeros(kvq_fp16_decode_workspace_bytes(cfg, batch, num_q_heads, max_len), dtype=torch.uint8,
                       device=device)


def kvq_fp16_decode_attention(cfg: CacheConfig, pool16: torch.Tensor, q: torch.Tensor, block_table: torch.Tensor,
                              seq_lens: torch.Tensor, max_len: int, softmax_scale: float, out: torch.Tensor,
                              workspace: torch.Tensor, stream=None) -> None:
    """Decode attention over the FP16 cache; arguments as kvq_decode_attention."""
    B, Hq = int(q.shape[0]), int(q.shape[1])
    rc = lib().kvq_fp16_decode_attention(
        C.byref(cfg), _dev(pool16, "pool16", torch.uint8), _dev(q, "q", torch.float16),
        _dev(block_table, "block_table", torch.int32), int(block_table.shape[1]),
        _dev(seq_lens, "seq_lens", torch.int32), B, Hq, int(max_len), float(softmax_scale),
        _dev(out, "out", torch.float32), _dev(workspace, "workspace", torch.uint8), workspace.numel(),
        _stream(stream))
    _check(rc)


def kvq_mixed_decode_workspace_bytes(cfg: CacheConfig, batch: int, num_q_heads: int, max_len: int,
                                     residual: int) -> int:
    n = int(lib().kvq_mixed_decode_workspace_bytes(C.byref(cfg), batch, num_q_heads, max_len, residual))
    if n == 0:
        raise KvqError(KVQ_EINVAL, kvq_last_error())
    return n


def kvq_mixed_decode_attention(cfg: CacheConfig, pool: torch.Tensor, block_table: torch.Tensor,
                               pool16: torch.Tensor, block_table16: torch.Tensor, num_pages16: int, q: torch.Tensor,
                               seq_lens: torch.Tensor, max_len: int, residual: int, softmax_scale: float,
                               out: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """Decode attention with the last `residual` positions read from the FP16 pool and the
    older ones from the INT4 pool."""
    B, Hq = int(q.shape[0]), int(q.shape[1])
    rc = lib().kvq_mixed_decode_attention(
        C.byref(cfg), _dev(pool, "pool", torch.uint8), _dev(block_table, "block_table", torch.int32),
        int(block_table.shape[1]), _dev(pool16, "pool16", torch.uint8),
        _dev(block_table16, "block_table16", torch.int32), int(block_table16.shape[1]), int(num_pages16),
        _dev(q, "q", torch.float16), _dev(seq_lens, "seq_lens", torch.int32), B, Hq, int(max_len), int(residual),
        float(softmax_scale), _dev(out, "out", torch.float32), _dev(workspace, "workspace", torch.uint8),
        workspace.numel(), _stream(stream))
    _check(rc)


# ---------------------------------------------------------------------------
# The INT8 per-row cache (one fp32 scale per token and kv head).
# ---------------------------------------------------------------------------

def kvq_int8_pool_bytes(cfg: CacheConfig) -> int:
    return int(lib().kvq_int8_pool_bytes(C.byref(cfg)))


def kvq_int8_quantize_append(cfg: CacheConfig, pool8: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                             block_table: torch.Tensor, start_pos: torch.Tensor, status: torch.Tensor | None = None,
                             stream=None) -> None:
    """Quantize fp16 rows k, v [B, n_new, Hkv, d] into the INT8 pool at start_pos[b] + t."""
    B, n = int(k.shape[0]), int(k.shape[1])
    rc = lib().kvq_int8_quantize_append(
        C.byref(cfg), _dev(pool8, "pool8", torch.uint8), _dev(k, "k", torch.float16), _dev(v, "v", torch.float16),
        _dev(block_table, "block_table", torch.int32), int(block_table.shape[1]),
        _dev(start_pos, "start_pos", torch.int32), B, n, None if status is None else _status(status),
        _stream(stream))
    _check(rc)


def kvq_int8_decode_workspace_bytes(cfg: CacheConfig, batch: int, num_q_heads: int, max_len: int) -> int:
    n = int(lib().kvq_int8_decode_workspace_bytes(C.byref(cfg), batch, num_q_heads, max_len))
    if n == 0:
        raise KvqError(KVQ_EINVAL, kvq_last_error())
    return n


def kvq_int8_decode_attention(cfg: CacheConfig, pool8: torch.Tensor, q: torch.Tensor, block_table: torch.Tensor,
                              seq_lens: torch.Tensor, max_len: int, softmax_scale: float, out: torch.Tensor,
                              workspace: torch.Tensor, stream=None) -> None:
    """Decode attention over the INT8 per-row cache; arguments as kvq_decode_attention."""
    B, Hq = int(q.shape[0]), int(q.shape[1])
    rc = lib().kvq_int8_decode_attention(
        C.byref(cfg), _dev(pool8, "pool8", torch.uint8), _dev(q, "q", torch.float16),
        _dev(block_table, "block_table", torch.int32), int(block_table.shape[1]),
        _dev(seq_lens, "seq_lens", torch.int32), B, Hq, int(max_len), float(softmax_scale),
        _dev(out, "out", torch.float32), _dev(workspace, "workspace", torch.uint8), workspace.numel(),
        _stream(stream))
    _check(rc)


# ---------------------------------------------------------------------------
# The rotated 4-bit cache ("LARQL KV cache engines", engine three: Walsh-Hadamard
# rotation and a Lloyd-Max codebook; layout and arithmetic in include/kvq.h)
# ---------------------------------------------------------------------------
def kvq_wht4_codebook() -> tuple[list[float], list[float]]:
    """The library's fp32 codebook: 16 levels (ascending) and the 15 thresholds between them."""
    lv = (C.c_float * 16)()
    tb = (C.c_float * 15)()
    lib().kvq_wht4_codebook(C.cast(lv, C.c_void_p), C.cast(tb, C.c_void_p))
    return list(lv), list(tb)


def kvq_wht4_pool_bytes(cfg: CacheConfig) -> int:
    return int(lib().kvq_wht4_pool_bytes(C.byref(cfg)))


def kvq_wht4_quantize_append(cfg: CacheConfig, pool: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                             block_table: torch.Tensor, start_pos: torch.Tensor, status: torch.Tensor | None = None,
                             stream=None) -> None:
    """Quantize fp16 rows k, v [B, n_new, Hkv, 128] into the rotated 4-bit pool at start_pos[b] + t."""
    B, n = int(k.shape[0]), int(k.shape[1])
    rc = lib().kvq_wht4_quantize_append(
        C.byref(cfg), _dev(pool, "pool", torch.uint8), _dev(k, "k", torch.float16), _dev(v, "v", torch.float16),
        _dev(block_table, "block_table", torch.int32), int(block_table.shape[1]),
        _dev(start_pos, "start_pos", torch.int32), B, n, None if status is None else _status(status),
        _stream(stream))
    _check(rc)


def kvq_wht4_dequantize(cfg: CacheConfig, pool: torch.Tensor, block_table: torch.Tensor, b: int, start: int, n: int,
                        out_k: torch.Tensor, out_v: torch.Tensor, status: torch.Tensor | None = None,
                        stream=None) -> None:
    """Positions [start, start + n) of sequence b to fp32 out_k, out_v [n, Hkv, 128]."""
    rc = lib().kvq_wht4_dequantize(
        C.byref(cfg), _dev(pool, "pool", torch.uint8), _dev(block_table, "block_table", torch.int32),
        int(block_table.shape[1]), int(b), int(start), int(n), _dev(out_k, "out_k", torch.float32),
        _dev(out_v, "out_v", torch.float32), None if status is None else _status(status), _stream(stream))
    _check(rc)


def kvq_wht4_decode_workspace_bytes(cfg: CacheConfig, batch: int, num_q_heads: int, max_len: int) -> int:
    n = int(lib().kvq_wht4_decode_workspace_bytes(C.byref(cfg), batch, num_q_heads, max_len))
    if n == 0:
        raise KvqError(KVQ_EINVAL, kvq_last_error())
    return n


def kvq_wht4_decode_attention(cfg: CacheConfig, pool: torch.Tensor, q: torch.Tensor, block_table: torch.Tensor,
                              seq_lens: torch.Tensor, max_len: int, softmax_scale: float, out: torch.Tensor,
                              workspace: torch.Tensor, stream=None) -> None:
    """Decode attention over the rotated 4-bit cache; arguments as kvq_decode_attention."""
    B, Hq = int(q.shape[0]), int(q.shape[1])
    rc = lib().kvq_wht4_decode_attention(
        C.byref(cfg), _dev(pool, "pool", torch.uint8), _dev(q, "q", torch.float16),
        _dev(block_table, "block_table", torch.int32), int(block_table.shape[1]),
        _dev(seq_lens, "seq_lens", torch.int32), B, Hq, int(max_len), float(softmax_scale),
        _dev(out, "out", torch.float32), _dev(workspace, "workspace", torch.uint8), workspace.numel(),
        _stream(stream))
    _check(rc)


def kvq_decode_step_host(cfg: CacheConfig, pool: torch.Tensor, host_in: torch.Tensor, dev_in: torch.Tensor,
                         append_pos: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor, batch: int,
                         num_q_heads: int, max_len: int, softmax_scale: float, out: torch.Tensor,
                         host_out: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """The decode step from host memory in one call: host_in (pinned fp16 q, k_new, v_new back to back)
    is copied to dev_in, the step runs, out is copied to host_out (pinned fp32)."""
    if host_in.is_cuda or host_out.is_cuda:
        raise ValueError("host_in and host_out must be host tensors")
    if host_in.dtype != torch.float16 or host_out.dtype != torch.float32:
        raise ValueError("host_in must be float16 and host_out float32")
    if host_in.numel() != dev_in.numel() or host_out.numel() != out.numel():
        raise ValueError("host and device buffers differ in size")
    rc = lib().kvq_decode_step_host(
        C.byref(cfg), _dev(pool, "pool", torch.uint8), host_in.data_ptr(), _dev(dev_in, "dev_in", torch.float16),
        _dev(append_pos, "append_pos", torch.int32), _dev(block_table, "block_table", torch.int32),
        int(block_table.shape[1]), _dev(seq_lens, "seq_lens", torch.int32), int(batch), int(num_q_heads),
        int(max_len), float(softmax_scale), _dev(out, "out", torch.float32), host_out.data_ptr(),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(rc)


def kvq_decode_step_host_pipelined(cfg: CacheConfig, pool: torch.Tensor, host_in: torch.Tensor, dev_in: torch.Tensor,
                                   append_pos: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                                   batch: int, num_q_heads: int, max_len: int, softmax_scale: float, out: torch.Tensor,
                                   host_out: torch.Tensor, workspace: torch.Tensor, stream, copy_in, copy_out,
                                   events) -> None:
    """kvq_decode_step_host with its copies on copy_in / copy_out: events are the staging slot's three
    torch.cuda.Event objects (input copied, step done, output copied), each recorded at least once so
    that it exists."""
    if host_in.is_cuda or host_out.is_cuda:
        raise ValueError("host_in and host_out must be host tensors")
    if host_in.dtype != torch.float16 or host_out.dtype != torch.float32:
        raise ValueError("host_in must be float16 and host_out float32")
    if host_in.numel() != dev_in.numel() or host_out.numel() != out.numel():
        raise ValueError("host and device buffers differ in size")
    handles = (C.c_void_p * 3)(*[int(ev.cuda_event) for ev in events])
    if not all(handles):
        raise ValueError("each event must have been recorded once (torch creates events on first record)")
    rc = lib().kvq_decode_step_host_pipelined(
        C.byref(cfg), _dev(pool, "pool", torch.uint8), host_in.data_ptr(), _dev(dev_in, "dev_in", torch.float16),
        _dev(append_pos, "append_pos", torch.int32), _dev(block_table, "block_table", torch.int32),
        int(block_table.shape[1]), _dev(seq_lens, "seq_lens", torch.int32), int(batch), int(num_q_heads),
        int(max_len), float(softmax_scale), _dev(out, "out", torch.float32), host_out.data_ptr(),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream), _stream(copy_in),
        _stream(copy_out), handles)
    _check(rc)


def kvq_test_decode_wait_timeout(cfg: CacheConfig, pool: torch.Tensor, q: torch.Tensor, block_table: torch.Tensor,
                                 seq_lens: torch.Tensor, max_len: int, softmax_scale: float, out: torch.Tensor,
                                 workspace: torch.Tensor, wait_limit_ns: int, stream=None) -> None:
    """The bounded-wait test of the decode kernel (the test suite's): its waits run out and it
    raises KVQ_FLAG_WAIT_TIMEOUT in the workspace status word."""
    B, Hq = int(q.shape[0]), int(q.shape[1])
    rc = lib().kvq_test_decode_wait_timeout(
        C.byref(cfg), _dev(pool, "pool", torch.uint8), _dev(q, "q", torch.float16),
        _dev(block_table, "block_table", torch.int32), int(block_table.shape[1]),
        _dev(seq_lens, "seq_lens", torch.int32), B, Hq, int(max_len), float(softmax_scale),
        _dev(out, "out", torch.float32), _dev(workspace, "workspace", torch.uint8), workspace.numel(),
        int(wait_limit_ns), _stream(stream))
    _check(rc)

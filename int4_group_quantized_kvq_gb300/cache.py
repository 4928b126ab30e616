"""One layer's INT4 paged KV cache on the GPU and its decode step.

A thin holder of device buffers (torch allocates them; the library allocates
nothing) around the C ABI calls of a decode step:

    quantize-on-append of the new token's K/V  ->  kvq_quantize_append
    decode attention over the packed cache      ->  kvq_decode_attention
    both in one call (append fused in)          ->  kvq_decode_step

With ``window > 0`` the attention is restricted to the last ``window`` positions and
the first ``sinks`` (``kvq_decode_attention_window`` / ``kvq_decode_step_window``).

``decode_step_host`` is the same step driven from pinned host buffers (``HostStaging``):
the step's q, K and V are copied in with one transfer and the output copied back, on
the same stream.
"""
from __future__ import annotations

import math

import torch

from . import binding as B


class PagedKVCache:
    def __init__(self, cfg: B.CacheConfig, block_table: torch.Tensor, num_q_heads: int, max_len: int,
                 device="cuda", pool: torch.Tensor | None = None, window: int = 0, sinks: int = 0):
        self.cfg = cfg
        self.window = int(window)
        self.sinks = int(sinks)
        self.device = torch.device(device)
        self.block_table = block_table.to(self.device, torch.int32).contiguous()
        self.batch = int(self.block_table.shape[0])
        self.num_q_heads = int(num_q_heads)
        self.max_len = int(max_len)
        nbytes = B.kvq_pool_bytes(cfg)
        if pool is None:
            pool = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
        if pool.numel() < nbytes:
            raise ValueError(f"pool has {pool.numel()} bytes, needs {nbytes}")
        self.pool = pool
        self.workspace = B.new_workspace(cfg, self.batch, self.num_q_heads, self.max_len, device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.softmax_scale = 1.0 / math.sqrt(cfg.head_dim)

    def append(self, k: torch.Tensor, v: torch.Tensor, start_pos: torch.Tensor, stream=None) -> None:
        """Quantize k, v [B, n, Hkv, d] fp16 into positions start_pos[b] .. start_pos[b] + n - 1."""
        B.kvq_quantize_append(self.cfg, self.pool, k, v, self.block_table, start_pos, status=self.status,
                              stream=stream)

    def attend(self, q: torch.Tensor, seq_lens: torch.Tensor, out: torch.Tensor, stream=None) -> None:
        """Decode attention of q [B, Hq, d] fp16 over positions 0 .. seq_lens[b]-1 into out (fp32)."""
        if self.window > 0:
            B.kvq_decode_attention_window(self.cfg, self.pool, q, self.block_table, seq_lens, self.max_len,
                                          self.softmax_scale, self.window, self.sinks, out, self.workspace,
                                          stream=stream)
        else:
            B.kvq_decode_attention(self.cfg, self.pool, q, self.block_table, seq_lens, self.max_len,
                                   self.softmax_scale, out, self.workspace, stream=stream)

    def decode_step(self, q, k_new, v_new, append_pos, seq_lens, out, stream=None) -> None:
        """Append one token per sequence at append_pos, then attend over seq_lens (which include it):
        one kvq_decode_step call."""
        if self.window > 0:
            B.kvq_decode_step_window(self.cfg, self.pool, k_new, v_new, append_pos, q, self.block_table, seq_lens,
                                     self.max_len, self.softmax_scale, self.window, self.sinks, out, self.workspace,
                                     stream=stream)
        else:
            B.kvq_decode_step(self.cfg, self.pool, k_new, v_new, append_pos, q, self.block_table, seq_lens,
                              self.max_len, self.softmax_scale, out, self.workspace, stream=stream)

    def decode_step_two_calls(self, q, k_new, v_new, append_pos, seq_lens, out, stream=None) -> None:
        """The same step as two calls: kvq_quantize_append, then kvq_decode_attention."""
        self.append(k_new, v_new, append_pos, stream)
        self.attend(q, seq_lens, out, stream)

    def decode_step_host(self, staging: "HostStaging", append_pos, seq_lens, stream=None) -> None:
        """The decode step from pinned host memory: one H2D copy of the step's q, K and V (staged
        back to back), the step (the decode and combine launches), one D2H copy of the output.
        All asynchronous on the step's stream; without a window, one kvq_decode_step_host call."""
        s = torch.cuda.current_stream() if stream is None else stream
        if self.window == 0:
            B.kvq_decode_step_host(self.cfg, self.pool, staging.host, staging.dev, append_pos, self.block_table,
                                   seq_lens, self.batch, self.num_q_heads, self.max_len, self.softmax_scale,
                                   staging.out, staging.out_host, self.workspace, stream=s)
            return
        with torch.cuda.stream(s):
            staging.dev.copy_(staging.host, non_blocking=True)
            self.decode_step(staging.q, staging.k_new, staging.v_new, append_pos, seq_lens, staging.out, stream=s)
            staging.out_host.copy_(staging.out, non_blocking=True)

    def flags(self) -> int:
        """Status flags of the last calls (synchronizes)."""
        return B.kvq_read_status(self.status) | B.kvq_read_status(self.workspace)


class HostStaging:
    """Pinned host buffers and their device twins for one decode step: q [B, Hq, d], k_new and
    v_new [B, Hkv, d] fp16 back to back (so a step copies its inputs in one transfer), and the
    fp32 output [B, Hq, d].  Fill `q_host`, `k_host`, `v_host` on the host; read `out_host`
    after the stream has passed the step."""

    def __init__(self, batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int, device="cuda"):
        nq = batch * num_q_heads * head_dim
        nk = batch * num_kv_heads * head_dim
        self.host = torch.empty(nq + 2 * nk, dtype=torch.float16).pin_memory()
        self.dev = torch.empty(nq + 2 * nk, dtype=torch.float16, device=device)
        shq = (batch, num_q_heads, head_dim)
        shk = (batch, num_kv_heads, head_dim)
        self.q_host = self.host[:nq].view(shq)
        self.k_host = self.host[nq:nq + nk].view(shk)
        self.v_host = self.host[nq + nk:].view(shk)
        self.q = self.dev[:nq].view(shq)
        self.k_new = self.dev[nq:nq + nk].view(shk)
        self.v_new = self.dev[nq + nk:].view(shk)
        self.out = torch.empty(shq, dtype=torch.float32, device=device)
        self.out_host = torch.empty(shq, dtype=torch.float32).pin_memory()

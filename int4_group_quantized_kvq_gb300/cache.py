"""One layer's INT4 paged KV cache on the GPU and its decode step.

A thin holder of device buffers (torch allocates them; the library allocates
nothing) around the C ABI calls of a decode step:

    quantize-on-append of the new token's K/V  ->  kvq_quantize_append
    decode attention over the packed cache      ->  kvq_decode_attention
    both in one call (append fused in)          ->  kvq_decode_step

With ``window > 0`` the attention is restricted to the last ``window`` positions and
the first ``sinks`` (``kvq_decode_attention_window`` / ``kvq_decode_step_window``).

``decode_step_host`` is the same step driven from pinned host buffers (``HostStaging``)
in one kvq_decode_step_host call: the step's q, K and V are copied in with one transfer
and the output copied back, on the same stream; ``HostPipeline`` overlaps those copies
with the neighbouring steps (kvq_decode_step_host_pipelined).
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
        """The decode step from pinned host memory in one kvq_decode_step_host call: one H2D copy of
        the step's q, K and V (staged back to back), the step, one D2H copy of the output, all
        asynchronous on the step's stream."""
        if self.window > 0:
            raise ValueError("the host step attends to every position (no window)")
        B.kvq_decode_step_host(self.cfg, self.pool, staging.host, staging.dev, append_pos, self.block_table, seq_lens,
                               self.batch, self.num_q_heads, self.max_len, self.softmax_scale, staging.out,
                               staging.out_host, self.workspace, stream=stream)

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


class HostPipeline:
    """Decode steps fed from pinned host memory with the copies overlapped with the kernels:
    one kvq_decode_step_host_pipelined call per step.

    Two staging slots alternate.  Step i (slot i % 2) copies its inputs host-to-device on an
    input copy stream, runs on the compute stream once that copy is done, and copies its
    output device-to-host on an output copy stream once the step is done; so step i + 1's
    inputs move while step i computes, and step i's output moves while step i + 1 computes.
    The slot's three events (input copied, step done, output copied) keep its device buffers
    from being overwritten while in use: a slot's input copy waits for the step two back to
    have read that slot, and its step waits for that step's output copy to have left the slot.
    The host side is the caller's: fill `slot(i)`'s host inputs before `step(i)` (for i >= 2,
    after `inputs_copied(i - 2)`), and read its `out_host` after `done(i)` and before
    `step(i + 2)`."""

    def __init__(self, cache: PagedKVCache, compute_stream=None):
        self.cache = cache
        dev = cache.device
        self.slots = [HostStaging(cache.batch, cache.num_q_heads, cache.cfg.num_kv_heads, cache.cfg.head_dim, dev)
                      for _ in range(2)]
        self.compute = torch.cuda.Stream(device=dev) if compute_stream is None else compute_stream
        self.copy_in = torch.cuda.Stream(device=dev)
        self.copy_out = torch.cuda.Stream(device=dev)
        # per slot: input copied, step done, output copied; recorded once so that they exist
        self.events = [[torch.cuda.Event() for _ in range(3)] for _ in range(2)]
        for evs in self.events:
            for ev in evs:
                ev.record(self.compute)
        self.compute.synchronize()

    def slot(self, i: int) -> HostStaging:
        return self.slots[i % 2]

    def step(self, i: int, append_pos: torch.Tensor, seq_lens: torch.Tensor, cache: PagedKVCache | None = None) -> None:
        """Step i on `cache` (default: the pipeline's), from slot(i)'s host inputs to its out_host."""
        cache = self.cache if cache is None else cache
        st = self.slots[i % 2]
        if cache.window > 0:
            raise ValueError("the pipelined host step attends to every position (no window)")
        B.kvq_decode_step_host_pipelined(cache.cfg, cache.pool, st.host, st.dev, append_pos, cache.block_table,
                                         seq_lens, cache.batch, cache.num_q_heads, cache.max_len,
                                         cache.softmax_scale, st.out, st.out_host, cache.workspace, self.compute,
                                         self.copy_in, self.copy_out, self.events[i % 2])

    def inputs_copied(self, i: int) -> torch.cuda.Event:
        """The event after which step i's host inputs have been read (slot(i) may be refilled)."""
        return self.events[i % 2][0]

    def done(self, i: int) -> torch.cuda.Event:
        """The event after which step i's output is in slot(i).out_host (until step i + 2 is issued)."""
        return self.events[i % 2][2]

    def synchronize(self) -> None:
        for s in (self.copy_in, self.compute, self.copy_out):
            s.synchronize()

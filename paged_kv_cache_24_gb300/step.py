"""DecodeStep: one serving decode step (slot mapping, append, decode) as a
replayable CUDA graph fed from pinned host memory.

With ``fused=True`` (the default) the step is ``pkv_append_decode`` -- the
new token of each sequence sits at position ``context_lens - 1`` -- in one
launch; ``fused=False`` runs the three separate calls.

A step's host inputs -- the queries, the new tokens' K and V, their positions,
the context lengths and (optionally) the block tables -- are packed into one
pinned staging buffer.  The kernels read the queries and the new K/V
straight from it over the host link, and the rest (positions, lengths, block
tables) reaches the device first in a single ``pkv_stage_copy`` kernel that
reads the pinned buffer directly (the copy engine where the GPU cannot reach
it); with ``direct_in=False`` everything is copied in that way.  The
attention output comes back in a second copy of that kind, or, with
``direct_out=True``, the decode kernels write it straight into a pinned host
buffer (the default when every context is planned as one split, so that no
combine pass writes the rows at the end).  The graph replays
``pkv_slot_mapping``, ``pkv_append`` and ``pkv_decode`` exactly as the eager
calls would run them.  The K/V pools stay resident on the device.

Several staging buffers can be kept (``num_buffers``), one graph each, so a
caller can fill the next step's inputs while the current one runs.

Usage::

    step = DecodeStep(k_cache, v_cache, num_seqs, num_q_heads, max_blocks,
                      window=0, scale=1 / math.sqrt(head_dim))
    step.host[0]["q"].copy_(q_cpu); step.host[0]["k"].copy_(k_cpu); ...
    out_cpu = step.run(0)          # waits for the result
"""
from __future__ import annotations

import torch

from ._binding import (cache_layout, pkv_append, pkv_append_decode, pkv_append_fp8,
                       pkv_append_int8, pkv_decode, pkv_decode_plan, pkv_device_address,
                       pkv_slot_mapping, pkv_stage_copy, PKV_ERR_UNSUPPORTED)

_ALIGN = 256


class DecodeStep:
    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor, num_seqs: int,
                 num_q_heads: int, max_blocks: int, window: int, scale: float,
                 copy_block_tables: bool = True, num_buffers: int = 1, use_graph: bool = True,
                 fused: bool = True, k_scale: torch.Tensor | None = None,
                 v_scale: torch.Tensor | None = None, direct_out: bool | None = None,
                 direct_in: bool = True):
        layout = cache_layout(k_cache)
        self.k_cache, self.v_cache = k_cache, v_cache
        self.window, self.scale = int(window), float(scale)
        self.block_size = layout.block_size
        # 8-bit pools (uint8 E4M3 / int8 codes) append through the quantising call
        self.q8 = k_cache.dtype in (torch.uint8, torch.int8)
        if self.q8 and fused:
            raise ValueError("8-bit pools append through pkv_append_fp8 / pkv_append_int8: "
                             "use fused=False")
        self.k_scale, self.v_scale = k_scale, v_scale
        self.fused = fused
        dev = k_cache.device
        dt = torch.float16 if self.q8 else k_cache.dtype
        B, hq, hkv, d = num_seqs, num_q_heads, layout.num_kv_heads, layout.head_dim
        shapes = {
            "q": ((B, hq, d), dt), "k": ((B, hkv, d), dt), "v": ((B, hkv, d), dt),
            "positions": ((B,), torch.int64), "context_lens": ((B,), torch.int32),
            "block_tables": ((B, max_blocks), torch.int32),
        }
        offsets, cur = {}, 0
        for name, (shape, t) in shapes.items():
            n = 1
            for s in shape:
                n *= s
            nbytes = n * torch.tensor([], dtype=t).element_size()
            offsets[name] = (cur, nbytes, shape, t)
            cur += (nbytes + _ALIGN - 1) // _ALIGN * _ALIGN
        # block tables sit last so that leaving them out shortens the copy
        self._staged_bytes = cur if copy_block_tables else offsets["block_tables"][0]

        def views(buf):
            return {name: buf[o:o + nb].view(t).view(shape)
                    for name, (o, nb, shape, t) in offsets.items()}

        self._host_bufs = [torch.empty(cur, dtype=torch.uint8).pin_memory()
                           for _ in range(num_buffers)]
        # direct_in: the decode (and, on the separate path, append) kernels read
        # the queries and the new K/V straight from the pinned buffer over the
        # host link; only the positions, lengths and block tables are copied
        # in first.
        # Measured on the MHA step: 0.3511 ms against 0.3658 with everything
        # copied in first (the copy of 1.5 MB no longer precedes the decode).
        self.direct_in = (direct_in and
                          all(pkv_device_address(b) is not None for b in self._host_bufs))
        self._stage_start = offsets["positions"][0] if self.direct_in else 0
        self.host = [views(b) for b in self._host_bufs]   # fill these, then run(i)
        self._dev_buf = torch.empty(cur, dtype=torch.uint8, device=dev)
        self.device = views(self._dev_buf)
        self.slots = torch.empty(B, dtype=torch.int64, device=dev)
        self.out = torch.empty((B, hq, d), dtype=dt, device=dev)
        self.host_out = torch.empty((B, hq, d), dtype=dt).pin_memory()
        # direct_out: the decode writes the result straight into the pinned
        # buffer where the GPU can address it, instead of a copy back after it.
        # By default only when the plan gives every context one split: then
        # the decode's CTAs write their rows over the host link while the
        # launch runs (the serving mix, 8 MB of output a step: 0.3030 ->
        # 0.2566 ms a step end to end); with a combine pass, that pass would
        # write every row over the link at the end, and the copy back is
        # faster (device time a step: the GQA step 0.704 against 0.728 ms,
        # the MHA step 0.3367 against 0.3382).
        if direct_out is None:
            direct_out = pkv_decode_plan(num_seqs, num_q_heads, layout, max_blocks,
                                         self.window)[1] == 1
        self.direct_out = direct_out and pkv_device_address(self.host_out) is not None
        self.h2d_bytes = self._staged_bytes
        self.d2h_bytes = self.host_out.numel() * self.host_out.element_size()
        # (the graphs are captured on a stream of their own and replayed on
        # the caller's)
        self.stream = torch.cuda.Stream(device=dev)
        self._device = dev.index if dev.index is not None else torch.cuda.current_device()
        self.graphs = None
        if use_graph:
            # an eager pass with empty contexts and no writes sizes the decode
            # workspace before capture
            for h in self.host:
                h["context_lens"].zero_()
                h["positions"].fill_(-1)
            self.stream.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(self.stream):
                self._enqueue(0)
            self.stream.synchronize()
            self.graphs = []
            for i in range(num_buffers):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.stream):
                    self._enqueue(i)
                self.graphs.append(g)

    def _copy(self, dst, src, n):
        # a kernel copy where the GPU reaches the pinned buffer directly (fewer
        # microseconds of fixed cost than a copy-engine transfer of these
        # sizes), else the copy engine
        if pkv_stage_copy(dst, src, n) == PKV_ERR_UNSUPPORTED:
            dst.view(-1)[:n // dst.element_size()].copy_(
                src.view(-1)[:n // src.element_size()], non_blocking=True)

    def _enqueue(self, i):
        a = self._stage_start
        self._copy(self._dev_buf[a:], self._host_bufs[i][a:], self._staged_bytes - a)
        dv = self.device
        src = self.host[i] if self.direct_in else dv
        out = self.host_out if self.direct_out else self.out
        if self.fused:
            # the new token sits at position context_lens - 1: one launch
            pkv_append_decode(src["q"], src["k"], src["v"], self.k_cache, self.v_cache,
                              dv["block_tables"], dv["context_lens"], self.window, self.scale,
                              out=out)
        else:
            pkv_slot_mapping(dv["block_tables"], dv["positions"], self.block_size,
                             out=self.slots)
            if self.q8:
                append = pkv_append_int8 if self.k_cache.dtype == torch.int8 else pkv_append_fp8
                append(src["k"], src["v"], self.slots, self.k_cache, self.v_cache, self.k_scale,
                       self.v_scale)
            else:
                pkv_append(src["k"], src["v"], self.slots, self.k_cache, self.v_cache)
            pkv_decode(src["q"], self.k_cache, self.v_cache, dv["block_tables"],
                       dv["context_lens"], self.window, self.scale, out=out,
                       k_scale=self.k_scale, v_scale=self.v_scale)
        if not self.direct_out:
            self._copy(self.host_out, self.out, self.d2h_bytes)

    def run(self, i: int = 0, wait: bool = True) -> torch.Tensor:
        """Run step i from staging buffer i on the caller's current stream
        (the pools' device must be current): after whatever the caller
        queued there, before whatever it queues next.  With ``wait`` the call
        returns once the output is in ``host_out``.  (Replaying on the
        caller's stream needs no cross-stream event a step: a GQA step end to
        end measured 0.711 ms this way, 0.724 through a stream of its own.)"""
        if torch.cuda.current_device() != self._device:
            raise RuntimeError("DecodeStep.run: make the pools' device current first")
        if self.graphs is not None:
            self.graphs[i].replay()
        else:
            self._enqueue(i)
        if wait:
            torch.cuda.current_stream(self._device).synchronize()
        return self.host_out

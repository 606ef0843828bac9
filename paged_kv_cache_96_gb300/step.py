"""One paged attention step on the GPU, driven through the C ABI.

A step, in the order the serving engine of the pages runs it
("vLLM源码解析(二)" §4.1 engine step; "PagedAttention & Continuous
Batching" §1.5, §1.6, §2.4, §2.5):

  1. slot mapping of the step's new tokens (one per running sequence for
     decode; a chunk of tokens per sequence for chunked prefill),
  2. reshape_and_cache of their K/V into the paged pools,
  3. copy-on-write block copies, when the step has any,
  4. attention: paged decode of every sequence over its whole context
     (single pass, or split-context partitions merged by a reduce; with a
     prefix plan, each group's shared prefix read once), or, for a prefill
     step, each chunk row over the context up to its own position.

A decode step with one new token per sequence runs 3 first and then 1, 2
and 4 in one call (the append fused into the attention pass), the order in
which the engine copies a shared block before writing into it.

Torch provides device memory and the stream; every step above is a kernel
of ``libpaged_attention.so``.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import binding as B
from .workloads import Workload


def _t16(a: np.ndarray, dtype: str, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    t = t.view(torch.float16 if dtype == "f16" else torch.bfloat16)
    return t.to(device)


def _ti(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


class DecodeStep:
    """Device state of one workload: pools holding the cached history,
    the step's inputs, and the output / workspace buffers."""

    def __init__(self, w: Workload, device: str = "cuda",
                 partition_size: Optional[int] = None, build_pools: bool = True):
        self.w = w
        self.device = torch.device(device)
        self.partition_size = (w.spec.partition_size if partition_size is None
                               else partition_size)
        dt = w.dtype
        self.torch_dtype = torch.float16 if dt == "f16" else torch.bfloat16
        self.max_context_len = int(w.context_lens.max())
        shape = w.pool_shape()
        self.fp8 = w.fp8
        self.kv_scale = float(w.spec.kv_scale)
        if self.fp8:
            # e4m3 codes; 0x7F is NaN
            self.key_cache = torch.full(shape, 0x7F, dtype=torch.uint8, device=self.device)
            self.value_cache = torch.full(shape, 0x7F, dtype=torch.uint8, device=self.device)
        else:
            fill = int(np.int16(np.uint16(w.fill).view(np.int16)))
            self.key_cache = torch.full(shape, fill, dtype=torch.int16,
                                        device=self.device).view(self.torch_dtype)
            self.value_cache = torch.full(shape, fill, dtype=torch.int16,
                                          device=self.device).view(self.torch_dtype)
        self.block_tables = _ti(w.block_tables, self.device)
        self.step_block_tables = _ti(w.step_block_tables, self.device)
        self.context_lens = _ti(w.context_lens, self.device)
        self.query = _t16(w.query, dt, self.device)
        self.new_seq = _ti(w.new_seq, self.device)
        self.new_pos = _ti(w.new_pos, self.device)
        self.new_key = _t16(w.new_key, dt, self.device)
        self.new_value = _t16(w.new_value, dt, self.device)
        self.cow_pairs = _ti(w.cow_pairs, self.device) if w.cow_pairs.shape[0] else None
        self.query_start = _ti(w.query_start, self.device)
        self.slots = torch.empty(w.new_seq.shape[0], dtype=torch.int32, device=self.device)
        self.out = torch.empty((w.T, w.H, w.D), dtype=self.torch_dtype, device=self.device)
        self.error_word = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.cascade = bool(w.spec.cascade)
        self.plan = None
        if w.prefill:
            self.workspace = None
        elif self.cascade:
            # host planner over the step's tables (the tables attention reads)
            plan, self.num_groups, self.num_members = B.pa_plan_prefix_groups(
                w.step_block_tables, w.context_lens, w.bs)
            self.plan = plan.to(self.device)
            n = B.pa_cascade_workspace_bytes(w.S, w.H, w.Hkv, w.D, self.max_context_len,
                                             self.partition_size)
            self.workspace = torch.zeros(n, dtype=torch.uint8, device=self.device)
        else:
            self.workspace = B.alloc_workspace(w.S, w.H, w.Hkv, w.D, self.max_context_len,
                                               self.partition_size, device=self.device)
        # Decode with one new token per sequence, at its last position, and
        # that position in the same block before and after copy-on-write: the
        # append runs inside the attention call.
        self.fused_append = False
        if not w.prefill and w.new_seq.shape[0] == w.S:
            last = w.context_lens.astype(np.int64) - 1
            if (np.array_equal(w.new_seq, np.arange(w.S)) and
                    np.array_equal(w.new_pos, last) and bool((last >= 0).all())):
                rows = np.arange(w.S)
                lb = last // w.bs
                self.fused_append = bool(np.array_equal(w.block_tables[rows, lb],
                                                        w.step_block_tables[rows, lb]))
        if build_pools:
            self.write_history()

    def write_history(self, chunk: int = 1 << 18) -> None:
        """Cache the workload's history tokens through the library's own
        slot mapping and reshape_and_cache (the prefill writes)."""
        w = self.w
        n = w.hist_seq.shape[0]
        for lo in range(0, n, chunk):
            hi = min(n, lo + chunk)
            seq = _ti(w.hist_seq[lo:hi], self.device)
            pos = _ti(w.hist_pos[lo:hi], self.device)
            k = _t16(w.hist_key[lo:hi], w.dtype, self.device)
            v = _t16(w.hist_value[lo:hi], w.dtype, self.device)
            slots = torch.empty(hi - lo, dtype=torch.int32, device=self.device)
            B.pa_slot_mapping(slots, self.block_tables, seq, pos, w.bs, w.num_blocks,
                              error_word=self.error_word)
            self._cache_write(k, v, slots)

    def _cache_write(self, k, v, slots, stream=None) -> None:
        if self.fp8:
            B.pa_reshape_and_cache_fp8(k, v, self.key_cache, self.value_cache, slots,
                                       self.kv_scale, self.kv_scale,
                                       error_word=self.error_word, stream=stream)
        else:
            B.pa_reshape_and_cache(k, v, self.key_cache, self.value_cache, slots,
                                   error_word=self.error_word, stream=stream)

    # individual steps ---------------------------------------------------------
    def slot_mapping(self, stream=None) -> None:
        B.pa_slot_mapping(self.slots, self.block_tables, self.new_seq, self.new_pos,
                          self.w.bs, self.w.num_blocks, error_word=self.error_word,
                          stream=stream)

    def reshape_and_cache(self, stream=None) -> None:
        self._cache_write(self.new_key, self.new_value, self.slots, stream)

    def copy_blocks(self, stream=None) -> None:
        if self.cow_pairs is not None:
            B.pa_copy_blocks(self.key_cache, self.value_cache, self.cow_pairs,
                             error_word=self.error_word, stream=stream)

    def attention(self, stream=None, partition_size: Optional[int] = None) -> None:
        w = self.w
        if w.prefill:
            B.pa_prefill_attention(self.out, self.query, self.key_cache, self.value_cache,
                                   self.step_block_tables, self.query_start,
                                   self.context_lens, self.max_context_len, w.scale,
                                   error_word=self.error_word, stream=stream,
                                   k_scale=self.kv_scale, v_scale=self.kv_scale)
            return
        P = self.partition_size if partition_size is None else partition_size
        if self.cascade:
            ws = self.workspace
            if P != self.partition_size:
                n = B.pa_cascade_workspace_bytes(w.S, w.H, w.Hkv, w.D, self.max_context_len, P)
                ws = torch.zeros(n, dtype=torch.uint8, device=self.device)
            B.pa_decode_attention_cascade(self.out, self.query, self.key_cache,
                                          self.value_cache, self.step_block_tables,
                                          self.context_lens, self.max_context_len, w.scale,
                                          self.plan, self.num_groups, self.num_members, P, ws,
                                          error_word=self.error_word, stream=stream,
                                          k_scale=self.kv_scale, v_scale=self.kv_scale)
            return
        ws = self.workspace
        if P != self.partition_size:
            ws = B.alloc_workspace(self.w.S, self.w.H, self.w.Hkv, self.w.D,
                                   self.max_context_len, P, device=self.device)
        if self.fp8:
            B.pa_decode_attention_fp8(self.out, self.query, self.key_cache, self.value_cache,
                                      self.step_block_tables, self.context_lens,
                                      self.max_context_len, self.w.scale, self.kv_scale,
                                      self.kv_scale, P, ws, error_word=self.error_word,
                                      stream=stream)
        else:
            B.pa_decode_attention(self.out, self.query, self.key_cache, self.value_cache,
                                  self.step_block_tables, self.context_lens,
                                  self.max_context_len, self.w.scale, P, ws,
                                  error_word=self.error_word, stream=stream)

    def slot_mapping_and_cache(self, stream=None) -> None:
        """Steps 1 and 2 in one launch (slots computed where they are used)."""
        B.pa_slot_mapping_and_cache(self.slots, self.block_tables, self.new_seq, self.new_pos,
                                    self.new_key, self.new_value, self.key_cache,
                                    self.value_cache, self.kv_scale, self.kv_scale,
                                    error_word=self.error_word, stream=stream)

    def append_attention(self, stream=None, partition_size: Optional[int] = None) -> None:
        """Steps 1, 2 and 4 of a decode step in one call: each sequence's new
        token goes to the pools inside the attention pass."""
        if not self.fused_append:
            raise RuntimeError("this step's new tokens are not one per sequence at its end")
        w = self.w
        P = self.partition_size if partition_size is None else partition_size
        ws = self.workspace
        if self.cascade:
            if P != self.partition_size:
                n = B.pa_cascade_workspace_bytes(w.S, w.H, w.Hkv, w.D, self.max_context_len, P)
                ws = torch.zeros(n, dtype=torch.uint8, device=self.device)
            B.pa_decode_attention_cascade_append(
                self.out, self.query, self.key_cache, self.value_cache, self.new_key,
                self.new_value, self.step_block_tables, self.context_lens, self.max_context_len,
                w.scale, self.plan, self.num_groups, self.num_members, P, ws,
                slot_mapping=self.slots, error_word=self.error_word, stream=stream,
                k_scale=self.kv_scale, v_scale=self.kv_scale)
            return
        if P != self.partition_size:
            ws = B.alloc_workspace(w.S, w.H, w.Hkv, w.D, self.max_context_len, P,
                                   device=self.device)
        B.pa_decode_attention_append(self.out, self.query, self.key_cache, self.value_cache,
                                     self.new_key, self.new_value, self.step_block_tables,
                                     self.context_lens, self.max_context_len, w.scale, P, ws,
                                     slot_mapping=self.slots, k_scale=self.kv_scale,
                                     v_scale=self.kv_scale, error_word=self.error_word,
                                     stream=stream)

    def run(self, stream=None) -> torch.Tensor:
        """One whole decode step; returns the attention output tensor.  A
        decode step whose new tokens are one per sequence copies its
        copy-on-write blocks first and then appends and attends in one call;
        other steps write, copy, then attend."""
        if self.fused_append:
            self.copy_blocks(stream)
            self.append_attention(stream)
            return self.out
        self.slot_mapping_and_cache(stream)
        self.copy_blocks(stream)
        self.attention(stream)
        return self.out

    def launches_per_step(self) -> int:
        """Kernels one run() launches: slot mapping with the cache write (unless
        fused into the attention pass), block copy (when the step has
        copy-on-write pairs), the attention pass (which merges split contexts
        of up to 8 partials itself), the shared-prefix pass (prefix-aware
        decode with at least one group), and the reduce (when a sequence may
        have more than 8 partials)."""
        n = (1 if self.fused_append else 2) + (1 if self.cow_pairs is not None else 0)
        if self.w.prefill:
            return n
        P = self.partition_size
        parts = -(-self.max_context_len // P) if P > 0 and self.max_context_len > 0 else 1
        if self.cascade and self.num_groups > 0:
            n += 1
            parts += 1  # the shared prefix's partial
        if parts > 8:
            n += 1
        return n


def to_bits(t: torch.Tensor) -> np.ndarray:
    """Device 16-bit tensor -> host uint16 bit patterns (uint8 stays uint8)."""
    if t.dtype == torch.uint8:
        return t.detach().contiguous().cpu().numpy()
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_float(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


class HostStepIO:
    """Decode steps driven from host memory, as a serving loop runs them:
    every step copies its inputs (query, new K/V, their sequence ids and
    positions, block tables, context lengths, copy-on-write pairs) from a
    pinned host staging buffer to the device in one transfer, runs the step,
    and copies the attention output back to a pinned host buffer.

    Uploads and read-backs each run on a stream of their own and are
    double-buffered: step i's inputs go into staging slot i % 2 (the step's
    input tensors become views into it, each at a 256-byte aligned offset, so
    the kernels read them in place) while step i - 1 computes, and step i's
    output is read back while step i + 1 computes.  A slot's inputs are
    refilled only after the step that last read them has finished, and its
    output is rewritten only after it has been read back.  The K/V pools stay
    resident on the device.  Bracket a run of steps with begin() and finish()
    so that the transfer streams are ordered inside it."""

    def __init__(self, st: DecodeStep):
        self.st = st
        names = ["query", "new_key", "new_value", "new_seq", "new_pos", "block_tables",
                 "step_block_tables", "context_lens"]
        if st.cow_pairs is not None:
            names.append("cow_pairs")
        if st.w.prefill:
            names.append("query_start")
        if st.plan is not None:
            names.append("plan")
        layout, total = [], 0
        for n in names:
            t = getattr(st, n)
            nbytes = t.numel() * t.element_size()
            layout.append((n, total, nbytes, t.dtype, t.shape))
            total += (nbytes + 255) & ~255
        self.dev_bufs = [torch.empty(total, dtype=torch.uint8, device=st.device)
                         for _ in range(2)]
        self.host_bufs = [torch.empty(total, dtype=torch.uint8, pin_memory=True)
                          for _ in range(2)]
        self.views = [{}, {}]
        for slot in range(2):
            for n, off, nbytes, dtype, shape in layout:
                t = getattr(st, n)
                self.host_bufs[slot][off:off + nbytes].view(dtype).view(shape).copy_(t)
                self.views[slot][n] = self.dev_bufs[slot][off:off + nbytes].view(dtype).view(shape)
        self.outs = [st.out, torch.empty_like(st.out)]
        self.host_outs = [torch.empty(st.out.shape, dtype=st.out.dtype, pin_memory=True)
                          for _ in range(2)]
        self.h2d_bytes = total
        self.d2h_bytes = self.host_outs[0].numel() * self.host_outs[0].element_size()
        self.up = torch.cuda.Stream(device=st.device)
        self.down = torch.cuda.Stream(device=st.device)
        self.in_ready = [torch.cuda.Event() for _ in range(2)]
        self.step_done = [torch.cuda.Event() for _ in range(2)]
        self.out_read = [torch.cuda.Event() for _ in range(2)]
        self.used = [False, False]
        self.i = 0

    def begin(self, stream: torch.cuda.Stream) -> None:
        """Order the transfer streams after everything queued so far on `stream`."""
        self.up.wait_stream(stream)
        self.down.wait_stream(stream)

    def finish(self, stream: torch.cuda.Stream) -> None:
        """Order `stream` after the last upload and read-back."""
        stream.wait_stream(self.up)
        stream.wait_stream(self.down)

    def step(self) -> torch.Tensor:
        slot = self.i % 2
        main = torch.cuda.current_stream(self.st.device)
        with torch.cuda.stream(self.up):
            if self.used[slot]:
                self.up.wait_event(self.step_done[slot])  # step i - 2 read these inputs
            self.dev_bufs[slot].copy_(self.host_bufs[slot], non_blocking=True)
            self.in_ready[slot].record(self.up)
        main.wait_event(self.in_ready[slot])
        if self.used[slot]:
            main.wait_event(self.out_read[slot])  # step i - 2's output has been read back
        for n, v in self.views[slot].items():
            setattr(self.st, n, v)
        self.st.out = self.outs[slot]
        out = self.st.run()
        self.step_done[slot].record(main)
        self.used[slot] = True
        with torch.cuda.stream(self.down):
            self.down.wait_event(self.step_done[slot])
            self.host_outs[slot].copy_(out, non_blocking=True)
            self.out_read[slot].record(self.down)
        self.i += 1
        return self.host_outs[slot]

    def capture(self, steps: int) -> None:
        """Record `steps` consecutive steps (transfers, kernels, read-backs,
        and their overlap) as one CUDA graph; replay() then runs them with a
        single launch from the host.  Run a few steps eagerly first, so every
        kernel's launch attributes are set before capture."""
        torch.cuda.synchronize(self.st.device)
        self.used = [False, False]  # dependencies inside one replay only
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            main = torch.cuda.current_stream(self.st.device)
            self.begin(main)
            for _ in range(steps):
                self.step()
            self.finish(main)
        self.graph_steps = steps

    def replay(self) -> None:
        """The captured steps; replays of one graph never overlap each other."""
        self.graph.replay()

"""Test helpers: the same decode step on the oracle (CPU) and on the GPU.

The oracle side builds its pools with its own slot mapping and
reshape_and_cache, applies the step's writes and copy-on-write copies, and
attends; the GPU side does the same through the C ABI.  Both start from the
same seeded workload arrays; nothing flows from the GPU into the oracle.
"""
from __future__ import annotations

import numpy as np

import oracle
from paged_kv_cache_96_gb300.workloads import Workload

# Attention tolerance of the contract: |gpu - oracle| <= ATOL + RTOL * |oracle|.
ATOL = 1e-2
RTOL = 1e-2


def odt(w: Workload) -> int:
    return oracle.F16 if w.dtype == "f16" else oracle.BF16


class OracleStep:
    def __init__(self, w: Workload):
        self.w = w
        kc, vc = w.empty_pools()
        self.hist_slots = oracle.slot_mapping(w.block_tables, w.hist_seq, w.hist_pos,
                                              w.bs)
        self._write(w.hist_key, w.hist_value, kc, vc, self.hist_slots)
        self.new_slots = oracle.slot_mapping(w.block_tables, w.new_seq, w.new_pos, w.bs)
        self._write(w.new_key, w.new_value, kc, vc, self.new_slots)
        if w.cow_pairs.shape[0]:
            if w.fp8:
                oracle.copy_blocks_u8(kc, vc, w.cow_pairs)
            else:
                oracle.copy_blocks(kc, vc, w.cow_pairs)
        self.key_cache, self.value_cache = kc, vc

    def _write(self, k, v, kc, vc, slots):
        w = self.w
        if w.fp8:
            oracle.reshape_and_cache_fp8(k, v, kc, vc, slots, odt(w), w.spec.kv_scale,
                                         w.spec.kv_scale)
        else:
            oracle.reshape_and_cache(k, v, kc, vc, slots)

    def attention(self, seqs=None, rows=None):
        """Decode: [S, H, d] (rows of `seqs` only, if given).  Prefill:
        [T, H, d] for every chunk row, or [len(rows), H, d] for the listed
        rows -- computed as a batch of one-row chunks, each with its own
        sequence's table and the context ending at the row's position."""
        w = self.w
        if w.prefill:
            if rows is None:
                return oracle.prefill_attention(w.query, self.key_cache, self.value_cache,
                                                w.step_block_tables, w.query_start,
                                                w.context_lens, w.scale, odt(w))
            rows = np.asarray(rows, dtype=np.int64)
            seq_of = np.searchsorted(w.query_start, rows, side="right") - 1
            q_len = w.query_start[seq_of + 1] - w.query_start[seq_of]
            pos = w.context_lens[seq_of] - q_len + (rows - w.query_start[seq_of])
            qs = np.arange(rows.shape[0] + 1, dtype=np.int32)
            return oracle.prefill_attention(
                np.ascontiguousarray(w.query[rows]), self.key_cache, self.value_cache,
                np.ascontiguousarray(w.step_block_tables[seq_of]), qs,
                (pos + 1).astype(np.int32), w.scale, odt(w))
        if w.fp8:
            return oracle.paged_attention_fp8(w.query, self.key_cache, self.value_cache,
                                              w.step_block_tables, w.context_lens, w.scale,
                                              odt(w), w.spec.kv_scale, w.spec.kv_scale,
                                              seqs=seqs)
        return oracle.paged_attention(w.query, self.key_cache, self.value_cache,
                                      w.step_block_tables, w.context_lens, w.scale,
                                      odt(w), seqs=seqs)

    def partitions(self, partition_size, max_parts, seqs=None):
        w = self.w
        return oracle.partition_pass(w.query, self.key_cache, self.value_cache,
                                     w.step_block_tables, w.context_lens, w.scale,
                                     odt(w), partition_size, max_parts, seqs=seqs)


def assert_attention_close(got: np.ndarray, want: np.ndarray, what: str = ""):
    """Element-wise contract tolerance; returns (max abs err, max rel err)."""
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite GPU output"
    err = np.abs(got - want)
    bound = ATOL + RTOL * np.abs(want)
    bad = err > bound
    if bad.any():
        idx = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance, "
                             f"first {idx}: gpu {got[idx]} oracle {want[idx]}")
    rel = err / np.maximum(np.abs(want), 1e-6)
    return float(err.max()), float(np.median(rel))

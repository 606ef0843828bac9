"""Test helpers: the same decode step on the oracle (CPU) and on the GPU.

The oracle side builds its pools with its own slot mapping and
reshape_and_cache, applies the step's writes and copy-on-write copies, and
attends; the GPU side does the same through the C ABI.  Both start from the
same seeded workload arrays; nothing flows from the GPU into the oracle.
"""
from __future__ import annotations

import os
import shutil
import tempfile
import types

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
            if w.fp8:
                def prefill(q, bt, qs, cl):
                    return oracle.prefill_attention_fp8(q, self.key_cache, self.value_cache,
                                                        bt, qs, cl, w.scale, odt(w),
                                                        w.spec.kv_scale, w.spec.kv_scale)
            else:
                def prefill(q, bt, qs, cl):
                    return oracle.prefill_attention(q, self.key_cache, self.value_cache,
                                                    bt, qs, cl, w.scale, odt(w))
            if rows is None:
                return prefill(w.query, w.step_block_tables, w.query_start, w.context_lens)
            rows = np.asarray(rows, dtype=np.int64)
            seq_of = np.searchsorted(w.query_start, rows, side="right") - 1
            q_len = w.query_start[seq_of + 1] - w.query_start[seq_of]
            pos = w.context_lens[seq_of] - q_len + (rows - w.query_start[seq_of])
            qs = np.arange(rows.shape[0] + 1, dtype=np.int32)
            return prefill(np.ascontiguousarray(w.query[rows]),
                           np.ascontiguousarray(w.step_block_tables[seq_of]), qs,
                           (pos + 1).astype(np.int32))
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


# ---- the oracle on every host core -------------------------------------------------
#
# Whole-step comparisons at full size: a spawn-context process pool (safe
# after CUDA has started in the test process) runs the unchanged oracle over
# disjoint, cost-balanced sets of sequences -- or, for a prefill step, of
# chunk rows -- against the OracleStep's pools, shared through files the
# workers map read-only.

_WORKER = {}


def _worker_init(folder, fields):
    import oracle as _oracle
    _oracle.load()
    arrays = {}
    for name in ("query", "query_start", "step_block_tables", "context_lens", "kc", "vc"):
        arrays[name] = np.load(os.path.join(folder, name + ".npy"), mmap_mode="r")
    w = types.SimpleNamespace(**fields, **{k: arrays[k] for k in (
        "query", "query_start", "step_block_tables", "context_lens")})
    w.spec = types.SimpleNamespace(kv_scale=fields["kv_scale"])
    ref = OracleStep.__new__(OracleStep)
    ref.w = w
    ref.key_cache = arrays["kc"]
    ref.value_cache = arrays["vc"]
    _WORKER["ref"] = ref


def _worker_task(job):
    kind, items = job
    ref = _WORKER["ref"]
    if kind == "rows":
        return items, ref.attention(rows=items)
    return items, ref.attention(seqs=items)[items]


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def attention_all(ref: OracleStep, workers: int = 0) -> np.ndarray:
    """The oracle's attention output of every sequence (decode, [S, H, d])
    or every chunk row (prefill, [T, H, d]), computed on `workers` processes
    (all host cores by default)."""
    import multiprocessing
    w = ref.w
    workers = workers or host_cores()
    if w.prefill:
        # a row's cost is its position + 1 keys; cut the rows into chunks of
        # similar cost
        qs = w.query_start.astype(np.int64)
        seq_of = np.searchsorted(qs, np.arange(w.T), side="right") - 1
        pos = w.context_lens[seq_of] - (qs[seq_of + 1] - qs[seq_of]) + (np.arange(w.T) - qs[seq_of])
        cost = np.maximum(pos + 1, 1).astype(np.float64)
        edges = np.searchsorted(np.cumsum(cost), np.linspace(0, cost.sum(), 8 * workers + 1)[1:-1])
        jobs = [("rows", [int(r) for r in c]) for c in np.split(np.arange(w.T), edges) if len(c)]
        out = np.full((w.T, w.H, w.D), np.nan)
    else:
        order = sorted(range(w.S), key=lambda s: -int(w.context_lens[s]))
        chunks = [[] for _ in range(min(w.S, 4 * workers))]
        load = [0] * len(chunks)
        for s in order:  # heaviest sequence to the lightest chunk
            i = load.index(min(load))
            chunks[i].append(s)
            load[i] += int(w.context_lens[s]) + 1
        jobs = [("seqs", sorted(c)) for c in chunks if c]
        out = np.full((w.S, w.H, w.D), np.nan)
    if workers <= 1:
        for kind, items in jobs:
            res = ref.attention(rows=items) if kind == "rows" else ref.attention(seqs=items)[items]
            out[items] = res
        return out
    base = "/dev/shm" if os.path.isdir("/dev/shm") else None
    d = tempfile.mkdtemp(prefix="pa_oracle_", dir=base)
    try:
        # every array goes through a file the workers map: arguments of the
        # workers' start are pickled into a pipe each child reads only once
        # it has imported this module, so large ones would start them one by
        # one
        for name, arr in (("kc", ref.key_cache), ("vc", ref.value_cache), ("query", w.query),
                          ("query_start", w.query_start),
                          ("step_block_tables", w.step_block_tables),
                          ("context_lens", w.context_lens)):
            np.save(os.path.join(d, name + ".npy"), np.ascontiguousarray(arr))
        fields = {"prefill": w.prefill, "fp8": w.fp8, "dtype": w.dtype, "scale": w.scale,
                  "kv_scale": float(w.spec.kv_scale)}
        ctx = multiprocessing.get_context("spawn")
        with ctx.Pool(workers, initializer=_worker_init, initargs=(d, fields)) as pool:
            # bounded: a pool whose workers cannot start would restart them
            # for ever
            for items, res in pool.map_async(_worker_task, jobs).get(timeout=1800):
                out[items] = res
        return out
    finally:
        shutil.rmtree(d, ignore_errors=True)

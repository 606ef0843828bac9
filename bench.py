#!/usr/bin/env python3
"""Paged decode step benchmark on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--partition P] [--separate-append] [--impl ours|reference]

A step is one pass of the whole hot path over one batch: slot mapping of
the step's new tokens, reshape_and_cache of their K/V, copy-on-write block
copies (when the workload has them) and paged decode attention (split-context
partitions merged by a reduce launch).  A decode step with one new token per
sequence copies its copy-on-write blocks first and then runs the slot
mapping, the cache write and attention as one call
(pa_decode_attention_append); `--separate-append` times the unfused order
instead (one launch for slot mapping and cache write, then copy-on-write,
then attention).  Default workload: the GQA 70B-like
decode layer (128 sequences, lognormal contexts, 64 query heads over 8 KV
heads, d 128, block 16, bf16).

Prints ONE JSON line.  `value` is the effective KV bandwidth of the whole
step (attended K and V bytes / step time, summed over ranks); the roofline
object reports the attention kernel alone against the measured HBM copy
bandwidth.  `--impl reference` times the CPU oracle (plain C, fp64) on a
bounded sample of the same workload.

The chunked-prefill workloads (`--config chunked`, `mixed`) report the
attention's tensor throughput instead (TFLOP/s of the step, roofline against
the measured sustained bf16 tensor rate); `prefix-cascade` is the
prefix-sharing step decoded with the shared prefix read once per group.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = ("paged decode attention effective KV GB/s and % of GB300 HBM peak; "
          "seqs/s per step")
PREFILL_METRIC = "chunked-prefill paged attention TFLOP/s; tokens/s per step"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="gqa70b",
                    choices=["tiny", "mha7b", "gqa70b", "longctx", "prefix", "gqa70b-fp8",
                             "longctx-fp8", "prefix-cascade", "prefix-cascade-fp8", "mixed",
                             "mixed-fp8", "chunked", "chunked-fp8"])
    ap.add_argument("--partition", type=int, default=None,
                    help="split-context partition tokens (0 = single pass)")
    ap.add_argument("--separate-append", action="store_true",
                    help="decode steps: write the new tokens with their own launch "
                         "before attention instead of inside it")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU, replicas: no data-path collective)

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def aggregate(elapsed_s: float, units: float, world: int, device=None):
    """Max elapsed and summed units over ranks (identity when world == 1)."""
    if world == 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ---------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 20

    def __init__(self, gpu_ids):
        """Samples nvidia-smi for the first of `gpu_ids` (UUID, then index)
        that nvidia-smi accepts."""
        self.samples = []
        self.proc = None
        self.thread = None
        self.error = None
        self.ids = [g for g in gpu_ids if g]
        self._start_next()

    def _start_next(self):
        while self.ids:
            gid = self.ids.pop(0)
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS), "-i", gid],
                    stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
            except (OSError, ValueError) as e:
                self.error = str(e)
                continue
            self.gpu_id = gid
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            return
        self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def wait_first(self, timeout: float = 10.0) -> bool:
        """Block until the first sample arrives (nvidia-smi takes a moment to
        start); try the next id if nvidia-smi refuses this one."""
        t_end = time.time() + timeout
        while time.time() < t_end:
            if self.samples:
                return True
            if self.proc is None:
                return False
            if self.proc.poll() is not None:  # refused this id
                err = self.proc.stderr.read().strip() if self.proc.stderr else ""
                self.error = f"nvidia-smi -i {self.gpu_id}: {err[:160]}"
                self._start_next()
                continue
            time.sleep(0.01)
        return bool(self.samples)

    def count(self, t0: float, t1: float) -> int:
        return sum(1 for (t, _) in self.samples if t0 <= t <= t1)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float, note: str = ""):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "note": self.error or "no nvidia-smi samples"}
        window = [p for (t, p) in self.samples if t0 <= t <= t1]
        note = note or f"sampled during the timed region ({self.PERIOD_MS} ms period)"
        if not window:
            window = [p for (_, p) in self.samples]
            note = "no sample inside the timed region: samples span the whole run"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in window if num(p[1]) is not None]
        mx = [num(p[2]) for p in window if num(p[2]) is not None]
        pw = [num(p[3]) for p in window if num(p[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in window for i in range(4)
                          if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(window), "note": note,
                "gpu": self.gpu_id}


def gpu_ids_for(torch, dev, local_rank):
    """nvidia-smi ids of a torch device: its UUID, then the physical index
    (CUDA_VISIBLE_DEVICES maps torch's index to it)."""
    ids = []
    uuid = str(getattr(torch.cuda.get_device_properties(dev), "uuid", "") or "")
    if uuid:
        ids.append(uuid if uuid.startswith("GPU-") or not re.fullmatch(r"[0-9a-f-]{36}", uuid)
                   else "GPU-" + uuid)
    vis = [v.strip() for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    idx = dev.index or 0
    ids.append(vis[idx] if idx < len(vis) else str(idx))
    return ids


# ---------------------------------------------------------------------------

def measured_tensor_peak():
    """Sustained bf16 tensor rate (a kernel timed inside a long loop)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured sustained"
    except (OSError, KeyError, ValueError):
        return 1700.0, "fallback sustained"


def measured_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# Per workload: the committed ncu summary whose DRAM bytes per launch the
# roofline's `traffic` reports, and the kernel sources it was captured from
# (a changed source voids the figure).
CSRC = os.path.join(ROOT, "paged_kv_cache_96_gb300", "csrc")
DECODE_SOURCES = ["pa_decode.cu", "pa_decode_common.cuh", "pa_ptx.cuh"]
PREFILL_SOURCES = ["pa_prefill.cu", "pa_tcgen05.cuh", "pa_decode_common.cuh", "pa_ptx.cuh"]
TRAFFIC_SUMMARIES = {
    "gqa70b": ("decode_gqa70b_ncu.md", DECODE_SOURCES),
    "gqa70b-fp8": ("decode_gqa70b_fp8_ncu.md", DECODE_SOURCES),
    "chunked": ("prefill_chunked_ncu.md", PREFILL_SOURCES),
    "chunked-fp8": ("prefill_chunked_fp8_ncu.md", PREFILL_SOURCES),
}


def _code_only(text: str) -> str:
    """C/C++/CUDA source with its comments and blank lines removed (the
    sources hold no comment markers inside string literals), so that a
    change of comments alone keeps a recorded capture valid."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def sources_sha256(names):
    """sha256 over the code (comments stripped) of the named kernel sources."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(CSRC, n), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()


def recorded_traffic(config: str, partition_is_default: bool = True):
    """DRAM bytes per launch of the attention call from the committed ncu
    summary of this workload -- only if its kernel sources are unchanged
    since the capture and the launch configuration is the captured one."""
    entry = TRAFFIC_SUMMARIES.get(config)
    if entry is None or not partition_is_default:
        return None
    try:
        text = open(os.path.join(ROOT, "profiles", entry[0])).read()
    except OSError:
        return None
    m_sha = re.search(r"kernel_sources_sha256:\s*([0-9a-f]{64})", text)
    m_b = re.search(r"dram_bytes_per_launch_full_workload:\s*([0-9.eE+]+)", text)
    if not (m_sha and m_b):
        return None
    return float(m_b.group(1)) if sources_sha256(entry[1]) == m_sha.group(1) else None


L2_BYTES = 129 * 1024 * 1024  # GB300 L2


def step_bytes(w) -> int:
    """Bytes one step touches: attended K/V (each physical block once) and the
    step's queries and outputs."""
    return w.unique_kv_bytes() + w.qo_bytes()


def l2_note(w) -> str:
    b = step_bytes(w)
    if b < L2_BYTES:
        return (f"step data {b / 1e6:.1f} MB < L2: L2 flushed before every timed step "
                f"(write of {2 * L2_BYTES >> 20} MiB, outside the timed intervals)")
    return f"inputs larger than L2: {b / 1e9:.2f} GB per step; no flush"


def workload_config(w, partition_size, world=1):
    kv = w.kv_bytes()
    if w.prefill:
        return {
            "workload": f"{w.spec.name}: {w.spec.description}",
            "num_seqs": w.S, "query_rows": w.T, "num_heads": w.H, "num_kv_heads": w.Hkv,
            "head_dim": w.D, "block_size": w.bs, "num_blocks": w.num_blocks,
            "context_tokens": int(w.context_lens.sum()),
            "attention_flops_per_step": w.prefill_flops(),
            "l2": l2_note(w),
            "parallelism": "replicas" if world > 1 else "single GPU",
            "kv_cache_dtype": "fp8-e4m3" if w.fp8 else w.dtype,
        }
    return {
        "workload": f"{w.spec.name}: {w.spec.description}",
        "num_seqs": w.S, "num_heads": w.H, "num_kv_heads": w.Hkv, "head_dim": w.D,
        "block_size": w.bs, "num_blocks": w.num_blocks, "partition_size": partition_size,
        "context_tokens": int(w.context_lens.sum()), "kv_bytes_per_step": kv,
        "l2": l2_note(w),
        "parallelism": "replicas" if world > 1 else "single GPU",
        "kv_cache_dtype": "fp8-e4m3" if w.fp8 else w.dtype,
    }


class OracleCache:
    """The oracle's own pools for a workload (history written through its
    slot mapping and cache write) and its step operations, 16-bit or FP8."""

    def __init__(self, w):
        import oracle
        self.o, self.w = oracle, w
        self.dt = oracle.F16 if w.dtype == "f16" else oracle.BF16
        self.kc, self.vc = w.empty_pools()
        slots = oracle.slot_mapping(w.block_tables, w.hist_seq, w.hist_pos, w.bs)
        self.write(w.hist_key, w.hist_value, slots)

    def write(self, k, v, slots):
        o, w = self.o, self.w
        if w.fp8:
            o.reshape_and_cache_fp8(k, v, self.kc, self.vc, slots, self.dt, w.spec.kv_scale,
                                    w.spec.kv_scale)
        else:
            o.reshape_and_cache(k, v, self.kc, self.vc, slots)

    def new_tokens(self, seqs):
        """The step's new tokens of the listed sequences (one each for
        decode, the chunk for prefill)."""
        o, w = self.o, self.w
        idx = np.nonzero(np.isin(w.new_seq, np.asarray(seqs, dtype=np.int32)))[0]
        sl = o.slot_mapping(w.block_tables, w.new_seq[idx], w.new_pos[idx], w.bs)
        self.write(w.new_key[idx], w.new_value[idx], sl)

    def copy_blocks(self):
        o, w = self.o, self.w
        if w.cow_pairs.shape[0]:
            (o.copy_blocks_u8 if w.fp8 else o.copy_blocks)(self.kc, self.vc, w.cow_pairs)

    def attention(self, seqs):
        o, w = self.o, self.w
        if w.prefill:
            # the listed sequences' chunk rows
            qs = w.query_start
            rows = np.concatenate([np.arange(qs[s], qs[s + 1]) for s in seqs]).astype(np.int64)
            sq = np.asarray(seqs, dtype=np.int64)
            sub_qs = np.zeros(len(seqs) + 1, dtype=np.int32)
            sub_qs[1:] = np.cumsum(qs[sq + 1] - qs[sq])
            args = (np.ascontiguousarray(w.query[rows]), self.kc, self.vc,
                    np.ascontiguousarray(w.step_block_tables[sq]), sub_qs,
                    np.ascontiguousarray(w.context_lens[sq]), w.scale, self.dt)
            if w.fp8:
                return o.prefill_attention_fp8(*args, w.spec.kv_scale, w.spec.kv_scale)
            return o.prefill_attention(*args)
        if w.fp8:
            return o.paged_attention_fp8(w.query, self.kc, self.vc, w.step_block_tables,
                                         w.context_lens, w.scale, self.dt, w.spec.kv_scale,
                                         w.spec.kv_scale, seqs=seqs)
        return o.paged_attention(w.query, self.kc, self.vc, w.step_block_tables,
                                 w.context_lens, w.scale, self.dt, seqs=seqs)


def _seq_flops(w, s):
    """Attention multiply-adds x 2 of sequence s's rows (prefill)."""
    n = int(w.query_start[s + 1] - w.query_start[s])
    pos1 = int(w.context_lens[s]) - n + np.arange(1, n + 1)
    return 4 * w.D * w.H * int(np.maximum(pos1, 0).sum())


def cpu_baseline_sample(w, target_s: float, keep: bool = False):
    """Time the oracle's step (new-token writes + attention) on the first
    sequences of the workload until about target_s seconds of CPU work
    (with keep, also return the oracle's pools)."""
    oc = OracleCache(w)
    done, tokens, elapsed, flops = [], 0, 0.0, 0
    for s in range(w.S):
        t0 = time.perf_counter()
        oc.new_tokens([s])
        oc.attention([s])
        elapsed += time.perf_counter() - t0
        done.append(s)
        tokens += int(w.context_lens[s])
        if w.prefill:
            flops += _seq_flops(w, s)
        if elapsed >= target_s:
            break
    if w.prefill:
        res = {"value": flops / elapsed / 1e12, "unit": "TFLOP/s", "cores": 1,
               "kind": "oracle",
               "sample": f"{len(done)} of {w.S} sequences ({flops / 1e9:.1f} GFLOP): "
                         f"chunk writes + fp64 attention of every chunk row, "
                         f"single-threaded C, {elapsed:.1f} s"}
    else:
        kv = tokens * w.Hkv * w.D * 2 * w.kv_elem_bytes
        res = {"value": kv / elapsed / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{len(done)} of {w.S} sequences ({tokens} attended tokens): "
                         f"new-token write + fp64 attention, single-threaded C, "
                         f"{elapsed:.1f} s"}
    return (res, oc) if keep else res


# The oracle on every host core: a spawn-context process pool (started after
# CUDA, so no fork) runs the unchanged oracle attention over disjoint,
# cost-balanced sets of sequences; the pools are shared through files the
# workers map read-only.  Wall-clock time of the whole pass.
_MC = {}


def _mc_init(folder, fields):
    import types

    import oracle
    oracle.load()
    arrays = {n: np.load(os.path.join(folder, n + ".npy"), mmap_mode="r")
              for n in ("query", "query_start", "step_block_tables", "context_lens", "kc", "vc")}
    w = types.SimpleNamespace(**fields, **{k: arrays[k] for k in (
        "query", "query_start", "step_block_tables", "context_lens")})
    w.spec = types.SimpleNamespace(kv_scale=fields["kv_scale"])
    oc = OracleCache.__new__(OracleCache)
    oc.o, oc.w = oracle, w
    oc.dt = oracle.F16 if w.dtype == "f16" else oracle.BF16
    oc.kc, oc.vc = arrays["kc"], arrays["vc"]
    _MC["oc"] = oc


def _mc_task(seqs):
    _MC["oc"].attention(list(seqs))
    return len(seqs)


def cpu_baseline_multicore(oc, w, cores: int):
    """(seconds of wall time for the whole step's attention on `cores`
    processes, sequences done)."""
    import multiprocessing
    import shutil
    import tempfile
    d = tempfile.mkdtemp(prefix="pa_oracle_",
                         dir="/dev/shm" if os.path.isdir("/dev/shm") else None)
    try:
        # every array through a file the workers map (start arguments go
        # through a pipe each child reads only after its imports, so large
        # ones would start the workers one by one)
        for name, arr in (("kc", oc.kc), ("vc", oc.vc), ("query", w.query),
                          ("query_start", w.query_start),
                          ("step_block_tables", w.step_block_tables),
                          ("context_lens", w.context_lens)):
            np.save(os.path.join(d, name + ".npy"), np.ascontiguousarray(arr))
        fields = {"prefill": w.prefill, "fp8": w.fp8, "dtype": w.dtype, "scale": w.scale,
                  "kv_scale": float(w.spec.kv_scale)}
        cost = [(_seq_flops(w, s) if w.prefill else int(w.context_lens[s]), s)
                for s in range(w.S)]
        cost.sort(reverse=True)
        chunks = [[] for _ in range(4 * cores)]
        load = [0] * len(chunks)
        for c, s in cost:  # greedy: heaviest sequence to the lightest chunk
            i = load.index(min(load))
            chunks[i].append(s)
            load[i] += c
        chunks = [c for c in chunks if c]
        ctx = multiprocessing.get_context("spawn")
        with ctx.Pool(cores, initializer=_mc_init, initargs=(d, fields)) as pool:
            # every worker started and loaded (bounded: a pool whose workers
            # cannot start would otherwise restart them for ever)
            pool.map_async(_mc_task, [[0]] * cores).get(timeout=120)
            t0 = time.perf_counter()
            done = sum(pool.map_async(_mc_task, chunks).get(timeout=600))
            el = time.perf_counter() - t0
        return el, done
    finally:
        shutil.rmtree(d, ignore_errors=True)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(w, target_s: float):
    """The oracle timed on the host: single-threaded on a bounded sample,
    then (when the host has more than one core) on every core over the whole
    step; the line reports the multi-core figure with the single-thread one
    beside it."""
    single, oc = cpu_baseline_sample(w, target_s, keep=True)
    cores = host_cores()
    if cores <= 1:
        return single
    try:
        oc.new_tokens(list(range(w.S)))  # the rest of the step's writes (setup)
        oc.copy_blocks()
        el, done = cpu_baseline_multicore(oc, w, cores)
    except Exception as e:  # keep the bench line; say why
        single["note"] = f"multi-core run failed: {e!r}"
        return single
    if w.prefill:
        work = sum(_seq_flops(w, s) for s in range(w.S))
        value, what = work / el / 1e12, f"{work / 1e9:.1f} GFLOP"
    else:
        work = int(w.context_lens.astype(np.int64).sum()) * w.Hkv * w.D * 2 * w.kv_elem_bytes
        value, what = work / el / 1e9, f"{work / 1e9:.2f} GB of K/V"
    return {"value": value, "unit": single["unit"], "cores": cores, "kind": "oracle",
            "sample": f"whole step's attention ({done} sequences, {what}) on {cores} "
                      f"processes of the unchanged single-threaded C oracle, "
                      f"{el:.2f} s wall; single thread: {single['value']:.4g} "
                      f"{single['unit']} ({single['sample']})",
            "single_thread": single["value"]}


# ---------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from paged_kv_cache_96_gb300 import workloads as W
    w = W.build(W.CONFIGS[args.config])
    oc = OracleCache(w)
    # per step: a bounded sample of sequences, sized so that the whole run
    # (warm-up + timed steps) takes about 2.5 minutes of CPU work, at most 2 s
    # per step
    cost = (lambda s: _seq_flops(w, s)) if w.prefill else (lambda s: int(w.context_lens[s]))
    t0 = time.perf_counter()
    oc.attention([0])
    per_unit = (time.perf_counter() - t0) / max(1, cost(0))
    budget = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    sample, toks, units = [], 0, 0
    for s in range(w.S):
        if sample and (units + cost(s)) * per_unit > budget:
            break
        sample.append(s)
        toks += int(w.context_lens[s])
        units += cost(s)

    def step():
        oc.new_tokens(sample)
        oc.copy_blocks()
        oc.attention(sample)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    if w.prefill:
        val, unit, metric = units * args.steps / el / 1e12, "TFLOP/s", PREFILL_METRIC
    else:
        kv = toks * w.Hkv * w.D * 2 * w.kv_elem_bytes
        val, unit, metric = kv * args.steps / el / 1e9, "GB/s", METRIC
    line = {
        "impl": "reference", "metric": metric, "value": val, "unit": unit,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, w.spec.partition_size if args.partition is None
                                  else args.partition),
        "cpu_baseline": {"value": val, "unit": unit, "cores": 1, "kind": "oracle",
                         "sample": f"{len(sample)} of {w.S} sequences ({toks} tokens) "
                                   "per step, fp64 single-threaded C"},
        "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank if world > 1 else 0)
    torch.cuda.set_device(dev)
    # clocks: started now, so that nvidia-smi is sampling before warm-up
    sampler = ClockSampler(gpu_ids_for(torch, dev, local_rank)) if rank == 0 else None

    from paged_kv_cache_96_gb300 import step as S
    from paged_kv_cache_96_gb300 import workloads as W
    w = W.build(W.CONFIGS[args.config])
    st = S.DecodeStep(w, device=str(dev), partition_size=args.partition)
    if args.separate_append:
        st.fused_append = False
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)

    for _ in range(max(args.warmup, 3)):
        st.run()
    torch.cuda.synchronize(dev)
    if sampler is not None:
        sampler.wait_first()
    if st.error_word.item() != 0:
        raise RuntimeError(f"device error word {int(st.error_word.item()):#x}")

    K = args.steps
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    # A step whose data fits in L2 gets L2 flushed before it (a write of twice
    # the L2 size, outside the timed intervals); larger steps need none.
    flush = None
    if step_bytes(w) < L2_BYTES:
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t_host0 = time.time()
    for i in range(K):
        if flush is not None:
            flush.zero_()
        ev_s[i].record(stream)
        if st.fused_append:
            # copy-on-write, then the new tokens' append fused into attention
            st.copy_blocks()
            ev_a[i].record(stream)
            st.append_attention()
        else:
            st.slot_mapping_and_cache()
            st.copy_blocks()
            ev_a[i].record(stream)
            st.attention()
        ev_b[i].record(stream)
    torch.cuda.synchronize(dev)
    t_host1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    step_s = sum(a.elapsed_time(b) for a, b in zip(ev_s, ev_b)) / 1e3
    attn_s = sum(a.elapsed_time(b) for a, b in zip(ev_a, ev_b)) / 1e3 / K
    clocks = None
    if sampler is not None:
        t_end, note = t_host1, ""
        if sampler.samples and sampler.count(t_host0, t_host1) < 3:
            # a timed region shorter than a few sampling periods: the same
            # steps keep running (untimed) until three samples have been
            # taken under that load, at most one second
            t_stop = time.time() + 1.0
            while sampler.count(t_host0, time.time()) < 3 and time.time() < t_stop:
                for _ in range(8):
                    st.run()
                torch.cuda.synchronize(dev)
            t_end = time.time()
            note = (f"timed region {1e3 * (t_host1 - t_host0):.1f} ms: sampled over it and "
                    f"the same steps run on, untimed, to {1e3 * (t_end - t_host0):.0f} ms "
                    f"({ClockSampler.PERIOD_MS} ms period)")
        sampler.stop()
        clocks = sampler.summary(t_host0, t_end, note)

    kv = w.kv_bytes()
    if w.prefill:
        per_unit, scale_u = w.prefill_flops(), 1e12   # TFLOP/s
    else:
        per_unit, scale_u = kv, 1e9                    # GB/s of attended K/V
    units = per_unit * K
    max_elapsed, total_units = aggregate(step_s, units, world, device=dev)
    value = total_units / max_elapsed / scale_u

    # end to end through the public API: pinned host inputs -> step -> host output
    e2e = None
    if rank == 0 and args.e2e_steps > 0:
        host = S.HostStepIO(st)
        host.begin(stream)
        for _ in range(3):
            host.step()
        host.finish(stream)
        torch.cuda.synchronize(dev)
        # the steps recorded as a CUDA graph of 32 overlapped steps, replayed
        # with one host launch each (eager steps when capture is refused)
        graph_steps = 32
        try:
            host.capture(graph_steps)
            host.replay()
            torch.cuda.synchronize(dev)
        except RuntimeError:
            graph_steps = 0
        Ke = max(1, args.e2e_steps // graph_steps) * graph_steps if graph_steps else args.e2e_steps
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if graph_steps:
            for _ in range(Ke // graph_steps):
                host.replay()
        else:
            host.begin(stream)   # the first input copy comes after e0
            for _ in range(Ke):
                host.step()
            host.finish(stream)  # e1 comes after the last output read-back
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_s = e0.elapsed_time(e1) / 1e3 / Ke
        e2e = {"value": per_unit / e2e_s / scale_u * world,
               "unit": "TFLOP/s" if w.prefill else "GB/s",
               "h2d_bytes_per_step": host.h2d_bytes, "d2h_bytes_per_step": host.d2h_bytes,
               "us_per_step": e2e_s * 1e6,
               "mode": (f"CUDA graph of {graph_steps} steps, transfers overlapped with "
                        "compute (copy stream, double-buffered staging)") if graph_steps
                       else "eager steps, transfers overlapped with compute"}

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds)
    per_step = step_s / K
    if w.prefill:
        tpeak, tpeak_kind = measured_tensor_peak()
        flops = w.prefill_flops()
        achieved = flops / attn_s / 1e12
        line = {
            "metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("fp8-e4m3 KV widened to fp16, tcgen05 kind::f16, fp32 accumulate"
                      if w.fp8 else f"{w.dtype} tcgen05 kind::f16, fp32 accumulate"),
            "data": "synthetic",
            "config": workload_config(w, 0, world),
            "tokens_per_s": w.T * world / per_step,
            "us_per_step": per_step * 1e6,
            "attention_us": attn_s * 1e6,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": tpeak,
                         "unit": "TFLOP/s", "frac": achieved / tpeak,
                         "traffic": recorded_traffic(args.config),
                         "kernel": "pa_prefill_attention (paged_mq_kernel)",
                         "peak_kind": f"{tpeak_kind} bf16 (cuBLAS)",
                         "algorithmic_flops_per_launch": flops},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": st.launches_per_step() * K,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
        return
    peak, peak_kind = measured_hbm_peak()
    # HBM minimum: each physical block once (a shared prefix counts once)
    attn_bytes = w.unique_kv_bytes() + w.qo_bytes()
    achieved = attn_bytes / attn_s / 1e9
    kernel = "pa_decode_attention (paged_decode_kernel, split contexts merged in the pass)"
    if st.fused_append:
        kernel = ("pa_decode_attention_append (paged_decode_kernel with the new tokens' "
                  "append, split contexts merged in the pass)")
    if st.cascade:
        kernel = ("pa_decode_attention_cascade (paged_decode_kernel + paged_mq_kernel "
                  "prefix pass, merges in whichever pass completes a sequence)")
        if st.fused_append:
            kernel = ("pa_decode_attention_cascade_append (paged_decode_kernel with the new "
                      "tokens' append + paged_mq_kernel prefix pass, merges in whichever "
                      "pass completes a sequence)")
    if st.launches_per_step() > (1 if st.fused_append else 2) + \
            (1 if st.cow_pairs is not None else 0) + (1 if st.cascade and st.num_groups else 0):
        kernel += " + paged_reduce_kernel"
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8-e4m3 KV, fp16 MMA, fp32 accumulate" if w.fp8 else w.dtype,
        "data": "synthetic",
        "config": workload_config(w, st.partition_size, world),
        "pct_of_hbm_peak_8tbps": 100.0 * value / world / NOMINAL_HBM_GBS,
        "pct_of_hbm_measured": 100.0 * value / world / peak,
        "seqs_per_s": w.S * world / per_step,
        "us_per_step": per_step * 1e6,
        "attention_us": attn_s * 1e6,
        "unique_kv_gbs": w.unique_kv_bytes() * world / per_step / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": recorded_traffic(
                         args.config, args.partition is None
                         or args.partition == w.spec.partition_size),
                     "kernel": kernel,
                     "peak_kind": f"{peak_kind} copy",
                     "algorithmic_bytes_per_launch": attn_bytes},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": st.launches_per_step() * K,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)
    rank, world, _ = dist_env()
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

"""Seeded synthetic decode workloads.

This module only *draws inputs*: context lengths, the physical block each
logical block of a sequence lives in (a seeded shuffle of the pool), query /
key / value values ~ N(0, 1) rounded to the storage dtype, the tokens that
are already cached before a step and the one new token per sequence that a
step writes, and copy-on-write (src, dst) block pairs.  It computes no slot,
no score and no softmax: both the CPU oracle and the CUDA path take these
inputs and do the method's arithmetic themselves.

Workload shapes follow the decode-step picture of "PagedAttention &
Continuous Batching" (gaoleia.github.io) §1.3-§1.6 and §2.4 (each running
sequence contributes one query token that attends to its whole cached
context), the shared-prefix picture of "vLLM 架构详解" (feifeigd.github.io,
"共享前缀的 Block 复用") and the copy-on-write steps of "vLLM源码解析(二)"
(lakecityint.com) §3.2.

Pool filling: every pool element that no cached token owns -- unassigned
blocks, the unused tail rows of each sequence's last block, and the block
that padding entries of the block tables point at -- holds a NaN pattern, so
a kernel that reads outside a sequence's context produces NaN instead of a
plausible number.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Callable, Dict, Optional

import numpy as np
import torch

F16_NAN = np.uint16(0x7E00)
BF16_NAN = np.uint16(0x7FC0)
FP8_NAN = np.uint8(0x7F)


@dataclasses.dataclass
class WorkloadSpec:
    name: str
    description: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str                      # "f16" or "bf16"
    context_lens: Callable[[np.random.Generator], np.ndarray]
    pool_factor: float = 1.25       # pool blocks = ceil(factor * blocks needed)
    num_blocks: Optional[int] = None  # fixed pool size (overrides pool_factor)
    shared_prefix_tokens: int = 0   # tokens of one prefix shared by every sequence
    cow_pairs: int = 0              # copy-on-write (src, dst) pairs per step
    partition_size: int = 512       # split-context partition (tokens); 0 = single pass
    seed: int = 0
    kv_dtype: str = "same"          # "same" (pools in dtype) or "fp8" (e4m3 codes)
    kv_scale: float = 0.0137        # per-pool scale of FP8 codes (K and V)
    # Chunked prefill / mixed batch: query rows (newest tokens) per sequence,
    # drawn from (rng, context_lens); None = decode, one row per sequence.
    query_lens: Optional[Callable[[np.random.Generator, np.ndarray], np.ndarray]] = None
    cascade: bool = False           # decode with the prefix-aware (cascade) path


@dataclasses.dataclass
class Workload:
    """Host arrays of one decode step.  16-bit values are raw bit patterns
    (uint16).  ``block_tables`` are the tables before the step; the step's
    copy-on-write remaps some entries, giving ``step_block_tables``, which
    attention reads."""
    spec: WorkloadSpec
    num_blocks: int
    max_blocks_per_seq: int
    scale: float
    context_lens: np.ndarray        # int32 [S]
    block_tables: np.ndarray        # int32 [S, MB]
    step_block_tables: np.ndarray   # int32 [S, MB]
    query: np.ndarray               # uint16 [T, H, d] (T = S for decode)
    hist_seq: np.ndarray            # int32 [Th]  tokens cached before the step
    hist_pos: np.ndarray            # int32 [Th]
    hist_key: np.ndarray            # uint16 [Th, Hkv, d]
    hist_value: np.ndarray          # uint16 [Th, Hkv, d]
    new_seq: np.ndarray             # int32 [T]   tokens the step writes
    new_pos: np.ndarray             # int32 [T]
    new_key: np.ndarray             # uint16 [T, Hkv, d]
    new_value: np.ndarray           # uint16 [T, Hkv, d]
    cow_pairs: np.ndarray           # int32 [P, 2]  (src, dst)
    pad_block: int                  # block id that table padding points at
    fill: np.uint16                 # NaN pattern of unowned pool elements
    query_start: np.ndarray = None  # int32 [S + 1]: query rows of each sequence

    # convenience -------------------------------------------------------
    @property
    def dtype(self) -> str:
        return self.spec.dtype

    @property
    def S(self) -> int:
        return self.spec.num_seqs

    @property
    def H(self) -> int:
        return self.spec.num_heads

    @property
    def Hkv(self) -> int:
        return self.spec.num_kv_heads

    @property
    def D(self) -> int:
        return self.spec.head_dim

    @property
    def bs(self) -> int:
        return self.spec.block_size

    def pool_shape(self):
        return (self.num_blocks, self.bs, self.Hkv, self.D)

    @property
    def fp8(self) -> bool:
        return self.spec.kv_dtype == "fp8"

    @property
    def prefill(self) -> bool:
        """Query rows are chunks of prompts (many per sequence), not one
        decode token per sequence."""
        return self.spec.query_lens is not None

    @property
    def T(self) -> int:
        """Query rows (= new tokens) of the step."""
        return int(self.query.shape[0])

    def prefill_flops(self) -> int:
        """Multiply-adds x 2 of the step's attention: each query row at
        position pos scores pos + 1 keys (q . k, d products) and sums as many
        value rows (d products), for every query head."""
        qs = self.query_start.astype(np.int64)
        ctx = self.context_lens.astype(np.int64)
        keys = 0
        for s in range(self.S):
            n = int(qs[s + 1] - qs[s])
            pos1 = ctx[s] - n + np.arange(1, n + 1)
            keys += int(np.maximum(pos1, 0).sum())
        return 4 * self.D * self.H * keys

    @property
    def kv_elem_bytes(self) -> int:
        return 1 if self.fp8 else 2

    def empty_pools(self):
        """Two pools filled with the NaN pattern (host): uint16 bit patterns,
        or uint8 e4m3 codes (0x7F is NaN) for FP8 pools."""
        if self.fp8:
            kc = np.full(self.pool_shape(), FP8_NAN, dtype=np.uint8)
            vc = np.full(self.pool_shape(), FP8_NAN, dtype=np.uint8)
            return kc, vc
        kc = np.full(self.pool_shape(), self.fill, dtype=np.uint16)
        vc = np.full(self.pool_shape(), self.fill, dtype=np.uint16)
        return kc, vc

    def kv_bytes(self) -> int:
        """Bytes of K and V the step's attention must read: one K row and
        one V row per (attended token, KV head)."""
        elem = self.kv_elem_bytes
        return int(self.context_lens.astype(np.int64).sum()) * self.Hkv * self.D * 2 * elem

    def unique_kv_bytes(self) -> int:
        """As kv_bytes, but each physical block counted once: the shared
        prefix once, plus the private copies made by copy-on-write (each
        remapped sequence reads its copy instead of the shared block)."""
        elem = self.kv_elem_bytes
        pre = self.spec.shared_prefix_tokens
        toks = int(self.context_lens.astype(np.int64).sum())
        if pre:
            toks -= pre * (self.S - 1)
            toks += self.cow_pairs.shape[0] * self.bs
        return toks * self.Hkv * self.D * 2 * elem

    def qo_bytes(self) -> int:
        return 2 * self.T * self.H * self.D * 2


# ---------------------------------------------------------------------------
# value drawing

def _round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 -> 16-bit bit patterns, round to nearest even."""
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _normal16(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    chunk = 1 << 24
    for i in range(0, n, chunk):
        m = min(chunk, n - i)
        out[i:i + m] = _round_to(rng.standard_normal(m, dtype=np.float32), dtype)
    return out.reshape(shape)


# ---------------------------------------------------------------------------
# building a workload

def build(spec: WorkloadSpec, seed: Optional[int] = None) -> Workload:
    rng = np.random.default_rng(spec.seed if seed is None else seed)
    S, H, Hkv, D, bs = (spec.num_seqs, spec.num_heads, spec.num_kv_heads,
                        spec.head_dim, spec.block_size)
    assert H % Hkv == 0
    ctx = np.asarray(spec.context_lens(rng), dtype=np.int64)
    assert ctx.shape == (S,) and (ctx >= 1).all()
    pre = spec.shared_prefix_tokens
    assert pre % bs == 0
    assert (ctx > pre).all() if pre else True
    pre_blocks = pre // bs

    # Blocks each sequence owns (the host block manager's allocation).
    nblk = -(-ctx // bs)
    private = nblk - pre_blocks
    needed = pre_blocks + int(private.sum())
    if spec.num_blocks is not None:
        N = spec.num_blocks
    else:
        N = int(math.ceil(spec.pool_factor * needed))
    # room for the copy-on-write destinations and a padding block
    N = max(N, needed + spec.cow_pairs + 1)
    MB = int(nblk.max())

    perm = rng.permutation(N).astype(np.int32)
    cursor = 0
    prefix_ids = perm[cursor:cursor + pre_blocks]
    cursor += pre_blocks
    tables = np.empty((S, MB), dtype=np.int32)
    free = perm[needed:]
    pad_block = int(free[-1])
    tables[:] = pad_block
    for s in range(S):
        tables[s, :pre_blocks] = prefix_ids
        k = int(private[s])
        tables[s, pre_blocks:pre_blocks + k] = perm[cursor:cursor + k]
        cursor += k
    assert cursor == needed

    # Query rows per sequence: its newest q_len tokens (one for decode).
    if spec.query_lens is not None:
        ql = np.asarray(spec.query_lens(rng, ctx), dtype=np.int64)
        assert ql.shape == (S,) and (ql >= 0).all() and (ql <= ctx - pre).all()
    else:
        ql = np.ones(S, dtype=np.int64)
    query_start = np.zeros(S + 1, dtype=np.int32)
    query_start[1:] = np.cumsum(ql)
    T = int(query_start[-1])

    # Tokens cached before the step: the shared prefix once (through
    # sequence 0, whose table names the shared blocks), then each
    # sequence's private history; the newest q_len positions of every
    # sequence are the tokens the step appends.
    hist_seq, hist_pos = [], []
    if pre:
        hist_seq.append(np.zeros(pre, dtype=np.int32))
        hist_pos.append(np.arange(pre, dtype=np.int32))
    for s in range(S):
        lo, hi = pre, int(ctx[s] - ql[s])
        if hi > lo:
            hist_seq.append(np.full(hi - lo, s, dtype=np.int32))
            hist_pos.append(np.arange(lo, hi, dtype=np.int32))
    hist_seq = np.concatenate(hist_seq) if hist_seq else np.zeros(0, np.int32)
    hist_pos = np.concatenate(hist_pos) if hist_pos else np.zeros(0, np.int32)
    Th = hist_seq.shape[0]
    new_seq = np.repeat(np.arange(S, dtype=np.int32), ql)
    new_pos = np.concatenate([np.arange(ctx[s] - ql[s], ctx[s]) for s in range(S)]
                             ).astype(np.int32) if T else np.zeros(0, np.int32)

    query = _normal16(rng, (T, H, D), spec.dtype)
    hist_key = _normal16(rng, (Th, Hkv, D), spec.dtype)
    hist_value = _normal16(rng, (Th, Hkv, D), spec.dtype)
    new_key = _normal16(rng, (T, Hkv, D), spec.dtype)
    new_value = _normal16(rng, (T, Hkv, D), spec.dtype)

    # Copy-on-write: distinct shared blocks are copied into distinct free
    # blocks, and one sequence per pair has its table entry remapped to the
    # private copy ("vLLM源码解析(二)" §3.2: allocate, copy, remap).
    step_tables = tables.copy()
    if spec.cow_pairs:
        P = spec.cow_pairs
        if pre_blocks < P or free.shape[0] - 1 < P or S < P:
            raise ValueError("cow_pairs needs that many shared blocks, free "
                             "blocks and sequences")
        logical = rng.choice(pre_blocks, size=P, replace=False)
        dst = rng.choice(free[:-1], size=P, replace=False)
        who = rng.choice(S, size=P, replace=False)
        src = prefix_ids[logical]
        cow = np.stack([src, dst], axis=1).astype(np.int32)
        for i in range(P):
            step_tables[who[i], logical[i]] = dst[i]
    else:
        cow = np.zeros((0, 2), dtype=np.int32)

    fill = F16_NAN if spec.dtype == "f16" else BF16_NAN
    return Workload(spec=spec, num_blocks=N, max_blocks_per_seq=MB,
                    scale=1.0 / math.sqrt(D), context_lens=ctx.astype(np.int32),
                    block_tables=tables, step_block_tables=step_tables,
                    query=query, hist_seq=hist_seq, hist_pos=hist_pos,
                    hist_key=hist_key, hist_value=hist_value, new_seq=new_seq,
                    new_pos=new_pos, new_key=new_key, new_value=new_value,
                    cow_pairs=cow, pad_block=pad_block, fill=fill, query_start=query_start)


# ---------------------------------------------------------------------------
# the five decode-layer workloads

def _fixed(values):
    return lambda rng: np.asarray(values, dtype=np.int64)


def _uniform(n, lo, hi):
    return lambda rng: rng.integers(lo, hi + 1, size=n)


def _lognormal(n, median, sigma, lo, hi):
    def draw(rng):
        x = np.exp(np.log(median) + sigma * rng.standard_normal(n))
        return np.clip(np.rint(x), lo, hi).astype(np.int64)
    return draw


def _long_skew(n_long, long_len, n_short, lo, hi):
    def draw(rng):
        lens = np.concatenate([np.full(n_long, long_len),
                               rng.integers(lo, hi + 1, size=n_short)])
        return lens[rng.permutation(lens.shape[0])]
    return draw


def _prefix_plus(n, prefix, lo, hi):
    return lambda rng: prefix + rng.integers(lo, hi + 1, size=n)


CONFIGS: Dict[str, WorkloadSpec] = {
    "tiny": WorkloadSpec(
        name="tiny", seed=9601,
        description="4 seqs, context {1,15,16,35}, 4 heads = 4 KV heads, d 64, "
                    "block 16, pool of 16 blocks, fp16",
        num_seqs=4, num_heads=4, num_kv_heads=4, head_dim=64, block_size=16,
        dtype="f16", context_lens=_fixed([1, 15, 16, 35]), num_blocks=16,
        partition_size=0),
    "mha7b": WorkloadSpec(
        name="mha7b", seed=9602,
        description="MHA 7B-like decode layer: 64 seqs, context U[128,2048], "
                    "32 heads, d 128, block 16, bf16, pool 1.25x",
        num_seqs=64, num_heads=32, num_kv_heads=32, head_dim=128, block_size=16,
        dtype="bf16", context_lens=_uniform(64, 128, 2048), partition_size=2048),
    "gqa70b": WorkloadSpec(
        name="gqa70b", seed=9603,
        description="GQA 70B-like decode layer: 128 seqs, context lognormal "
                    "(median 1500, sigma 0.8) clipped [16,8192], 64 query heads "
                    "over 8 KV heads, d 128, block 16, bf16, pool 1.25x",
        num_seqs=128, num_heads=64, num_kv_heads=8, head_dim=128, block_size=16,
        dtype="bf16", context_lens=_lognormal(128, 1500.0, 0.8, 16, 8192),
        partition_size=1024),
    "longctx": WorkloadSpec(
        name="longctx", seed=9604,
        description="long-context skew: 16 seqs (4 x 32768, 12 x U[64,512]), "
                    "32 query heads over 8 KV heads, d 128, block 32, bf16, "
                    "512-token partitions + reduce",
        num_seqs=16, num_heads=32, num_kv_heads=8, head_dim=128, block_size=32,
        dtype="bf16", context_lens=_long_skew(4, 32768, 12, 64, 512)),
    "prefix": WorkloadSpec(
        name="prefix", seed=9605,
        description="prefix-sharing step: 256 seqs sharing one 1024-token prefix "
                    "(64 blocks) + private suffix U[1,1024], 32 query heads over "
                    "8 KV heads, d 128, block 16, bf16; 32 copy-on-write pairs",
        num_seqs=256, num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
        dtype="bf16", context_lens=_prefix_plus(256, 1024, 1, 1024),
        shared_prefix_tokens=1024, cow_pairs=32, partition_size=2048),
}


def _fixed_q(values):
    return lambda rng, ctx: np.asarray(values, dtype=np.int64)


# Prefill-side workloads ("PagedAttention & Continuous Batching" §2.4, §2.5)
# and the prefix-aware decode of the prefix-sharing step.
CONFIGS["mixed"] = WorkloadSpec(
    name="mixed", seed=9606,
    description="mixed batch of the continuous-batching iteration: 2 decode requests "
                "(1 token; contexts 37, 70) + 2 fresh prompts prefilled whole (50 and "
                "30 tokens), 8 query heads over 2 KV heads, d 64, block 16, fp16",
    num_seqs=4, num_heads=8, num_kv_heads=2, head_dim=64, block_size=16, dtype="f16",
    context_lens=_fixed([37, 70, 50, 30]), query_lens=_fixed_q([1, 1, 50, 30]),
    partition_size=0)
CONFIGS["chunked"] = WorkloadSpec(
    name="chunked", seed=9607,
    description="chunked-prefill iteration: four 2048-token prompts, each at a "
                "different 512-token chunk (contexts 512, 1024, 1536, 2048; 2048 "
                "batched tokens), 64 query heads over 8 KV heads, d 128, block 16, bf16",
    num_seqs=4, num_heads=64, num_kv_heads=8, head_dim=128, block_size=16, dtype="bf16",
    context_lens=_fixed([512, 1024, 1536, 2048]), query_lens=_fixed_q([512] * 4),
    partition_size=0)
CONFIGS["prefix-cascade"] = dataclasses.replace(
    CONFIGS["prefix"], name="prefix-cascade", cascade=True, partition_size=1024,
    description=CONFIGS["prefix"].description + "; prefix-aware decode (shared "
    "prefix read once per group)")


def fp8_variant(spec: WorkloadSpec) -> WorkloadSpec:
    """The same workload with e4m3 KV pools ("--kv-cache-dtype fp8")."""
    return dataclasses.replace(spec, name=spec.name + "-fp8", kv_dtype="fp8",
                               description=spec.description + "; KV cache FP8 e4m3 "
                               f"(per-pool scale {spec.kv_scale})")


def small_variant(name: str, seed: int = 0) -> WorkloadSpec:
    """A reduced copy of one of the five workloads -- same head layout,
    dtype and block size, fewer and shorter sequences -- that the oracle
    finishes in seconds while still spanning several tiles, partitions and a
    ragged tail."""
    if name.endswith("-fp8"):
        return fp8_variant(small_variant(name[:-4], seed))
    base = CONFIGS[name]
    if name == "tiny":
        return dataclasses.replace(base, seed=seed or base.seed)
    if name == "mha7b":
        return dataclasses.replace(base, name="mha7b-small", seed=seed or 19602,
                                   num_seqs=5, num_heads=8, num_kv_heads=8,
                                   context_lens=_uniform(5, 1, 700),
                                   partition_size=128)
    if name == "gqa70b":
        return dataclasses.replace(base, name="gqa70b-small", seed=seed or 19603,
                                   num_seqs=6, num_heads=16, num_kv_heads=2,
                                   context_lens=_lognormal(6, 300.0, 0.8, 1, 900),
                                   partition_size=128)
    if name == "longctx":
        return dataclasses.replace(base, name="longctx-small", seed=seed or 19604,
                                   num_seqs=5, num_heads=8, num_kv_heads=2,
                                   context_lens=_long_skew(2, 1500, 3, 1, 120),
                                   partition_size=256)
    if name == "mixed":
        return dataclasses.replace(base, seed=seed or base.seed)
    if name == "chunked":
        return dataclasses.replace(base, name="chunked-small", seed=seed or 19607,
                                   num_seqs=4, num_heads=16, num_kv_heads=2,
                                   context_lens=_fixed([100, 300, 513, 7]),
                                   query_lens=_fixed_q([100, 64, 129, 1]))
    if name in ("prefix", "prefix-cascade"):
        return dataclasses.replace(base, name=name + "-small", seed=seed or 19605,
                                   num_seqs=6, num_heads=8, num_kv_heads=2,
                                   context_lens=_prefix_plus(6, 128, 1, 200),
                                   shared_prefix_tokens=128, cow_pairs=4,
                                   partition_size=128)
    raise KeyError(name)


CONFIGS["gqa70b-fp8"] = fp8_variant(CONFIGS["gqa70b"])
CONFIGS["longctx-fp8"] = fp8_variant(CONFIGS["longctx"])
CONFIGS["chunked-fp8"] = fp8_variant(CONFIGS["chunked"])
CONFIGS["prefix-cascade-fp8"] = fp8_variant(CONFIGS["prefix-cascade"])
CONFIGS["mixed-fp8"] = fp8_variant(CONFIGS["mixed"])

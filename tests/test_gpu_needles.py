"""Needle parity: cases where one token decides the output, placed at every
boundary the kernels tile by.

"PagedAttention & Continuous Batching" §1.6 attends exactly positions
[0, context_len) of a sequence.  On random N(0, 1) inputs a kernel that
drops one 16-token tile, or counts the appended token twice, moves each
output by about 1 % of its size and could pass the contract tolerance.
Here the inputs make a single position matter:

  * dominant needle -- for one (sequence, KV head), the G query heads of the
    group are one row q0 and the key at position p is q0 scaled so that its
    score is 20 (the others score about N(0, 1)); its value row is a
    distinctive constant pattern.  The output is that row, and a kernel that
    misses position p is off by O(1).
  * balanced needle -- every other key of that KV head is zero (score 0,
    weight 1 each) and the needle's score is ln(context - 1), so the needle
    holds exactly half of the softmax mass.  Counting it twice moves the
    output by a sixth of the needle's value row; dropping it, by a half.

Needles sit at token 0, both sides of 16-token tile edges and block edges,
both sides of partition edges, the middle, the last cached row and the
appended position context - 1; for prefix-aware decode also both sides of
the shared-prefix end and inside the shared blocks; for chunked prefill at
64-token tile edges, before and inside the chunk.  Each case runs the
decode step (fused append and separate write; single pass and split),
prefix-aware decode and chunked prefill, each over 16-bit and FP8 pools,
and compares every
output element with the oracle at the contract tolerance; dominant needles
are also checked against their value row directly.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from paged_kv_cache_96_gb300 import workloads as W  # noqa: E402
from stepping import OracleStep, assert_attention_close  # noqa: E402


def _fixed(values):
    return lambda rng: np.asarray(values, dtype=np.int64)


def _fixed_q(values):
    return lambda rng, ctx: np.asarray(values, dtype=np.int64)


SPECS = {
    # GQA, group 8, bf16, 16-token blocks
    "gqa": W.WorkloadSpec(
        name="needle-gqa", description="needles, GQA", seed=7701, num_seqs=16,
        num_heads=16, num_kv_heads=2, head_dim=128, block_size=16, dtype="bf16",
        context_lens=_fixed([1, 2, 16, 17, 32, 33, 63, 64, 65, 129, 200, 256, 257, 700,
                             1025, 2100]), partition_size=64),
    # group 2, head_dim 64, fp16, 32-token blocks (block edges off the tile grid)
    "d64": W.WorkloadSpec(
        name="needle-d64", description="needles, d 64, block 32", seed=7702, num_seqs=8,
        num_heads=4, num_kv_heads=2, head_dim=64, block_size=32, dtype="f16",
        context_lens=_fixed([1, 31, 32, 33, 100, 300, 513, 1000]), partition_size=128),
    # prefix-aware decode: 128 shared tokens, group 4, four KV heads
    "cascade": W.WorkloadSpec(
        name="needle-cascade", description="needles, shared prefix", seed=7703,
        num_seqs=8, num_heads=16, num_kv_heads=4, head_dim=128, block_size=16,
        dtype="bf16", context_lens=_fixed([129, 130, 143, 144, 145, 192, 193, 328]),
        shared_prefix_tokens=128, cascade=True, partition_size=64),
    # chunked prefill: chunks mid-context, a whole prompt, a decode row
    "prefill": W.WorkloadSpec(
        name="needle-prefill", description="needles, chunked prefill", seed=7704,
        num_seqs=4, num_heads=16, num_kv_heads=2, head_dim=128, block_size=16,
        dtype="bf16", context_lens=_fixed([100, 300, 513, 70]),
        query_lens=_fixed_q([100, 64, 129, 1]), partition_size=0),
}
SPECS["gqa-fp8"] = W.fp8_variant(SPECS["gqa"])
SPECS["d64-fp8"] = W.fp8_variant(SPECS["d64"])
SPECS["cascade-fp8"] = W.fp8_variant(SPECS["cascade"])
SPECS["prefill-fp8"] = W.fp8_variant(SPECS["prefill"])
SPECS["prefill-d64-fp8"] = W.fp8_variant(dataclasses.replace(
    SPECS["prefill"], name="needle-prefill-d64", head_dim=64, block_size=32))

DOMINANT_SCORE = 20.0
VROW = np.array([3.0, 3.25, 3.5, 3.75])   # exact in fp16 and bf16
BALANCED_V = 4.0


# ---- host-side value handling (bit patterns <-> float64) ----------------------

def _vals(bits: np.ndarray, dtype: str) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return b.view(np.float16).astype(np.float64)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bits(x: np.ndarray, dtype: str) -> np.ndarray:
    return W._round_to(np.asarray(x, dtype=np.float32), dtype)


def _vrow(d: int) -> np.ndarray:
    return np.tile(VROW, d // 4)


def _rows_of(w, s, p):
    """(array name, index) holding the K/V of position p of sequence s: the
    step's new tokens, a private history token, or -- inside a shared
    prefix -- the prefix token written once through sequence 0."""
    hit = np.nonzero((w.new_seq == s) & (w.new_pos == p))[0]
    if hit.size:
        return "new", int(hit[0])
    pre = w.spec.shared_prefix_tokens
    owner = 0 if p < pre else s
    hit = np.nonzero((w.hist_seq == owner) & (w.hist_pos == p))[0]
    assert hit.size == 1, (s, p)
    return "hist", int(hit[0])


def _set_kv(w, s, kh, p, k, v):
    kind, i = _rows_of(w, s, p)
    getattr(w, kind + "_key")[i, kh] = _bits(k, w.dtype)
    getattr(w, kind + "_value")[i, kh] = _bits(v, w.dtype)


def _query_rows(w, s):
    return range(int(w.query_start[s]), int(w.query_start[s + 1]))


def _equalise_group(w, seqs, kh, q0_bits):
    """Every query row of the listed sequences gets q0 in each head of KV
    head kh's group."""
    G = w.H // w.Hkv
    for s in seqs:
        for r in _query_rows(w, s):
            w.query[r, kh * G:(kh + 1) * G] = q0_bits


def _needle_key(w, q0_bits, score):
    """A key whose score against q0 is `score` (before rounding)."""
    q0 = _vals(q0_bits, w.dtype)
    return q0 * (score / (w.scale * float(q0 @ q0)))


def plant_dominant(w, s, kh, p, share=None):
    """Dominant needle at position p of (s, kh); with `share`, p is a shared
    prefix position and every listed sequence gets the same group query."""
    seqs = [s] if share is None else share
    q0_bits = w.query[int(w.query_start[s]), kh * (w.H // w.Hkv)].copy()
    _equalise_group(w, seqs, kh, q0_bits)
    _set_kv(w, s, kh, p, _needle_key(w, q0_bits, DOMINANT_SCORE), _vrow(w.D))


def zero_keys(w, kh):
    w.hist_key[:, kh] = 0
    w.new_key[:, kh] = 0


def plant_balanced(w, s, kh, p):
    """Balanced needle (keys of kh already zero): half the softmax mass."""
    c = int(w.context_lens[s])
    q0_bits = w.query[int(w.query_start[s]), kh * (w.H // w.Hkv)].copy()
    _equalise_group(w, [s], kh, q0_bits)
    score = float(np.log(c - 1)) if c > 1 else 0.0
    _set_kv(w, s, kh, p, _needle_key(w, q0_bits, score), np.full(w.D, BALANCED_V))


# ---- needle positions ------------------------------------------------------------

def positions(c, bs, P, pre=0, own_only=False, shared_only=False):
    cand = {0, 1, 15, 16, 17, bs - 1, bs, bs + 1, c // 2, c - 2, c - 1}
    if P:
        cand |= {P - 1, P, P + 1, 2 * P - 1, 2 * P}
    if pre:
        cand |= {pre - 16, pre - 1, pre, pre + 15, pre + 16, pre + P - 1, pre + P}
    lo = pre if own_only else 0
    hi = pre if shared_only else c
    return sorted(x for x in cand if lo <= x < hi)


def _decode_rounds(spec, P):
    """Per round: [(seq, dominant position, balanced position)]."""
    ctx = np.asarray(spec.context_lens(None))
    lists = [positions(int(c), spec.block_size, P) for c in ctx]
    R = max(len(x) for x in lists)
    return [[(s, L[(r + s) % len(L)], L[(r + s + len(L) // 2) % len(L)])
             for s, L in enumerate(lists)] for r in range(R)]


# ---- running a case on both sides -----------------------------------------------

@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_96_gb300 import step
    return step


def _dequant_row(w, v):
    """What an FP8 pool holds for value row v (torch's e4m3 cast of
    v / scale, times the scale)."""
    x = torch.from_numpy(np.asarray(v, dtype=np.float32) * np.float32(1.0 / w.spec.kv_scale))
    return x.to(torch.float8_e4m3fn).to(torch.float64).numpy() * w.spec.kv_scale


def _check_dominant(w, got, want, s, kh, rows=None):
    G = w.H // w.Hkv
    row = _vrow(w.D)
    if w.fp8:
        row = _dequant_row(w, row)
    rows = [s] if rows is None else rows
    for r in rows:
        for h in range(kh * G, (kh + 1) * G):
            # the oracle confirms the construction; the GPU must give the row
            assert np.abs(want[r, h] - row).max() < 1e-3, (s, kh, r, h)
            assert np.abs(got[r, h] - row).max() <= 0.02 + 0.01 * np.abs(row).max(), \
                (s, kh, r, h, got[r, h][:4])


def _run(S, w, P, how):
    st = S.DecodeStep(w, partition_size=P)
    if how == "append":
        st.copy_blocks()
        st.append_attention()
    else:
        st.slot_mapping_and_cache()
        st.copy_blocks()
        st.attention()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    return S.to_float(st.out)


DECODE_CASES = [(n, P, how) for n in ("gqa", "d64", "gqa-fp8", "d64-fp8")
                for P in (0, SPECS[n].partition_size, 16)
                for how in ("append", "separate")]


@pytest.mark.parametrize("name,P,how", DECODE_CASES, ids=lambda x: str(x))
def test_decode_needles(S, name, P, how):
    spec = SPECS[name]
    for r, plan in enumerate(_decode_rounds(spec, P)):
        w = W.build(spec)
        zero_keys(w, 1)
        for s, pd, pb in plan:
            plant_dominant(w, s, 0, pd)
            plant_balanced(w, s, 1, pb)
        got = _run(S, w, P, how)
        want = OracleStep(w).attention()
        assert_attention_close(got, want, f"{name} P {P} {how} round {r} {plan}")
        for s, pd, _ in plan:
            _check_dominant(w, got, want, s, 0)


@pytest.mark.parametrize("name", ["cascade", "cascade-fp8"])
@pytest.mark.parametrize("how", ["append", "separate"])
def test_cascade_needles(S, how, name):
    """Prefix-aware decode.  KV head 0: a dominant needle in each sequence's
    own tokens; head 1: one dominant needle inside the shared prefix, every
    sequence's group query set to the same row; head 2: balanced needles
    (keys of head 2 zero everywhere, the shared prefix included); head 3:
    untouched."""
    spec = SPECS[name]
    pre, P = spec.shared_prefix_tokens, spec.partition_size
    ctx = np.asarray(spec.context_lens(None))
    own = [positions(int(c), spec.block_size, P, pre, own_only=True) for c in ctx]
    shared = positions(int(ctx.min()), spec.block_size, P, pre, shared_only=True)
    R = max(max(len(x) for x in own), len(shared))
    for r in range(R):
        w = W.build(spec)
        zero_keys(w, 2)
        plan = []
        for s, L in enumerate(own):
            pd = L[(r + s) % len(L)]
            pb = L[(r + s + len(L) // 2) % len(L)]
            plant_dominant(w, s, 0, pd)
            plant_balanced(w, s, 2, pb)
            plan.append((s, pd, pb))
        ps = shared[r % len(shared)]
        plant_dominant(w, 0, 1, ps, share=list(range(w.S)))
        got = _run(S, w, P, how)
        want = OracleStep(w).attention()
        assert_attention_close(got, want, f"{name} {how} round {r} {plan} shared {ps}")
        for s, _, _ in plan:
            _check_dominant(w, got, want, s, 0)
            _check_dominant(w, got, want, s, 1)


@pytest.mark.parametrize("name", ["prefill", "prefill-fp8", "prefill-d64-fp8"])
def test_prefill_needles(S, name):
    """Chunked prefill: a dominant needle per (sequence, KV head) -- before
    the chunk, at its first row, at 64-token tile edges, inside it -- with
    every chunk row's group query set to one row; rows at or past the needle
    give its value row, rows before it must not see it."""
    spec = SPECS[name]
    ctx = np.asarray(spec.context_lens(None))
    ql = np.asarray(spec.query_lens(None, ctx))
    lists = []
    for c, q in zip(ctx, ql):
        c0 = int(c - q)
        cand = {0, 15, 16, 63, 64, 65, 127, 128, c0 - 1, c0, c0 + 1, c0 + 63, c0 + 64,
                int(c) - 1, int(c) // 2}
        lists.append(sorted(x for x in cand if 0 <= x < c))
    R = max(len(x) for x in lists)
    for r in range(R):
        w = W.build(spec)
        plan = []
        for s, L in enumerate(lists):
            p0, p1 = L[(r + s) % len(L)], L[(r + s + len(L) // 2) % len(L)]
            plant_dominant(w, s, 0, p0)
            plant_dominant(w, s, 1, p1)
            plan.append((s, p0, p1))
        got = _run(S, w, 0, "separate")
        want = OracleStep(w).attention()
        assert_attention_close(got, want, f"{name} round {r} {plan}")
        for s, p0, p1 in plan:
            c, q = int(w.context_lens[s]), int(ql[s])
            for kh, p in ((0, p0), (1, p1)):
                seen = [int(w.query_start[s]) + i for i in range(q) if c - q + i >= p]
                _check_dominant(w, got, want, s, kh, rows=seen)

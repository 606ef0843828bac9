"""Pins of the CPU oracle to facts outside itself.

Each ``pin_*`` function takes a loaded oracle library (the real one, or a
deliberately broken copy in the mutation tests) and raises AssertionError
when the oracle disagrees with:

  * a value the pages print (the worked slot example of "PagedAttention &
    Continuous Batching" §1.5, stored under tests/golden/),
  * the exact IEEE / bfloat16 conversions of numpy and torch,
  * structural invariants of the block-table picture (§1.4, §1.5),
  * a library routine on a special case (torch's scaled-dot-product
    attention in float64 on the gathered, contiguous K/V -- the §1.6
    "gather, then attend" definition),
  * closed forms (one token, constant values, equal keys, a two-token
    logistic weight, disjoint per-head values),
  * invariants (physical placement, shared vs private prefix blocks,
    split-then-merge vs unsplit, softmax rows summing to one, large
    scores staying finite).

The layouts built here use numpy slicing of whole blocks (block b of a
sequence holds its tokens b*bs .. b*bs+bs-1), never the oracle's own index
arithmetic.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------
# helpers (test-side, independent of the oracle's arithmetic)

def f16_bits(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def bf16_bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f16_vals(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def place_sequences(logical, tables, num_blocks, bs, fill=np.uint16(0x7E00)):
    """Pool [N, bs, Hkv, d] holding each sequence's logical rows
    [ctx, Hkv, d] block by block: block b of the sequence -> pool[table[b]]."""
    Hkv, d = logical[0].shape[1:]
    pool = np.full((num_blocks, bs, Hkv, d), fill, dtype=np.uint16)
    for rows, table in zip(logical, tables):
        ctx = rows.shape[0]
        for b in range(-(-ctx // bs)):
            chunk = rows[b * bs:(b + 1) * bs]
            pool[table[b], :chunk.shape[0]] = chunk
    return pool


def sdpa_reference(q_bits, k_logical, v_logical, scale, decode_np):
    """torch scaled_dot_product_attention in float64 on contiguous K/V.
    q_bits [S, H, d]; k/v_logical: list of [ctx, Hkv, d] bit arrays."""
    S, H, d = q_bits.shape
    out = np.zeros((S, H, d))
    for s in range(S):
        k = torch.from_numpy(decode_np(k_logical[s]))      # [ctx, Hkv, d]
        v = torch.from_numpy(decode_np(v_logical[s]))
        ctx, Hkv, _ = k.shape
        if ctx == 0:
            continue
        g = H // Hkv
        k = k.permute(1, 0, 2).repeat_interleave(g, dim=0)  # [H, ctx, d]
        v = v.permute(1, 0, 2).repeat_interleave(g, dim=0)
        q = torch.from_numpy(decode_np(q_bits[s]))[:, None, :]  # [H, 1, d]
        o = torch.nn.functional.scaled_dot_product_attention(
            q[None], k[None], v[None], scale=scale)[0, :, 0, :]
        out[s] = o.numpy()
    return out


def random_paged_case(rng, ctxs, H, Hkv, d, bs, extra_blocks=3, dtype="f16",
                      spread=1.0):
    """Random GQA decode case with shuffled physical blocks."""
    S = len(ctxs)
    nblk = [-(-c // bs) for c in ctxs]
    N = sum(nblk) + extra_blocks
    perm = rng.permutation(N)
    tables = np.full((S, max(max(nblk), 1)), perm[-1], dtype=np.int32)
    cur = 0
    for s in range(S):
        tables[s, :nblk[s]] = perm[cur:cur + nblk[s]]
        cur += nblk[s]
    conv = f16_bits if dtype == "f16" else bf16_bits
    kl = [conv(rng.standard_normal((c, Hkv, d))) for c in ctxs]
    vl = [conv(rng.standard_normal((c, Hkv, d))) for c in ctxs]
    q = conv(spread * rng.standard_normal((S, H, d)))
    fill = np.uint16(0x7E00) if dtype == "f16" else np.uint16(0x7FC0)
    kc = place_sequences(kl, tables, N, bs, fill)
    vc = place_sequences(vl, tables, N, bs, fill)
    return dict(q=q, kc=kc, vc=vc, tables=tables,
                ctx=np.asarray(ctxs, dtype=np.int32), kl=kl, vl=vl, N=N)


def _dec(dtype):
    if dtype == "f16":
        return f16_vals
    return lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(
        torch.bfloat16).to(torch.float64).numpy()


def _close(a, b, rtol=1e-12, atol=1e-12, what=""):
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    ok = np.abs(a - b) <= atol + rtol * np.abs(b)
    assert ok.all(), f"{what}: max abs err {np.nanmax(np.abs(a - b))}"


# ---------------------------------------------------------------------------
# pins

def pin_worked_slot_example(lib):
    """"PagedAttention & Continuous Batching" §1.5: position 35,
    block_size 16, block_table[2] = 9 -> slot 147."""
    with open(os.path.join(GOLDEN, "slot_worked_example.json")) as f:
        g = json.load(f)
    got = oracle.slot_for_position(g["block_table"], g["position"],
                                   g["block_size"], lib=lib)
    assert got == g["slot"], (got, g["slot"])
    got = oracle.slot_mapping(np.asarray([g["block_table"]]), [0], [g["position"]],
                              g["block_size"], lib=lib)
    assert int(got[0]) == g["slot"]


def pin_slot_structure(lib):
    """§1.4/§1.5: the slots of a sequence's positions tile exactly the
    physical blocks its table names, block_size consecutive slots per block,
    in position order."""
    rng = np.random.default_rng(5)
    for bs in (1, 4, 16, 32):
        nblk = 6
        table = rng.permutation(50)[:nblk].astype(np.int32)
        n = nblk * bs - (bs // 2)
        slots = oracle.slot_mapping(table[None, :], np.zeros(n, np.int32),
                                    np.arange(n, dtype=np.int32), bs, lib=lib)
        assert len(set(slots.tolist())) == n
        for b in range(nblk):
            seg = slots[b * bs:min((b + 1) * bs, n)]
            want = np.arange(table[b] * bs, table[b] * bs + seg.shape[0])
            assert np.array_equal(seg, want), (bs, b, seg[:4], want[:4])


def pin_fp16_decode_exact(lib):
    """Every binary16 pattern decodes to numpy's float16 -> float64 value."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits, oracle.F16, lib=lib)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def pin_bf16_decode_exact(lib):
    """Every bfloat16 pattern decodes to torch's bfloat16 -> float64 value."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits, oracle.BF16, lib=lib)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(
        torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def pin_reshape_and_cache_gather_roundtrip(lib):
    """Writing every token of a sequence through its slots, then gathering
    whole blocks in table order and truncating to the context (§1.6's
    gather), gives back the logical rows; nothing else in the pool moves;
    negative slots write nothing."""
    rng = np.random.default_rng(7)
    bs, Hkv, d, N = 4, 3, 8, 20
    ctxs = [1, 4, 9, 14]
    S = len(ctxs)
    perm = rng.permutation(N)
    tables = np.full((S, 4), perm[-1], dtype=np.int32)
    cur = 0
    for s, c in enumerate(ctxs):
        k = -(-c // bs)
        tables[s, :k] = perm[cur:cur + k]
        cur += k
    seq = np.concatenate([np.full(c, s) for s, c in enumerate(ctxs)]).astype(np.int32)
    pos = np.concatenate([np.arange(c) for c in ctxs]).astype(np.int32)
    T = seq.shape[0]
    key = rng.integers(0, 0x7C00, size=(T, Hkv, d)).astype(np.uint16)
    val = rng.integers(0, 0x7C00, size=(T, Hkv, d)).astype(np.uint16)
    kc = np.full((N, bs, Hkv, d), 0xFFFF, dtype=np.uint16)
    vc = kc.copy()
    slots = oracle.slot_mapping(tables, seq, pos, bs, lib=lib)
    slots_pad = np.concatenate([slots, [-1, -7]])
    key_pad = np.concatenate([key, np.zeros((2, Hkv, d), np.uint16)])
    val_pad = np.concatenate([val, np.zeros((2, Hkv, d), np.uint16)])
    oracle.reshape_and_cache(key_pad, val_pad, kc, vc, slots_pad, lib=lib)
    off = 0
    for s, c in enumerate(ctxs):
        nb = -(-c // bs)
        gk = np.concatenate([kc[tables[s, b]] for b in range(nb)])[:c]
        gv = np.concatenate([vc[tables[s, b]] for b in range(nb)])[:c]
        assert np.array_equal(gk, key[off:off + c]), s
        assert np.array_equal(gv, val[off:off + c]), s
        off += c
    written = int((kc != 0xFFFF).any(axis=(2, 3)).sum())
    assert written == T, (written, T)
    assert int((vc != 0xFFFF).any(axis=(2, 3)).sum()) == T


def pin_copy_blocks(lib):
    """"vLLM源码解析(二)" §3.2: after the copy every destination block holds
    its source block's K and V bytes; every other block is unchanged."""
    rng = np.random.default_rng(11)
    N, bs, Hkv, d = 12, 4, 2, 8
    kc = rng.integers(0, 65536, size=(N, bs, Hkv, d)).astype(np.uint16)
    vc = rng.integers(0, 65536, size=(N, bs, Hkv, d)).astype(np.uint16)
    k0, v0 = kc.copy(), vc.copy()
    pairs = np.array([[3, 7], [0, 11], [5, 2]], dtype=np.int32)
    oracle.copy_blocks(kc, vc, pairs, lib=lib)
    for src, dst in pairs:
        assert np.array_equal(kc[dst], k0[src]) and np.array_equal(vc[dst], v0[src])
    others = [b for b in range(N) if b not in pairs[:, 1]]
    assert np.array_equal(kc[others], k0[others]) and np.array_equal(vc[others], v0[others])


def pin_copy_blocks_u8(lib):
    """"vLLM源码解析(二)" §3.2 on 1-byte (FP8) pools: the result equals numpy
    whole-block slice copies made pair by pair -- every destination block
    holds the source block's K and V codes, byte for byte over the whole
    block, and every other block keeps its bytes.  Several shapes, so that a
    block length taken from the wrong sizes (or halved) shows."""
    rng = np.random.default_rng(17)
    for N, bs, Hkv, d, npairs in ((12, 4, 2, 8, 3), (9, 16, 3, 128, 4), (20, 1, 1, 16, 7)):
        kc = rng.integers(0, 256, size=(N, bs, Hkv, d)).astype(np.uint8)
        vc = rng.integers(0, 256, size=(N, bs, Hkv, d)).astype(np.uint8)
        ids = rng.permutation(N)[:2 * npairs]
        pairs = np.stack([ids[:npairs], ids[npairs:]], axis=1).astype(np.int32)
        want_k, want_v = kc.copy(), vc.copy()
        for src, dst in pairs:
            want_k[dst] = want_k[src]
            want_v[dst] = want_v[src]
        oracle.copy_blocks_u8(kc, vc, pairs, lib=lib)
        assert np.array_equal(kc, want_k) and np.array_equal(vc, want_v), (N, bs, Hkv, d)


def pin_attention_matches_sdpa(lib):
    """§1.6 on random GQA inputs with shuffled blocks equals torch's
    float64 scaled-dot-product attention on the gathered contiguous K/V."""
    rng = np.random.default_rng(13)
    for dtype, (H, Hkv, d, bs) in (("f16", (4, 2, 16, 4)), ("bf16", (6, 3, 8, 8)),
                                   ("f16", (2, 2, 32, 16))):
        c = random_paged_case(rng, [1, 5, 9, 13, 23], H, Hkv, d, bs, dtype=dtype)
        scale = 1.0 / math.sqrt(d)
        dt = oracle.F16 if dtype == "f16" else oracle.BF16
        got = oracle.paged_attention(c["q"], c["kc"], c["vc"], c["tables"], c["ctx"],
                                     scale, dt, lib=lib)
        want = sdpa_reference(c["q"], c["kl"], c["vl"], scale, _dec(dtype))
        _close(got, want, 1e-11, 1e-12, f"sdpa {dtype} {H}/{Hkv}")


def pin_attention_closed_forms(lib):
    """One token -> its value row; constant value rows -> that row; equal
    keys -> mean of the values; two tokens with scores 0 and x*scale ->
    v0 + sigmoid(x*scale) (v1 - v0)."""
    d, bs, N = 8, 4, 6
    dec = f16_vals
    rng = np.random.default_rng(17)
    scale = 0.25
    tables = np.array([[4, 1]], dtype=np.int32)
    # one token
    k = f16_bits(rng.standard_normal((1, 1, d)))
    v = f16_bits(rng.standard_normal((1, 1, d)))
    q = f16_bits(rng.standard_normal((1, 1, d)))
    kc = place_sequences([k], tables, N, bs)
    vc = place_sequences([v], tables, N, bs)
    o = oracle.paged_attention(q, kc, vc, tables, [1], scale, oracle.F16, lib=lib)
    assert np.array_equal(o[0, 0], dec(v[0, 0])), "one token"
    # constant values, random keys (7 tokens across two blocks)
    k = f16_bits(rng.standard_normal((7, 1, d)))
    c_row = f16_bits(rng.standard_normal(d))
    v = np.broadcast_to(c_row, (7, 1, d)).copy()
    kc = place_sequences([k], tables, N, bs)
    vc = place_sequences([v], tables, N, bs)
    o = oracle.paged_attention(q, kc, vc, tables, [7], scale, oracle.F16, lib=lib)
    _close(o[0, 0], dec(c_row), 1e-14, 1e-14, "constant values")
    # equal keys
    k = np.broadcast_to(f16_bits(rng.standard_normal(d)), (7, 1, d)).copy()
    v = f16_bits(rng.standard_normal((7, 1, d)))
    kc = place_sequences([k], tables, N, bs)
    vc = place_sequences([v], tables, N, bs)
    o = oracle.paged_attention(q, kc, vc, tables, [7], scale, oracle.F16, lib=lib)
    _close(o[0, 0], dec(v[:, 0]).mean(axis=0), 1e-13, 1e-14, "equal keys")
    # two tokens: k0 = 0 (score 0), k1 = e_0 (score q_0 * scale)
    for x in (3.0, -2.5, 0.75):
        q = np.zeros((1, 1, d), np.uint16)
        q[0, 0, 0] = f16_bits(x)
        k = np.zeros((2, 1, d), np.uint16)
        k[1, 0, 0] = f16_bits(1.0)
        v = f16_bits(rng.standard_normal((2, 1, d)))
        kc = place_sequences([k], tables, N, bs)
        vc = place_sequences([v], tables, N, bs)
        o = oracle.paged_attention(q, kc, vc, tables, [2], scale, oracle.F16, lib=lib)
        w1 = 1.0 / (1.0 + math.exp(-x * scale))
        want = dec(v[0, 0]) + w1 * (dec(v[1, 0]) - dec(v[0, 0]))
        _close(o[0, 0], want, 1e-13, 1e-14, f"two tokens x={x}")


def pin_gqa_head_groups(lib):
    """Query heads 0..G-1 read KV head 0, heads G..2G-1 read KV head 1:
    with every value row of KV head j equal to (j+1), the output of query
    head h is (h // G) + 1."""
    H, Hkv, d, bs, N = 6, 3, 8, 4, 8
    rng = np.random.default_rng(19)
    ctx = 6
    tables = np.array([[5, 2]], dtype=np.int32)
    k = f16_bits(rng.standard_normal((ctx, Hkv, d)))
    v = np.zeros((ctx, Hkv, d), np.uint16)
    for j in range(Hkv):
        v[:, j, :] = f16_bits(j + 1.0)
    q = f16_bits(rng.standard_normal((1, H, d)))
    kc = place_sequences([k], tables, N, bs)
    vc = place_sequences([v], tables, N, bs)
    o = oracle.paged_attention(q, kc, vc, tables, [ctx], 0.3, oracle.F16, lib=lib)
    for h in range(H):
        _close(o[0, h], np.full(d, h // (H // Hkv) + 1.0), 1e-14, 1e-14, f"head {h}")


def pin_block_placement_invariance(lib):
    """Output is identical (bit for bit) under any permutation of where the
    physical blocks sit in the pool."""
    rng = np.random.default_rng(23)
    c = random_paged_case(rng, [3, 17, 30], 4, 2, 16, 4)
    scale = 0.25
    base = oracle.paged_attention(c["q"], c["kc"], c["vc"], c["tables"], c["ctx"],
                                  scale, oracle.F16, lib=lib)
    for _ in range(3):
        p = rng.permutation(c["N"])           # new location of block b is p[b]
        kc2 = np.empty_like(c["kc"])
        vc2 = np.empty_like(c["vc"])
        kc2[p] = c["kc"]
        vc2[p] = c["vc"]
        t2 = p[c["tables"]].astype(np.int32)
        o = oracle.paged_attention(c["q"], kc2, vc2, t2, c["ctx"], scale, oracle.F16,
                                   lib=lib)
        assert np.array_equal(o, base)


def pin_shared_prefix_equals_private(lib):
    """"vLLM 架构详解" shared-prefix blocks: two tables naming the same
    prefix blocks give the same output as private copies of them."""
    rng = np.random.default_rng(29)
    bs, Hkv, H, d = 4, 2, 4, 8
    pre = f16_bits(rng.standard_normal((8, Hkv, d)))      # 2 shared blocks
    vpre = f16_bits(rng.standard_normal((8, Hkv, d)))
    sa = f16_bits(rng.standard_normal((3, Hkv, d)))
    sb = f16_bits(rng.standard_normal((5, Hkv, d)))
    va = f16_bits(rng.standard_normal((3, Hkv, d)))
    vb = f16_bits(rng.standard_normal((5, Hkv, d)))
    kA, kB = np.concatenate([pre, sa]), np.concatenate([pre, sb])
    vA, vB = np.concatenate([vpre, va]), np.concatenate([vpre, vb])
    q = f16_bits(rng.standard_normal((2, H, d)))
    shared = np.array([[0, 1, 4, 9], [0, 1, 5, 6]], dtype=np.int32)
    private = np.array([[7, 8, 4, 9], [2, 3, 5, 6]], dtype=np.int32)
    N = 10
    kc_s = place_sequences([kA, kB], shared, N, bs)
    vc_s = place_sequences([vA, vB], shared, N, bs)
    kc_p = place_sequences([kA, kB], private, N, bs)
    vc_p = place_sequences([vA, vB], private, N, bs)
    ctx = [11, 13]
    o_s = oracle.paged_attention(q, kc_s, vc_s, shared, ctx, 0.35, oracle.F16, lib=lib)
    o_p = oracle.paged_attention(q, kc_p, vc_p, private, ctx, 0.35, oracle.F16, lib=lib)
    assert np.array_equal(o_s, o_p)


def pin_softmax_rows(lib):
    """Softmax weights are non-negative, sum to one, and the weighted sum
    of the gathered value rows is the attention output."""
    rng = np.random.default_rng(31)
    c = random_paged_case(rng, [1, 6, 21], 4, 2, 16, 4)
    scale = 0.25
    out = oracle.paged_attention(c["q"], c["kc"], c["vc"], c["tables"], c["ctx"],
                                 scale, oracle.F16, lib=lib)
    for s in range(3):
        for h in range(4):
            w = oracle.attention_weights(c["q"], c["kc"], c["tables"], c["ctx"], s, h,
                                         scale, oracle.F16, lib=lib)
            assert (w >= 0).all() and abs(w.sum() - 1.0) < 1e-13
            v = f16_vals(c["vl"][s][:, h // 2, :])
            _close(w @ v, out[s, h], 1e-12, 1e-13, "weights @ V")


def pin_split_merge_equals_unsplit(lib):
    """Partition pass + log-sum-exp merge equals unsplit attention for any
    partition size; each partition's (m, l, o) equals attention restricted to
    that partition's tokens."""
    rng = np.random.default_rng(37)
    ctxs = [1, 7, 16, 33, 50]
    c = random_paged_case(rng, ctxs, 4, 2, 16, 4)
    scale = 0.25
    full = oracle.paged_attention(c["q"], c["kc"], c["vc"], c["tables"], c["ctx"],
                                  scale, oracle.F16, lib=lib)
    for P in (1, 4, 5, 16, 64):
        nparts = np.array([oracle.num_partitions(x, P, lib=lib) for x in ctxs])
        assert np.array_equal(nparts, [-(-x // P) for x in ctxs])
        Pm = int(nparts.max())
        m, l, o = oracle.partition_pass(c["q"], c["kc"], c["vc"], c["tables"],
                                        c["ctx"], scale, oracle.F16, P, Pm, lib=lib)
        merged = oracle.partition_merge(m, l, o, nparts, lib=lib)
        _close(merged, full, 1e-12, 1e-13, f"merge P={P}")
        # partition j of sequence s against sdpa on that slice
        for s, x in enumerate(ctxs):
            for j in range(nparts[s]):
                lo, hi = j * P, min(x, (j + 1) * P)
                ks, vs = c["kl"][s][lo:hi], c["vl"][s][lo:hi]
                want = sdpa_reference(c["q"][s:s + 1], [ks], [vs], scale, f16_vals)[0]
                _close(o[s, :, j, :], want, 1e-11, 1e-12, f"partial P={P} s={s} j={j}")
                qd = f16_vals(c["q"][s])                              # [H, d]
                kd = f16_vals(ks).repeat(2, axis=1)                    # [n, H, d]
                sc = scale * np.einsum("hd,nhd->hn", qd, kd)
                lse = np.log(np.exp(sc - sc.max(axis=1, keepdims=True)).sum(axis=1)) \
                    + sc.max(axis=1)
                _close(m[s, :, j] + np.log(l[s, :, j]), lse, 1e-12, 1e-12, "lse")


def pin_large_scores_stable(lib):
    """Queries scaled x30 (scores of order 1e3) stay finite and match
    torch's float64 attention, unsplit and split."""
    rng = np.random.default_rng(41)
    c = random_paged_case(rng, [9, 40], 4, 2, 16, 4, spread=30.0)
    scale = 4.0
    # the case really reaches scores where exp() overflows without the
    # running-max shift
    top = max(np.abs(scale * np.einsum("hd,nhd->hn", f16_vals(c["q"][s]),
                                       f16_vals(c["kl"][s]).repeat(2, axis=1))).max()
              for s in range(2))
    assert top > 800.0, top
    got = oracle.paged_attention(c["q"], c["kc"], c["vc"], c["tables"], c["ctx"],
                                 scale, oracle.F16, lib=lib)
    assert np.isfinite(got).all()
    want = sdpa_reference(c["q"], c["kl"], c["vl"], scale, f16_vals)
    _close(got, want, 1e-9, 1e-10, "stable")
    m, l, o = oracle.partition_pass(c["q"], c["kc"], c["vc"], c["tables"], c["ctx"],
                                    scale, oracle.F16, 8, 5, lib=lib)
    merged = oracle.partition_merge(m, l, o, [2, 5], lib=lib)
    assert np.isfinite(merged).all()
    _close(merged, want, 1e-9, 1e-10, "stable split")


def pin_empty_context(lib):
    """A sequence with no context gives an all-zero output row and no
    partitions."""
    rng = np.random.default_rng(43)
    c = random_paged_case(rng, [5, 3], 2, 2, 8, 4)
    ctx = np.array([0, 3], dtype=np.int32)
    o = oracle.paged_attention(c["q"], c["kc"], c["vc"], c["tables"], ctx, 0.5,
                               oracle.F16, lib=lib)
    assert np.array_equal(o[0], np.zeros_like(o[0]))
    assert oracle.num_partitions(0, 16, lib=lib) == 0


# ---------------------------------------------------------------------------
# FP8 (e4m3) KV cache

def _torch_e4m3(x_f32: np.ndarray) -> np.ndarray:
    """torch's float32 -> float8_e4m3fn codes (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def _e4m3_values() -> np.ndarray:
    c = np.arange(256, dtype=np.uint8)
    return torch.from_numpy(c).view(torch.float8_e4m3fn).double().numpy()


def pin_e4m3_decode_exact(lib):
    """Every e4m3 code decodes to torch's float8_e4m3fn value (NaN for
    S.1111.111)."""
    got = oracle.decode_e4m3(np.arange(256, dtype=np.uint8), lib=lib)
    want = _e4m3_values()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def pin_e4m3_encode_matches_torch(lib):
    """Every finite fp16 value below 448 in magnitude (plenty of exact ties)
    encodes to torch's round-to-nearest-even code; larger ones saturate to
    +-448; NaN stays NaN."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16).astype(np.float32)
    got = oracle.quantize_e4m3(bits, oracle.F16, 1.0, lib=lib)
    fin = np.isfinite(vals)
    small = fin & (np.abs(vals) < 448)
    assert np.array_equal(got[small], _torch_e4m3(vals[small]))
    big = fin & (np.abs(vals) >= 448)
    assert np.array_equal(got[big], np.where(vals[big] > 0, 0x7E, 0xFE).astype(np.uint8))
    assert (got[np.isnan(vals)] & 0x7F == 0x7F).all()


def pin_e4m3_encode_nearest_brute_force(lib):
    """Encoding picks the nearest representable value (ties to the even
    code), checked against an exhaustive nearest search, including the
    fp32 product with a non-trivial inverse scale."""
    rng = np.random.default_rng(47)
    x = f16_bits(np.concatenate([rng.standard_normal(3000) * 50,
                                 rng.standard_normal(1000) * 0.01]))
    inv = np.float32(1.0) / np.float32(0.37)
    got = oracle.quantize_e4m3(x, oracle.F16, float(inv), lib=lib)
    v = (f16_vals(x).astype(np.float32) * inv).astype(np.float64)
    table = _e4m3_values()
    codes = np.arange(127)                       # non-negative finite codes
    mags = table[codes]
    want = []
    for a in v:
        m = min(abs(a), 448.0)
        err = np.abs(mags - m)
        best = np.flatnonzero(err == err.min())
        c = int(best[0]) if len(best) == 1 else int(best[best % 2 == 0][0])
        want.append(c | (0x80 if (a < 0 or (a == 0 and np.signbit(a))) else 0))
    assert np.array_equal(got, np.asarray(want, dtype=np.uint8))


def pin_fp8_reshape_and_cache(lib):
    """FP8 cache write: gathering whole blocks in table order gives back the
    codes torch makes from float(x) * (1/scale) in fp32."""
    rng = np.random.default_rng(53)
    bs, Hkv, d, N = 4, 2, 8, 9
    ctx = 11
    table = np.array([[6, 1, 4]], dtype=np.int32)
    key = bf16_bits(rng.standard_normal((ctx, Hkv, d)) * 3)
    val = bf16_bits(rng.standard_normal((ctx, Hkv, d)) * 3)
    ks, vs = 0.02, 0.015
    kc = np.zeros((N, bs, Hkv, d), np.uint8)
    vc = np.zeros((N, bs, Hkv, d), np.uint8)
    slots = oracle.slot_mapping(table, np.zeros(ctx, np.int32), np.arange(ctx, dtype=np.int32),
                                bs, lib=lib)
    oracle.reshape_and_cache_fp8(key, val, kc, vc, slots, oracle.BF16, ks, vs, lib=lib)
    dec = _dec("bf16")
    for pool, src, sc in ((kc, key, ks), (vc, val, vs)):
        gathered = np.concatenate([pool[b] for b in table[0]])[:ctx]
        inv = np.float32(1.0) / np.float32(sc)
        want = _torch_e4m3(np.clip(dec(src).astype(np.float32) * inv, -448, 448))
        assert np.array_equal(gathered, want)


def pin_fp8_attention_matches_sdpa(lib):
    """Attention over FP8 pools equals torch's float64 attention on the
    dequantised K and V (codes from torch's conversion)."""
    rng = np.random.default_rng(59)
    H, Hkv, d, bs = 4, 2, 16, 4
    ctxs = [1, 6, 13]
    ks, vs = 0.011, 0.013
    perm = rng.permutation(12)
    tables = np.array([perm[0:4], perm[4:8], perm[8:12]], dtype=np.int32)
    kl = [_torch_e4m3(rng.standard_normal((c, Hkv, d)).astype(np.float32) * 60) for c in ctxs]
    vl = [_torch_e4m3(rng.standard_normal((c, Hkv, d)).astype(np.float32) * 60) for c in ctxs]
    q = bf16_bits(rng.standard_normal((3, H, d)))
    kc = place_sequences(kl, tables, 12, bs, fill=np.uint8(0x7F)).astype(np.uint8)
    vc = place_sequences(vl, tables, 12, bs, fill=np.uint8(0x7F)).astype(np.uint8)
    got = oracle.paged_attention_fp8(q, kc, vc, tables, ctxs, 0.25, oracle.BF16, ks, vs,
                                     lib=lib)
    table = _e4m3_values()
    want = np.zeros_like(got)
    for i in range(3):
        kd = torch.from_numpy(table[kl[i]] * float(np.float32(ks)))
        vd = torch.from_numpy(table[vl[i]] * float(np.float32(vs)))
        kd = kd.permute(1, 0, 2).repeat_interleave(H // Hkv, 0)
        vd = vd.permute(1, 0, 2).repeat_interleave(H // Hkv, 0)
        qd = torch.from_numpy(_dec("bf16")(q[i]))[:, None, :]
        want[i] = torch.nn.functional.scaled_dot_product_attention(
            qd[None], kd[None], vd[None], scale=0.25)[0, :, 0, :].numpy()
    _close(got, want, 1e-11, 1e-12, "fp8 sdpa")


def _prefill_case(rng, ctxs, q_lens, H, Hkv, d, bs, dtype="f16"):
    """A mixed batch: sequence s has its newest q_lens[s] tokens as query
    rows (stacked into [T, H, d]) and all ctxs[s] tokens in the pool."""
    c = random_paged_case(rng, ctxs, H, Hkv, d, bs, dtype=dtype)
    conv = f16_bits if dtype == "f16" else bf16_bits
    qs = np.zeros(len(ctxs) + 1, dtype=np.int32)
    qs[1:] = np.cumsum(q_lens)
    c["qrows"] = conv(rng.standard_normal((int(qs[-1]), H, d)))
    c["qs"] = qs
    return c


def _causal_sdpa(c, scale, dec):
    """torch float64 SDPA per sequence with an explicit mask: chunk row i
    (position ctx - q_len + i) may see key positions <= its own."""
    T, H, d = c["qrows"].shape
    out = np.zeros((T, H, d))
    for s, ctx in enumerate(c["ctx"]):
        q0, q1 = int(c["qs"][s]), int(c["qs"][s + 1])
        n = q1 - q0
        if n == 0:
            continue
        k = torch.from_numpy(dec(c["kl"][s]))
        v = torch.from_numpy(dec(c["vl"][s]))
        g = H // k.shape[1]
        k = k.permute(1, 0, 2).repeat_interleave(g, dim=0)   # [H, ctx, d]
        v = v.permute(1, 0, 2).repeat_interleave(g, dim=0)
        q = torch.from_numpy(dec(c["qrows"][q0:q1])).permute(1, 0, 2)  # [H, n, d]
        pos = int(ctx) - n + torch.arange(n)[:, None]
        mask = torch.arange(int(ctx))[None, :] <= pos          # [n, ctx]
        o = torch.nn.functional.scaled_dot_product_attention(
            q[None], k[None], v[None], attn_mask=mask[None, None], scale=scale)[0]
        out[q0:q1] = o.permute(1, 0, 2).numpy()
    return out


def pin_prefill_matches_causal_sdpa(lib):
    """Chunked prefill (GAO §2.4, §2.5): each chunk row attends the cached
    tokens up to its own position -- torch float64 SDPA with a boolean mask
    on the gathered K/V; a mixed batch with decode rows (q_len 1), whole
    prompts (q_len = ctx), chunks in mid-context and an empty chunk."""
    rng = np.random.default_rng(31)
    for dtype, (H, Hkv, d, bs) in (("f16", (4, 2, 16, 4)), ("bf16", (6, 3, 8, 8)),
                                   ("f16", (2, 2, 32, 16))):
        ctxs, q_lens = [7, 5, 20, 41, 9, 3], [1, 5, 3, 16, 0, 3]
        c = _prefill_case(rng, ctxs, q_lens, H, Hkv, d, bs, dtype)
        scale = 1.0 / math.sqrt(d)
        dt = oracle.F16 if dtype == "f16" else oracle.BF16
        got = oracle.prefill_attention(c["qrows"], c["kc"], c["vc"], c["tables"], c["qs"],
                                       c["ctx"], scale, dt, lib=lib)
        want = _causal_sdpa(c, scale, _dec(dtype))
        _close(got, want, 1e-11, 1e-12, f"causal sdpa {dtype} {H}/{Hkv}")


def pin_fp8_prefill_matches_causal_sdpa(lib):
    """Chunked prefill over FP8 pools (the FP8 KV cache of "vLLM 架构详解"'s
    deployment options, read by GAO §2.4/§2.5's chunk rows): torch float64
    SDPA with the causal mask on the dequantised gathered codes (torch's e4m3
    values times each pool's scale); a mixed batch with decode rows, whole
    prompts, mid-context chunks and an empty chunk."""
    rng = np.random.default_rng(61)
    table = _e4m3_values()
    ks, vs = 0.011, 0.013
    for dtype, (H, Hkv, d, bs) in (("bf16", (4, 2, 16, 4)), ("f16", (6, 3, 8, 8))):
        ctxs, q_lens = [7, 5, 20, 33, 9], [1, 5, 3, 16, 0]
        c = _prefill_case(rng, ctxs, q_lens, H, Hkv, d, bs, dtype)
        kl = [_torch_e4m3(rng.standard_normal((n, Hkv, d)).astype(np.float32) * 60)
              for n in ctxs]
        vl = [_torch_e4m3(rng.standard_normal((n, Hkv, d)).astype(np.float32) * 60)
              for n in ctxs]
        kc = place_sequences(kl, c["tables"], c["N"], bs, fill=np.uint8(0x7F)).astype(np.uint8)
        vc = place_sequences(vl, c["tables"], c["N"], bs, fill=np.uint8(0x7F)).astype(np.uint8)
        scale = 1.0 / math.sqrt(d)
        dt = oracle.F16 if dtype == "f16" else oracle.BF16
        got = oracle.prefill_attention_fp8(c["qrows"], kc, vc, c["tables"], c["qs"], c["ctx"],
                                           scale, dt, ks, vs, lib=lib)
        # the same rows through the mask-based reference, K/V dequantised
        c2 = dict(c, kl=[table[k] * float(np.float32(ks)) for k in kl],
                  vl=[table[v] * float(np.float32(vs)) for v in vl])
        want = _causal_sdpa(c2, scale, lambda x, dd=_dec(dtype): (
            x if x.dtype == np.float64 else dd(x)))
        _close(got, want, 1e-11, 1e-12, f"fp8 causal sdpa {dtype} {H}/{Hkv}")


def pin_prefill_causal_closed_forms(lib):
    """A whole prompt as one chunk: its first row sees only token 0, so its
    output is v_0 exactly; poisoning (NaN) the K/V of the last token leaves
    every earlier row finite and unchanged and makes only the last row NaN."""
    rng = np.random.default_rng(37)
    H, Hkv, d, bs, ctx = 4, 2, 16, 4, 11
    c = _prefill_case(rng, [ctx], [ctx], H, Hkv, d, bs)
    scale = 0.3
    args = (c["tables"], c["qs"], c["ctx"], scale, oracle.F16)
    o = oracle.prefill_attention(c["qrows"], c["kc"], c["vc"], *args, lib=lib)
    for h in range(H):
        assert np.array_equal(o[0, h], f16_vals(c["vl"][0][0, h // (H // Hkv)])), "row 0"
    last_blk, last_off = c["tables"][0][(ctx - 1) // bs], (ctx - 1) % bs
    kc, vc = c["kc"].copy(), c["vc"].copy()
    kc[last_blk, last_off] = np.uint16(0x7E00)
    vc[last_blk, last_off] = np.uint16(0x7E00)
    o2 = oracle.prefill_attention(c["qrows"], kc, vc, *args, lib=lib)
    assert np.array_equal(o2[:-1], o[:-1]), "earlier rows changed by a later token"
    assert np.isnan(o2[-1]).all(), "the last row must see its own token"


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]

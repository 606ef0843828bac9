"""GPU path against the CPU oracle on the reduced workloads (all sequences,
every element): slots, pools and copy-on-write bit-exact; attention within
the contract tolerance; plus the invariants the pages imply."""
import json
import math
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from paged_kv_cache_96_gb300 import workloads as W  # noqa: E402
from stepping import OracleStep, assert_attention_close, odt  # noqa: E402

NAMES = ["tiny", "mha7b", "gqa70b", "longctx", "prefix",
         "mha7b-fp8", "gqa70b-fp8", "longctx-fp8", "prefix-fp8"]


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_96_gb300 import binding
    return binding


@pytest.fixture(scope="module")
def S():
    from paged_kv_cache_96_gb300 import step
    return step


def _cases():
    out = []
    for n in NAMES:
        spec = W.small_variant(n)
        parts = sorted({0, spec.partition_size, 16, 48})
        for P in parts:
            out.append((n, P))
    return out


@pytest.fixture(scope="module")
def small():
    cache = {}

    def get(name):
        if name not in cache:
            w = W.build(W.small_variant(name))
            cache[name] = (w, OracleStep(w))
        return cache[name]
    return get


def test_worked_slot_example_gpu(B):
    with open(os.path.join(os.path.dirname(__file__), "golden",
                           "slot_worked_example.json")) as f:
        g = json.load(f)
    dev = "cuda"
    table = torch.tensor([g["block_table"]], dtype=torch.int32, device=dev)
    seq = torch.zeros(1, dtype=torch.int32, device=dev)
    pos = torch.tensor([g["position"]], dtype=torch.int32, device=dev)
    slots = torch.empty(1, dtype=torch.int32, device=dev)
    B.pa_slot_mapping(slots, table, seq, pos, g["block_size"], 16)
    assert int(slots.item()) == g["slot"]


@pytest.mark.parametrize("name,P", _cases(), ids=lambda x: str(x))
def test_step_matches_oracle(B, S, small, name, P):
    w, ref = small(name)
    st = S.DecodeStep(w, partition_size=P)
    out = st.run()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    # slots of the step's new tokens: exact
    assert np.array_equal(st.slots.cpu().numpy().astype(np.int64), ref.new_slots)
    # pools after history writes, the step's writes and copy-on-write: exact,
    # every byte including the untouched NaN fill
    assert np.array_equal(S.to_bits(st.key_cache), ref.key_cache)
    assert np.array_equal(S.to_bits(st.value_cache), ref.value_cache)
    # attention: every sequence, head and element
    want = ref.attention()
    got = S.to_float(out)
    assert_attention_close(got, want, f"{name} P={P}")


@pytest.mark.parametrize("name", ["gqa70b", "longctx", "mha7b", "prefix"])
def test_partition_partials_match_oracle(B, S, small, name):
    """The split-context pass's partials (m, l, o) in the workspace, for the
    sequences that span more than one partition."""
    w, ref = small(name)
    P = w.spec.partition_size
    st = S.DecodeStep(w, partition_size=P)
    st.run()
    torch.cuda.synchronize()
    Pm = math.ceil(int(w.context_lens.max()) / P)
    m_o, l_o, o_o = ref.partitions(P, Pm)
    ws = st.workspace
    assert ws is not None
    S_, H, D = w.S, w.H, w.D

    def region(off, count):
        return ws[off:off + 4 * count].view(torch.float32).cpu().numpy().astype(np.float64)

    def a256(x):
        return (x + 255) // 256 * 256
    # the arrival counters come first (and are back at zero after the call)
    n_cnt = max(1 << 18, S_ * w.Hkv)
    assert int(ws[:4 * n_cnt].view(torch.int32).abs().sum().item()) == 0
    base = a256(4 * n_cnt)
    n_ml = S_ * H * Pm
    m_g = region(base, n_ml).reshape(S_, H, Pm)
    l_g = region(base + a256(4 * n_ml), n_ml).reshape(S_, H, Pm)
    o_g = region(base + 2 * a256(4 * n_ml), n_ml * D).reshape(S_, H, Pm, D)
    multi = [s for s in range(S_) if oracle.num_partitions(int(w.context_lens[s]), P) > 1]
    assert multi, "reduced workload should have multi-partition sequences"
    for s in multi:
        n = oracle.num_partitions(int(w.context_lens[s]), P)
        lse_g = m_g[s, :, :n] + np.log(l_g[s, :, :n])
        lse_o = m_o[s, :, :n] + np.log(l_o[s, :, :n])
        assert np.allclose(lse_g, lse_o, atol=1e-3, rtol=1e-4), s
        assert_attention_close(o_g[s, :, :n], o_o[s, :, :n], f"partials s={s}")


def test_single_token_context_is_value_row(B, S, small):
    """Context 1: the output is that token's value row, bit for bit."""
    w, _ = small("tiny")
    st = S.DecodeStep(w)
    out = st.run()
    s = int(np.where(w.context_lens == 1)[0][0])
    G = w.H // w.Hkv
    got = S.to_bits(out)[s]
    for h in range(w.H):
        assert np.array_equal(got[h], w.new_value[s, h // G])


def _attend(B, st, tables, P, kc=None, vc=None, ctx=None):
    w = st.w
    ws = B.alloc_workspace(w.S, w.H, w.Hkv, w.D, st.max_context_len, P)
    out = torch.full_like(st.out, float("nan"))
    B.pa_decode_attention(out, st.query, st.key_cache if kc is None else kc,
                          st.value_cache if vc is None else vc, tables,
                          st.context_lens if ctx is None else ctx, st.max_context_len,
                          w.scale, P, ws)
    return out


def test_block_placement_invariance_gpu(B, S, small):
    """Moving physical blocks around the pool (and renaming them in the
    tables) leaves the output bit-identical."""
    w, _ = small("gqa70b")
    st = S.DecodeStep(w)
    st.run()
    g = torch.Generator().manual_seed(3)
    perm = torch.randperm(w.num_blocks, generator=g).to("cuda")  # block b -> perm[b]
    kc2 = torch.empty_like(st.key_cache)
    vc2 = torch.empty_like(st.value_cache)
    kc2[perm] = st.key_cache
    vc2[perm] = st.value_cache
    t2 = perm[st.step_block_tables.long()].to(torch.int32)
    for P in (0, w.spec.partition_size, 32):
        a = _attend(B, st, st.step_block_tables, P)
        b = _attend(B, st, t2, P, kc2, vc2)
        assert torch.equal(a, b), P


def test_shared_prefix_equals_private_copies(B, S, small):
    """Sequences naming the same prefix blocks give the same output as
    sequences holding private copies of those blocks."""
    w, _ = small("prefix")
    st = S.DecodeStep(w)
    st.run()
    pre = w.spec.shared_prefix_tokens // w.bs
    N = w.num_blocks
    kc = torch.cat([st.key_cache, torch.empty((w.S * pre,) + tuple(st.key_cache.shape[1:]),
                                              dtype=st.key_cache.dtype, device="cuda")])
    vc = torch.cat([st.value_cache, torch.empty_like(kc[N:])])
    tables = st.step_block_tables.clone()
    nxt = N
    for s in range(w.S):
        for b in range(pre):
            src = int(tables[s, b])
            kc[nxt] = kc[src]
            vc[nxt] = vc[src]
            tables[s, b] = nxt
            nxt += 1
    for P in (0, w.spec.partition_size):
        a = _attend(B, st, st.step_block_tables, P)
        b = _attend(B, st, tables, P, kc, vc)
        assert torch.equal(a, b), P


def test_split_agrees_with_single_pass(B, S, small):
    w, _ = small("longctx")
    st = S.DecodeStep(w)
    st.run()
    outs = []
    for P in (0, 16, 32, 256, 1024):
        st.attention(partition_size=P)
        outs.append(S.to_float(st.out))
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() < 2e-2


def test_repeated_calls_are_identical(B, S, small):
    """Re-running the step (same writes, same copies, same attention) gives
    bit-identical output, single pass and split."""
    w, _ = small("longctx")
    st = S.DecodeStep(w)
    st.run()
    for P in (0, w.spec.partition_size):
        st.attention(partition_size=P)
        a = st.out.clone()
        for _ in range(3):
            st.run()
            st.attention(partition_size=P)
            assert torch.equal(a, st.out), P


def test_empty_context_gives_zero_row(B, S, small):
    w, _ = small("gqa70b")
    st = S.DecodeStep(w)
    st.run()
    ctx = st.context_lens.clone()
    ctx[1] = 0
    ctx[4] = 0
    for P in (0, w.spec.partition_size):
        ws = B.alloc_workspace(w.S, w.H, w.Hkv, w.D, st.max_context_len, P)
        out = torch.full_like(st.out, float("nan"))
        B.pa_decode_attention(out, st.query, st.key_cache, st.value_cache,
                              st.step_block_tables, ctx, st.max_context_len, w.scale,
                              P, ws)
        o = S.to_float(out)
        assert (o[1] == 0).all() and (o[4] == 0).all()
        assert np.isfinite(o).all()


def test_large_scores_stay_finite(B, S, small):
    """Queries x30: scores far from zero, a peaky softmax."""
    import dataclasses
    w, _ = small("gqa70b")
    rng = np.random.default_rng(5)
    qx = W._round_to(rng.standard_normal(w.query.shape).astype(np.float32) * 30, w.dtype)
    w2 = dataclasses.replace(w, query=qx)
    ref = OracleStep(w2).attention()
    st = S.DecodeStep(w2)
    st.run()
    for P in (0, w.spec.partition_size):
        got = S.to_float(_attend(B, st, st.step_block_tables, P))
        assert_attention_close(got, ref, f"x30 P={P}")


def test_device_index_errors_are_flagged_not_faulted(B, S, small):
    w, _ = small("gqa70b")
    st = S.DecodeStep(w)
    st.run()
    torch.cuda.synchronize()
    # a block-table entry outside the pool
    tables = st.step_block_tables.clone()
    tables[2, 0] = w.num_blocks + 5
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.pa_decode_attention(st.out, st.query, st.key_cache, st.value_cache, tables,
                          st.context_lens, st.max_context_len, w.scale,
                          w.spec.partition_size, st.workspace, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & B.DEVERR_BLOCK_RANGE
    # a context longer than max_context_len
    err.zero_()
    ctx = st.context_lens.clone()
    ctx[0] = st.max_context_len + 100
    B.pa_decode_attention(st.out, st.query, st.key_cache, st.value_cache,
                          st.step_block_tables, ctx, st.max_context_len, w.scale,
                          w.spec.partition_size, st.workspace, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & B.DEVERR_CONTEXT_RANGE
    # a slot outside the pool, a negative slot (skipped silently)
    err.zero_()
    before = st.key_cache.clone()
    slots = torch.tensor([-1, w.num_blocks * w.bs + 3], dtype=torch.int32, device="cuda")
    B.pa_reshape_and_cache(st.new_key[:2], st.new_value[:2], st.key_cache, st.value_cache,
                           slots, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == B.DEVERR_SLOT_RANGE
    assert torch.equal(before.view(torch.int16), st.key_cache.view(torch.int16))
    # a copy pair outside the pool
    err.zero_()
    pairs = torch.tensor([[0, w.num_blocks]], dtype=torch.int32, device="cuda")
    B.pa_copy_blocks(st.key_cache, st.value_cache, pairs, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == B.DEVERR_PAIR_RANGE
    # a token whose position is past its table
    err.zero_()
    out = torch.empty(1, dtype=torch.int32, device="cuda")
    B.pa_slot_mapping(out, st.block_tables,
                      torch.zeros(1, dtype=torch.int32, device="cuda"),
                      torch.tensor([w.max_blocks_per_seq * w.bs], dtype=torch.int32,
                                   device="cuda"), w.bs, w.num_blocks, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == B.DEVERR_TOKEN_RANGE and int(out.item()) == -1
    assert torch.cuda.is_available()  # the context is still usable


def test_host_argument_errors(B, S, small):
    w, _ = small("gqa70b")
    st = S.DecodeStep(w)
    with pytest.raises(B.PAError) as e:
        B.pa_decode_attention(st.out, st.query, st.key_cache, st.value_cache,
                              st.step_block_tables, st.context_lens, st.max_context_len,
                              w.scale, w.spec.partition_size, None)
    assert e.value.status == B.PA_ERR_WORKSPACE
    with pytest.raises(B.PAError) as e:
        B.pa_decode_attention(st.out, st.query, st.key_cache, st.value_cache,
                              st.step_block_tables, st.context_lens, st.max_context_len,
                              w.scale, 24, None)
    assert e.value.status == B.PA_ERR_UNSUPPORTED


def test_fp8_query_beyond_fp16_range_is_flagged(B, S, small):
    """FP8 pools take the query in fp16 for the tensor-core products: a bf16
    query element past the fp16 range is flagged on the device (and a query
    inside it is not)."""
    w, _ = small("gqa70b-fp8")
    st = S.DecodeStep(w, partition_size=w.spec.partition_size)
    st.run()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    assert st.query.dtype == torch.bfloat16
    st.query[1, 3, 17] = 1.0e5   # bf16 holds it, fp16 does not
    st.attention()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) & B.DEVERR_QUERY_RANGE



@pytest.mark.parametrize("P", [128, 0])
def test_fp8_query_heads_far_apart_in_magnitude(B, S, small, P):
    """FP8 pools with bf16 queries, every head's row scaled by its own power
    of two from 2^-30 to 2^12 (rows below the fp16 range vanish in fp16, as
    their scores do in the oracle's softmax), and one row whose elements
    span 2^-14 .. 2^0 of its largest: the decode matches the oracle."""
    w, ref = small("gqa70b-fp8")
    st = S.DecodeStep(w, partition_size=w.spec.partition_size)
    st.run()
    torch.cuda.synchronize()
    rng = np.random.default_rng(96)
    ex = torch.tensor(rng.integers(-30, 13, size=(w.S, w.H)), dtype=torch.float32)
    q = (st.query.float() * torch.exp2(ex).to("cuda")[..., None]).to(torch.bfloat16)
    row = q[0, 5].float()
    spread = torch.exp2(-(torch.arange(w.D, device="cuda", dtype=torch.float32) % 15))
    q[0, 5] = (row * spread).to(torch.bfloat16)
    out = torch.full_like(st.out, float("nan"))
    ws = B.alloc_workspace(w.S, w.H, w.Hkv, w.D, st.max_context_len, P, device=st.device)
    B.pa_decode_attention_fp8(out, q, st.key_cache, st.value_cache, st.step_block_tables,
                              st.context_lens, st.max_context_len, w.scale, st.kv_scale,
                              st.kv_scale, P, ws, error_word=st.error_word)
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    qbits = q.view(torch.int16).cpu().numpy().view(np.uint16)
    want = oracle.paged_attention_fp8(qbits, ref.key_cache, ref.value_cache,
                                      w.step_block_tables, w.context_lens, w.scale, odt(w),
                                      w.spec.kv_scale, w.spec.kv_scale)
    assert_attention_close(S.to_float(out), want, f"fp8 heads 2^-30..2^12 P={P}")

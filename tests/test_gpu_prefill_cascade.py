"""Chunked prefill / mixed batches and prefix-aware (cascade) decode on the
GPU against the CPU oracle: slots and pools bit-exact; attention within the
contract tolerance on every row; invariants; plan and index errors flagged
on the device without a fault."""
import dataclasses

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from paged_kv_cache_96_gb300 import workloads as W  # noqa: E402
from stepping import OracleStep, assert_attention_close  # noqa: E402


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


@pytest.fixture(scope="module")
def small():
    cache = {}

    def get(name):
        if name not in cache:
            w = W.build(W.small_variant(name))
            cache[name] = (w, OracleStep(w))
        return cache[name]
    return get


# ---- chunked prefill / mixed batch ------------------------------------------------

@pytest.mark.parametrize("name", ["mixed", "chunked", "chunked-fp8", "mixed-fp8"])
def test_prefill_step_matches_oracle(B, S, small, name):
    w, ref = small(name)
    st = S.DecodeStep(w)
    out = st.run()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    assert np.array_equal(st.slots.cpu().numpy().astype(np.int64), ref.new_slots)
    assert np.array_equal(S.to_bits(st.key_cache), ref.key_cache)
    assert np.array_equal(S.to_bits(st.value_cache), ref.value_cache)
    assert_attention_close(S.to_float(out), ref.attention(), name)


def test_prefill_rows_subset_matches_whole(B, S, small):
    """The sampled-row oracle used at full size agrees with the whole-batch
    oracle (and so with the GPU) on the reduced workload."""
    w, ref = small("chunked")
    rows = [0, 1, 99, 100, 163, 164, 200, 292, 293]
    assert np.array_equal(ref.attention(rows=rows), ref.attention()[rows])


def test_prompt_first_row_is_value_row(B, S, small):
    """A prompt prefilled whole: its first row sees only token 0, so the
    output is that token's value row, bit for bit."""
    w, _ = small("mixed")
    st = S.DecodeStep(w)
    out = S.to_bits(st.run())
    G = w.H // w.Hkv
    whole = [s for s in range(w.S)
             if w.query_start[s + 1] - w.query_start[s] == w.context_lens[s]]
    assert whole
    for s in whole:
        r = int(w.query_start[s])
        for h in range(w.H):
            assert np.array_equal(out[r, h], w.new_value[r, h // G])


@pytest.mark.parametrize("name", ["chunked", "chunked-fp8"])
def test_prefill_block_placement_invariance(B, S, small, name):
    w, _ = small(name)
    st = S.DecodeStep(w)
    a = st.run().clone()
    g = torch.Generator().manual_seed(5)
    perm = torch.randperm(w.num_blocks, generator=g).to("cuda")
    kc2 = torch.empty_like(st.key_cache)
    vc2 = torch.empty_like(st.value_cache)
    kc2[perm] = st.key_cache
    vc2[perm] = st.value_cache
    t2 = perm[st.step_block_tables.long()].to(torch.int32)
    b = torch.full_like(a, float("nan"))
    B.pa_prefill_attention(b, st.query, kc2, vc2, t2, st.query_start, st.context_lens,
                           st.max_context_len, w.scale, k_scale=st.kv_scale,
                           v_scale=st.kv_scale)
    assert torch.equal(a, b)


def _many_segments(n, qmax, cmax, fp8, dtype="bf16"):
    """A prefill batch of n sequences (16 query heads over 2 KV heads, d 128)
    with unsorted and tied contexts, a fifth of them single-token rows, and
    two single-token rows past 64 key tiles (the deal's last sort bucket);
    more row-tile units than one round of CTAs takes."""
    rng = np.random.default_rng(9700 + n)
    q = rng.integers(1, qmax, size=n)
    q[::5] = 1
    ctx = q + rng.integers(0, cmax, size=n)
    q[3], ctx[3] = 1, 4500
    q[8], ctx[8] = 1, 4100
    spec = dataclasses.replace(W.CONFIGS["chunked"], name=f"chunked-{n}seg", seed=9700 + n,
                               num_seqs=n, num_heads=16, num_kv_heads=2, dtype=dtype,
                               context_lens=lambda r, c=ctx: c.copy(),
                               query_lens=lambda r, c, qq=q: qq.copy())
    return W.fp8_variant(spec) if fp8 else spec


@pytest.mark.parametrize("n,qmax,cmax,fp8,dtype", [(56, 160, 500, False, "bf16"),
                                                   (56, 160, 500, True, "bf16"),
                                                   (56, 160, 500, True, "f16"),
                                                   (520, 3, 100, False, "bf16")],
                         ids=["56seg", "56seg-fp8", "56seg-fp8-f16", "520seg"])
def test_prefill_many_segments(B, S, n, qmax, cmax, fp8, dtype):
    """Segments numbered longest context first and dealt boustrophedon over
    more than one round (56 sequences, 500 units), the query tiles by TMA
    (FP8 pools: bf16 tiles rounded to fp16 in place, fp16 tiles as they
    land); past 512 sequences the natural order and round-robin deal (520
    sequences, 1,040 units)."""
    w = W.build(_many_segments(n, qmax, cmax, fp8, dtype))
    ref = OracleStep(w)
    st = S.DecodeStep(w)
    out = st.run()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    assert_attention_close(S.to_float(out), ref.attention(), w.spec.name)


@pytest.mark.parametrize("name", ["chunked", "mixed"])
def test_prefill_output_alignment_paths(B, S, small, name):
    """The output goes out in 32-byte stores when it is 32-byte aligned and
    in 16-byte stores otherwise; the query tiles come by TMA from any
    16-byte aligned query (chunked: more units than one round of CTAs) or
    from the row warps' loads (mixed, one round): every combination gives
    the same bits, and a query off the 16-byte grid is refused on the host
    (nothing is launched)."""
    w, _ = small(name)
    st = S.DecodeStep(w)
    ref = st.run().clone()
    for q_shift, o_shift in [(8, 0), (0, 8), (8, 8)]:  # elements of 2 bytes
        qbuf = torch.empty(st.query.numel() + 16, dtype=st.query.dtype, device="cuda")
        obuf = torch.full((st.out.numel() + 16,), float("nan"), dtype=st.out.dtype, device="cuda")
        q = qbuf[q_shift:q_shift + st.query.numel()].view(st.query.shape)
        o = obuf[o_shift:o_shift + st.out.numel()].view(st.out.shape)
        q.copy_(st.query)
        B.pa_prefill_attention(o, q, st.key_cache, st.value_cache, st.step_block_tables,
                               st.query_start, st.context_lens, st.max_context_len, w.scale,
                               error_word=st.error_word)
        torch.cuda.synchronize()
        assert int(st.error_word.item()) == 0
        assert torch.equal(o, ref), (q_shift, o_shift)
    q = qbuf[4:4 + st.query.numel()].view(st.query.shape)
    with pytest.raises(B.PAError) as e:
        B.pa_prefill_attention(st.out, q, st.key_cache, st.value_cache, st.step_block_tables,
                               st.query_start, st.context_lens, st.max_context_len, w.scale)
    assert e.value.status == B.PA_ERR_INVALID_ARG


def test_prefill_group_not_dividing_row_tile(B, S):
    """12 query heads over 2 KV heads: a group of 6 does not divide the
    128-row tile, so the row warps write the query tiles (rows of a tile
    straddle tokens) -- against the oracle."""
    spec = dataclasses.replace(W.small_variant("chunked"), name="chunked-g6", num_heads=12,
                               num_kv_heads=2)
    w = W.build(spec)
    ref = OracleStep(w)
    st = S.DecodeStep(w)
    out = st.run()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    assert_attention_close(S.to_float(out), ref.attention(), "chunked, group 6")


@pytest.mark.parametrize("H,Hkv,counts,extra", [
    (4, 4, [1300] * 8, 300),
    (4, 2, [1250] * 8, 300),
    (32, 2, [160, 200, 240, 180, 220, 260, 150, 190], 400)], ids=["group1", "group2", "group16"])
def test_prefill_query_tiles_by_tma_groups(B, S, H, Hkv, counts, extra):
    """More units than one round of CTAs, so the query tiles arrive by TMA as
    boxes of 64 elements x G heads x 128 / G tokens: groups 1, 2 and 16
    (boxes of 128 tokens x 1 head down to 8 tokens x 16 heads), most chunks
    ending in a partial row tile, against the oracle on every row."""
    from stepping import attention_all
    rng = np.random.default_rng(9800 + H)
    q = np.array(counts)
    ctx = q + rng.integers(0, extra, size=len(q))
    spec = dataclasses.replace(W.small_variant("chunked"), name=f"chunked-g{H // Hkv}",
                               seed=9800 + H, num_seqs=len(q), num_heads=H, num_kv_heads=Hkv,
                               context_lens=lambda r, c=ctx: c.copy(),
                               query_lens=lambda r, c, qq=q: qq.copy())
    w = W.build(spec)
    st = S.DecodeStep(w)
    out = st.run()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    assert_attention_close(S.to_float(out), attention_all(OracleStep(w)), spec.name)


def test_prefill_fp8_query_by_tma_beyond_fp16_is_flagged(B, S):
    """FP8 pools, a multi-round batch: the bf16 query tiles arrive by TMA and
    the row warps round them to fp16 in place; a bf16 element past the fp16
    range is flagged there too (and a query inside it is not)."""
    w = W.build(_many_segments(56, 160, 500, True))
    st = S.DecodeStep(w)
    st.run()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    assert st.query.dtype == torch.bfloat16
    st.query[w.T - 3, 5, 17] = 1.0e5   # bf16 holds it, fp16 does not
    st.attention()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) & B.DEVERR_QUERY_RANGE


def test_prefill_fp8_query_beyond_fp16_is_flagged(B, S, small):
    """The FP8 prefill rounds the query to fp16 for the tensor-core tiles: a
    bf16 query element beyond the fp16 range is flagged, not silently
    saturated."""
    w, _ = small("chunked-fp8")
    st = S.DecodeStep(w)
    st.run()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    assert st.query.dtype == torch.bfloat16
    st.query[5, 3, 17] = 1.0e5
    st.attention()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) & B.DEVERR_QUERY_RANGE


def test_prefill_fp8_scales_enter_as_stated(B, S, small):
    """Doubling v_scale doubles every output (bit for bit: a power of two);
    doubling k_scale equals doubling the softmax scale."""
    w, _ = small("chunked-fp8")
    st = S.DecodeStep(w)
    st.run()
    torch.cuda.synchronize()
    args = (st.query, st.key_cache, st.value_cache, st.step_block_tables, st.query_start,
            st.context_lens, st.max_context_len)
    a = torch.empty_like(st.out)
    b = torch.empty_like(st.out)
    c = torch.empty_like(st.out)
    k, v = st.kv_scale, st.kv_scale
    B.pa_prefill_attention(a, *args, w.scale, k_scale=k, v_scale=v)
    B.pa_prefill_attention(b, *args, w.scale, k_scale=k, v_scale=2 * v)
    B.pa_prefill_attention(c, *args, 2 * w.scale, k_scale=k, v_scale=v)
    d = torch.empty_like(st.out)
    B.pa_prefill_attention(d, *args, w.scale, k_scale=2 * k, v_scale=v)
    torch.cuda.synchronize()
    assert torch.equal(b, 2 * a)
    assert torch.equal(c, d)


def test_prefill_index_errors_are_flagged(B, S, small):
    w, _ = small("chunked")
    st = S.DecodeStep(w)
    st.run()
    torch.cuda.synchronize()
    tables = st.step_block_tables.clone()
    tables[2, 1] = w.num_blocks + 7
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(st.out)
    B.pa_prefill_attention(out, st.query, st.key_cache, st.value_cache, tables,
                           st.query_start, st.context_lens, st.max_context_len, w.scale,
                           error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & B.DEVERR_BLOCK_RANGE
    ctx = st.context_lens.clone()
    ctx[0] = st.max_context_len + 50
    err.zero_()
    B.pa_prefill_attention(out, st.query, st.key_cache, st.value_cache,
                           st.step_block_tables, st.query_start, ctx, st.max_context_len,
                           w.scale, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & B.DEVERR_CONTEXT_RANGE


def test_prefill_host_errors(B, S, small):
    w, _ = small("chunked")
    st = S.DecodeStep(w, build_pools=False)
    with pytest.raises(ValueError):
        B.pa_prefill_attention(st.out, st.query, st.key_cache, st.value_cache,
                               st.step_block_tables, st.query_start[:-1], st.context_lens,
                               st.max_context_len, w.scale)
    lib = B.lib()
    r = lib.pa_prefill_attention(None, None, None, None, None, 1, None, None, 16, 1, 1, 8, 2,
                                 96, 16, 4, 1.0, 1, None, None)
    assert r == B.PA_ERR_UNSUPPORTED or r == B.PA_ERR_INVALID_ARG
    r = lib.pa_prefill_attention(None, None, None, None, None, 1, None, None, 16, 1, 1, 8, 3,
                                 128, 16, 4, 1.0, 1, None, None)
    assert r == B.PA_ERR_INVALID_ARG


# ---- prefix-aware (cascade) decode -------------------------------------------------

@pytest.mark.parametrize("name", ["prefix-cascade", "prefix-cascade-fp8"])
@pytest.mark.parametrize("P", [0, 48, 128])
def test_cascade_step_matches_oracle(B, S, small, P, name):
    w, ref = small(name)
    st = S.DecodeStep(w, partition_size=P)
    assert st.num_groups >= 1
    assert st.fused_append
    out = st.run()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    assert np.array_equal(st.slots.cpu().numpy().astype(np.int64), ref.new_slots)
    assert np.array_equal(S.to_bits(st.key_cache), ref.key_cache)
    assert np.array_equal(S.to_bits(st.value_cache), ref.value_cache)
    assert_attention_close(S.to_float(out), ref.attention(), f"{name} P={P}")


@pytest.mark.parametrize("name", ["prefix-cascade", "prefix-cascade-fp8"])
def test_cascade_separate_write_matches_oracle(B, S, small, name):
    """The step with its writes as their own launch and the prefix-aware
    decode without append: same pools, same attention."""
    w, ref = small(name)
    st = S.DecodeStep(w)
    st.slot_mapping_and_cache()
    st.copy_blocks()
    st.attention()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    assert np.array_equal(S.to_bits(st.key_cache), ref.key_cache)
    assert np.array_equal(S.to_bits(st.value_cache), ref.value_cache)
    assert_attention_close(S.to_float(st.out), ref.attention(), f"{name} separate")


@pytest.mark.parametrize("fp8", [False, True])
def test_cascade_head_dim_64(B, S, fp8):
    """Prefix-aware decode at head_dim 64 (16-bit and FP8 pools), fused append
    and separate write, against the oracle."""
    import dataclasses
    spec = W.small_variant("prefix-cascade-fp8" if fp8 else "prefix-cascade")
    spec = dataclasses.replace(spec, name=spec.name + "-d64", head_dim=64)
    w = W.build(spec)
    ref = OracleStep(w)
    for how in ("append", "separate"):
        st = S.DecodeStep(w)
        assert st.num_groups >= 1
        if how == "append":
            st.copy_blocks()
            st.append_attention()
        else:
            st.slot_mapping_and_cache()
            st.copy_blocks()
            st.attention()
        torch.cuda.synchronize()
        assert int(st.error_word.item()) == 0
        assert np.array_equal(S.to_bits(st.key_cache), ref.key_cache)
        assert_attention_close(S.to_float(st.out), ref.attention(), f"d64 fp8={fp8} {how}")


def test_cascade_fp8_query_beyond_fp16_is_flagged(B, S, small):
    w, _ = small("prefix-cascade-fp8")
    st = S.DecodeStep(w)
    st.run()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    members = st.plan.cpu().numpy()[w.S + 2 * st.num_groups + 1:]
    st.query[int(members[0]), 1, 5] = 1.0e5
    st.slot_mapping_and_cache()
    st.attention()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) & B.DEVERR_QUERY_RANGE


@pytest.mark.parametrize("P", [0, 64])
def test_cascade_prefix_partial_matches_oracle(B, S, small, P):
    """The first partials of every grouped (sequence, head) are the attention
    over the group's shared prefix [0, L), in partitions of P tokens (P = 0:
    one): the oracle's partitions of that size over a context of L tokens."""
    w, ref = small("prefix-cascade")
    st = S.DecodeStep(w, partition_size=P)
    st.run()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    plan = st.plan.cpu().numpy()
    Sn, H, D = w.S, w.H, w.D
    ng = st.num_groups
    gstart = plan[Sn:Sn + ng + 1]
    gprefix = plan[Sn + ng + 1:Sn + 2 * ng + 1]
    members = plan[Sn + 2 * ng + 1:]
    mc = st.max_context_len
    split = P > 0 and mc > P
    Q = P if split else (mc + 15) // 16 * 16  # tokens per prefix partition
    parts = (-(-mc // P) if split else 1) + 1  # the workspace's partials per (sequence, head)
    ws = st.workspace
    assert ws.numel() == B.pa_cascade_workspace_bytes(Sn, H, w.Hkv, D, mc, P)

    def a256(x):
        return (x + 255) // 256 * 256
    n_ml = Sn * H * parts
    # the arrival counters come first (zero before and after the call)
    n_cnt = max(1 << 18, Sn * w.Hkv)
    assert int(ws[:4 * n_cnt].view(torch.int32).abs().sum().item()) == 0
    base = a256(4 * n_cnt)

    def region(off, count):
        return ws[off:off + 4 * count].view(torch.float32).cpu().numpy().astype(np.float64)
    m_g = region(base, n_ml).reshape(Sn, H, parts)
    l_g = region(base + a256(4 * n_ml), n_ml).reshape(Sn, H, parts)
    o_g = region(base + 2 * a256(4 * n_ml), n_ml * D).reshape(Sn, H, parts, D)
    for g in range(ng):
        L = int(gprefix[g])
        mem = members[gstart[g]:gstart[g + 1]].tolist()
        n = -(-L // Q)
        ctx_l = np.full(Sn, L, dtype=np.int32)
        m_o, l_o, o_o = oracle.partition_pass(w.query, ref.key_cache, ref.value_cache,
                                              w.step_block_tables, ctx_l, w.scale,
                                              oracle.BF16 if w.dtype == "bf16" else oracle.F16,
                                              Q, n, seqs=mem)
        for s in mem:
            for j in range(n):
                lse_g = m_g[s, :, j] + np.log(l_g[s, :, j])
                lse_o = m_o[s, :, j] + np.log(l_o[s, :, j])
                assert np.allclose(lse_g, lse_o, atol=1e-3, rtol=1e-4), (s, j)
                assert_attention_close(o_g[s, :, j], o_o[s, :, j], f"prefix partial s={s} j={j}")


def test_cascade_without_groups_is_plain_decode(B, S, small):
    w, _ = small("gqa70b")
    st = S.DecodeStep(w)
    st.run()
    plan, ng, nm = B.pa_plan_prefix_groups(w.step_block_tables, w.context_lens, w.bs)
    assert ng == 0
    P = w.spec.partition_size
    ws = torch.zeros(B.pa_cascade_workspace_bytes(w.S, w.H, w.Hkv, w.D, st.max_context_len, P),
                     dtype=torch.uint8, device="cuda")
    a = torch.empty_like(st.out)
    B.pa_decode_attention_cascade(a, st.query, st.key_cache, st.value_cache,
                                  st.step_block_tables, st.context_lens, st.max_context_len,
                                  w.scale, plan.cuda(), ng, nm, P, ws)
    st.attention()
    assert torch.equal(a, st.out)


def test_cascade_bad_plan_is_flagged(B, S, small):
    """A plan whose member records another prefix length, or whose member's
    table differs from the leader's on the prefix, sets the plan error bit;
    nothing faults."""
    w, _ = small("prefix-cascade")
    st = S.DecodeStep(w)
    st.run()
    torch.cuda.synchronize()
    Sn = w.S
    ng = st.num_groups
    plan = st.plan.clone()
    member = int(plan[Sn + 2 * ng + 1 + 1])
    plan[member] = plan[member] + w.bs  # seq_prefix_len disagrees with its group
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(st.out)
    B.pa_decode_attention_cascade(out, st.query, st.key_cache, st.value_cache,
                                  st.step_block_tables, st.context_lens, st.max_context_len,
                                  w.scale, plan, ng, st.num_members, 0, st.workspace,
                                  error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & B.DEVERR_PREFIX_PLAN
    tables = st.step_block_tables.clone()
    tables[member, 0] = (int(tables[member, 0]) + 1) % w.num_blocks
    err.zero_()
    B.pa_decode_attention_cascade(out, st.query, st.key_cache, st.value_cache, tables,
                                  st.context_lens, st.max_context_len, w.scale, st.plan, ng,
                                  st.num_members, 0, st.workspace, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & B.DEVERR_PREFIX_PLAN

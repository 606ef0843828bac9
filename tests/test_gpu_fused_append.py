"""pa_decode_attention_append (and its FP8 form) -- the decode step's slot
mapping and reshape_and_cache fused into the attention pass -- against the
calls it replaces (pa_slot_mapping_and_cache, copy-on-write, then
pa_decode_attention): the same slots and bit-identical pools, and outputs
that agree within the attention tolerance (the new token's term is summed
in another order), over the reduced workloads and several partition sizes
(the new token then falls on every row of a 16-token tile, alone in its
partition, and in the last partition of both single- and multi-partition
sequences).  The oracle comparison of the fused step itself is the step
parity test, whose run() takes this path.  Edge rows: a context of 0
(nothing appended, slot -1, a zero output row) and a new token whose block
is outside the pool (slot -1, nothing written, PA_DEVERR_BLOCK_RANGE); for
the prefix-aware form, a plan whose shared prefix reaches a new token
(PA_DEVERR_PREFIX_PLAN)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from paged_kv_cache_96_gb300 import workloads as W  # noqa: E402
from stepping import assert_attention_close  # noqa: E402

NAMES = ["tiny", "mha7b", "gqa70b", "longctx", "prefix", "prefix-cascade",
         "gqa70b-fp8", "longctx-fp8", "prefix-fp8"]


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
        for P in sorted({0, 16, 48, spec.partition_size}):
            out.append((n, P))
    return out


@pytest.mark.parametrize("name,P", _cases(), ids=lambda x: str(x))
def test_fused_append_matches_separate_calls(B, S, name, P):
    w = W.build(W.small_variant(name))
    a = S.DecodeStep(w, partition_size=P)
    b = S.DecodeStep(w, partition_size=P)
    assert b.fused_append
    a.slot_mapping_and_cache()
    a.copy_blocks()
    a.attention()
    b.slots.fill_(12345)
    b.out.fill_(float("nan"))
    out = b.run()
    torch.cuda.synchronize()
    assert int(a.error_word.item()) == 0 and int(b.error_word.item()) == 0
    assert torch.equal(a.slots, b.slots)
    assert np.array_equal(S.to_bits(a.key_cache), S.to_bits(b.key_cache))
    assert np.array_equal(S.to_bits(a.value_cache), S.to_bits(b.value_cache))
    assert_attention_close(S.to_float(out), S.to_float(a.out).astype(np.float64),
                           f"{name} P={P}")


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("P", [0, 16, 32])
def test_append_empty_context_and_bad_block(B, S, fp8, P):
    name = "gqa70b-fp8" if fp8 else "tiny"
    w = W.build(W.small_variant(name))
    a = S.DecodeStep(w, partition_size=P)
    b = S.DecodeStep(w, partition_size=P)
    dev = a.device
    ctx = w.context_lens.copy()
    zero = 0                    # this sequence's context becomes 0
    bad = w.S - 1               # this one's new token lands on a bad entry
    ctx[zero] = 0
    tables = w.step_block_tables.copy()
    tables[bad, (int(ctx[bad]) - 1) // w.bs] = w.num_blocks + 5
    ctx_t = torch.from_numpy(ctx.astype(np.int32)).to(dev)
    tab_t = torch.from_numpy(tables.astype(np.int32)).to(dev)
    keep = [s for s in range(w.S) if s not in (zero, bad)]

    # reference: the other sequences' tokens written by the separate call,
    # then attention with the same contexts and tables
    idx = torch.tensor(keep, dtype=torch.long, device=dev)
    slots_a = torch.empty(len(keep), dtype=torch.int32, device=dev)
    B.pa_slot_mapping_and_cache(slots_a, tab_t, a.new_seq[idx].contiguous(),
                                a.new_pos[idx].contiguous(), a.new_key[idx].contiguous(),
                                a.new_value[idx].contiguous(), a.key_cache, a.value_cache,
                                a.kv_scale, a.kv_scale, error_word=a.error_word)
    ws = B.alloc_workspace(w.S, w.H, w.Hkv, w.D, a.max_context_len, P, device=dev)
    if fp8:
        B.pa_decode_attention_fp8(a.out, a.query, a.key_cache, a.value_cache, tab_t, ctx_t,
                                  a.max_context_len, w.scale, a.kv_scale, a.kv_scale, P, ws,
                                  error_word=a.error_word)
    else:
        B.pa_decode_attention(a.out, a.query, a.key_cache, a.value_cache, tab_t, ctx_t,
                              a.max_context_len, w.scale, P, ws, error_word=a.error_word)

    slots_b = torch.full((w.S,), 777, dtype=torch.int32, device=dev)
    out_b = torch.full_like(b.out, float("nan"))
    ws_b = B.alloc_workspace(w.S, w.H, w.Hkv, w.D, b.max_context_len, P, device=dev)
    B.pa_decode_attention_append(out_b, b.query, b.key_cache, b.value_cache, b.new_key,
                                 b.new_value, tab_t, ctx_t, b.max_context_len, w.scale, P,
                                 ws_b, slot_mapping=slots_b, k_scale=b.kv_scale,
                                 v_scale=b.kv_scale, error_word=b.error_word)
    torch.cuda.synchronize()
    sb = slots_b.cpu().numpy()
    assert sb[zero] == -1 and sb[bad] == -1
    assert np.array_equal(sb[keep], slots_a.cpu().numpy())
    assert int(b.error_word.item()) & B.DEVERR_BLOCK_RANGE
    assert np.array_equal(S.to_bits(a.key_cache), S.to_bits(b.key_cache))
    assert np.array_equal(S.to_bits(a.value_cache), S.to_bits(b.value_cache))
    got, want = S.to_float(out_b), S.to_float(a.out).astype(np.float64)
    assert_attention_close(got[keep], want[keep], f"{name} P={P} kept rows")
    assert not got[zero].any()


def test_append_argument_checks(B, S):
    w = W.build(W.small_variant("tiny"))
    st = S.DecodeStep(w)
    with pytest.raises(ValueError):
        B.pa_decode_attention_append(st.out, st.query, st.key_cache, st.value_cache,
                                     st.new_key[:1], st.new_value, st.step_block_tables,
                                     st.context_lens, st.max_context_len, w.scale)
    with pytest.raises(B.PAError):
        B.pa_decode_attention_append(st.out, st.query, st.key_cache, st.value_cache,
                                     st.new_key, st.new_value, st.step_block_tables,
                                     st.context_lens, st.max_context_len, float("nan"))


def test_cascade_append_prefix_must_end_before_new_token(B, S):
    w = W.build(W.small_variant("prefix-cascade"))
    st = S.DecodeStep(w)
    assert st.cascade and st.fused_append and st.num_groups >= 1
    ng = st.num_groups
    plan = st.plan.cpu().numpy()
    member = int(plan[w.S + 2 * ng + 1 + 1])   # a group's second member
    ctx = st.context_lens.clone()
    ctx[member] = int(plan[member])            # its context now ends with the prefix
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.pa_decode_attention_cascade_append(st.out, st.query, st.key_cache, st.value_cache,
                                         st.new_key, st.new_value, st.step_block_tables, ctx,
                                         st.max_context_len, w.scale, st.plan, ng,
                                         st.num_members, st.partition_size, st.workspace,
                                         error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & B.DEVERR_PREFIX_PLAN

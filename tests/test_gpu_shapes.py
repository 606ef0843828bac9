"""Shapes the five workloads do not reach, against the oracle: query-head
groups that do not fill an 8-head tile (2, 3, 5, 12) and the 16-head tile
variant, head_dim 64 and 128 in both 16-bit types, block sizes 16 to 256,
several partition sizes, FP8 pools with wide and odd groups at head_dim 64
and 128 (fp16 and bf16 queries), chunked prefill
with the same groups and block sizes, and batches of thousands of sequences
(past 10,000 the decode pass falls back to one ring stage per warp to fit
the per-sequence arrays in shared memory).  Slots and pools bit-exact;
attention within the contract tolerance on every (or every sampled) row."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from paged_kv_cache_96_gb300 import workloads as W  # noqa: E402
from stepping import OracleStep, assert_attention_close  # noqa: E402


def _spec(name, S, H, Hkv, D, bs, dtype, ctx, P=0, kv="same", q_lens=None, seed=1):
    return W.WorkloadSpec(
        name=name, description=name, num_seqs=S, num_heads=H, num_kv_heads=Hkv,
        head_dim=D, block_size=bs, dtype=dtype, context_lens=ctx, partition_size=P,
        seed=seed, kv_dtype=kv, query_lens=q_lens)


def _uni(n, lo, hi):
    return lambda rng: rng.integers(lo, hi + 1, size=n)


DECODE = [
    # (name, S, H, Hkv, D, bs, dtype, partitions)
    ("g2_d64_bs64_f16", 5, 4, 2, 64, 64, "f16", (0, 64)),
    ("g3_d128_bs16_bf16", 5, 9, 3, 128, 16, "bf16", (0, 48)),
    ("g5_d64_bs32_bf16", 4, 10, 2, 64, 32, "bf16", (0, 96)),
    ("g12_d128_bs128_f16", 4, 24, 2, 128, 128, "f16", (0, 160)),
    ("g16_d128_bs16_bf16", 5, 32, 2, 128, 16, "bf16", (0, 32, 256)),
    ("g16_d64_bs256_f16", 4, 16, 1, 64, 256, "f16", (0, 512)),
]


@pytest.mark.parametrize("case", DECODE, ids=[c[0] for c in DECODE])
def test_decode_shapes(case):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_96_gb300 import step as St
    name, S, H, Hkv, D, bs, dt, parts = case
    w = W.build(_spec(name, S, H, Hkv, D, bs, dt, _uni(S, 1, 700)))
    ref = OracleStep(w)
    want = ref.attention()
    for P in parts:
        st = St.DecodeStep(w, partition_size=P)
        out = st.run()
        torch.cuda.synchronize()
        assert int(st.error_word.item()) == 0
        assert np.array_equal(St.to_bits(st.key_cache), ref.key_cache)
        assert np.array_equal(St.to_bits(st.value_cache), ref.value_cache)
        assert_attention_close(St.to_float(out), want, f"{name} P={P}")


FP8 = [
    # (name, S, H, Hkv, bs, partitions, head_dim, query dtype)
    ("fp8_g16_bs16", 4, 32, 2, 16, (0, 64), 128, "bf16"),
    ("fp8_g3_bs64", 5, 6, 2, 64, (0, 128), 128, "bf16"),
    ("fp8_g1_bs32", 4, 4, 4, 32, (0, 32), 128, "bf16"),
    ("fp8_d64_g8_bs16", 5, 16, 2, 16, (0, 64), 64, "bf16"),
    ("fp8_d64_g4_bs32_f16", 4, 8, 2, 32, (0, 96), 64, "f16"),
    ("fp8_d64_g16_bs16", 4, 16, 1, 16, (0, 48), 64, "bf16"),
    ("fp8_d64_g3_bs64", 5, 9, 3, 64, (0, 128), 64, "f16"),
]


@pytest.mark.parametrize("case", FP8, ids=[c[0] for c in FP8])
def test_fp8_decode_shapes(case):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_96_gb300 import step as St
    name, S, H, Hkv, bs, parts, D, dt = case
    w = W.build(_spec(name, S, H, Hkv, D, bs, dt, _uni(S, 1, 600), kv="fp8"))
    ref = OracleStep(w)
    want = ref.attention()
    for P in parts:
        st = St.DecodeStep(w, partition_size=P)
        out = st.run()
        torch.cuda.synchronize()
        assert int(st.error_word.item()) == 0
        assert np.array_equal(St.to_bits(st.key_cache), ref.key_cache)
        assert_attention_close(St.to_float(out), want, f"{name} P={P}")


PREFILL = [
    # (name, H, Hkv, D, bs, dtype, contexts, query rows)
    ("pf_g16_d64_bs64", 16, 1, 64, 64, "f16", [200, 65, 300], [200, 1, 37]),
    ("pf_g3_d128_bs256", 6, 2, 128, 256, "bf16", [300, 257], [140, 257]),
    ("pf_g12_d128_bs16", 24, 2, 128, 16, "bf16", [90, 33, 1], [90, 0, 1]),
]


@pytest.mark.parametrize("case", PREFILL, ids=[c[0] for c in PREFILL])
def test_prefill_shapes(case):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_96_gb300 import step as St
    name, H, Hkv, D, bs, dt, ctx, ql = case
    w = W.build(_spec(name, len(ctx), H, Hkv, D, bs, dt, lambda rng: np.asarray(ctx),
                      q_lens=lambda rng, c: np.asarray(ql)))
    ref = OracleStep(w)
    st = St.DecodeStep(w)
    out = st.run()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    assert np.array_equal(St.to_bits(st.key_cache), ref.key_cache)
    assert_attention_close(St.to_float(out), ref.attention(), name)


@pytest.mark.parametrize("S,P", [(3000, 0), (11000, 0), (11000, 16)])
def test_many_sequences(S, P):
    """Thousands of short sequences (past 10,000 the decode pass runs with one
    ring stage per warp); sampled sequences against the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_96_gb300 import step as St
    w = W.build(_spec(f"many{S}", S, 8, 2, 128, 16, "bf16", _uni(S, 1, 40)))
    st = St.DecodeStep(w, partition_size=P)
    out = st.run()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    ref = OracleStep(w)
    assert np.array_equal(St.to_bits(st.key_cache), ref.key_cache)
    rng = np.random.default_rng(3)
    seqs = sorted({0, S - 1} | {int(x) for x in rng.choice(S, size=40, replace=False)})
    want = ref.attention(seqs=seqs)
    assert_attention_close(St.to_float(out)[seqs], want[seqs], f"S={S} P={P}")


def test_many_prefill_segments():
    """A mixed batch of 2,500 decode rows and two prompt chunks (2,502
    sequences for the multi-query kernel's unit table)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_96_gb300 import step as St
    S = 2502
    ctx = np.concatenate([np.arange(1, 2501) % 37 + 1, [300, 129]])
    ql = np.concatenate([np.ones(2500, np.int64), [300, 64]])
    w = W.build(_spec("manyseg", S, 16, 2, 128, 16, "bf16", lambda rng: ctx,
                      q_lens=lambda rng, c: ql))
    st = St.DecodeStep(w)
    out = St.to_float(st.run())
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    ref = OracleStep(w)
    qs = w.query_start
    rows = sorted({0, 1, 2499, int(qs[2500]), int(qs[2501]) - 1, int(qs[2501]),
                   w.T - 1} | set(range(1000, 1010)))
    assert_attention_close(out[rows], ref.attention(rows=rows), "many segments")

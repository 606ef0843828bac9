"""The seeded workload generator (host logic, no GPU)."""
import numpy as np
import pytest

from paged_kv_cache_96_gb300 import workloads as W

NAMES = ["tiny", "mha7b", "gqa70b", "longctx", "prefix"]


@pytest.mark.parametrize("name", NAMES)
def test_small_variant_structure(name):
    w = W.build(W.small_variant(name))
    S, MB, bs = w.S, w.max_blocks_per_seq, w.bs
    nblk = -(-w.context_lens.astype(np.int64) // bs)
    pre = w.spec.shared_prefix_tokens // bs
    owned = []
    for s in range(S):
        row = w.block_tables[s]
        assert (row[nblk[s]:] == w.pad_block).all()
        owned.append(row[pre:nblk[s]])
    owned = np.concatenate(owned)
    # private blocks are distinct, never the shared or padding block
    assert len(set(owned.tolist())) == owned.shape[0]
    shared = set(w.block_tables[0, :pre].tolist())
    assert not shared & set(owned.tolist())
    assert w.pad_block not in set(owned.tolist()) | shared
    assert (w.block_tables >= 0).all() and (w.block_tables < w.num_blocks).all()
    # every sequence shares the same prefix blocks
    assert (w.block_tables[:, :pre] == w.block_tables[0, :pre]).all()
    # history + new tokens cover [0, ctx) of every sequence exactly once
    for s in range(S):
        pos = np.concatenate([w.hist_pos[w.hist_seq == s], w.new_pos[w.new_seq == s]])
        if pre and s != 0:
            pos = np.concatenate([np.arange(pre * bs), pos])
        assert np.array_equal(np.sort(pos), np.arange(w.context_lens[s]))
    # copy-on-write pairs: shared sources, free distinct destinations, remapped
    if w.spec.cow_pairs:
        src, dst = w.cow_pairs[:, 0], w.cow_pairs[:, 1]
        assert set(src.tolist()) <= shared
        assert len(set(dst.tolist())) == dst.shape[0]
        assert not set(dst.tolist()) & (set(owned.tolist()) | shared | {w.pad_block})
        diff = np.argwhere(w.step_block_tables != w.block_tables)
        assert diff.shape[0] == w.spec.cow_pairs
        for s, b in diff:
            i = int(np.where(dst == w.step_block_tables[s, b])[0][0])
            assert w.block_tables[s, b] == src[i]


def test_seeded_reproducible():
    a = W.build(W.small_variant("gqa70b"))
    b = W.build(W.small_variant("gqa70b"))
    for f in ("context_lens", "block_tables", "query", "hist_key", "new_value"):
        assert np.array_equal(getattr(a, f), getattr(b, f))


def test_full_config_lengths():
    """Context-length recipes of the five full workloads (no values drawn)."""
    rng = np.random.default_rng(9603)
    c = W.CONFIGS["gqa70b"].context_lens(rng)
    assert c.shape == (128,) and c.min() >= 16 and c.max() <= 8192
    c = W.CONFIGS["longctx"].context_lens(np.random.default_rng(1))
    assert sorted(c.tolist())[-4:] == [32768] * 4 and c.min() >= 64
    c = W.CONFIGS["prefix"].context_lens(np.random.default_rng(1))
    assert c.min() >= 1025 and c.max() <= 2048
    assert W.CONFIGS["tiny"].context_lens(None).tolist() == [1, 15, 16, 35]

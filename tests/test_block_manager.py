"""The library's C++ host block manager against the reference block manager
(oracle/block_manager.py), operation by operation: slots, copy-on-write pairs,
tables, token counts, reference counts, free blocks and refusals must be
identical.  Host code only: runs without a GPU."""
import numpy as np
import pytest

try:
    from paged_kv_cache_96_gb300 import binding as B
except ImportError as e:  # library not built
    pytest.skip(f"library missing: {e}", allow_module_level=True)

from oracle import block_manager as M


def _same_state(bm, ref, live):
    assert bm.num_free() == ref.num_free()
    assert [bm.ref(b) for b in range(ref.num_blocks)] == ref.ref
    for s in live:
        assert bm.table(s) == ref.table(s)
        assert bm.length(s) == ref.length(s)


@pytest.mark.parametrize("seed", range(12))
def test_random_sessions_match_reference(seed):
    rng = np.random.default_rng(1000 + seed)
    bs = int(rng.choice([1, 4, 16, 32]))
    N = int(rng.integers(8, 200))
    MB = int(rng.integers(2, 40))
    bm, ref = B.BlockManager(N, bs, MB), M.BlockManager(N, bs, MB)
    live, nxt = [], 0
    for _ in range(400):
        op = int(rng.integers(0, 6))
        if op == 0 or not live:
            bm.add_sequence(nxt)
            ref.add_sequence(nxt)
            live.append(nxt)
            nxt += int(rng.integers(1, 4))      # ids need not be dense
        elif op == 1:
            p = int(rng.choice(live))
            bm.fork(p, nxt)
            ref.fork(p, nxt)
            live.append(nxt)
            nxt += 1
        elif op in (2, 3):
            s = int(rng.choice(live))
            n = int(rng.integers(0, 3 * bs + 2))
            assert bm.blocks_needed(s, n) == ref.blocks_needed(s, n)
            try:
                want = ref.append_tokens(s, n)
                err = None
            except M.OutOfBlocks:
                err = B.PA_ERR_OUT_OF_BLOCKS
            except M.TableFull:
                err = B.PA_ERR_TABLE_FULL
            if err is None:
                slots, pairs = bm.append_tokens(s, n)
                assert slots.tolist() == want[0] and pairs == want[1]
            else:
                with pytest.raises(B.PAError) as ex:
                    bm.append_tokens(s, n)
                assert ex.value.status == err
        elif op == 4:
            # one step's appends for a random subset (forked sharers included)
            k = int(rng.integers(1, len(live) + 1))
            seqs = [int(x) for x in rng.choice(live, size=k, replace=False)]
            counts = [int(rng.integers(0, 2 * bs + 2)) for _ in seqs]
            try:
                want = ref.append_batch(seqs, counts)
                err = None
            except M.OutOfBlocks:
                err = B.PA_ERR_OUT_OF_BLOCKS
            except M.TableFull:
                err = B.PA_ERR_TABLE_FULL
            if err is None:
                slots, pairs = bm.append_batch(seqs, counts)
                assert slots.tolist() == want[0] and pairs == want[1]
            else:
                with pytest.raises(B.PAError) as ex:
                    bm.append_batch(seqs, counts)
                assert ex.value.status == err
        else:
            s = live.pop(int(rng.integers(0, len(live))))
            bm.free_sequence(s)
            ref.free_sequence(s)
        _same_state(bm, ref, live)
    # step inputs for the live batch
    if live:
        pad = N - 1
        tab, lens = bm.build_batch(live, MB, pad)
        want_t, want_l = ref.build_batch(live, MB, pad)
        assert tab.tolist() == want_t and lens.tolist() == want_l
    bm.close()


def test_refusals_change_nothing():
    bm = B.BlockManager(4, 4, 4)
    bm.add_sequence(7)
    bm.append_tokens(7, 5)
    bm.fork(7, 9)
    before = (bm.table(7), bm.table(9), [bm.ref(b) for b in range(4)], bm.num_free())
    with pytest.raises(B.PAError) as ex:          # 2 new blocks + a copy, 2 free
        bm.append_tokens(9, 8)
    assert ex.value.status == B.PA_ERR_OUT_OF_BLOCKS
    with pytest.raises(B.PAError) as ex:          # would need 5 blocks, max 4
        bm.append_tokens(7, 12)
    assert ex.value.status == B.PA_ERR_TABLE_FULL
    for bad in (lambda: bm.add_sequence(7), lambda: bm.add_sequence(-1),
                lambda: bm.fork(3, 4), lambda: bm.fork(7, 9),
                lambda: bm.free_sequence(11), lambda: bm.append_tokens(11, 1)):
        with pytest.raises(B.PAError) as ex:
            bad()
        assert ex.value.status == B.PA_ERR_INVALID_ARG
    with pytest.raises(B.PAError) as ex:          # a table longer than the batch rows
        bm.build_batch([7], 1, 0)
    assert ex.value.status == B.PA_ERR_WORKSPACE
    assert (bm.table(7), bm.table(9), [bm.ref(b) for b in range(4)], bm.num_free()) == before
    lib = B.lib()
    assert lib.pa_bm_create(0, 16, 4, None) == B.PA_ERR_INVALID_ARG
    assert lib.pa_bm_ref_count(bm._h, 4) == -1 and lib.pa_bm_blocks_needed(bm._h, 11, 1) == -1


def test_batch_where_every_sharer_appends():
    """Three tables on one partly filled block all append in one step: the
    first two copy it, the last writes in place; a repeated id is refused."""
    bm = B.BlockManager(16, 4, 8)
    bm.add_sequence(0)
    bm.append_tokens(0, 6)
    bm.fork(0, 1)
    bm.fork(0, 2)
    shared = bm.table(0)[1]
    slots, pairs = bm.append_batch([2, 0, 1], [1, 1, 1])
    assert [p[0] for p in pairs] == [shared, shared]
    assert bm.table(1)[1] == shared and bm.ref(shared) == 1
    assert slots[2] == shared * 4 + 2
    with pytest.raises(B.PAError) as ex:
        bm.append_batch([0, 0], [1, 1])
    assert ex.value.status == B.PA_ERR_INVALID_ARG


def test_copy_on_write_needs_room_for_the_pair():
    import ctypes
    bm = B.BlockManager(8, 4, 4)
    bm.add_sequence(0)
    bm.append_tokens(0, 2)
    bm.fork(0, 1)
    slots = np.zeros(1, np.int32)
    ncow = ctypes.c_int(-1)
    r = B.lib().pa_bm_append_tokens(bm._h, 1, 1, slots.ctypes.data_as(ctypes.c_void_p), None,
                                    0, ctypes.byref(ncow))
    assert r == B.PA_ERR_WORKSPACE and bm.table(1) == bm.table(0) and bm.length(1) == 2


def test_large_pool_is_fast():
    """A serving-size pool: 200k blocks, 2k sequences sharing a prompt, 256
    decode tokens each; host time stays small."""
    import time
    bm = B.BlockManager(200_000, 16, 512)
    bm.add_sequence(0)
    bm.append_tokens(0, 1000)
    t0 = time.perf_counter()
    for s in range(1, 2000):
        bm.fork(0, s)
    for step in range(256):
        for s in range(0, 2000, 8):
            bm.append_tokens(s, 1)
    el = time.perf_counter() - t0
    assert bm.ref(0) == 2000 and el < 30.0

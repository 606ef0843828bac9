"""Pins of the reference block manager (oracle/block_manager.py) to facts
outside itself: the pages' printed shared-prefix reference counts and slot
example, the copy-on-write steps of "vLLM源码解析(二)" §3.2, and invariants
recounted by brute force from the tables.  Each pin takes the module under
test (the oracle, or a deliberately broken copy of it)."""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def recount(bm):
    """Reference counts and free blocks recounted from the tables alone."""
    ref = [0] * bm.num_blocks
    for t in bm.tables.values():
        for b in t:
            ref[b] += 1
    return ref


def pin_shared_prefix_refcounts(M):
    """FEI "共享前缀的 Block 复用": A and B share four blocks; each then
    appends into a fresh block -> counts 2, 2, 2, 2, 1, 1."""
    g = json.load(open(os.path.join(GOLDEN, "shared_prefix_refcounts.json")))
    bs = g["block_size"]
    bm = M.BlockManager(16, bs, 8)
    bm.add_sequence(0)
    bm.append_tokens(0, 4 * bs)
    bm.fork(0, 1)
    bm.append_tokens(0, 1)
    bm.append_tokens(1, 1)
    names = {}
    for name, b in zip(g["table_a"], bm.table(0)):
        names[name] = b
    for name, b in zip(g["table_b"], bm.table(1)):
        assert names.setdefault(name, b) == b, "shared names must be shared blocks"
    assert len(set(names.values())) == 6
    for name, want in g["ref_counts"].items():
        assert bm.ref[names[name]] == want, (name, bm.ref[names[name]], want)


def pin_worked_slot_example(M):
    """GAO §1.5: position 35, block size 16, table[2] = 9 -> slot 147."""
    g = json.load(open(os.path.join(GOLDEN, "slot_worked_example.json")))
    assert M.slot_for_position(g["block_table"], g["position"], g["block_size"]) == g["slot"]


def pin_slots_are_table_positions(M):
    """Every appended token's slot is its position through its own table."""
    bm = M.BlockManager(40, 4, 10)
    bm.add_sequence(3)
    got = []
    for n in (1, 3, 5, 2, 4):
        s, pairs = bm.append_tokens(3, n)
        assert pairs == []
        got += s
    t = bm.table(3)
    assert got == [t[p // 4] * 4 + p % 4 for p in range(15)]
    assert len(t) == 4 and len(set(t)) == 4


def pin_copy_on_write(M):
    """LAKE §3.2 on a shared, partly filled last block: the sequence that
    appends first gets a new block, a (shared, new) copy pair, its table
    remapped, and the old block loses one reference; the other sequence then
    appends in place."""
    bs = 4
    bm = M.BlockManager(10, bs, 6)
    bm.add_sequence(0)
    bm.append_tokens(0, 6)                  # blocks b0 (full), b1 (2 of 4)
    b0, b1 = bm.table(0)
    bm.fork(0, 1)
    assert bm.ref[b0] == 2 and bm.ref[b1] == 2
    slots, pairs = bm.append_tokens(1, 1)
    assert len(pairs) == 1 and pairs[0][0] == b1
    new = pairs[0][1]
    assert new not in (b0, b1) and bm.table(1) == [b0, new]
    assert slots == [new * bs + 2]
    assert bm.ref[b1] == 1 and bm.ref[new] == 1 and bm.ref[b0] == 2
    slots, pairs = bm.append_tokens(0, 1)
    assert pairs == [] and slots == [b1 * bs + 2] and bm.table(0) == [b0, b1]
    # three tables on b1: the first to append copies it; once only one
    # table names b1 again, that one appends in place and then opens a new
    # block when b1 is full
    bm.fork(0, 2)
    assert bm.ref[b1] == 2
    s0, p0 = bm.append_tokens(0, 1)
    assert len(p0) == 1 and p0[0][0] == b1 and bm.ref[b1] == 1
    s2, p2 = bm.append_tokens(2, 2)
    assert p2 == [] and s2[0] == b1 * bs + 3 and bm.table(2)[:2] == [b0, b1]
    assert len(bm.table(2)) == 3 and s2[1] == bm.table(2)[2] * bs


def pin_free_returns_blocks(M):
    """P1 §3.1: blocks go back to the pool when no table names them."""
    bm = M.BlockManager(12, 4, 6)
    bm.add_sequence(0)
    bm.append_tokens(0, 9)
    bm.fork(0, 1)
    bm.append_tokens(1, 3)
    used = bm.num_blocks - bm.num_free()
    bm.free_sequence(0)
    assert bm.num_blocks - bm.num_free() == len(bm.table(1)), "shared blocks stay"
    bm.free_sequence(1)
    assert bm.num_free() == bm.num_blocks and used > 0


def pin_lowest_free_block_first(M):
    bm = M.BlockManager(8, 2, 8)
    bm.add_sequence(0)
    bm.append_tokens(0, 6)
    assert bm.table(0) == [0, 1, 2]
    bm.add_sequence(1)
    bm.append_tokens(1, 2)
    bm.free_sequence(0)
    bm.add_sequence(2)
    bm.append_tokens(2, 3)
    assert bm.table(2) == [0, 1]


def pin_out_of_blocks_changes_nothing(M):
    bm = M.BlockManager(3, 4, 8)
    bm.add_sequence(0)
    bm.append_tokens(0, 6)
    bm.fork(0, 1)
    before = (bm.table(0), bm.table(1), list(bm.ref), bm.length(1))
    try:
        bm.append_tokens(1, 7)   # copy-on-write + 2 new blocks, only 1 free
        raise AssertionError("append must fail")
    except M.OutOfBlocks:
        pass
    assert (bm.table(0), bm.table(1), list(bm.ref), bm.length(1)) == before


def pin_random_invariants(M):
    """Random sessions: reference counts equal a recount from the tables,
    tables hold exactly ceil(len / bs) distinct-per-table blocks, slots
    decode back to their positions, no block is written by two sequences."""
    rng = np.random.default_rng(5)
    for trial in range(20):
        bs = int(rng.choice([1, 2, 4, 16]))
        bm = M.BlockManager(64, bs, 32)
        live, nxt = [], 0
        for _ in range(120):
            op = rng.integers(0, 4)
            if op == 0 or not live:
                bm.add_sequence(nxt)
                live.append(nxt)
                nxt += 1
            elif op == 1:
                bm.fork(int(rng.choice(live)), nxt)
                live.append(nxt)
                nxt += 1
            elif op == 2:
                s = int(rng.choice(live))
                n = int(rng.integers(1, 3 * bs + 1))
                try:
                    slots, pairs = bm.append_tokens(s, n)
                except (M.OutOfBlocks, M.TableFull):
                    continue
                L = bm.length(s)
                t = bm.table(s)
                assert slots == [t[p // bs] * bs + p % bs for p in range(L - n, L)]
                # the written blocks are this sequence's alone
                for sl in slots:
                    assert bm.ref[sl // bs] == 1
            else:
                s = live.pop(int(rng.integers(0, len(live))))
                bm.free_sequence(s)
            assert recount(bm) == bm.ref
            for s in live:
                t = bm.table(s)
                assert len(t) == -(-bm.length(s) // bs) and len(set(t)) == len(t)


def _state(bm):
    return (list(bm.ref), {k: list(v) for k, v in bm.tables.items()}, dict(bm.lengths))


def _session(M, seed, num_blocks, bs):
    """A manager with a few sequences, some forked (shared, partly filled
    last blocks), built by single-sequence appends only."""
    rng = np.random.default_rng(seed)
    bm = M.BlockManager(num_blocks, bs, 12)
    bm.add_sequence(0)
    bm.append_tokens(0, int(rng.integers(1, 3 * bs)))
    nxt = 1
    for _ in range(5):
        if rng.integers(0, 2):
            bm.fork(int(rng.integers(0, nxt)), nxt)
        else:
            bm.add_sequence(nxt)
            bm.append_tokens(nxt, int(rng.integers(1, 2 * bs)))
        nxt += 1
    return bm, rng


def pin_append_batch_is_sequential_appends(M):
    """A step's batch append equals single-sequence appends made one after
    another in batch order ([FEI] "Block Table 实现", [LAKE] §3.2): same
    slots, same copy-on-write pairs, same tables, counts and lengths.  The
    single appends run on an independent deep copy of the manager."""
    import copy
    cow = 0
    for seed in range(12):
        bm, rng = _session(M, 100 + seed, 64, int(rng_bs(seed)))
        ref_bm = copy.deepcopy(bm)
        seqs = [int(s) for s in rng.permutation(sorted(bm.tables))]
        counts = [int(rng.integers(0, 2 * bm.block_size)) for _ in seqs]
        slots, pairs = bm.append_batch(seqs, counts)
        want_slots, want_pairs = [], []
        for s, n in zip(seqs, counts):
            sl, pr = ref_bm.append_tokens(s, n)
            want_slots += sl
            want_pairs += pr
        assert slots == want_slots and pairs == want_pairs, seed
        assert _state(bm) == _state(ref_bm), seed
        assert recount(bm) == bm.ref
        cow += len(pairs)
    assert cow > 0, "the sessions must exercise copy-on-write"


def rng_bs(seed):
    return (1, 2, 4, 16)[seed % 4]


def pin_append_batch_rolls_back(M):
    """All or nothing: a batch that runs out of blocks part-way -- after
    earlier sequences of the batch have taken blocks and copy-on-write
    copies -- leaves every count, table and length exactly as before."""
    bs = 4
    bm = M.BlockManager(7, bs, 8)
    bm.add_sequence(0)
    bm.append_tokens(0, 6)          # 2 blocks, last one half full
    bm.fork(0, 1)                   # shares both
    bm.add_sequence(2)
    bm.append_tokens(2, 4)          # 1 full block; 4 blocks free
    before = _state(bm)
    # seq 1: copy-on-write (1 block) + 1 new; seq 2: 2 new; seq 0: 2 more
    # -> 6 blocks wanted, 4 free: the first two succeed, the third fails
    try:
        bm.append_batch([1, 2, 0], [3, 8, 8])
        raise AssertionError("batch must fail")
    except M.OutOfBlocks:
        pass
    assert _state(bm) == before
    assert recount(bm) == bm.ref
    # the same batch without its last member goes through
    slots, pairs = bm.append_batch([1, 2], [3, 8])
    assert len(pairs) == 1 and len(slots) == 11


def pin_append_batch_refusal_order(M):
    """Refusals come in a fixed order, each leaving the manager unchanged:
    an unknown or repeated sequence first, then a table past
    max_blocks_per_seq (checked for the whole batch before any append),
    then running out of blocks."""
    bm = M.BlockManager(4, 2, 3)
    bm.add_sequence(0)
    bm.add_sequence(1)
    bm.append_tokens(0, 3)          # 2 blocks; 2 free
    before = _state(bm)
    cases = [
        # an unknown id beside a table-full and an out-of-blocks member
        (([0, 9, 1], [4, 1, 6]), KeyError),
        # a repeated id whose total would also pass the table limit
        (([1, 1], [7, 1]), KeyError),
        # seq 1 alone would run out of blocks (3 wanted, 2 free), seq 0
        # would pass the table (7 tokens = 4 blocks > 3): the table wins
        (([1, 0], [6, 4]), M.TableFull),
        # seq 0 takes a block, then seq 1 wants 2 with 1 left
        (([0, 1], [2, 3]), M.OutOfBlocks),
    ]
    for (seqs, counts), exc in cases:
        try:
            bm.append_batch(seqs, counts)
            raise AssertionError(f"{seqs} {counts} must fail")
        except exc:
            pass
        assert _state(bm) == before, (seqs, counts)


def pin_build_batch_rows(M):
    """Step inputs ([GAO] §1.4): row i is the table of seqs[i] followed by
    pad_block up to max_blocks, and the context length is the sequence's
    token count (not the FEI sketch's len(blocks) * block_size)."""
    bm, rng = _session(M, 7, 64, 4)
    seqs = [int(s) for s in rng.permutation(sorted(bm.tables))]
    width = max(len(bm.table(s)) for s in seqs) + 3
    tables, lens = bm.build_batch(seqs, width, -5)
    assert len(tables) == len(seqs) and len(lens) == len(seqs)
    for i, s in enumerate(seqs):
        t = bm.table(s)
        assert tables[i] == t + [-5] * (width - len(t)), s
        assert lens[i] == bm.length(s)
    # token counts that are not whole blocks are kept as counts
    assert any(n % bm.block_size for n in lens)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]

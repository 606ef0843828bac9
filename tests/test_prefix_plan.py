"""The host prefix planner (pa_plan_prefix_groups): plan layout and
invariants on random batches with shared leading blocks, and optimality
against exhaustive search over every grouping of small batches.  Host code
only: runs without a GPU."""
import itertools

import numpy as np
import pytest

try:
    from paged_kv_cache_96_gb300 import binding as B
except ImportError as e:  # library not built
    pytest.skip(f"library missing: {e}", allow_module_level=True)


def _decode_plan(plan, S, ng, nm):
    plan = np.asarray(plan)
    assert plan.shape[0] == S + 2 * ng + 1 + nm
    seq_prefix = plan[:S]
    gstart = plan[S:S + ng + 1]
    gprefix = plan[S + ng + 1:S + 2 * ng + 1]
    members = plan[S + 2 * ng + 1:]
    groups = [(int(gprefix[g]), members[gstart[g]:gstart[g + 1]].tolist()) for g in range(ng)]
    return seq_prefix, groups


def _random_batch(rng, S, MB, bs, families=3):
    """Sequences drawn from a few families sharing leading blocks, with
    random divergence points and some copy-on-write style single-block
    remaps inside shared prefixes."""
    tables = np.zeros((S, MB), np.int32)
    ctx = np.zeros(S, np.int32)
    nxt = 1000
    fam_rows = [rng.integers(0, 500, MB) for _ in range(families)]
    for s in range(S):
        f = int(rng.integers(0, families + 1))
        if f < families:
            keep = int(rng.integers(0, MB + 1))
            row = fam_rows[f].copy()
            row[keep:] = np.arange(nxt, nxt + MB - keep)
            nxt += MB
            if rng.random() < 0.3 and keep > 1:
                row[int(rng.integers(0, keep))] = nxt
                nxt += 1
        else:
            row = np.arange(nxt, nxt + MB)
            nxt += MB
        tables[s] = row
        ctx[s] = int(rng.integers(1, MB * bs + 1))
    return tables, ctx


def _cap(ctx, bs, MB):
    return np.minimum(np.maximum(ctx - 1, 0) // bs, MB)


def _savings(tables, ctx, bs, MB, groups):
    total = 0
    for L, mem in groups:
        total += (len(mem) - 1) * (L // bs)
    return total


def _check_invariants(tables, ctx, bs, MB, min_blocks, plan, ng, nm):
    S = tables.shape[0]
    seq_prefix, groups = _decode_plan(plan, S, ng, nm)
    seen = set()
    cap = _cap(ctx, bs, MB)
    for L, mem in groups:
        assert len(mem) >= 2
        assert L % bs == 0 and L // bs >= min_blocks
        lead = mem[0]
        for s in mem:
            assert s not in seen
            seen.add(s)
            assert seq_prefix[s] == L
            assert L // bs <= cap[s], "prefix must end before the last token"
            assert L < ctx[s]
            assert (tables[s, :L // bs] == tables[lead, :L // bs]).all()
    for s in range(S):
        if s not in seen:
            assert seq_prefix[s] == 0
    return groups


@pytest.mark.parametrize("seed", range(20))
def test_plan_invariants_random(seed):
    rng = np.random.default_rng(seed)
    S, MB, bs = int(rng.integers(1, 40)), int(rng.integers(1, 12)), 16
    tables, ctx = _random_batch(rng, S, MB, bs)
    for min_blocks in (1, 2, 4):
        plan, ng, nm = B.pa_plan_prefix_groups(tables, ctx, bs, min_blocks)
        _check_invariants(tables, ctx, bs, MB, min_blocks, plan, ng, nm)


def _best_exhaustive(tables, ctx, bs, MB, min_blocks):
    """Maximum saved block reads over every set partition of the sequences
    (a group's prefix = the longest one all members share, capped)."""
    S = tables.shape[0]
    cap = _cap(ctx, bs, MB)

    def group_value(mem):
        if len(mem) < 2:
            return 0
        L = min(int(cap[s]) for s in mem)
        lead = tables[mem[0]]
        k = 0
        while k < L and all(tables[s][k] == lead[k] for s in mem):
            k += 1
        return (len(mem) - 1) * k if k >= min_blocks else 0

    best = 0

    def rec(i, groups):
        nonlocal best
        if i == S:
            best = max(best, sum(group_value(g) for g in groups))
            return
        for g in groups:
            g.append(i)
            rec(i + 1, groups)
            g.pop()
        groups.append([i])
        rec(i + 1, groups)
        groups.pop()

    rec(0, [])
    return best


@pytest.mark.parametrize("seed", range(25))
def test_plan_optimal_small(seed):
    rng = np.random.default_rng(100 + seed)
    S, MB, bs = int(rng.integers(2, 8)), int(rng.integers(1, 6)), 16
    tables, ctx = _random_batch(rng, S, MB, bs, families=2)
    for min_blocks in (1, 2):
        plan, ng, nm = B.pa_plan_prefix_groups(tables, ctx, bs, min_blocks)
        groups = _check_invariants(tables, ctx, bs, MB, min_blocks, plan, ng, nm)
        assert _savings(tables, ctx, bs, MB, groups) == _best_exhaustive(
            tables, ctx, bs, MB, min_blocks)


def test_plan_prefix_sharing_step_shape():
    """The prefix-sharing picture: 8 sequences share 4 blocks; one of them
    had block 2 copied on write (its table names the copy), one shares only
    the first block, one shares nothing.  The planner groups the six with
    the whole prefix and leaves the others to their own tables."""
    bs = 16
    shared = [10, 11, 12, 13]
    rows = []
    for s in range(6):
        rows.append(shared + [100 + s])
    rows.append([10, 11, 99, 13, 200])   # copied on write at block 2
    rows.append([10, 300, 301, 302, 303])
    rows.append([400, 401, 402, 403, 404])
    tables = np.array(rows, np.int32)
    ctx = np.full(tables.shape[0], 5 * bs, np.int32)
    plan, ng, nm = B.pa_plan_prefix_groups(tables, ctx, bs)
    seq_prefix, groups = _decode_plan(plan, tables.shape[0], ng, nm)
    assert [(L, sorted(m)) for L, m in groups] == [(4 * bs, [0, 1, 2, 3, 4, 5])]
    assert seq_prefix.tolist() == [64] * 6 + [0, 0, 0]


def test_plan_edge_cases():
    bs = 16
    # empty batch, single sequence, contexts too short to share anything
    plan, ng, nm = B.pa_plan_prefix_groups(np.zeros((0, 3), np.int32),
                                           np.zeros(0, np.int32), bs)
    assert (ng, nm) == (0, 0) and plan.numel() == 1
    plan, ng, nm = B.pa_plan_prefix_groups(np.array([[1, 2]], np.int32),
                                           np.array([32], np.int32), bs)
    assert (ng, nm) == (0, 0)
    t = np.array([[1, 2], [1, 2]], np.int32)
    plan, ng, nm = B.pa_plan_prefix_groups(t, np.array([16, 16], np.int32), bs)
    assert (ng, nm) == (0, 0), "a prefix must end before each member's last token"
    plan, ng, nm = B.pa_plan_prefix_groups(t, np.array([17, 40], np.int32), bs)
    assert (ng, nm) == (1, 2) and plan.tolist() == [16, 16, 0, 2, 16, 0, 1]

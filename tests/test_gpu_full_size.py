"""Every benchmarked workload at full size, in the launch configuration the
benchmark times (each workload's own partition size): slots and both pools
-- after the history writes, the step's writes and its copy-on-write copies
-- bit-exact against the oracle; attention of sampled sequences (the
longest, the shortest and seeded random ones, every head and element), or
for a prefill step sampled chunk rows (each chunk's first and last row and
seeded random ones), within the contract tolerance."""
import numpy as np
import pytest
import torch

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

from paged_kv_cache_96_gb300 import workloads as W  # noqa: E402
from stepping import OracleStep, assert_attention_close  # noqa: E402

NAMES = ["tiny", "mha7b", "gqa70b", "longctx", "prefix", "gqa70b-fp8", "longctx-fp8",
         "prefix-cascade", "mixed", "chunked"]


def _sample(w, k=6, seed=7):
    ctx = w.context_lens
    order = np.argsort(ctx)
    picks = {int(order[0]), int(order[-1]), int(order[len(order) // 2])}
    rng = np.random.default_rng(seed)
    picks.update(int(x) for x in rng.choice(w.S, size=min(k, w.S), replace=False))
    return sorted(picks)


@pytest.mark.parametrize("name", NAMES)
def test_full_size_step(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_96_gb300 import step as S
    w = W.build(W.CONFIGS[name])
    st = S.DecodeStep(w)  # the workload's own partition size, as the benchmark runs it
    out = st.run()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0

    ref = OracleStep(w)
    assert np.array_equal(st.slots.cpu().numpy().astype(np.int64), ref.new_slots)
    assert np.array_equal(S.to_bits(st.key_cache), ref.key_cache)
    assert np.array_equal(S.to_bits(st.value_cache), ref.value_cache)

    got = S.to_float(out)
    if w.prefill:
        qs = w.query_start
        rows = {int(qs[s]) for s in range(w.S) if qs[s + 1] > qs[s]}
        rows |= {int(qs[s + 1]) - 1 for s in range(w.S) if qs[s + 1] > qs[s]}
        rng = np.random.default_rng(11)
        rows |= {int(x) for x in rng.choice(w.T, size=min(8, w.T), replace=False)}
        rows = sorted(rows)
        assert_attention_close(got[rows], ref.attention(rows=rows), f"{name} rows {rows}")
        return
    seqs = _sample(w)
    want = ref.attention(seqs=seqs)
    assert_attention_close(got[seqs], want[seqs], f"{name} seqs {seqs}")

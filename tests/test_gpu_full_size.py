"""Every benchmarked workload at full size, in the launch configuration the
benchmark times (each workload's own partition size): slots and both pools
-- after the history writes, the step's writes and its copy-on-write copies
-- bit-exact against the oracle; attention of every sequence (every head
and element), or for a prefill step of every chunk row, within the contract
tolerance -- the oracle runs on all host cores (a spawn-context process
pool)."""
import numpy as np
import pytest
import torch

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

from paged_kv_cache_96_gb300 import workloads as W  # noqa: E402
from stepping import OracleStep, assert_attention_close, attention_all  # noqa: E402

NAMES = ["tiny", "mha7b", "gqa70b", "longctx", "prefix", "gqa70b-fp8", "longctx-fp8",
         "prefix-cascade", "mixed", "chunked", "chunked-fp8", "prefix-cascade-fp8", "mixed-fp8"]


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
    want = attention_all(ref)
    assert_attention_close(got, want, f"{name} (all {'rows' if w.prefill else 'sequences'})")

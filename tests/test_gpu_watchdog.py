"""The attention kernels' bounded waits, made to run out on purpose.

Every wait of the decode pass, the prefix pass and the chunked-prefill
kernel for staged data is bounded (the watchdog; the pages have no
counterpart).  Here a test hook leaves the first K/V fill of every CTA
unissued -- a barrier that nothing completes -- with a short stage-wait
limit, so that wait certainly runs out.  Checked for each path: the call
returns and the stream completes, PA_DEVERR_TIMEOUT is in the error word,
and the same call made normally right after it on the same stream (which,
for the tensor-core kernel, has to allocate the tensor memory the aborted
launch released) matches the oracle with a clean error word.  Nothing here
faults or hangs a GPU: the withheld fill is a wait with a limit.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from paged_kv_cache_96_gb300 import workloads as W  # noqa: E402
from stepping import OracleStep, assert_attention_close  # noqa: E402

LIMIT_NS = 2_000_000  # 2 ms: short, but far above any real fill's latency

CASES = [
    ("gqa70b", 128, "attention"),
    ("gqa70b", 0, "append"),
    ("longctx", 256, "append"),
    ("gqa70b-fp8", 128, "attention"),
    ("gqa70b-fp8", 128, "append"),
    ("prefix-cascade", 64, "attention"),
    ("prefix-cascade", 64, "append"),
    ("prefix-cascade-fp8", 64, "attention"),
    ("prefix-cascade-fp8", 64, "append"),
    ("chunked", 0, "prefill"),
    ("chunked-fp8", 0, "prefill"),
    ("mixed", 0, "prefill"),
    ("mixed-fp8", 0, "prefill"),
]


@pytest.fixture(scope="module")
def mods():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_96_gb300 import binding, step
    return binding, step


def _call(st, how):
    if how == "append":
        st.copy_blocks()
        st.append_attention()
    else:
        st.attention()


@pytest.mark.parametrize("name,P,how", CASES, ids=lambda x: str(x))
def test_wait_runs_out_then_recovers(mods, name, P, how):
    B, S = mods
    w = W.build(W.small_variant(name))
    ref = OracleStep(w)
    st = S.DecodeStep(w, partition_size=P)
    if how != "append":
        # the step's writes first, then attention alone
        st.slot_mapping_and_cache()
        st.copy_blocks()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    try:
        B.pa_set_stage_wait_limit_ns(LIMIT_NS)
        B.pa_debug_withhold_first_fill(True)
        _call(st, how)
    finally:
        B.pa_debug_withhold_first_fill(False)
        B.pa_set_stage_wait_limit_ns(0)
    torch.cuda.synchronize()  # the aborted launch has returned
    err = int(st.error_word.item())
    assert err & B.DEVERR_TIMEOUT, hex(err)
    assert err & ~B.DEVERR_TIMEOUT == 0, hex(err)

    # the same call, normally, on the same stream (a timed-out call may leave
    # the prefix pass's arrival counters short: the workspace is zeroed again,
    # as the interface asks)
    st.error_word.zero_()
    if st.workspace is not None:
        st.workspace.zero_()
    _call(st, how)
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    got = S.to_float(st.out)
    want = ref.attention()
    assert_attention_close(got, want, f"{name} after a timed-out call")
    assert np.array_equal(S.to_bits(st.key_cache), ref.key_cache)
    assert np.array_equal(S.to_bits(st.value_cache), ref.value_cache)

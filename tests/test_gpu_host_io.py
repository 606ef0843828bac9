"""The end-to-end path a serving loop runs (step.HostStepIO): inputs copied
from pinned host staging buffers, the step, the output read back into pinned
host memory, with uploads and read-backs on their own streams overlapped with
the neighbouring steps and double-buffered -- run eagerly and as a captured
CUDA graph.  Every step of the workload recomputes the same output (the cache
write of the step's tokens is idempotent), so each host output must equal,
bit for bit, the output of a plain device-side step, and match the oracle."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from paged_kv_cache_96_gb300 import workloads as W  # noqa: E402
from stepping import OracleStep, assert_attention_close  # noqa: E402


@pytest.mark.parametrize("name", ["gqa70b", "prefix-cascade", "chunked", "gqa70b-fp8"])
def test_host_step_io_matches_device_step(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_96_gb300 import step as S
    w = W.build(W.small_variant(name))
    st = S.DecodeStep(w)
    want = st.run().clone()
    torch.cuda.synchronize()
    assert int(st.error_word.item()) == 0
    want_bits = want.view(torch.int16).cpu().numpy()

    host = S.HostStepIO(st)
    stream = torch.cuda.current_stream()
    host.begin(stream)
    outs = [host.step() for _ in range(5)]
    host.finish(stream)
    torch.cuda.synchronize()
    # the last two steps' host buffers hold steps 3 and 4
    for out in outs[-2:]:
        assert np.array_equal(out.view(torch.int16).numpy(), want_bits), name

    host.capture(4)
    for _ in range(3):
        host.replay()
    torch.cuda.synchronize()
    for slot in range(2):
        assert np.array_equal(host.host_outs[slot].view(torch.int16).numpy(), want_bits), name
    assert int(st.error_word.item()) == 0

    ref = OracleStep(w)
    assert_attention_close(S.to_float(host.host_outs[0]), ref.attention(), name)

"""The allocation-free decode entry point, through the C ABI.

pa_decode_attention_noalloc serves callers that may not allocate device
memory on their decode path (a plugin inside an engine that owns every
device allocation, a loop that cannot take an allocation's implicit
synchronisation, a C interface with no way to pass a workspace).  It keeps
its split-context partials in a fixed-size device array inside the library.
This test checks, on two calls in a row, that its output matches the
regular entry point's (same kernels, caller-provided workspace) within the
attention tolerance, and that sizes needing more scratch than the array
holds are refused before anything runs.  The file is named so that pytest
collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from paged_kv_cache_96_gb300 import workloads as W  # noqa: E402
from stepping import ATOL, RTOL  # noqa: E402


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_96_gb300 import binding
    return binding


def _raw_noalloc(L, st, P, stream):
    w = st.w
    return L.pa_decode_attention_noalloc(
        ctypes.c_void_p(st.out.data_ptr()), ctypes.c_void_p(st.query.data_ptr()),
        ctypes.c_void_p(st.key_cache.data_ptr()), ctypes.c_void_p(st.value_cache.data_ptr()),
        ctypes.c_void_p(st.step_block_tables.data_ptr()), w.max_blocks_per_seq,
        ctypes.c_void_p(st.context_lens.data_ptr()), st.max_context_len, w.S, w.H, w.Hkv,
        w.D, w.bs, w.num_blocks, ctypes.c_float(w.scale), P, 1 if w.dtype == "bf16" else 0,
        None, ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("name", ["longctx", "gqa70b"])
def test_noalloc_matches_workspace_entry_point(B, name):
    from paged_kv_cache_96_gb300 import step as S
    w = W.build(W.small_variant(name))
    P = 32  # several partitions per sequence, so the scratch array is used
    st = S.DecodeStep(w, partition_size=P)
    st.run()
    st.attention(partition_size=P)
    torch.cuda.synchronize()
    ref = S.to_float(st.out)
    L = B.lib()
    stream = torch.cuda.current_stream()
    for call in range(2):
        st.out.fill_(float("nan"))
        assert _raw_noalloc(L, st, P, stream) == B.PA_OK, call
        torch.cuda.synchronize()
        got = S.to_float(st.out)
        assert np.isfinite(got).all(), call
        assert (np.abs(got - ref) <= ATOL + RTOL * np.abs(ref)).all(), call


def test_noalloc_refuses_oversized_workspace(B):
    from paged_kv_cache_96_gb300 import step as S
    w = W.build(W.small_variant("gqa70b"))
    st = S.DecodeStep(w, partition_size=16)
    L = B.lib()
    # a maximum context that would need more partials than the array holds
    big = B.NOALLOC_WORKSPACE_BYTES
    per_part = w.S * w.H * (w.D + 2) * 4
    ctx_needed = (big // per_part + 2) * 16
    need = B.pa_decode_workspace_bytes(w.S, w.H, w.Hkv, w.D, ctx_needed, 16)
    assert need > big
    r = L.pa_decode_attention_noalloc(
        ctypes.c_void_p(st.out.data_ptr()), ctypes.c_void_p(st.query.data_ptr()),
        ctypes.c_void_p(st.key_cache.data_ptr()), ctypes.c_void_p(st.value_cache.data_ptr()),
        ctypes.c_void_p(st.step_block_tables.data_ptr()), w.max_blocks_per_seq,
        ctypes.c_void_p(st.context_lens.data_ptr()), ctx_needed, w.S, w.H, w.Hkv, w.D, w.bs,
        w.num_blocks, ctypes.c_float(w.scale), 16, 1, None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert r == B.PA_ERR_WORKSPACE

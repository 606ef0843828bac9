"""The allocation-free decode entry point, through the C ABI.

pa_decode_attention_noalloc serves callers that may not allocate device
memory on their decode path (a plugin inside an engine that owns every
device allocation, a loop that cannot take an allocation's implicit
synchronisation, a C interface with no way to pass a workspace).  It keeps
its split-context partials in a fixed-size device array inside the library,
shared by every call.  This test runs it on workloads of different sizes one
after another -- long context, then GQA, then long context again, so that a
call finds the array holding another call's partials -- through the raw C
ABI and through the Python binding, and checks each output bit for bit
against the regular entry point's (the same kernels with a caller-provided
workspace and the same partitions give the same bits); it also checks that
sizes needing more scratch than the array holds are refused before anything
runs.  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from paged_kv_cache_96_gb300 import workloads as W  # noqa: E402


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


def _step(name, P):
    from paged_kv_cache_96_gb300 import step as S
    w = W.build(W.small_variant(name))
    st = S.DecodeStep(w, partition_size=P)
    st.run()  # the step's writes; then attention alone through each entry point
    st.attention(partition_size=P)
    torch.cuda.synchronize()
    return st, st.out.clone()


def test_noalloc_matches_workspace_entry_point(B):
    P = 32  # several partitions per sequence, so the scratch array is used
    steps = {n: _step(n, P) for n in ("longctx", "gqa70b")}
    L = B.lib()
    stream = torch.cuda.current_stream()
    for call, name in enumerate(["longctx", "gqa70b", "longctx"]):
        st, ref = steps[name]
        st.out.fill_(float("nan"))
        if call == 1:
            B.pa_decode_attention_noalloc(st.out, st.query, st.key_cache, st.value_cache,
                                          st.step_block_tables, st.context_lens,
                                          st.max_context_len, st.w.scale, P)
        else:
            assert _raw_noalloc(L, st, P, stream) == B.PA_OK, call
        torch.cuda.synchronize()
        assert torch.isfinite(st.out.float()).all(), (call, name)
        assert torch.equal(st.out, ref), (call, name)


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

"""The C ABI on the host (no GPU): the library builds, loads and exports
every entry point the header declares; host-side argument checks return
their status before anything is launched; workspace sizes follow the
documented layout."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "paged_attention.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_96_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


@pytest.fixture(scope="module")
def B(lib):
    from paged_kv_cache_96_gb300 import binding
    return binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("pa_slot_mapping", "pa_reshape_and_cache", "pa_copy_blocks",
              "pa_decode_attention", "pa_decode_workspace_bytes"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(B):
    L = B.lib()
    assert L.pa_status_string(0) == b"PA_OK"
    assert L.pa_status_string(3) == b"PA_ERR_WORKSPACE"
    assert L.pa_version() >= 100


FAKE = ctypes.c_void_p(0x10000)      # never dereferenced: checks fail first
FAKE_ODD = ctypes.c_void_p(0x10002)  # not 16-byte aligned


def _decode(L, **kw):
    a = dict(out=FAKE, query=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, mb=4, ctx=FAKE, maxctx=64,
             S=2, H=8, Hkv=2, D=128, bs=16, N=8, scale=0.1, P=0, ws=None, wsb=0, dt=1,
             err=None, stream=None)
    a.update(kw)
    return L.pa_decode_attention(a["out"], a["query"], a["kc"], a["vc"], a["bt"], a["mb"],
                                 a["ctx"], a["maxctx"], a["S"], a["H"], a["Hkv"], a["D"],
                                 a["bs"], a["N"], a["scale"], a["P"], a["ws"], a["wsb"],
                                 a["dt"], a["err"], a["stream"])


def test_decode_argument_checks(B):
    L = B.lib()
    assert _decode(L, out=None) == B.PA_ERR_INVALID_ARG
    assert _decode(L, query=FAKE_ODD) == B.PA_ERR_INVALID_ARG
    assert _decode(L, H=6, Hkv=4) == B.PA_ERR_INVALID_ARG
    assert _decode(L, dt=7) == B.PA_ERR_INVALID_ARG
    assert _decode(L, scale=float("nan")) == B.PA_ERR_INVALID_ARG
    assert _decode(L, D=96) == B.PA_ERR_UNSUPPORTED
    assert _decode(L, bs=8) == B.PA_ERR_UNSUPPORTED
    assert _decode(L, bs=48) == B.PA_ERR_UNSUPPORTED
    assert _decode(L, H=34, Hkv=2) == B.PA_ERR_UNSUPPORTED      # group 17
    assert _decode(L, P=24) == B.PA_ERR_UNSUPPORTED
    # split path needs a workspace
    assert _decode(L, P=16, maxctx=64) == B.PA_ERR_WORKSPACE
    need = L.pa_decode_workspace_bytes(2, 8, 2, 128, 64, 16)
    assert _decode(L, P=16, ws=FAKE, wsb=need - 1) == B.PA_ERR_WORKSPACE
    assert _decode(L, P=16, ws=ctypes.c_void_p(0x10010), wsb=need) == B.PA_ERR_WORKSPACE
    # no sequences: nothing to do
    assert _decode(L, S=0, out=None) == B.PA_OK


def test_cache_op_argument_checks(B):
    L = B.lib()
    assert L.pa_slot_mapping(None, None, 4, None, None, 0, 1, 16, 8, None, None) == B.PA_OK
    assert L.pa_slot_mapping(None, FAKE, 4, FAKE, FAKE, 3, 1, 16, 8, None, None) == \
        B.PA_ERR_INVALID_ARG
    assert L.pa_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 8, 16, 2, 128, 1,
                                  None, None) == B.PA_OK
    assert L.pa_reshape_and_cache(FAKE_ODD, FAKE, FAKE, FAKE, FAKE, 2, 8, 16, 2, 128, 1,
                                  None, None) == B.PA_ERR_INVALID_ARG
    assert L.pa_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 16, 1, 4, 1,
                                  None, None) == B.PA_ERR_UNSUPPORTED  # 8-byte rows
    assert L.pa_copy_blocks(FAKE, FAKE, FAKE, 0, 8, 16, 2, 128, 1, None, None) == B.PA_OK
    assert L.pa_copy_blocks(FAKE, FAKE, None, 3, 8, 16, 2, 128, 1, None, None) == \
        B.PA_ERR_INVALID_ARG
    assert L.pa_copy_blocks(FAKE, FAKE, FAKE, 3, 8, 16, 2, 128, 5, None, None) == \
        B.PA_ERR_INVALID_ARG


def test_fused_cache_argument_checks(B):
    """pa_slot_mapping_and_cache(_fp8): the slot-mapping checks, then the
    cache-write checks, all before any launch."""
    L = B.lib()
    f = L.pa_slot_mapping_and_cache
    f8 = L.pa_slot_mapping_and_cache_fp8
    # (slots, tables, mb, seq, pos, T, S, key, value, kc, vc, N, bs, Hkv, d, dtype, err, stream)
    ok = (FAKE, FAKE, 4, FAKE, FAKE, 3, 2, FAKE, FAKE, FAKE, FAKE, 8, 16, 2, 128, 1, None, None)
    assert f(*ok[:5], 0, *ok[6:]) == B.PA_OK                          # no tokens
    assert f(None, *ok[1:]) == B.PA_ERR_INVALID_ARG                   # no slot array
    assert f(*ok[:3], None, *ok[4:]) == B.PA_ERR_INVALID_ARG          # no sequence ids
    assert f(*ok[:2], 0, *ok[3:]) == B.PA_ERR_INVALID_ARG             # empty table rows
    assert f(*ok[:7], FAKE_ODD, *ok[8:]) == B.PA_ERR_INVALID_ARG      # unaligned keys
    assert f(*ok[:13], 1, 4, *ok[15:]) == B.PA_ERR_UNSUPPORTED        # 8-byte rows
    assert f(*ok[:15], 5, *ok[16:]) == B.PA_ERR_INVALID_ARG           # not a 16-bit type
    assert f(*ok[:11], 1 << 20, 1 << 12, *ok[13:]) == B.PA_ERR_UNSUPPORTED  # 2^32 slots
    ok8 = ok[:16] + (0.5, 0.5) + ok[16:]
    assert f8(*ok8[:5], 0, *ok8[6:]) == B.PA_OK
    assert f8(*ok8[:16], 0.0, 0.5, *ok8[18:]) == B.PA_ERR_INVALID_ARG  # zero K scale
    assert f8(*ok8[:16], 0.5, float("inf"), *ok8[18:]) == B.PA_ERR_INVALID_ARG
    assert f8(*ok8[:3], None, *ok8[4:]) == B.PA_ERR_INVALID_ARG


def test_append_argument_checks(B):
    """pa_decode_attention_append(_fp8): the decode checks, then the new-row
    buffers, all before any launch."""
    L = B.lib()
    f = L.pa_decode_attention_append
    f8 = L.pa_decode_attention_append_fp8
    # (out, query, kc, vc, new_key, new_value, slots, tables, mb, ctx, maxctx, S, H, Hkv,
    #  d, bs, N, scale, P, ws, ws_bytes, dtype, err, stream)
    ok = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 4, FAKE, 64, 2, 8, 2, 128, 16, 8,
          0.1, 0, None, 0, 1, None, None)
    assert f(*ok[:11], 0, *ok[12:]) == B.PA_OK                        # no sequences
    assert f(*ok[:4], None, *ok[5:]) == B.PA_ERR_INVALID_ARG          # no new keys
    assert f(*ok[:5], None, *ok[6:]) == B.PA_ERR_INVALID_ARG          # no new values
    assert f(*ok[:4], FAKE_ODD, *ok[5:]) == B.PA_ERR_INVALID_ARG      # unaligned rows
    assert f(*ok[:21], 7, *ok[22:]) == B.PA_ERR_INVALID_ARG           # not a 16-bit type
    assert f(*ok[:14], 96, *ok[15:]) == B.PA_ERR_UNSUPPORTED          # head_dim 96
    assert f(*ok[:18], 16, *ok[19:]) == B.PA_ERR_WORKSPACE            # split, no workspace
    ok8 = ok[:18] + (0.5, 0.5) + ok[18:]
    assert f8(*ok8[:11], 0, *ok8[12:]) == B.PA_OK
    assert f8(*ok8[:18], 0.0, 0.5, *ok8[20:]) == B.PA_ERR_INVALID_ARG  # zero K scale
    assert f8(*ok8[:18], 0.5, float("nan"), *ok8[20:]) == B.PA_ERR_INVALID_ARG
    assert f8(*ok8[:14], 96, *ok8[15:]) == B.PA_ERR_UNSUPPORTED         # FP8: d 64 or 128
    assert f8(*ok8[:5], None, *ok8[6:]) == B.PA_ERR_INVALID_ARG


def test_cascade_append_argument_checks(B):
    L = B.lib()
    f = L.pa_decode_attention_cascade_append
    # (out, query, kc, vc, new_key, new_value, slots, tables, mb, ctx, maxctx, S, H, Hkv,
    #  d, bs, N, scale, plan, groups, members, P, ws, ws_bytes, dtype, err, stream)
    ok = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 4, FAKE, 64, 2, 8, 2, 128, 16, 8,
          0.1, FAKE, 1, 2, 16, None, 0, 1, None, None)
    assert f(*ok[:4], None, *ok[5:]) == B.PA_ERR_INVALID_ARG          # no new keys
    assert f(*ok[:5], None, *ok[6:]) == B.PA_ERR_INVALID_ARG          # no new values
    assert f(*ok[:24], 2, *ok[25:]) == B.PA_ERR_UNSUPPORTED           # FP8 pools
    assert f(*ok[:19], 1, 1, *ok[21:]) == B.PA_ERR_INVALID_ARG        # group of one
    assert f(*ok[:18], None, *ok[19:]) == B.PA_ERR_WORKSPACE          # no workspace first
    assert f(*ok[:11], 0, *ok[12:]) == B.PA_OK                        # no sequences
    # FP8 pools: k_scale, v_scale after scale
    f8 = L.pa_decode_attention_cascade_append_fp8
    ok8 = ok[:18] + (0.5, 0.5) + ok[18:]
    assert f8(*ok8[:11], 0, *ok8[12:]) == B.PA_OK                      # no sequences
    assert f8(*ok8[:18], 0.0, 0.5, *ok8[20:]) == B.PA_ERR_INVALID_ARG  # zero K scale
    assert f8(*ok8[:18], 0.5, float("inf"), *ok8[20:]) == B.PA_ERR_INVALID_ARG
    assert f8(*ok8[:26], 2, *ok8[27:]) == B.PA_ERR_INVALID_ARG         # query not 16-bit
    assert f8(*ok8[:5], None, *ok8[6:]) == B.PA_ERR_INVALID_ARG        # no new values
    assert f8(*ok8[:21], 1, 1, *ok8[23:]) == B.PA_ERR_INVALID_ARG      # group of one
    assert f8(*ok8[:20], None, *ok8[21:]) == B.PA_ERR_WORKSPACE        # no workspace
    ws = (ctypes.c_uint8 * (1 << 22))()
    wsp = (ctypes.addressof(ws) + 255) // 256 * 256
    okw = ok8[:24] + (wsp, (1 << 22) - 256) + ok8[26:]
    assert f8(*okw[:14], 96, *okw[15:]) == B.PA_ERR_UNSUPPORTED        # head_dim 96
    g8 = L.pa_decode_attention_cascade_fp8
    # (out, query, kc, vc, tables, mb, ctx, maxctx, S, H, Hkv, d, bs, N, scale, k_scale,
    #  v_scale, plan, groups, members, P, ws, ws_bytes, dtype, err, stream)
    okc = (FAKE, FAKE, FAKE, FAKE, FAKE, 4, FAKE, 64, 2, 8, 2, 128, 16, 8, 0.1, 0.5, 0.5,
           FAKE, 1, 2, 16, None, 0, 1, None, None)
    assert g8(*okc[:8], 0, *okc[9:]) == B.PA_OK
    assert g8(*okc[:15], -1.0, *okc[16:]) == B.PA_ERR_INVALID_ARG
    assert g8(*okc[:21], None, *okc[22:]) == B.PA_ERR_WORKSPACE
    assert g8(*okc[:11], 96, *okc[12:]) == B.PA_ERR_UNSUPPORTED


def test_prefill_argument_checks(B):
    """pa_prefill_attention(_fp8): sizes, scales and types, before any launch."""
    L = B.lib()
    f = L.pa_prefill_attention
    f8 = L.pa_prefill_attention_fp8
    # (out, query, kc, vc, tables, mb, query_start, ctx, maxctx, S, T, H, Hkv, d, bs, N,
    #  scale, dtype, err, stream)
    ok = (FAKE, FAKE, FAKE, FAKE, FAKE, 4, FAKE, FAKE, 64, 2, 10, 8, 2, 128, 16, 8, 0.1, 1,
          None, None)
    assert f(*ok[:10], 0, *ok[11:]) == B.PA_OK                        # no tokens
    assert f(*ok[:16], 0.0, *ok[17:]) == B.PA_ERR_INVALID_ARG         # scale 0
    assert f(*ok[:17], 2, *ok[18:]) == B.PA_ERR_UNSUPPORTED           # FP8 pools: _fp8
    assert f(*ok[:13], 96, *ok[14:]) == B.PA_ERR_UNSUPPORTED          # head_dim 96
    assert f(*ok[:12], 3, *ok[13:]) == B.PA_ERR_INVALID_ARG           # 8 heads over 3
    ok8 = ok[:17] + (0.5, 0.5) + ok[17:]
    assert f8(*ok8[:10], 0, *ok8[11:]) == B.PA_OK
    assert f8(*ok8[:17], 0.0, 0.5, *ok8[19:]) == B.PA_ERR_INVALID_ARG  # zero K scale
    assert f8(*ok8[:17], 0.5, float("nan"), *ok8[19:]) == B.PA_ERR_INVALID_ARG
    assert f8(*ok8[:19], 2, *ok8[20:]) == B.PA_ERR_INVALID_ARG         # query not 16-bit
    assert f8(*ok8[:13], 96, *ok8[14:]) == B.PA_ERR_UNSUPPORTED        # head_dim 96
    assert f8(*ok8[:2], FAKE_ODD, *ok8[3:]) == B.PA_ERR_INVALID_ARG    # unaligned pool


def test_workspace_layout_sizes(B):
    L = B.lib()
    a256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    # long-context workload: 16 seqs, 32 heads over 8, d 128, 32768 tokens / 512
    S, H, Hkv, D, P = 16, 32, 8, 128, 64
    counters = a256(4 * max(1 << 18, S * Hkv))
    want = counters + 2 * a256(S * H * P * 4) + a256(S * H * P * D * 4)
    assert L.pa_decode_workspace_bytes(S, H, Hkv, D, 32768, 512) == want
    # a batch whose counters pass the fixed region
    S2, P2 = 40000, 3
    counters2 = a256(4 * S2 * Hkv)
    assert counters2 > 4 << 18
    assert L.pa_decode_workspace_bytes(S2, H, Hkv, D, 3 * 512, 512) == \
        counters2 + 2 * a256(S2 * H * P2 * 4) + a256(S2 * H * P2 * D * 4)
    # prefix-aware decode: the shared prefix and the own tokens each in
    # partitions of P (P = 0: one of each), ceil(max_ctx / P) + 1 partials
    def cascade(S_, mc, P_):
        parts = (-(-mc // P_) if P_ > 0 and mc > 0 else 1) + 1
        return a256(4 * max(1 << 18, S_ * Hkv)) + 2 * a256(S_ * H * parts * 4) + \
            a256(S_ * H * parts * D * 4)
    for S_, mc, P_ in ((256, 2048, 1024), (256, 2048, 0), (6, 328, 0), (6, 328, 64),
                       (16, 32768, 512), (3, 100, 48), (1, 1, 0)):
        assert L.pa_cascade_workspace_bytes(S_, H, Hkv, D, mc, P_) == cascade(S_, mc, P_), \
            (S_, mc, P_)
    # everything fits one partition, or single pass: no workspace
    assert L.pa_decode_workspace_bytes(S, H, Hkv, D, 512, 512) == 0
    assert L.pa_decode_workspace_bytes(S, H, Hkv, D, 32768, 0) == 0
    assert L.pa_decode_workspace_bytes(-1, H, Hkv, D, 32768, 512) == 0


@pytest.mark.parametrize("name,fused", [("tiny", True), ("mha7b", True), ("gqa70b", True),
                                        ("longctx", True), ("prefix", True),
                                        ("prefix-cascade", True), ("gqa70b-fp8", True),
                                        ("prefix-cascade-fp8", True),
                                        ("chunked", False), ("chunked-fp8", False),
                                        ("mixed", False), ("mixed-fp8", False)])
def test_step_takes_the_fused_append(lib, name, fused):
    """Host logic of the step: a decode step whose new tokens are one per
    sequence at its last position (in the same block before and after
    copy-on-write) runs the fused append; prefill steps, a second new token
    or a remapped last block send it back to the separate write."""
    from paged_kv_cache_96_gb300 import step as S
    from paged_kv_cache_96_gb300 import workloads as W
    w = W.build(W.small_variant(name))
    st = S.DecodeStep(w, device="cpu", build_pools=False)
    assert st.fused_append is fused
    n_attn = st.launches_per_step()
    assert n_attn >= (1 if fused else 2)
    if not fused:
        return
    # a step whose new token is not the last position
    w2 = W.build(W.small_variant(name))
    w2.new_pos = w2.new_pos - 1
    assert S.DecodeStep(w2, device="cpu", build_pools=False).fused_append is False
    # a step whose copy-on-write remaps the block holding a new token
    w3 = W.build(W.small_variant(name))
    s0 = 0
    lb = (int(w3.context_lens[s0]) - 1) // w3.bs
    w3.step_block_tables = w3.step_block_tables.copy()
    w3.step_block_tables[s0, lb] = (int(w3.step_block_tables[s0, lb]) + 1) % w3.num_blocks
    assert S.DecodeStep(w3, device="cpu", build_pools=False).fused_append is False


def test_stage_wait_limit_setting(B):
    """The watchdog limit is process-wide, settable, and 0 restores the
    default of one second."""
    default = B.pa_stage_wait_limit_ns()
    assert default == 1_000_000_000
    try:
        B.pa_set_stage_wait_limit_ns(250)
        assert B.pa_stage_wait_limit_ns() == 250
        B.pa_set_stage_wait_limit_ns(0)
        assert B.pa_stage_wait_limit_ns() == default
    finally:
        B.pa_set_stage_wait_limit_ns(0)


def test_noalloc_checks_arguments_before_its_size(B):
    """The allocation-free entry point answers bad arguments as
    pa_decode_attention does, even where their workspace would not fit its
    array; only valid sizes that do not fit are refused for their size."""
    L = B.lib()

    def call(**kw):
        a = dict(out=FAKE, query=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, mb=1 << 14, ctx=FAKE,
                 maxctx=1 << 18, S=64, H=32, Hkv=8, D=128, bs=16, N=1 << 16, scale=0.1, P=16,
                 dt=1)
        a.update(kw)
        return L.pa_decode_attention_noalloc(
            a["out"], a["query"], a["kc"], a["vc"], a["bt"], a["mb"], a["ctx"], a["maxctx"],
            a["S"], a["H"], a["Hkv"], a["D"], a["bs"], a["N"], a["scale"], a["P"], a["dt"],
            None, None)

    need = B.pa_decode_workspace_bytes(64, 32, 8, 128, 1 << 18, 16)
    assert need > B.NOALLOC_WORKSPACE_BYTES
    assert call() == B.PA_ERR_WORKSPACE
    assert call(P=24) == B.PA_ERR_UNSUPPORTED        # not a multiple of 16 tokens
    assert call(D=96) == B.PA_ERR_UNSUPPORTED
    assert call(out=None) == B.PA_ERR_INVALID_ARG
    assert call(query=FAKE_ODD) == B.PA_ERR_INVALID_ARG
    assert call(H=30) == B.PA_ERR_INVALID_ARG         # not a multiple of the KV heads
    assert call(dt=2) == B.PA_ERR_INVALID_ARG
    assert call(S=0) == B.PA_OK

"""ctypes binding of ``libpaged_attention.so`` (the C ABI declared in
``include/paged_attention.h``).

Argument marshalling only: every function takes torch CUDA tensors, checks
their dtype, device and contiguity, and passes raw pointers, sizes and the
current CUDA stream to the library of the same name.  All computation runs
in the library's kernels.  There is no fallback: if the library has not been
built, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.environ.get("PA_LIBRARY",
                           os.path.join(_HERE, "lib", "libpaged_attention.so"))

(PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA,
 PA_ERR_OUT_OF_BLOCKS, PA_ERR_TABLE_FULL) = range(7)
PA_F16, PA_BF16, PA_FP8_E4M3 = 0, 1, 2

DEVERR_SLOT_RANGE = 0x01
DEVERR_BLOCK_RANGE = 0x02
DEVERR_PAIR_RANGE = 0x04
DEVERR_CONTEXT_RANGE = 0x08
DEVERR_TOKEN_RANGE = 0x10
DEVERR_TIMEOUT = 0x20
DEVERR_PREFIX_PLAN = 0x40
DEVERR_QUERY_RANGE = 0x80


class PAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        name = _lib.pa_status_string(status).decode()
        extra = ""
        if status == PA_ERR_CUDA:
            extra = ": " + _lib.pa_last_cuda_error().decode()
        super().__init__(f"{fn} returned {name}{extra}")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def _load() -> ctypes.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"CUDA library {_LIB_PATH} is missing; build it with "
            "`python -m paged_kv_cache_96_gb300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(_LIB_PATH)
    P, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sigs = {
        "pa_slot_mapping": (i32, [P, P, i32, P, P, i32, i32, i32, i32, P, P]),
        "pa_reshape_and_cache": (i32, [P, P, P, P, P, i32, i32, i32, i32, i32, i32, P, P]),
        "pa_copy_blocks": (i32, [P, P, P, i32, i32, i32, i32, i32, i32, P, P]),
        "pa_decode_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32]),
        "pa_decode_attention": (i32, [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32,
                                      i32, i32, f32, i32, P, sz, i32, P, P]),
        "pa_decode_attention_noalloc": (i32, [P, P, P, P, P, i32, P, i32, i32, i32, i32,
                                              i32, i32, i32, f32, i32, i32, P, P]),
        "pa_reshape_and_cache_fp8": (i32, [P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32,
                                           f32, P, P]),
        "pa_slot_mapping_and_cache": (i32, [P, P, i32, P, P, i32, i32, P, P, P, P, i32, i32,
                                            i32, i32, i32, P, P]),
        "pa_slot_mapping_and_cache_fp8": (i32, [P, P, i32, P, P, i32, i32, P, P, P, P, i32,
                                                i32, i32, i32, i32, f32, f32, P, P]),
        "pa_decode_attention_fp8": (i32, [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32,
                                          i32, i32, f32, f32, f32, i32, P, sz, i32, P, P]),
        "pa_decode_attention_append": (i32, [P, P, P, P, P, P, P, P, i32, P, i32, i32, i32,
                                             i32, i32, i32, i32, f32, i32, P, sz, i32, P, P]),
        "pa_decode_attention_append_fp8": (i32, [P, P, P, P, P, P, P, P, i32, P, i32, i32,
                                                 i32, i32, i32, i32, i32, f32, f32, f32, i32,
                                                 P, sz, i32, P, P]),
        "pa_prefill_attention": (i32, [P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32,
                                       i32, i32, i32, f32, i32, P, P]),
        "pa_prefill_attention_fp8": (i32, [P, P, P, P, P, i32, P, P, i32, i32, i32, i32,
                                           i32, i32, i32, i32, f32, f32, f32, i32, P, P]),
        "pa_prefix_plan_ints": (sz, [i32, i32, i32]),
        "pa_plan_prefix_groups": (i32, [P, i32, P, i32, i32, i32, P, sz, P, P]),
        "pa_cascade_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32]),
        "pa_decode_attention_cascade": (i32, [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32,
                                              i32, i32, f32, P, i32, i32, i32, P, sz, i32, P,
                                              P]),
        "pa_decode_attention_cascade_append": (i32, [P, P, P, P, P, P, P, P, i32, P, i32,
                                                     i32, i32, i32, i32, i32, i32, f32, P,
                                                     i32, i32, i32, P, sz, i32, P, P]),
        "pa_decode_attention_cascade_fp8": (i32, [P, P, P, P, P, i32, P, i32, i32, i32, i32,
                                                  i32, i32, i32, f32, f32, f32, P, i32, i32,
                                                  i32, P, sz, i32, P, P]),
        "pa_decode_attention_cascade_append_fp8": (i32, [P, P, P, P, P, P, P, P, i32, P, i32,
                                                         i32, i32, i32, i32, i32, i32, f32,
                                                         f32, f32, P, i32, i32, i32, P, sz,
                                                         i32, P, P]),
        "pa_bm_create": (i32, [i32, i32, i32, P]),
        "pa_bm_destroy": (None, [P]),
        "pa_bm_num_free_blocks": (i32, [P]),
        "pa_bm_add_sequence": (i32, [P, i32]),
        "pa_bm_fork": (i32, [P, i32, i32]),
        "pa_bm_append_tokens": (i32, [P, i32, i32, P, P, i32, P]),
        "pa_bm_append_batch": (i32, [P, P, P, i32, P, P, i32, P]),
        "pa_bm_blocks_needed": (i32, [P, i32, i32]),
        "pa_bm_free_sequence": (i32, [P, i32]),
        "pa_bm_sequence_info": (i32, [P, i32, P, P]),
        "pa_bm_block_table": (i32, [P, i32, P, i32]),
        "pa_bm_ref_count": (i32, [P, i32]),
        "pa_bm_build_batch": (i32, [P, P, i32, P, i32, P, i32]),
        "pa_status_string": (ctypes.c_char_p, [i32]),
        "pa_last_cuda_error": (ctypes.c_char_p, []),
        "pa_version": (i32, []),
        "pa_set_stage_wait_limit_ns": (None, [ctypes.c_uint64]),
        "pa_stage_wait_limit_ns": (ctypes.c_uint64, []),
        "pa_debug_withhold_first_fill": (None, [i32]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def lib() -> ctypes.CDLL:
    """The loaded C library (for callers that pass raw pointers)."""
    return _lib


def pa_set_stage_wait_limit_ns(limit_ns: int) -> None:
    """Process-wide limit of one stage wait in the attention kernels (0: the
    default of one second)."""
    _lib.pa_set_stage_wait_limit_ns(int(limit_ns))


def pa_stage_wait_limit_ns() -> int:
    return int(_lib.pa_stage_wait_limit_ns())


def pa_debug_withhold_first_fill(enable: bool) -> None:
    """Test hook of the time-out path: while enabled, every CTA of each
    attention launch leaves its first K/V fill unissued, so its wait runs out."""
    _lib.pa_debug_withhold_first_fill(1 if enable else 0)


# ---------------------------------------------------------------------------

def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return PA_F16
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype == torch.uint8:
        return PA_FP8_E4M3
    raise TypeError(f"fp16 / bf16 tensor (or uint8 FP8 pool) expected, got {t.dtype}")


def _dev(t: torch.Tensor, name: str, dtype: Optional[torch.dtype] = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: torch.Tensor expected")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: {dtype} expected, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _opt(t: Optional[torch.Tensor], name: str):
    return None if t is None else _dev(t, name, torch.int32)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, status: int) -> None:
    if status != PA_OK:
        raise PAError(fn, status)


def pa_slot_mapping(slot_mapping: torch.Tensor, block_tables: torch.Tensor,
                    token_seq: torch.Tensor, token_pos: torch.Tensor,
                    block_size: int, num_blocks: int,
                    error_word: Optional[torch.Tensor] = None, stream=None) -> None:
    """slot_mapping[t] = block_tables[s][p // bs] * bs + p % bs (int32)."""
    S, MB = block_tables.shape
    T = token_seq.shape[0]
    _check("pa_slot_mapping", _lib.pa_slot_mapping(
        _dev(slot_mapping, "slot_mapping", torch.int32),
        _dev(block_tables, "block_tables", torch.int32), MB,
        _dev(token_seq, "token_seq", torch.int32),
        _dev(token_pos, "token_pos", torch.int32), T, S, block_size, num_blocks,
        _opt(error_word, "error_word"), _stream(stream)))


def pa_reshape_and_cache(key: torch.Tensor, value: torch.Tensor,
                         key_cache: torch.Tensor, value_cache: torch.Tensor,
                         slot_mapping: torch.Tensor,
                         error_word: Optional[torch.Tensor] = None,
                         stream=None) -> None:
    """Write key/value [T, Hkv, d] into the pools [N, bs, Hkv, d] at their slots."""
    T, Hkv, d = key.shape
    N, bs, Hkv2, d2 = key_cache.shape
    if (Hkv, d) != (Hkv2, d2) or value.shape != key.shape or value_cache.shape != key_cache.shape:
        raise ValueError("shape mismatch between new tokens and pools")
    dt = _dtype_code(key_cache)
    _check("pa_reshape_and_cache", _lib.pa_reshape_and_cache(
        _dev(key, "key", key_cache.dtype), _dev(value, "value", key_cache.dtype),
        _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache", key_cache.dtype),
        _dev(slot_mapping, "slot_mapping", torch.int32), T, N, bs, Hkv, d, dt,
        _opt(error_word, "error_word"), _stream(stream)))


def pa_slot_mapping_and_cache(slot_mapping: torch.Tensor, block_tables: torch.Tensor,
                              token_seq: torch.Tensor, token_pos: torch.Tensor,
                              key: torch.Tensor, value: torch.Tensor,
                              key_cache: torch.Tensor, value_cache: torch.Tensor,
                              k_scale: float = 1.0, v_scale: float = 1.0,
                              error_word: Optional[torch.Tensor] = None,
                              stream=None) -> None:
    """pa_slot_mapping and the cache write in one launch: slot_mapping gets
    the slots, the pools the new tokens' K/V (e4m3 codes with the scales when
    the pools are uint8)."""
    S, MB = block_tables.shape
    T, Hkv, d = key.shape
    N, bs, Hkv2, d2 = key_cache.shape
    if (Hkv, d) != (Hkv2, d2) or value.shape != key.shape or value_cache.shape != key_cache.shape:
        raise ValueError("shape mismatch between new tokens and pools")
    if token_seq.shape[0] != T or token_pos.shape[0] != T or slot_mapping.shape[0] != T:
        raise ValueError("one sequence id, position and slot per new token expected")
    head = (_dev(slot_mapping, "slot_mapping", torch.int32),
            _dev(block_tables, "block_tables", torch.int32), MB,
            _dev(token_seq, "token_seq", torch.int32), _dev(token_pos, "token_pos", torch.int32),
            T, S)
    if key_cache.dtype == torch.uint8:
        _check("pa_slot_mapping_and_cache_fp8", _lib.pa_slot_mapping_and_cache_fp8(
            *head, _dev(key, "key"), _dev(value, "value", key.dtype),
            _dev(key_cache, "key_cache", torch.uint8),
            _dev(value_cache, "value_cache", torch.uint8), N, bs, Hkv, d, _dtype_code(key),
            float(k_scale), float(v_scale), _opt(error_word, "error_word"), _stream(stream)))
        return
    _check("pa_slot_mapping_and_cache", _lib.pa_slot_mapping_and_cache(
        *head, _dev(key, "key", key_cache.dtype), _dev(value, "value", key_cache.dtype),
        _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache", key_cache.dtype),
        N, bs, Hkv, d, _dtype_code(key_cache), _opt(error_word, "error_word"),
        _stream(stream)))


def pa_copy_blocks(key_cache: torch.Tensor, value_cache: torch.Tensor,
                   block_mapping: torch.Tensor,
                   error_word: Optional[torch.Tensor] = None, stream=None) -> None:
    """For each (src, dst) row of block_mapping [P, 2]: block dst := block src."""
    N, bs, Hkv, d = key_cache.shape
    P = block_mapping.shape[0]
    _check("pa_copy_blocks", _lib.pa_copy_blocks(
        _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache", key_cache.dtype),
        _dev(block_mapping, "block_mapping", torch.int32), P, N, bs, Hkv, d,
        _dtype_code(key_cache), _opt(error_word, "error_word"), _stream(stream)))


def pa_decode_workspace_bytes(num_seqs: int, num_heads: int, num_kv_heads: int,
                              head_dim: int, max_context_len: int,
                              partition_size: int) -> int:
    return int(_lib.pa_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads,
                                              head_dim, max_context_len, partition_size))


def pa_decode_attention(out: torch.Tensor, query: torch.Tensor,
                        key_cache: torch.Tensor, value_cache: torch.Tensor,
                        block_tables: torch.Tensor, context_lens: torch.Tensor,
                        max_context_len: int, scale: float, partition_size: int = 0,
                        workspace: Optional[torch.Tensor] = None,
                        error_word: Optional[torch.Tensor] = None,
                        stream=None) -> None:
    """Paged decode attention; out and query are [S, H, d]."""
    S, H, d = query.shape
    N, bs, Hkv, d2 = key_cache.shape
    MB = block_tables.shape[1]
    if d != d2 or out.shape != query.shape:
        raise ValueError("shape mismatch")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr = _dev(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    if key_cache.dtype == torch.uint8:
        raise TypeError("FP8 pools: use pa_decode_attention_fp8")
    _check("pa_decode_attention", _lib.pa_decode_attention(
        _dev(out, "out", query.dtype), _dev(query, "query", key_cache.dtype),
        _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache", key_cache.dtype),
        _dev(block_tables, "block_tables", torch.int32), MB,
        _dev(context_lens, "context_lens", torch.int32), int(max_context_len), S, H, Hkv,
        d, bs, N, float(scale), int(partition_size), ws_ptr, ws_bytes,
        _dtype_code(key_cache), _opt(error_word, "error_word"), _stream(stream)))


def pa_decode_attention_noalloc(out: torch.Tensor, query: torch.Tensor,
                                key_cache: torch.Tensor, value_cache: torch.Tensor,
                                block_tables: torch.Tensor, context_lens: torch.Tensor,
                                max_context_len: int, scale: float, partition_size: int = 0,
                                error_word: Optional[torch.Tensor] = None,
                                stream=None) -> None:
    """As pa_decode_attention, with the library's static device workspace
    (for callers that cannot allocate one)."""
    S, H, d = query.shape
    N, bs, Hkv, d2 = key_cache.shape
    MB = block_tables.shape[1]
    if d != d2 or out.shape != query.shape:
        raise ValueError("shape mismatch")
    _check("pa_decode_attention_noalloc", _lib.pa_decode_attention_noalloc(
        _dev(out, "out", query.dtype), _dev(query, "query", key_cache.dtype),
        _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache", key_cache.dtype),
        _dev(block_tables, "block_tables", torch.int32), MB,
        _dev(context_lens, "context_lens", torch.int32), int(max_context_len), S, H, Hkv,
        d, bs, N, float(scale), int(partition_size), _dtype_code(key_cache),
        _opt(error_word, "error_word"), _stream(stream)))


NOALLOC_WORKSPACE_BYTES = 32 * 1024 * 1024


def pa_reshape_and_cache_fp8(key: torch.Tensor, value: torch.Tensor,
                             key_cache: torch.Tensor, value_cache: torch.Tensor,
                             slot_mapping: torch.Tensor, k_scale: float, v_scale: float,
                             error_word: Optional[torch.Tensor] = None,
                             stream=None) -> None:
    """Quantise key/value [T, Hkv, d] (fp16/bf16) into uint8 e4m3 pools."""
    T, Hkv, d = key.shape
    N, bs, Hkv2, d2 = key_cache.shape
    if (Hkv, d) != (Hkv2, d2) or value.shape != key.shape or value_cache.shape != key_cache.shape:
        raise ValueError("shape mismatch between new tokens and pools")
    _check("pa_reshape_and_cache_fp8", _lib.pa_reshape_and_cache_fp8(
        _dev(key, "key"), _dev(value, "value", key.dtype),
        _dev(key_cache, "key_cache", torch.uint8), _dev(value_cache, "value_cache", torch.uint8),
        _dev(slot_mapping, "slot_mapping", torch.int32), T, N, bs, Hkv, d, _dtype_code(key),
        float(k_scale), float(v_scale), _opt(error_word, "error_word"), _stream(stream)))


def pa_decode_attention_fp8(out: torch.Tensor, query: torch.Tensor,
                            key_cache: torch.Tensor, value_cache: torch.Tensor,
                            block_tables: torch.Tensor, context_lens: torch.Tensor,
                            max_context_len: int, scale: float, k_scale: float,
                            v_scale: float, partition_size: int = 0,
                            workspace: Optional[torch.Tensor] = None,
                            error_word: Optional[torch.Tensor] = None,
                            stream=None) -> None:
    """Paged decode attention over uint8 e4m3 pools."""
    S, H, d = query.shape
    N, bs, Hkv, d2 = key_cache.shape
    MB = block_tables.shape[1]
    if d != d2 or out.shape != query.shape:
        raise ValueError("shape mismatch")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr = _dev(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    _check("pa_decode_attention_fp8", _lib.pa_decode_attention_fp8(
        _dev(out, "out", query.dtype), _dev(query, "query"),
        _dev(key_cache, "key_cache", torch.uint8), _dev(value_cache, "value_cache", torch.uint8),
        _dev(block_tables, "block_tables", torch.int32), MB,
        _dev(context_lens, "context_lens", torch.int32), int(max_context_len), S, H, Hkv,
        d, bs, N, float(scale), float(k_scale), float(v_scale), int(partition_size),
        ws_ptr, ws_bytes, _dtype_code(query), _opt(error_word, "error_word"),
        _stream(stream)))


def pa_decode_attention_append(out: torch.Tensor, query: torch.Tensor,
                               key_cache: torch.Tensor, value_cache: torch.Tensor,
                               new_key: torch.Tensor, new_value: torch.Tensor,
                               block_tables: torch.Tensor, context_lens: torch.Tensor,
                               max_context_len: int, scale: float, partition_size: int = 0,
                               workspace: Optional[torch.Tensor] = None,
                               slot_mapping: Optional[torch.Tensor] = None,
                               k_scale: float = 1.0, v_scale: float = 1.0,
                               error_word: Optional[torch.Tensor] = None,
                               stream=None) -> None:
    """One decode step in one call: each sequence's new token (new_key /
    new_value [S, Hkv, d], at position context_lens[s] - 1) is written to the
    pools, then attention runs over the whole context.  uint8 pools take the
    e4m3 path with k_scale / v_scale."""
    S, H, d = query.shape
    N, bs, Hkv, d2 = key_cache.shape
    MB = block_tables.shape[1]
    if d != d2 or out.shape != query.shape:
        raise ValueError("shape mismatch")
    if new_key.shape != (S, Hkv, d) or new_value.shape != new_key.shape:
        raise ValueError("new_key / new_value must be [num_seqs, num_kv_heads, head_dim]")
    if slot_mapping is not None and slot_mapping.shape[0] != S:
        raise ValueError("one slot per sequence expected")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr = _dev(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    fp8 = key_cache.dtype == torch.uint8
    head = (_dev(out, "out", query.dtype), _dev(query, "query"),
            _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache", key_cache.dtype),
            _dev(new_key, "new_key", query.dtype), _dev(new_value, "new_value", query.dtype),
            _opt(slot_mapping, "slot_mapping"),
            _dev(block_tables, "block_tables", torch.int32), MB,
            _dev(context_lens, "context_lens", torch.int32), int(max_context_len), S, H, Hkv,
            d, bs, N, float(scale))
    if fp8:
        _check("pa_decode_attention_append_fp8", _lib.pa_decode_attention_append_fp8(
            *head, float(k_scale), float(v_scale), int(partition_size), ws_ptr, ws_bytes,
            _dtype_code(query), _opt(error_word, "error_word"), _stream(stream)))
        return
    if query.dtype != key_cache.dtype:
        raise TypeError("query and pools must share one 16-bit type")
    _check("pa_decode_attention_append", _lib.pa_decode_attention_append(
        *head, int(partition_size), ws_ptr, ws_bytes, _dtype_code(key_cache),
        _opt(error_word, "error_word"), _stream(stream)))


def alloc_workspace(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                    max_context_len: int, partition_size: int,
                    device="cuda") -> Optional[torch.Tensor]:
    """Zero-initialised workspace for pa_decode_attention (None if not needed)."""
    n = pa_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim,
                                  max_context_len, partition_size)
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=device)


def pa_prefill_attention(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                         value_cache: torch.Tensor, block_tables: torch.Tensor,
                         query_start: torch.Tensor, context_lens: torch.Tensor,
                         max_context_len: int, scale: float,
                         error_word: Optional[torch.Tensor] = None, stream=None,
                         k_scale: float = 1.0, v_scale: float = 1.0) -> None:
    """Chunked prefill / mixed batch: out and query are [T, H, d]; sequence s
    owns rows [query_start[s], query_start[s+1]), its newest tokens.  uint8
    pools take the e4m3 path (pa_prefill_attention_fp8) with k_scale /
    v_scale."""
    T, H, d = query.shape
    N, bs, Hkv, d2 = key_cache.shape
    MB = block_tables.shape[1]
    S = context_lens.shape[0]
    if d != d2 or out.shape != query.shape or query_start.shape[0] != S + 1:
        raise ValueError("shape mismatch")
    fp8 = key_cache.dtype == torch.uint8
    if not fp8 and query.dtype != key_cache.dtype:
        raise TypeError("query and pools must share one 16-bit type")
    head = (_dev(out, "out", query.dtype), _dev(query, "query"),
            _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache", key_cache.dtype),
            _dev(block_tables, "block_tables", torch.int32), MB,
            _dev(query_start, "query_start", torch.int32),
            _dev(context_lens, "context_lens", torch.int32), int(max_context_len), S, T, H,
            Hkv, d, bs, N, float(scale))
    if fp8:
        _check("pa_prefill_attention_fp8", _lib.pa_prefill_attention_fp8(
            *head, float(k_scale), float(v_scale), _dtype_code(query),
            _opt(error_word, "error_word"), _stream(stream)))
        return
    _check("pa_prefill_attention", _lib.pa_prefill_attention(
        *head, _dtype_code(key_cache), _opt(error_word, "error_word"), _stream(stream)))


def pa_plan_prefix_groups(block_tables, context_lens, block_size: int,
                          min_shared_blocks: int = 1):
    """Host planner of prefix-aware decode on host (numpy-convertible) int32
    block tables [S, MB] and context lengths [S].  Returns (plan, num_groups,
    num_members); plan is an int32 CPU tensor in the layout the cascade
    decode takes (copy it to the device)."""
    import numpy as np
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    cl = np.ascontiguousarray(np.asarray(context_lens, dtype=np.int32))
    S, MB = bt.shape
    cap = 3 * S + 1
    plan = np.zeros(max(cap, 1), dtype=np.int32)
    ng, nm = ctypes.c_int(0), ctypes.c_int(0)
    _check("pa_plan_prefix_groups", _lib.pa_plan_prefix_groups(
        bt.ctypes.data_as(ctypes.c_void_p), MB, cl.ctypes.data_as(ctypes.c_void_p), S,
        int(block_size), int(min_shared_blocks), plan.ctypes.data_as(ctypes.c_void_p), cap,
        ctypes.byref(ng), ctypes.byref(nm)))
    n = int(_lib.pa_prefix_plan_ints(S, ng.value, nm.value))
    return torch.from_numpy(plan[:n].copy()), ng.value, nm.value


def pa_cascade_workspace_bytes(num_seqs: int, num_heads: int, num_kv_heads: int,
                               head_dim: int, max_context_len: int,
                               partition_size: int) -> int:
    return int(_lib.pa_cascade_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim,
                                               max_context_len, partition_size))


def pa_decode_attention_cascade(out: torch.Tensor, query: torch.Tensor,
                                key_cache: torch.Tensor, value_cache: torch.Tensor,
                                block_tables: torch.Tensor, context_lens: torch.Tensor,
                                max_context_len: int, scale: float, prefix_plan: torch.Tensor,
                                num_groups: int, num_members: int, partition_size: int,
                                workspace: torch.Tensor,
                                error_word: Optional[torch.Tensor] = None,
                                stream=None, k_scale: float = 1.0,
                                v_scale: float = 1.0) -> None:
    """Prefix-aware decode: pa_decode_attention's result with each planned
    group's shared prefix read once (prefix_plan on the device).  uint8
    pools take the e4m3 path with k_scale / v_scale."""
    S, H, d = query.shape
    N, bs, Hkv, d2 = key_cache.shape
    MB = block_tables.shape[1]
    if d != d2 or out.shape != query.shape:
        raise ValueError("shape mismatch")
    fp8 = key_cache.dtype == torch.uint8
    if not fp8 and query.dtype != key_cache.dtype:
        raise TypeError("query and pools must share one 16-bit type")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr = _dev(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    head = (_dev(out, "out", query.dtype), _dev(query, "query"),
            _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache", key_cache.dtype),
            _dev(block_tables, "block_tables", torch.int32), MB,
            _dev(context_lens, "context_lens", torch.int32), int(max_context_len), S, H, Hkv,
            d, bs, N, float(scale))
    tail = (_dev(prefix_plan, "prefix_plan", torch.int32), int(num_groups),
            int(num_members), int(partition_size), ws_ptr, ws_bytes, _dtype_code(query),
            _opt(error_word, "error_word"), _stream(stream))
    if fp8:
        _check("pa_decode_attention_cascade_fp8", _lib.pa_decode_attention_cascade_fp8(
            *head, float(k_scale), float(v_scale), *tail))
        return
    _check("pa_decode_attention_cascade", _lib.pa_decode_attention_cascade(*head, *tail))


def pa_decode_attention_cascade_append(out: torch.Tensor, query: torch.Tensor,
                                       key_cache: torch.Tensor, value_cache: torch.Tensor,
                                       new_key: torch.Tensor, new_value: torch.Tensor,
                                       block_tables: torch.Tensor, context_lens: torch.Tensor,
                                       max_context_len: int, scale: float,
                                       prefix_plan: torch.Tensor, num_groups: int,
                                       num_members: int, partition_size: int,
                                       workspace: torch.Tensor,
                                       slot_mapping: Optional[torch.Tensor] = None,
                                       error_word: Optional[torch.Tensor] = None,
                                       stream=None, k_scale: float = 1.0,
                                       v_scale: float = 1.0) -> None:
    """Prefix-aware decode step in one call: each sequence's new token
    (new_key / new_value [S, Hkv, d], position context_lens[s] - 1) written
    to the pools and attended, each planned group's shared prefix read once.
    uint8 pools take the e4m3 path with k_scale / v_scale."""
    S, H, d = query.shape
    N, bs, Hkv, d2 = key_cache.shape
    MB = block_tables.shape[1]
    if d != d2 or out.shape != query.shape:
        raise ValueError("shape mismatch")
    if new_key.shape != (S, Hkv, d) or new_value.shape != new_key.shape:
        raise ValueError("new_key / new_value must be [num_seqs, num_kv_heads, head_dim]")
    if slot_mapping is not None and slot_mapping.shape[0] != S:
        raise ValueError("one slot per sequence expected")
    fp8 = key_cache.dtype == torch.uint8
    if not fp8 and query.dtype != key_cache.dtype:
        raise TypeError("query and pools must share one 16-bit type")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr = _dev(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    head = (_dev(out, "out", query.dtype), _dev(query, "query"),
            _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache", key_cache.dtype),
            _dev(new_key, "new_key", query.dtype), _dev(new_value, "new_value", query.dtype),
            _opt(slot_mapping, "slot_mapping"), _dev(block_tables, "block_tables", torch.int32),
            MB, _dev(context_lens, "context_lens", torch.int32), int(max_context_len), S, H,
            Hkv, d, bs, N, float(scale))
    tail = (_dev(prefix_plan, "prefix_plan", torch.int32), int(num_groups),
            int(num_members), int(partition_size), ws_ptr, ws_bytes, _dtype_code(query),
            _opt(error_word, "error_word"), _stream(stream))
    if fp8:
        _check("pa_decode_attention_cascade_append_fp8",
               _lib.pa_decode_attention_cascade_append_fp8(*head, float(k_scale),
                                                           float(v_scale), *tail))
        return
    _check("pa_decode_attention_cascade_append",
           _lib.pa_decode_attention_cascade_append(*head, *tail))


class BlockManager:
    """The library's host block manager (C++): block tables, reference
    counts, copy-on-write decisions and slot mapping for a pool of
    num_blocks blocks of block_size tokens.  Host memory only."""

    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int):
        self._h = ctypes.c_void_p()
        _check("pa_bm_create", _lib.pa_bm_create(num_blocks, block_size, max_blocks_per_seq,
                                                 ctypes.byref(self._h)))
        self.num_blocks, self.block_size = num_blocks, block_size
        self.max_blocks_per_seq = max_blocks_per_seq

    def close(self):
        if self._h:
            _lib.pa_bm_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free(self) -> int:
        return int(_lib.pa_bm_num_free_blocks(self._h))

    def add_sequence(self, seq: int) -> None:
        _check("pa_bm_add_sequence", _lib.pa_bm_add_sequence(self._h, int(seq)))

    def fork(self, parent: int, child: int) -> None:
        _check("pa_bm_fork", _lib.pa_bm_fork(self._h, int(parent), int(child)))

    def blocks_needed(self, seq: int, n: int) -> int:
        return int(_lib.pa_bm_blocks_needed(self._h, int(seq), int(n)))

    def append_tokens(self, seq: int, n: int):
        """(slots int32 array [n], copy-on-write pairs [(src, dst)])."""
        import numpy as np
        slots = np.zeros(max(n, 1), dtype=np.int32)
        pairs = np.zeros(2, dtype=np.int32)
        ncow = ctypes.c_int(0)
        _check("pa_bm_append_tokens", _lib.pa_bm_append_tokens(
            self._h, int(seq), int(n), slots.ctypes.data_as(ctypes.c_void_p),
            pairs.ctypes.data_as(ctypes.c_void_p), 1, ctypes.byref(ncow)))
        return slots[:n], [(int(pairs[0]), int(pairs[1]))] if ncow.value else []

    def append_batch(self, seqs, counts):
        """One step's appends in one call: (slots int32 array in batch order,
        copy-on-write pairs [(src, dst)])."""
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
        cnt = np.ascontiguousarray(np.asarray(counts, dtype=np.int32))
        total = int(cnt.sum()) if cnt.size else 0
        slots = np.zeros(max(total, 1), dtype=np.int32)
        cap = max(ids.shape[0], 1)
        pairs = np.zeros(2 * cap, dtype=np.int32)
        ncow = ctypes.c_int(0)
        _check("pa_bm_append_batch", _lib.pa_bm_append_batch(
            self._h, ids.ctypes.data_as(ctypes.c_void_p), cnt.ctypes.data_as(ctypes.c_void_p),
            ids.shape[0], slots.ctypes.data_as(ctypes.c_void_p),
            pairs.ctypes.data_as(ctypes.c_void_p), cap, ctypes.byref(ncow)))
        return slots[:total], [(int(pairs[2 * i]), int(pairs[2 * i + 1]))
                               for i in range(ncow.value)]

    def free_sequence(self, seq: int) -> None:
        _check("pa_bm_free_sequence", _lib.pa_bm_free_sequence(self._h, int(seq)))

    def length(self, seq: int) -> int:
        t, b = ctypes.c_int(0), ctypes.c_int(0)
        _check("pa_bm_sequence_info", _lib.pa_bm_sequence_info(self._h, int(seq),
                                                               ctypes.byref(t), ctypes.byref(b)))
        return t.value

    def table(self, seq: int):
        import numpy as np
        t, b = ctypes.c_int(0), ctypes.c_int(0)
        _check("pa_bm_sequence_info", _lib.pa_bm_sequence_info(self._h, int(seq),
                                                               ctypes.byref(t), ctypes.byref(b)))
        row = np.zeros(max(b.value, 1), dtype=np.int32)
        _check("pa_bm_block_table", _lib.pa_bm_block_table(
            self._h, int(seq), row.ctypes.data_as(ctypes.c_void_p), b.value))
        return row[:b.value].tolist()

    def ref(self, block: int) -> int:
        return int(_lib.pa_bm_ref_count(self._h, int(block)))

    def build_batch(self, seqs, max_blocks: int, pad_block: int):
        """(block_tables int32 [n, max_blocks], context_lens int32 [n])."""
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
        n = ids.shape[0]
        tables = np.zeros((max(n, 1), max_blocks), dtype=np.int32)
        lens = np.zeros(max(n, 1), dtype=np.int32)
        _check("pa_bm_build_batch", _lib.pa_bm_build_batch(
            self._h, ids.ctypes.data_as(ctypes.c_void_p), n,
            tables.ctypes.data_as(ctypes.c_void_p), max_blocks,
            lens.ctypes.data_as(ctypes.c_void_p), int(pad_block)))
        return tables[:n], lens[:n]


"""CPU oracle for the paged KV-cache decode path -- TEST INFRASTRUCTURE ONLY.

This package wraps ``pa_oracle.c`` (plain single-threaded C, fp64
arithmetic) with ctypes and numpy.  Only the tests, the package smoke check
and the benchmark's CPU-baseline leg may import it.  The CUDA product path
never does, and nothing here imports the product package.

Every function states the page passage it restates; the C source carries the
full citations and the readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

F16 = 0
BF16 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpa_oracle.so")
_lock = threading.Lock()
_lib = None


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle C source into a shared library with gcc.

    Plain ``-O2``: no fast-math, no contraction of a*b+c into fused
    multiply-adds, so every double operation rounds as written.
    """
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _needs_build() -> bool:
    return (not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load (building first if stale) the oracle library.

    ``path`` loads another build of the oracle (used by the mutation tests,
    which compile deliberately broken copies of the source).
    """
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _needs_build():
                compile_oracle()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    sig = {
        "oracle_decode": (None, [P, P, i64, i32]),
        "oracle_slot_for_position": (i64, [P, i64, i32]),
        "oracle_slot_mapping": (None, [P, P, i32, P, P, i32, i32]),
        "oracle_reshape_and_cache": (None, [P, P, P, P, P, i32, i32, i32, i32]),
        "oracle_copy_blocks": (None, [P, P, P, i32, i32, i32, i32]),
        "oracle_paged_attention": (None, [P, P, P, P, P, i32, P, i32, i32, i32,
                                          i32, i32, dbl, i32, P, i32]),
        "oracle_attention_weights": (None, [P, P, P, P, i32, P, i32, i32, i32,
                                            i32, i32, i32, dbl, i32]),
        "oracle_num_partitions": (i32, [i64, i32]),
        "oracle_partition_pass": (None, [P, P, P, P, P, P, P, i32, P, i32, i32,
                                         i32, i32, i32, dbl, i32, i32, i32, P,
                                         i32]),
        "oracle_partition_merge": (None, [P, P, P, P, P, i32, i32, i32, i32]),
        "oracle_decode_e4m3": (None, [P, P, i64]),
        "oracle_quantize_e4m3": (None, [P, P, i64, i32, ctypes.c_float]),
        "oracle_reshape_and_cache_fp8": (None, [P, P, P, P, P, i32, i32, i32, i32, i32,
                                                ctypes.c_float, ctypes.c_float]),
        "oracle_paged_attention_fp8": (None, [P, P, P, P, P, i32, P, i32, i32, i32, i32,
                                              i32, dbl, i32, dbl, dbl, P, i32]),
        "oracle_copy_blocks_u8": (None, [P, P, P, i32, i32, i32, i32]),
        "oracle_prefill_attention_fp8": (None, [P, P, P, P, P, i32, P, P, i32, i32, i32,
                                                i32, i32, dbl, i32, dbl, dbl]),
        "oracle_prefill_attention": (None, [P, P, P, P, P, i32, P, P, i32, i32, i32,
                                            i32, i32, dbl, i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype in (np.uint16, np.int16), a.dtype
    return a.view(np.uint16)


def _inplace_u16(a: np.ndarray) -> np.ndarray:
    """A uint16 view of an array the oracle writes in place."""
    if not (isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"]
            and a.dtype in (np.uint16, np.int16)):
        raise TypeError("pools written in place must be C-contiguous 16-bit arrays")
    return a.view(np.uint16)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


# ---------------------------------------------------------------------------
# Element decoding

def decode(bits: np.ndarray, dtype: int, lib=None) -> np.ndarray:
    """Exact fp16 / bf16 bit patterns -> float64 (same shape)."""
    lib = lib or load()
    b = _u16(bits)
    out = np.empty(b.shape, dtype=np.float64)
    lib.oracle_decode(_ptr(out), _ptr(b), b.size, dtype)
    return out


# ---------------------------------------------------------------------------
# Slot mapping -- "PagedAttention & Continuous Batching" §1.5

def slot_for_position(block_table_row: Sequence[int], position: int,
                      block_size: int, lib=None) -> int:
    lib = lib or load()
    row = _i32(block_table_row)
    return int(lib.oracle_slot_for_position(_ptr(row), position, block_size))


def slot_mapping(block_tables: np.ndarray, token_seq: np.ndarray,
                 token_pos: np.ndarray, block_size: int, lib=None) -> np.ndarray:
    """Slots (int64) of tokens (token_seq[t], token_pos[t])."""
    lib = lib or load()
    bt = _i32(block_tables)
    ts, tp = _i32(token_seq), _i32(token_pos)
    out = np.empty(ts.shape[0], dtype=np.int64)
    lib.oracle_slot_mapping(_ptr(out), _ptr(bt), bt.shape[1], _ptr(ts), _ptr(tp),
                            ts.shape[0], block_size)
    return out


# ---------------------------------------------------------------------------
# reshape_and_cache -- §1.5 of the same page; "Block Table 实现" (feifeigd)

def reshape_and_cache(key: np.ndarray, value: np.ndarray, key_cache: np.ndarray,
                      value_cache: np.ndarray, slots: np.ndarray,
                      lib=None) -> None:
    """In place: write key/value [T, Hkv, d] rows into the pools
    [N, bs, Hkv, d] at their slots; negative slots are skipped."""
    lib = lib or load()
    k, v = _u16(key), _u16(value)
    kc, vc = _inplace_u16(key_cache), _inplace_u16(value_cache)
    sl = np.ascontiguousarray(slots, dtype=np.int64)
    T, Hkv, d = k.shape
    bs = kc.shape[1]
    lib.oracle_reshape_and_cache(_ptr(k), _ptr(v), _ptr(kc), _ptr(vc), _ptr(sl),
                                 T, Hkv, d, bs)


# ---------------------------------------------------------------------------
# copy_blocks -- "vLLM源码解析(二)" §3.2 copy-on-write

def copy_blocks(key_cache: np.ndarray, value_cache: np.ndarray,
                block_mapping: np.ndarray, lib=None) -> None:
    """In place: for each (src, dst) pair in order, block dst := block src."""
    lib = lib or load()
    kc, vc = _inplace_u16(key_cache), _inplace_u16(value_cache)
    bm = _i32(block_mapping).reshape(-1, 2)
    N, bs, Hkv, d = kc.shape
    lib.oracle_copy_blocks(_ptr(kc), _ptr(vc), _ptr(bm), bm.shape[0], bs, Hkv, d)


# ---------------------------------------------------------------------------
# Paged decode attention -- "PagedAttention & Continuous Batching" §1.6

def paged_attention(query: np.ndarray, key_cache: np.ndarray,
                    value_cache: np.ndarray, block_tables: np.ndarray,
                    context_lens: np.ndarray, scale: float, dtype: int,
                    seqs: Optional[Sequence[int]] = None,
                    lib=None) -> np.ndarray:
    """fp64 output [S, H, d].  With ``seqs`` only those rows are computed
    (the others are NaN)."""
    lib = lib or load()
    q = _u16(query)
    kc, vc = _u16(key_cache), _u16(value_cache)
    bt, cl = _i32(block_tables), _i32(context_lens)
    S, H, d = q.shape
    N, bs, Hkv, d2 = kc.shape
    assert d == d2 and H % Hkv == 0
    out = np.full((S, H, d), np.nan, dtype=np.float64)
    sub = None if seqs is None else _i32(list(seqs))
    lib.oracle_paged_attention(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt),
                               bt.shape[1], _ptr(cl), S, H, Hkv, d, bs,
                               float(scale), dtype, _ptr(sub),
                               0 if sub is None else sub.shape[0])
    return out


def prefill_attention(query: np.ndarray, key_cache: np.ndarray,
                      value_cache: np.ndarray, block_tables: np.ndarray,
                      query_start: np.ndarray, context_lens: np.ndarray,
                      scale: float, dtype: int, lib=None) -> np.ndarray:
    """Chunked prefill / mixed batch: fp64 output [T, H, d] for the query rows
    [T, H, d]; sequence s owns rows [query_start[s], query_start[s+1]), the
    newest tokens of its context, each attending its own position and the
    earlier ones."""
    lib = lib or load()
    q = _u16(query)
    kc, vc = _u16(key_cache), _u16(value_cache)
    bt, qs, cl = _i32(block_tables), _i32(query_start), _i32(context_lens)
    T, H, d = q.shape
    N, bs, Hkv, d2 = kc.shape
    S = cl.shape[0]
    assert d == d2 and H % Hkv == 0 and qs.shape[0] == S + 1 and int(qs[-1]) == T
    out = np.full((T, H, d), np.nan, dtype=np.float64)
    lib.oracle_prefill_attention(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt),
                                 bt.shape[1], _ptr(qs), _ptr(cl), S, H, Hkv, d, bs,
                                 float(scale), dtype)
    return out


def attention_weights(query: np.ndarray, key_cache: np.ndarray,
                      block_tables: np.ndarray, context_lens: np.ndarray,
                      seq: int, head: int, scale: float, dtype: int,
                      lib=None) -> np.ndarray:
    """Softmax weights [context_lens[seq]] of one (sequence, head)."""
    lib = lib or load()
    q = _u16(query)
    kc = _u16(key_cache)
    bt, cl = _i32(block_tables), _i32(context_lens)
    S, H, d = q.shape
    N, bs, Hkv, _ = kc.shape
    w = np.zeros(max(int(cl[seq]), 1), dtype=np.float64)
    lib.oracle_attention_weights(_ptr(w), _ptr(q), _ptr(kc), _ptr(bt), bt.shape[1],
                                 _ptr(cl), seq, head, H, Hkv, d, bs, float(scale),
                                 dtype)
    return w[: int(cl[seq])]


def num_partitions(context_len: int, partition_size: int, lib=None) -> int:
    lib = lib or load()
    return int(lib.oracle_num_partitions(int(context_len), int(partition_size)))


def partition_pass(query: np.ndarray, key_cache: np.ndarray,
                   value_cache: np.ndarray, block_tables: np.ndarray,
                   context_lens: np.ndarray, scale: float, dtype: int,
                   partition_size: int, max_partitions: int,
                   seqs: Optional[Sequence[int]] = None, lib=None):
    """Split-context partials: (m [S,H,P], l [S,H,P], o [S,H,P,d]) in fp64;
    entries past a sequence's partition count are NaN."""
    lib = lib or load()
    q = _u16(query)
    kc, vc = _u16(key_cache), _u16(value_cache)
    bt, cl = _i32(block_tables), _i32(context_lens)
    S, H, d = q.shape
    N, bs, Hkv, _ = kc.shape
    m = np.full((S, H, max_partitions), np.nan)
    l = np.full((S, H, max_partitions), np.nan)
    o = np.full((S, H, max_partitions, d), np.nan)
    sub = None if seqs is None else _i32(list(seqs))
    lib.oracle_partition_pass(_ptr(m), _ptr(l), _ptr(o), _ptr(q), _ptr(kc), _ptr(vc),
                              _ptr(bt), bt.shape[1], _ptr(cl), S, H, Hkv, d, bs,
                              float(scale), dtype, partition_size, max_partitions,
                              _ptr(sub), 0 if sub is None else sub.shape[0])
    return m, l, o


def partition_merge(m: np.ndarray, l: np.ndarray, o: np.ndarray,
                    nparts: np.ndarray, lib=None) -> np.ndarray:
    """Log-sum-exp merge of partials -> fp64 output [S, H, d]."""
    lib = lib or load()
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    o = np.ascontiguousarray(o, dtype=np.float64)
    npart = _i32(nparts)
    S, H, P, d = o.shape
    out = np.empty((S, H, d), dtype=np.float64)
    lib.oracle_partition_merge(_ptr(out), _ptr(m), _ptr(l), _ptr(o), _ptr(npart),
                               S, H, d, P)
    return out


# ---------------------------------------------------------------------------
# FP8 (e4m3) KV cache -- the "--kv-cache-dtype fp8" option of "vLLM 架构详解"
# (deployment flags); format and rounding readings are in pa_oracle.c.

def decode_e4m3(codes: np.ndarray, lib=None) -> np.ndarray:
    """e4m3 codes (uint8) -> exact float64 values."""
    lib = lib or load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib.oracle_decode_e4m3(_ptr(out), _ptr(c), c.size)
    return out


def quantize_e4m3(x_bits: np.ndarray, dtype: int, inv_scale: float, lib=None) -> np.ndarray:
    """16-bit values -> e4m3 codes of float(x) * inv_scale (fp32 product)."""
    lib = lib or load()
    x = _u16(x_bits)
    out = np.empty(x.shape, dtype=np.uint8)
    lib.oracle_quantize_e4m3(_ptr(out), _ptr(x), x.size, dtype, float(inv_scale))
    return out


def _inplace_u8(a: np.ndarray) -> np.ndarray:
    if not (isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"] and a.dtype == np.uint8):
        raise TypeError("FP8 pools written in place must be C-contiguous uint8 arrays")
    return a


def reshape_and_cache_fp8(key: np.ndarray, value: np.ndarray, key_cache: np.ndarray,
                          value_cache: np.ndarray, slots: np.ndarray, dtype: int,
                          k_scale: float, v_scale: float, lib=None) -> None:
    """In place: quantise key/value [T, Hkv, d] into FP8 pools [N, bs, Hkv, d]."""
    lib = lib or load()
    k, v = _u16(key), _u16(value)
    kc, vc = _inplace_u8(key_cache), _inplace_u8(value_cache)
    sl = np.ascontiguousarray(slots, dtype=np.int64)
    T, Hkv, d = k.shape
    lib.oracle_reshape_and_cache_fp8(_ptr(k), _ptr(v), _ptr(kc), _ptr(vc), _ptr(sl), T, Hkv,
                                     d, kc.shape[1], dtype, _f32_inv(k_scale),
                                     _f32_inv(v_scale))


def _f32_inv(scale: float) -> float:
    """1 / scale rounded to fp32 (the inverse both sides multiply by)."""
    return float(np.float32(1.0) / np.float32(scale))


def paged_attention_fp8(query: np.ndarray, key_cache: np.ndarray, value_cache: np.ndarray,
                        block_tables: np.ndarray, context_lens: np.ndarray, scale: float,
                        dtype: int, k_scale: float, v_scale: float,
                        seqs: Optional[Sequence[int]] = None, lib=None) -> np.ndarray:
    """fp64 attention over FP8 pools (dequantised codes)."""
    lib = lib or load()
    q = _u16(query)
    kc = np.ascontiguousarray(key_cache, dtype=np.uint8)
    vc = np.ascontiguousarray(value_cache, dtype=np.uint8)
    bt, cl = _i32(block_tables), _i32(context_lens)
    S, H, d = q.shape
    N, bs, Hkv, _ = kc.shape
    out = np.full((S, H, d), np.nan, dtype=np.float64)
    sub = None if seqs is None else _i32(list(seqs))
    lib.oracle_paged_attention_fp8(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt),
                                   bt.shape[1], _ptr(cl), S, H, Hkv, d, bs, float(scale),
                                   dtype, float(np.float32(k_scale)),
                                   float(np.float32(v_scale)), _ptr(sub),
                                   0 if sub is None else sub.shape[0])
    return out


def copy_blocks_u8(key_cache: np.ndarray, value_cache: np.ndarray,
                   block_mapping: np.ndarray, lib=None) -> None:
    lib = lib or load()
    kc, vc = _inplace_u8(key_cache), _inplace_u8(value_cache)
    bm = _i32(block_mapping).reshape(-1, 2)
    N, bs, Hkv, d = kc.shape
    lib.oracle_copy_blocks_u8(_ptr(kc), _ptr(vc), _ptr(bm), bm.shape[0], bs, Hkv, d)


def prefill_attention_fp8(query: np.ndarray, key_cache: np.ndarray, value_cache: np.ndarray,
                          block_tables: np.ndarray, query_start: np.ndarray,
                          context_lens: np.ndarray, scale: float, dtype: int,
                          k_scale: float, v_scale: float, lib=None) -> np.ndarray:
    """Chunked prefill over FP8 pools (uint8 e4m3 codes, one scale per
    pool): fp64 output [T, H, d], as prefill_attention with K and V the
    dequantised codes."""
    lib = lib or load()
    q = _u16(query)
    kc = np.ascontiguousarray(key_cache, dtype=np.uint8)
    vc = np.ascontiguousarray(value_cache, dtype=np.uint8)
    bt, qs, cl = _i32(block_tables), _i32(query_start), _i32(context_lens)
    T, H, d = q.shape
    N, bs, Hkv, d2 = kc.shape
    S = cl.shape[0]
    assert d == d2 and H % Hkv == 0 and qs.shape[0] == S + 1 and int(qs[-1]) == T
    out = np.full((T, H, d), np.nan, dtype=np.float64)
    lib.oracle_prefill_attention_fp8(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt),
                                     bt.shape[1], _ptr(qs), _ptr(cl), S, H, Hkv, d, bs,
                                     float(scale), dtype, float(np.float32(k_scale)),
                                     float(np.float32(v_scale)))
    return out

"""CPU fp64 oracle for paged decode attention (TEST INFRASTRUCTURE ONLY).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The product path (the CUDA library in
``paged_kv_cache_32_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``pa_oracle.c`` (plain loops in double, see its header
for the page citations); this module only marshals numpy arrays to it.
``brute.py`` is a second, pure-Python implementation for tiny inputs.

Storage conventions for the arrays passed in:
  * ``'f32'``  -> numpy float32
  * ``'f16'``  -> numpy float16 (IEEE binary16 bits)
  * ``'bf16'`` -> numpy uint16 holding bfloat16 bit patterns
Layouts: ``'ours'`` = [blocks][kv_heads][block_size][head_size];
``'prior'`` = the prior-art key [blocks, kv_heads, head_size/x, block_size, x]
and value [blocks, kv_heads, head_size, block_size] layouts described in
"PagedAttention 详解：缓存的存储结构", section "软件地址翻译".
"""
from __future__ import annotations

import contextlib
import ctypes

import numpy as np

from . import build as _build

DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2, "fp8": 3}
LAYOUT_CODE = {"ours": 0, "prior": 1, "fp8": 2}
NP_STORAGE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "fp8": np.uint8}

_lib = None


def _load(path: str) -> ctypes.CDLL:
    L = ctypes.CDLL(path)
    i32, i64, dbl, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
    L.pao_f16_to_f64.argtypes = [ctypes.c_uint16]
    L.pao_f16_to_f64.restype = dbl
    L.pao_bf16_to_f64.argtypes = [ctypes.c_uint16]
    L.pao_bf16_to_f64.restype = dbl
    L.pao_locate.argtypes = [vp, i32, i64, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
    L.pao_locate.restype = None
    L.pao_offset_ours.argtypes = [i64, i64, i64, i64, i32, i32, i32]
    L.pao_offset_ours.restype = i64
    L.pao_key_offset_prior.argtypes = [i64, i64, i64, i64, i32, i32, i32, i32]
    L.pao_key_offset_prior.restype = i64
    L.pao_value_offset_prior.argtypes = [i64, i64, i64, i64, i32, i32, i32]
    L.pao_value_offset_prior.restype = i64
    L.pao_attention.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp] + [i32] * 7 + [dbl, i32, i32, vp]
    L.pao_attention.restype = i32
    L.pao_prefill_attention.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp] + [i32] * 7 + [dbl, i32]
    L.pao_prefill_attention.restype = i32
    L.pao_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32]
    L.pao_reshape_and_cache.restype = i32
    L.pao_copy_blocks.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32]
    L.pao_copy_blocks.restype = i32
    L.pao_max_threads.argtypes = []
    L.pao_max_threads.restype = i32
    L.pao_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    L.pao_e4m3_to_f64.restype = dbl
    L.pao_f32_to_e4m3_sat.argtypes = [ctypes.c_float]
    L.pao_f32_to_e4m3_sat.restype = ctypes.c_uint8
    L.pao_f32_to_e4m3_array.argtypes = [vp, vp, i64]
    L.pao_f32_to_e4m3_array.restype = None
    L.pao_attention_fp8.argtypes = [vp, vp, vp, vp, vp, vp] + [i32] * 7 + [dbl, dbl, dbl, i32, i32, vp]
    L.pao_attention_fp8.restype = i32
    L.pao_reshape_and_cache_fp8.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float,
                                            ctypes.c_float]
    L.pao_reshape_and_cache_fp8.restype = i32
    return L


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = _load(_build.build())
    return _lib


@contextlib.contextmanager
def use_library(path: str):
    """Temporarily route every oracle call to another build of pa_oracle.c
    (the mutation tests use this to run the pins against planted mistakes)."""
    global _lib
    saved = lib()
    _lib = _load(path)
    try:
        yield _lib
    finally:
        _lib = saved


class OracleError(RuntimeError):
    pass


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _check_storage(a: np.ndarray, dtype: str, name: str) -> None:
    if a.dtype != NP_STORAGE[dtype]:
        raise TypeError(f"{name}: expected storage {NP_STORAGE[dtype]} for {dtype}, got {a.dtype}")
    if not a.flags.c_contiguous:
        raise ValueError(f"{name} must be C-contiguous")


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact conversion of stored values to float64."""
    if dtype == "f32":
        return a.astype(np.float64)
    if dtype == "f16":
        return a.astype(np.float64)  # numpy's binary16 -> double is exact
    if dtype == "fp8":
        table = np.array([lib().pao_e4m3_to_f64(c) for c in range(256)], dtype=np.float64)
        return table[np.ascontiguousarray(a)]
    # bfloat16 is the upper half of an IEEE binary32
    return (np.ascontiguousarray(a).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def locate(table_row: np.ndarray, block_size: int, i: int) -> tuple[int, int]:
    """(physical block, offset) of token i through one block-table row."""
    row = np.ascontiguousarray(table_row, dtype=np.int32)
    blk, off = ctypes.c_int32(), ctypes.c_int32()
    lib().pao_locate(_ptr(row), block_size, i, ctypes.byref(blk), ctypes.byref(off))
    return blk.value, off.value


def offset_ours(block, head, slot, d, num_kv_heads, block_size, head_size) -> int:
    return lib().pao_offset_ours(block, head, slot, d, num_kv_heads, block_size, head_size)


def key_offset_prior(block, head, slot, d, num_kv_heads, block_size, head_size, x) -> int:
    return lib().pao_key_offset_prior(block, head, slot, d, num_kv_heads, block_size, head_size, x)


def value_offset_prior(block, head, slot, d, num_kv_heads, block_size, head_size) -> int:
    return lib().pao_value_offset_prior(block, head, slot, d, num_kv_heads, block_size, head_size)


def paged_attention(q, k_cache, v_cache, block_tables, seq_lens, *, dtype: str, num_kv_heads: int,
                    block_size: int, scale: float, layout: str = "ours", partition_size: int = 0,
                    threads: int = 0, alibi_slopes=None) -> np.ndarray:
    """out[s, h, :] = softmax(scale * q[s,h] . K_s^T) V_s, in float64.

    q: [N, Hq, D]; k_cache/v_cache: the whole pool in ``layout``;
    block_tables: int32 [N, M]; seq_lens: int32 [N].
    partition_size > 0 evaluates the partitioned form with the log-sum-exp merge.
    alibi_slopes: optional per-query-head slopes; score_i += slope * (i - (L - 1)).
    """
    q = np.ascontiguousarray(q)
    _check_storage(q, dtype, "q")
    _check_storage(k_cache, dtype, "k_cache")
    _check_storage(v_cache, dtype, "v_cache")
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    N, Hq, D = q.shape
    M = bt.shape[1] if bt.ndim == 2 else 0
    per_block = num_kv_heads * block_size * D
    num_blocks = k_cache.size // per_block
    out = np.zeros((N, Hq, D), dtype=np.float64)
    slopes = None if alibi_slopes is None else np.ascontiguousarray(alibi_slopes, dtype=np.float64)
    if slopes is not None and slopes.shape != (Hq,):
        raise ValueError("alibi_slopes must have one entry per query head")
    rc = lib().pao_attention(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), DTYPE_CODE[dtype],
                             LAYOUT_CODE[layout], _ptr(bt), _ptr(sl), N, Hq, num_kv_heads, D, block_size, M,
                             num_blocks, float(scale), int(partition_size), int(threads),
                             None if slopes is None else _ptr(slopes))
    if rc != 0:
        raise OracleError(f"pao_attention failed: {rc}")
    return out


def prefill_attention(q, k_cache, v_cache, block_tables, seq_lens, query_start, *, dtype: str, num_kv_heads: int,
                      block_size: int, scale: float, threads: int = 0) -> np.ndarray:
    """Chunked prefill over the paged cache, float64 [total_q, Hq, D].

    q: packed [total_q, Hq, D]; query_start: int32 [N + 1] offsets of each
    sequence's chunk in q; seq_lens: int32 [N] cached tokens including the
    chunk.  Query j of sequence s attends causally to cache positions
    0 .. seq_lens[s] - n_s + j.
    """
    q = np.ascontiguousarray(q)
    _check_storage(q, dtype, "q")
    _check_storage(k_cache, dtype, "k_cache")
    _check_storage(v_cache, dtype, "v_cache")
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    T, Hq, D = q.shape
    N = len(sl)
    assert qs.shape == (N + 1,) and qs[-1] == T
    M = bt.shape[1] if bt.ndim == 2 else 0
    num_blocks = k_cache.size // (num_kv_heads * block_size * D)
    out = np.zeros((T, Hq, D), dtype=np.float64)
    rc = lib().pao_prefill_attention(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), DTYPE_CODE[dtype], _ptr(bt),
                                     _ptr(sl), _ptr(qs), N, Hq, num_kv_heads, D, block_size, M, num_blocks,
                                     float(scale), int(threads))
    if rc != 0:
        raise OracleError(f"pao_prefill_attention failed: {rc}")
    return out


def reshape_and_cache(k_cache, v_cache, key, value, slot_mapping, *, dtype: str, num_kv_heads: int,
                      block_size: int) -> None:
    """In place on the host pools: key/value [T, Hkv, D] -> slots of slot_mapping."""
    for a, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (key, "key"), (value, "value")):
        _check_storage(a, dtype, n)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, Hkv, D = key.shape
    num_blocks = k_cache.size // (Hkv * block_size * D)
    rc = lib().pao_reshape_and_cache(_ptr(k_cache), _ptr(v_cache), _ptr(key), _ptr(value), _ptr(sm), T,
                                     DTYPE_CODE[dtype], Hkv, D, block_size, num_blocks)
    if rc != 0:
        raise OracleError(f"pao_reshape_and_cache failed: {rc}")


def copy_blocks(k_cache, v_cache, pairs, *, dtype: str, num_kv_heads: int, block_size: int,
                head_size: int) -> None:
    """In place on the host pools: block dst <- block src for each (src, dst) pair, in order."""
    _check_storage(k_cache, dtype, "k_cache")
    _check_storage(v_cache, dtype, "v_cache")
    pr = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
    num_blocks = k_cache.size // (num_kv_heads * block_size * head_size)
    rc = lib().pao_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(pr), pr.shape[0], DTYPE_CODE[dtype],
                               num_kv_heads, head_size, block_size, num_blocks)
    if rc != 0:
        raise OracleError(f"pao_copy_blocks failed: {rc}")


def max_threads() -> int:
    return lib().pao_max_threads()


def e4m3_to_f64(code: int) -> float:
    """Value of one E4M3 code (NaN for S.1111.111)."""
    return lib().pao_e4m3_to_f64(int(code))


def quantize_e4m3(r) -> np.ndarray:
    """E4M3 codes nearest to the float32 values r (ties to even, saturating at +-448)."""
    r = np.ascontiguousarray(r, dtype=np.float32)
    out = np.empty(r.shape, dtype=np.uint8)
    lib().pao_f32_to_e4m3_array(_ptr(r), _ptr(out), r.size)
    return out


def quantize_cache_fp8(cache_f16: np.ndarray, scale: float, values: bool) -> np.ndarray:
    """An fp16 pool [blocks][kv_heads][B][D] as E4M3 codes of x / scale (fp32 division),
    in the FP8 layout: keys [blocks][kv_heads][B][D], values [blocks][kv_heads][B/16][D][16]."""
    x = np.ascontiguousarray(cache_f16, dtype=np.float16).astype(np.float32)
    codes = quantize_e4m3(x / np.float32(scale))
    return values_to_fp8_layout(codes) if values else codes


def values_to_fp8_layout(v: np.ndarray) -> np.ndarray:
    """[blocks][kv_heads][B][D] -> [blocks][kv_heads][B/16][D][16] (the FP8 value layout)."""
    nb, h, B, D = v.shape
    return np.ascontiguousarray(v.reshape(nb, h, B // 16, 16, D).transpose(0, 1, 2, 4, 3))


def values_from_fp8_layout(v: np.ndarray) -> np.ndarray:
    """[blocks][kv_heads][B/16][D][16] -> [blocks][kv_heads][B][D]."""
    nb, h, g, D, _ = v.shape
    return np.ascontiguousarray(v.transpose(0, 1, 2, 4, 3).reshape(nb, h, g * 16, D))


def paged_attention_fp8(q, k_cache, v_cache, block_tables, seq_lens, *, num_kv_heads: int, block_size: int,
                        scale: float, k_scale: float, v_scale: float, partition_size: int = 0, threads: int = 0,
                        alibi_slopes=None) -> np.ndarray:
    """Decode attention over an FP8 (E4M3) cache in float64: fp16 q [N, Hq, D]; key codes
    [blocks][kv_heads][B][D], value codes [blocks][kv_heads][B/16][D][16]; k = k_scale * e4m3(code),
    v = v_scale * e4m3(code)."""
    q = np.ascontiguousarray(q)
    _check_storage(q, "f16", "q")
    _check_storage(k_cache, "fp8", "k_cache")
    _check_storage(v_cache, "fp8", "v_cache")
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    N, Hq, D = q.shape
    M = bt.shape[1] if bt.ndim == 2 else 0
    num_blocks = k_cache.size // (num_kv_heads * block_size * D)
    out = np.zeros((N, Hq, D), dtype=np.float64)
    slopes = None if alibi_slopes is None else np.ascontiguousarray(alibi_slopes, dtype=np.float64)
    rc = lib().pao_attention_fp8(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(sl), N, Hq,
                                 num_kv_heads, D, block_size, M, num_blocks, float(scale), float(k_scale),
                                 float(v_scale), int(partition_size), int(threads),
                                 None if slopes is None else _ptr(slopes))
    if rc != 0:
        raise OracleError(f"pao_attention_fp8 failed: {rc}")
    return out


def reshape_and_cache_fp8(k_cache, v_cache, key, value, slot_mapping, *, num_kv_heads: int, block_size: int,
                          k_scale: float, v_scale: float) -> None:
    """In place on the host FP8 pools: fp16 key/value [T, Hkv, D] -> E4M3 codes at the slots."""
    _check_storage(k_cache, "fp8", "k_cache")
    _check_storage(v_cache, "fp8", "v_cache")
    key = np.ascontiguousarray(key, dtype=np.float16)
    value = np.ascontiguousarray(value, dtype=np.float16)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, Hkv, D = key.shape
    num_blocks = k_cache.size // (Hkv * block_size * D)
    rc = lib().pao_reshape_and_cache_fp8(_ptr(k_cache), _ptr(v_cache), _ptr(key), _ptr(value), _ptr(sm), T, Hkv, D,
                                         block_size, num_blocks, float(k_scale), float(v_scale))
    if rc != 0:
        raise OracleError(f"pao_reshape_and_cache_fp8 failed: {rc}")

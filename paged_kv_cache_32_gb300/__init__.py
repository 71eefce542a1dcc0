"""paged_kv_cache_32_gb300 - paged decode attention for GB300 (sm_103a).

Thin Python binding of the C ABI in ``include/pa.h`` (``libpa.so``), with the
same entry-point names.  It only marshals arguments: torch tensors provide
device memory and the current CUDA stream; every step of the computation runs
in the library's CUDA kernels.  There is no CPU or PyTorch fallback: if the
library has not been built, every entry point raises.

Cache layout expected by every call: K and V are each a dense tensor
[num_blocks, num_kv_heads, block_size, head_size] of float32, float16 or
bfloat16 on the GPU.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

PA_F32, PA_F16, PA_BF16, PA_FP8_E4M3 = 0, 1, 2, 3
PA_OK = 0
PA_DEVERR = {0: "none", 1: "block id out of range", 2: "slot out of range", 3: "copy pair id out of range",
             4: "wait on an asynchronous copy timed out", 5: "prefill chunk inconsistent with q, grid or sequence"}

EXPORTED = ("pa_decode", "pa_decode_ex", "pa_decode_append", "pa_decode_partition_size", "pa_decode_workspace_size",
            "pa_reshape_and_cache", "pa_copy_blocks", "pa_status_string", "pa_version", "pa_decode_noalloc", "pa_prefill",
            "pa_reshape_and_cache_fp8")


PA_DECODE_TEST_EXPIRE_FIRST_WAIT = 1


class pa_decode_options(ctypes.Structure):
    _fields_ = [("alibi_slopes", ctypes.c_void_p), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
                ("test_flags", ctypes.c_uint32)]


class pa_cache_desc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_size", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class PaError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} (status {status})")
        self.status = status


_lib = None


def lib_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded libpa.so.  Raises if it has not been built (no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise ImportError(f"libpa.so is not built ({_build.LIB}); run paged_kv_cache_32_gb300.build.build()")
        L = ctypes.CDLL(_build.LIB)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        desc_p = ctypes.POINTER(pa_cache_desc)
        L.pa_decode.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, desc_p, ctypes.c_float, i32, vp, sz, vp, vp]
        L.pa_decode.restype = ctypes.c_int
        L.pa_decode_ex.argtypes = L.pa_decode.argtypes + [ctypes.POINTER(pa_decode_options)]
        L.pa_decode_ex.restype = ctypes.c_int
        L.pa_decode_append.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, desc_p, ctypes.c_float, i32, vp, sz,
                                       vp, vp, ctypes.POINTER(pa_decode_options)]
        L.pa_decode_append.restype = ctypes.c_int
        L.pa_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, desc_p, ctypes.c_float, vp, vp]
        L.pa_prefill.restype = ctypes.c_int
        L.pa_decode_partition_size.argtypes = [i32, desc_p, i32]
        L.pa_decode_partition_size.restype = i32
        L.pa_decode_workspace_size.argtypes = [i32, i32, i32, desc_p, i32]
        L.pa_decode_workspace_size.restype = sz
        L.pa_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i32, desc_p, vp, vp]
        L.pa_reshape_and_cache.restype = ctypes.c_int
        L.pa_copy_blocks.argtypes = [vp, vp, vp, i32, desc_p, vp, vp]
        L.pa_reshape_and_cache_fp8.argtypes = [vp, vp, vp, vp, vp, i32, desc_p, ctypes.c_float, ctypes.c_float, vp, vp]
        L.pa_reshape_and_cache_fp8.restype = ctypes.c_int
        L.pa_copy_blocks.restype = ctypes.c_int
        L.pa_status_string.argtypes = [ctypes.c_int]
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_version.argtypes = []
        L.pa_version.restype = ctypes.c_int
        _lib = L
    return _lib


def build(force: bool = False) -> str:
    """Compile libpa.so in-tree for sm_103a (see build.py)."""
    global _lib
    path = _build.build(force=force)
    _lib = None
    return path


def status_string(status: int) -> str:
    return lib().pa_status_string(int(status)).decode()


def version() -> int:
    return lib().pa_version()


# ---------------------------------------------------------------- marshalling helpers
def _dtype_code(t) -> int:
    import torch
    codes = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16, torch.uint8: PA_FP8_E4M3}
    if hasattr(torch, "float8_e4m3fn"):
        codes[torch.float8_e4m3fn] = PA_FP8_E4M3
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return codes[t.dtype]


def cache_desc(k_cache) -> pa_cache_desc:
    """Descriptor of a [num_blocks, num_kv_heads, block_size, head_size] key-cache tensor
    (uint8 or float8_e4m3fn storage means an FP8 E4M3 cache, whose values are
    [num_blocks, num_kv_heads, block_size / 16, head_size, 16])."""
    if k_cache.dim() != 4:
        raise ValueError("cache must be [num_blocks, num_kv_heads, block_size, head_size]")
    nb, hkv, bs, d = (int(x) for x in k_cache.shape)
    return pa_cache_desc(nb, bs, hkv, d, _dtype_code(k_cache))


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


def _dense(t, name: str):
    if t is not None and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    return int(getattr(stream, "cuda_stream", stream))


def _check(status: int, where: str) -> None:
    if status != PA_OK:
        raise PaError(status, where)


# ---------------------------------------------------------------- entry points
def pa_decode_partition_size(max_blocks_per_seq: int, desc: pa_cache_desc, partition_size: int = 0) -> int:
    r = lib().pa_decode_partition_size(int(max_blocks_per_seq), ctypes.byref(desc), int(partition_size))
    if r < 0:
        raise PaError(-r, "pa_decode_partition_size")
    return r


def pa_decode_workspace_size(num_seqs: int, num_q_heads: int, max_blocks_per_seq: int, desc: pa_cache_desc,
                             partition_size: int = 0) -> int:
    return int(lib().pa_decode_workspace_size(int(num_seqs), int(num_q_heads), int(max_blocks_per_seq),
                                              ctypes.byref(desc), int(partition_size)))


def pa_decode(out, q, k_cache, v_cache, block_tables, seq_lens, scale: float, partition_size: int = 0,
              workspace=None, err_flag=None, stream=None, desc: pa_cache_desc | None = None,
              alibi_slopes=None, k_scale: float | None = None, v_scale: float | None = None,
              test_flags: int = 0) -> None:
    """out[s, h] = softmax(scale * q[s, h] K_s^T) V_s over seq_lens[s] paged tokens.

    out, q: [num_seqs, num_q_heads, head_size] (cache dtype); block_tables: int32
    [num_seqs, max_blocks_per_seq]; seq_lens: int32 [num_seqs].  ``workspace`` is a
    uint8 device tensor of at least pa_decode_workspace_size(...) bytes; when None
    and one is needed, it is allocated with torch.  ``alibi_slopes``: optional
    float32 device tensor [num_q_heads] (calls pa_decode_ex).  ``k_scale`` /
    ``v_scale``: dequantisation scales of an FP8 cache (q and out are fp16 then).
    ``test_flags``: 0, or PA_DECODE_TEST_EXPIRE_FIRST_WAIT in tests of the bounded waits.
    """
    desc = desc or cache_desc(k_cache)
    for t, n in ((out, "out"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (block_tables, "block_tables"), (seq_lens, "seq_lens")):
        _dense(t, n)
    num_seqs, num_q_heads = int(q.shape[0]), int(q.shape[1])
    max_blocks = int(block_tables.shape[1]) if block_tables.dim() == 2 else 0
    need = pa_decode_workspace_size(num_seqs, num_q_heads, max_blocks, desc, partition_size)
    if workspace is None and need > 0:
        import torch
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = (_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(seq_lens), num_seqs,
            num_q_heads, max_blocks, ctypes.byref(desc), float(scale), int(partition_size), _ptr(workspace), ws_bytes,
            _ptr(err_flag), _stream(stream))
    if alibi_slopes is None and k_scale is None and v_scale is None and not test_flags:
        _check(lib().pa_decode(*args), "pa_decode")
    else:
        _dense(alibi_slopes, "alibi_slopes")
        opts = pa_decode_options(_ptr(alibi_slopes), float(k_scale or 0.0), float(v_scale or 0.0), int(test_flags))
        _check(lib().pa_decode_ex(*args, ctypes.byref(opts)), "pa_decode_ex")


def pa_decode_append(out, q, k_cache, v_cache, key, value, block_tables, seq_lens, scale: float,
                     partition_size: int = 0, workspace=None, err_flag=None, stream=None,
                     desc: pa_cache_desc | None = None, alibi_slopes=None, k_scale: float | None = None,
                     v_scale: float | None = None) -> None:
    """A decode step with its append: key/value [num_seqs, num_kv_heads, head_size] are each
    sequence's new token, stored at position seq_lens[s] - 1 of both caches (through the block
    table) and attended in the same call.  fp16/bf16 caches, and FP8 caches (key/value fp16,
    quantised with k_scale / v_scale as pa_reshape_and_cache_fp8 does)."""
    desc = desc or cache_desc(k_cache)
    for t, n in ((out, "out"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (key, "key"), (value, "value"),
                 (block_tables, "block_tables"), (seq_lens, "seq_lens")):
        _dense(t, n)
    num_seqs, num_q_heads = int(q.shape[0]), int(q.shape[1])
    max_blocks = int(block_tables.shape[1]) if block_tables.dim() == 2 else 0
    need = pa_decode_workspace_size(num_seqs, num_q_heads, max_blocks, desc, partition_size)
    if workspace is None and need > 0:
        import torch
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    opts = None
    if alibi_slopes is not None or k_scale is not None or v_scale is not None:
        _dense(alibi_slopes, "alibi_slopes")
        opts = ctypes.byref(pa_decode_options(_ptr(alibi_slopes), float(k_scale or 0.0), float(v_scale or 0.0), 0))
    _check(lib().pa_decode_append(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(key), _ptr(value),
                                  _ptr(block_tables), _ptr(seq_lens), num_seqs, num_q_heads, max_blocks,
                                  ctypes.byref(desc), float(scale), int(partition_size), _ptr(workspace), ws_bytes,
                                  _ptr(err_flag), _stream(stream), opts), "pa_decode_append")


def pa_prefill(out, q, k_cache, v_cache, block_tables, seq_lens, query_start, max_query_len: int, scale: float,
               err_flag=None, stream=None, desc: pa_cache_desc | None = None) -> None:
    """Chunked prefill: the queries q[query_start[s]:query_start[s+1]] are the last
    n_s of seq_lens[s] cached tokens; query j attends to positions 0..L-n_s+j.

    out, q: [num_query_tokens, num_q_heads, 128] (f16/bf16); block_tables int32
    [num_seqs, max_blocks_per_seq]; seq_lens int32 [num_seqs]; query_start int32
    [num_seqs + 1]; max_query_len bounds every n_s (it sizes the grid).
    """
    desc = desc or cache_desc(k_cache)
    for t, n in ((out, "out"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (block_tables, "block_tables"), (seq_lens, "seq_lens"), (query_start, "query_start")):
        _dense(t, n)
    num_seqs = int(seq_lens.shape[0])
    max_blocks = int(block_tables.shape[1]) if block_tables.dim() == 2 else 0
    status = lib().pa_prefill(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(seq_lens),
                              _ptr(query_start), num_seqs, int(q.shape[0]), int(q.shape[1]), max_blocks,
                              int(max_query_len), ctypes.byref(desc), float(scale), _ptr(err_flag), _stream(stream))
    _check(status, "pa_prefill")


def pa_reshape_and_cache(k_cache, v_cache, key, value, slot_mapping, err_flag=None, stream=None,
                         desc: pa_cache_desc | None = None) -> None:
    """Write key/value [num_tokens, num_kv_heads, head_size] into the slots of slot_mapping (int64)."""
    desc = desc or cache_desc(k_cache)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (key, "key"), (value, "value"),
                 (slot_mapping, "slot_mapping")):
        _dense(t, n)
    status = lib().pa_reshape_and_cache(_ptr(k_cache), _ptr(v_cache), _ptr(key), _ptr(value), _ptr(slot_mapping),
                                        int(slot_mapping.shape[0]), ctypes.byref(desc), _ptr(err_flag),
                                        _stream(stream))
    _check(status, "pa_reshape_and_cache")


def pa_reshape_and_cache_fp8(k_cache, v_cache, key, value, slot_mapping, k_scale: float, v_scale: float,
                             err_flag=None, stream=None, desc: pa_cache_desc | None = None) -> None:
    """Write fp16 key/value [num_tokens, num_kv_heads, head_size] into an FP8 cache as
    E4M3 codes of x / k_scale and x / v_scale (values at [block, head, offset / 16, d, offset % 16])."""
    desc = desc or cache_desc(k_cache)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (key, "key"), (value, "value"),
                 (slot_mapping, "slot_mapping")):
        _dense(t, n)
    status = lib().pa_reshape_and_cache_fp8(_ptr(k_cache), _ptr(v_cache), _ptr(key), _ptr(value), _ptr(slot_mapping),
                                            int(slot_mapping.shape[0]), ctypes.byref(desc), float(k_scale),
                                            float(v_scale), _ptr(err_flag), _stream(stream))
    _check(status, "pa_reshape_and_cache_fp8")


def pa_copy_blocks(k_cache, v_cache, block_pairs, err_flag=None, stream=None, desc: pa_cache_desc | None = None) -> None:
    """For each (src, dst) row of block_pairs (int32 [n, 2]) copy whole block src to dst in both caches."""
    desc = desc or cache_desc(k_cache)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (block_pairs, "block_pairs")):
        _dense(t, n)
    status = lib().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(block_pairs), int(block_pairs.shape[0]),
                                  ctypes.byref(desc), _ptr(err_flag), _stream(stream))
    _check(status, "pa_copy_blocks")

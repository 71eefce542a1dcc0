"""Chunked prefill attention in float64 with library matmuls (TEST INFRASTRUCTURE ONLY).

The same definition as ``pa_oracle.c``'s prefill, written with numpy so that a
whole benchmark-size workload (tens of thousands of query tokens over
contexts of a few thousand) is checked in seconds rather than minutes: the
plain loops of the C oracle visit every (query, key, dimension) triple
through a per-element gather.

Per sequence s and kv head, in the pages' order:
  1. gather the L = seq_lens[s] cached keys and values: token i lives at offset
     i % B of block block_tables[s][i // B] ("PagedAttention 详解：缓存的存储结构",
     sections "Block Table" and "软件地址翻译");
  2. scores S = scale * Q K^T for the chunk's n queries of each query head of
     that kv head (consecutive query heads share a kv head), one matmul;
  3. the causal mask of a chunk at the end of the context: query j sits at
     position L - n + j and sees positions 0 .. L - n + j ("vLLM 核心工程深度剖析",
     section "6.1": long prompts are prefilled in chunks; "PagedAttention 详解：
     缓存的存储结构", section "使用流程": cached blocks take part directly);
  4. the max-subtracted softmax in two passes (row max, then exp and its sum),
     P = exp(S - max) / sum ("vLLM 核心工程深度剖析", section "3.1 Kernel 签名与
     分块策略");
  5. out = P V, one matmul.
Stored 16-bit values are converted exactly to float64 first.  Nothing is
blocked, fused or reordered beyond the matmuls.  It shares no code with the
CUDA library; the tests pin it to the C oracle and to the pure-Python brute
force on small inputs.
"""
from __future__ import annotations

import numpy as np

from . import to_f64


def gather_tokens(cache: np.ndarray, table_row: np.ndarray, L: int, kv_head: int, block_size: int) -> np.ndarray:
    """[L, D] rows of one kv head: token i at offset i % B of block table_row[i // B]."""
    i = np.arange(L)
    blocks = np.asarray(table_row, dtype=np.int64)[i // block_size]
    if L and (blocks.min() < 0 or blocks.max() >= cache.shape[0]):
        raise ValueError("block id outside the pool")
    return cache[blocks, kv_head, i % block_size, :]


def prefill_attention(q, k_cache, v_cache, block_tables, seq_lens, query_start, *, dtype: str, num_kv_heads: int,
                      block_size: int, scale: float) -> np.ndarray:
    """float64 [total_q, Hq, D]: the chunk of sequence s is q[query_start[s]:query_start[s+1]],
    the last n_s of its seq_lens[s] cached tokens; query j attends to positions 0 .. L - n_s + j."""
    T, Hq, D = q.shape
    G = Hq // num_kv_heads
    kc = k_cache.reshape(-1, num_kv_heads, block_size, D)
    vc = v_cache.reshape(-1, num_kv_heads, block_size, D)
    qs = np.asarray(query_start, dtype=np.int64)
    out = np.zeros((T, Hq, D), dtype=np.float64)
    for s in range(len(seq_lens)):
        t0, t1, L = int(qs[s]), int(qs[s + 1]), int(seq_lens[s])
        n = t1 - t0
        if n == 0:
            continue
        if n > L:
            raise ValueError("a chunk longer than its sequence")
        pos = L - n + np.arange(n)                         # the queries' positions
        visible = np.arange(L)[None, :] <= pos[:, None]    # [n, L]
        for hkv in range(num_kv_heads):
            K = to_f64(gather_tokens(kc, block_tables[s], L, hkv, block_size), dtype)   # [L, D]
            V = to_f64(gather_tokens(vc, block_tables[s], L, hkv, block_size), dtype)
            for h in range(hkv * G, (hkv + 1) * G):
                Q = to_f64(q[t0:t1, h, :], dtype)          # [n, D]
                S = np.where(visible, scale * (Q @ K.T), -np.inf)
                E = np.exp(S - S.max(axis=1, keepdims=True))
                P = E / E.sum(axis=1, keepdims=True)
                out[t0:t1, h, :] = P @ V
    return out

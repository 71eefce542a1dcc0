"""Pure-Python brute force of paged decode attention for tiny inputs (TEST INFRASTRUCTURE ONLY).

A second implementation, independent of ``pa_oracle.c``: it decodes stored
bits with ``struct`` (binary16 via the 'e' format, bfloat16 by padding to a
binary32), builds each sequence's contiguous key and value lists by walking the
block table token by token, and evaluates softmax(scale * q k^T) v with Python
floats (IEEE double) and ``math.exp``.

Source: "PagedAttention 详解：缓存的存储结构", sections "Block Table" and
"软件地址翻译" (token i lives at offset i % B of block block_tables[s][i // B]);
"vLLM 核心工程深度剖析", section "3.1 Kernel 签名与分块策略" (the scaled
softmax and the value-weighted sum).
"""
from __future__ import annotations

import math
import struct


def _decode(bits_or_value, dtype: str) -> float:
    if dtype == "f32":
        return float(bits_or_value)
    if dtype == "f16":
        return struct.unpack("<e", struct.pack("<H", int(bits_or_value)))[0]
    return struct.unpack("<f", struct.pack("<I", int(bits_or_value) << 16))[0]


def _flat_values(arr, dtype: str) -> list[float]:
    """Python floats of an array given as float32 values, float16 values or bf16 bit patterns."""
    if dtype == "f16":
        return [_decode(int(b), "f16") for b in arr.reshape(-1).view("uint16")]
    return [_decode(x, dtype) for x in arr.reshape(-1).tolist()]


def paged_attention(q, k_cache, v_cache, block_tables, seq_lens, *, dtype: str, num_kv_heads: int,
                    block_size: int, scale: float, alibi_slopes=None) -> list:
    """Nested lists out[s][h][d]; cache layout [blocks][kv_heads][block_size][head_size].
    With alibi_slopes, score i of head h gains slope_h * (i - (L - 1)) (linear
    bias towards the query's own position, read from the per-head alibi_slopes
    of "vLLM 核心工程深度剖析", section "3.1 Kernel 签名与分块策略")."""
    N, Hq, D = q.shape
    G = Hq // num_kv_heads
    qf = _flat_values(q, dtype)
    kf = _flat_values(k_cache, dtype)
    vf = _flat_values(v_cache, dtype)

    def row(cache, blk, head, slot):
        base = ((blk * num_kv_heads + head) * block_size + slot) * D
        return cache[base:base + D]

    out = []
    for s in range(N):
        L = int(seq_lens[s])
        per_head = []
        for h in range(Hq):
            hkv = h // G
            qv = qf[(s * Hq + h) * D:(s * Hq + h + 1) * D]
            keys, values = [], []
            for i in range(L):
                blk = int(block_tables[s][i // block_size])
                off = i % block_size
                keys.append(row(kf, blk, hkv, off))
                values.append(row(vf, blk, hkv, off))
            if L == 0:
                per_head.append([0.0] * D)
                continue
            scores = [scale * sum(a * b for a, b in zip(qv, k)) for k in keys]
            if alibi_slopes is not None:
                scores = [x + float(alibi_slopes[h]) * (i - (L - 1)) for i, x in enumerate(scores)]
            mx = max(scores)
            ex = [math.exp(x - mx) for x in scores]
            den = sum(ex)
            per_head.append([sum(e * v[d] for e, v in zip(ex, values)) / den for d in range(D)])
        out.append(per_head)
    return out


def prefill_attention(q, k_cache, v_cache, block_tables, seq_lens, query_start, *, dtype: str, num_kv_heads: int,
                      block_size: int, scale: float) -> list:
    """Chunked prefill by brute force: query j of sequence s (chunk of n_s tokens
    at the end of its seq_lens[s] cached tokens) attends to cache positions
    0 .. seq_lens[s] - n_s + j, evaluated as a one-query problem each."""
    import numpy as np
    out = []
    for s in range(len(seq_lens)):
        n = int(query_start[s + 1]) - int(query_start[s])
        for j in range(n):
            t = int(query_start[s]) + j
            pos = int(seq_lens[s]) - n + j
            res = paged_attention(q[t:t + 1], k_cache, v_cache, [list(block_tables[s])], [pos + 1], dtype=dtype,
                                  num_kv_heads=num_kv_heads, block_size=block_size, scale=scale)
            out.append(res[0])
    return out


def e4m3_value(code: int) -> float:
    """E4M3 code -> float from its fields: sign, 4 exponent bits (bias 7), 3 mantissa bits;
    exponent 0 is subnormal (m/8 * 2^-6), S.1111.111 is NaN."""
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def paged_attention_fp8(q_f16, k_codes, v_codes, block_tables, seq_lens, *, num_kv_heads: int, block_size: int,
                        scale: float, k_scale: float, v_scale: float) -> list:
    """Decode attention over an FP8 cache by brute force: keys [blocks][Hkv][B][D] and values
    [blocks][Hkv][B/16][D][16] of E4M3 codes standing for k_scale (v_scale) times their value."""
    N, Hq, D = q_f16.shape
    G = Hq // num_kv_heads
    qf = _flat_values(q_f16, "f16")
    kc = [int(c) for c in k_codes.reshape(-1)]
    vc = [int(c) for c in v_codes.reshape(-1)]
    out = []
    for s in range(N):
        L = int(seq_lens[s])
        per_head = []
        for h in range(Hq):
            hkv = h // G
            qv = qf[(s * Hq + h) * D:(s * Hq + h + 1) * D]
            if L == 0:
                per_head.append([0.0] * D)
                continue
            scores, values = [], []
            for i in range(L):
                blk, off = int(block_tables[s][i // block_size]), i % block_size
                base = (blk * num_kv_heads + hkv) * block_size * D
                key = [k_scale * e4m3_value(kc[base + off * D + d]) for d in range(D)]
                vbase = base + (off // 16) * D * 16 + off % 16
                values.append([v_scale * e4m3_value(vc[vbase + d * 16]) for d in range(D)])
                scores.append(scale * sum(a * b for a, b in zip(qv, key)))
            mx = max(scores)
            ex = [math.exp(x - mx) for x in scores]
            den = sum(ex)
            per_head.append([sum(e * v[d] for e, v in zip(ex, values)) / den for d in range(D)])
        out.append(per_head)
    return out

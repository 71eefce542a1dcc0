"""Test-side glue: run a workload step through the CUDA library and through the oracle.

The two sides receive the same host arrays from ``workloads``; nothing the GPU
computes is ever fed to the oracle.
"""
from __future__ import annotations

import numpy as np

import oracle as O
import workloads as W

TOL = {"f32": 1e-5, "f16": 3e-3, "bf16": 3e-3}
MANTISSA_BITS = {"f16": 10, "bf16": 7}


# Error of the fp32 result before its final rounding to the output type, allowed on top
# of half an output ulp where that half ulp alone exceeds the stated tolerance (bf16
# outputs with |out| >= 1, reached only by very short sequences).  What bounds it there:
# probabilities enter the value contraction as two bf16 terms, hi + lo, whose sum is
# within 2^-16 p of the fp32 weight p (prefill: hi truncated, so p - hi < 2^-7 p and lo
# rounds that to 8 bits) or 2^-18 p (decode: hi rounded), while the normaliser sums the
# fp32 weights; the output therefore moves by at most 2^-16 max|v|, 1.2e-4 for the
# N(0,1) values here (|v| < 8).  The fp32 roundings of scores, exponentials and sums
# over the few tokens of such a sequence are orders of magnitude smaller.  2^-12 =
# 2.4e-4 keeps a factor of two over that term.
PRE_ROUNDING_EXCESS = 2.0 ** -12


def rising_keys(w: W.Workload, c: float, seed: int, positions=None) -> None:
    """Make a decode workload's scores rise along each sequence (in place): every query
    becomes one vector u (N(0,1) entries) and key i of each sequence gains c * i * u,
    so a query's score for key i grows by about c * |u|^2 per token.  The kernels' running
    maxima then move on some slabs or tiles and stay on others.  ``positions``: for a
    prefill workload, the number of cached tokens before each chunk (keys of the chunk
    are the new_key rows, in query order)."""
    rng = np.random.default_rng(seed)
    u = rng.standard_normal(w.head_size)
    B = w.block_size
    k = O.to_f64(w.k_cache, w.dtype)
    nk = O.to_f64(w.new_key, w.dtype) if w.new_key is not None else None
    for s, L in enumerate(w.seq_lens):
        L = int(L)
        if positions is None:  # decode: with an append, position L - 1 arrives as new_key[s]
            cached = L - 1 if (nk is not None and L > 0) else L
            if nk is not None and L > 0:
                nk[s] += c * (L - 1) * u
        else:  # prefill: chunk token j (position cached + j) is new_key[query_start[s] + j]
            cached = int(positions[s])
            q0 = int(w.query_start[s])
            for j in range(L - cached):
                nk[q0 + j] += c * (cached + j) * u
        for i in range(cached):
            k[w.block_tables[s][i // B], :, i % B, :] += c * i * u
    w.k_cache = W.to_storage(k, w.dtype)
    if nk is not None:
        w.new_key = W.to_storage(nk, w.dtype)
    w.q = W.to_storage(np.broadcast_to(u, w.q.shape), w.dtype)


def bound(ref: np.ndarray, dtype: str) -> np.ndarray:
    """Per-element error bound against the fp64 result.

    The stated tolerance (1e-5 fp32, 3e-3 fp16/bf16).  Rounding the output to a
    16-bit type alone costs half an ulp of |out|; for bf16 that exceeds 3e-3 once
    |out| >= 1 (half an ulp on [1, 2) is 2^-8), which very short sequences can
    reach.  There the bound is that half ulp plus PRE_ROUNDING_EXCESS; for
    |out| < 1 (every output of the five benchmark workloads) it is exactly the
    stated tolerance."""
    tol = TOL[dtype]
    if dtype == "f32":
        return np.full(ref.shape, tol)
    e = np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -14)))
    half_ulp = 2.0 ** (e - MANTISSA_BITS[dtype] - 1)
    return np.maximum(tol, half_ulp + PRE_ROUNDING_EXCESS)


def within_bound(got: np.ndarray, ref: np.ndarray, dtype: str):
    """(ok, max abs error, worst error / bound)."""
    if ref.size == 0:
        return True, 0.0, 0.0
    err = np.abs(got - ref)
    ratio = err / bound(ref, dtype)
    return bool(np.all(ratio <= 1.0)), float(err.max()), float(ratio.max())


def to_torch(a: np.ndarray, dtype: str, device="cuda"):
    import torch
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(device)


def to_numpy_storage(t, dtype: str) -> np.ndarray:
    import torch
    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def out_f64(t) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


class GpuStep:
    """Device copies of a workload's inputs plus the calls of one decode step."""

    def __init__(self, w: W.Workload, device="cuda"):
        import torch
        import paged_kv_cache_32_gb300 as pa
        self.w, self.pa = w, pa
        self.k = to_torch(w.k_cache, w.dtype, device)
        self.v = to_torch(w.v_cache, w.dtype, device)
        self.q = to_torch(w.q, w.dtype, device)
        self.tables = torch.from_numpy(w.block_tables).to(device)
        self.lens = torch.from_numpy(w.seq_lens).to(device)
        self.out = torch.empty_like(self.q)
        self.pairs = torch.from_numpy(w.copy_pairs).to(device) if w.copy_pairs is not None else None
        self.slots = torch.from_numpy(w.slot_mapping).to(device) if w.slot_mapping is not None else None
        self.nk = to_torch(w.new_key, w.dtype, device) if w.new_key is not None else None
        self.nv = to_torch(w.new_value, w.dtype, device) if w.new_value is not None else None
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.desc = pa.cache_desc(self.k)
        need = pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.max_blocks_per_seq, self.desc,
                                           w.partition_size)
        self.ws = torch.empty(max(need, 1), dtype=torch.uint8, device=device)

    def writes(self, stream=None):
        if self.pairs is not None and len(self.pairs):
            self.pa.pa_copy_blocks(self.k, self.v, self.pairs, err_flag=self.err, stream=stream, desc=self.desc)
        if self.slots is not None and len(self.slots):
            self.pa.pa_reshape_and_cache(self.k, self.v, self.nk, self.nv, self.slots, err_flag=self.err,
                                         stream=stream, desc=self.desc)

    def decode(self, stream=None, partition_size=None):
        part = self.w.partition_size if partition_size is None else partition_size
        ws = self.ws
        if partition_size is not None:
            import torch
            need = self.pa.pa_decode_workspace_size(self.w.num_seqs, self.w.num_q_heads, self.w.max_blocks_per_seq,
                                                    self.desc, part)
            if need > ws.numel():
                ws = torch.empty(need, dtype=torch.uint8, device=self.q.device)
        self.pa.pa_decode(self.out, self.q, self.k, self.v, self.tables, self.lens, self.w.scale,
                          partition_size=part, workspace=ws, err_flag=self.err, stream=stream, desc=self.desc)

    def step(self, stream=None):
        self.writes(stream)
        self.decode(stream)


def oracle_step(w: W.Workload, threads: int = 0):
    """Host pools after the step's writes, and the fp64 attention output."""
    k, v = w.k_cache.copy(), w.v_cache.copy()
    kw = dict(dtype=w.dtype, num_kv_heads=w.num_kv_heads, block_size=w.block_size)
    W.apply_writes_host(
        w, k, v,
        lambda kk, vv, pairs: O.copy_blocks(kk, vv, pairs, head_size=w.head_size, **kw),
        lambda kk, vv, nk, nv, slots: O.reshape_and_cache(kk, vv, nk, nv, slots, **kw))
    out = O.paged_attention(w.q, k, v, w.block_tables, w.seq_lens, scale=w.scale, threads=threads, **kw)
    return k, v, out


def max_abs_err(gpu_out, ref: np.ndarray) -> float:  # noqa: E302
    return float(np.max(np.abs(out_f64(gpu_out) - ref))) if ref.size else 0.0

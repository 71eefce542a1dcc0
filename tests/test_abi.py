"""The C ABI without a GPU: the library builds, loads, exports every declared
symbol, and rejects invalid arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_32_gb300 as pa


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pa.build()
    return pa.lib()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"\b(pa_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert {"pa_decode", "pa_reshape_and_cache", "pa_copy_blocks", "pa_decode_workspace_size"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(pa.EXPORTED) <= set(names)


def test_version_and_status_strings(lib):
    assert pa.version() >= 100
    for code in range(8):
        assert pa.status_string(code)
    assert pa.status_string(999) == "unknown status"


def desc(nb=16, bs=16, hkv=2, d=128, dtype=pa.PA_F16):
    return pa.pa_cache_desc(nb, bs, hkv, d, dtype)


FAKE = 0x10000  # never dereferenced: every call below is rejected before any CUDA call


def call_decode(lib, d, out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, sl=FAKE, n=2, hq=4, m=4, scale=0.1, part=0,
                ws=None, ws_bytes=0):
    return lib.pa_decode(out, q, k, v, bt, sl, n, hq, m, ctypes.byref(d), scale, part, ws, ws_bytes, None, None)


def test_decode_argument_errors(lib):
    assert call_decode(lib, desc(d=96)) == 2                         # head_size unsupported
    assert call_decode(lib, desc(dtype=7)) == 2                      # dtype unsupported
    assert call_decode(lib, desc(bs=24)) == 2                        # f16: B = 8 or a multiple of 16
    assert call_decode(lib, desc(bs=8, dtype=pa.PA_FP8_E4M3)) == 2   # fp8: B a multiple of 16
    assert call_decode(lib, desc(bs=8), part=8) == 3                 # partitions are whole 16-token slabs
    assert call_decode(lib, desc(), hq=3) == 3                       # Hq % Hkv != 0
    assert call_decode(lib, desc(), n=-1) == 3
    assert call_decode(lib, desc(), scale=float("nan")) == 3
    assert call_decode(lib, desc(), out=None) == 1
    assert call_decode(lib, desc(), bt=None) == 1
    assert call_decode(lib, desc(), part=24) == 3                    # not a multiple of B
    assert call_decode(lib, desc(), m=100) == 4                      # split needs a workspace
    assert call_decode(lib, desc(), m=100, ws=FAKE, ws_bytes=16) == 4
    assert call_decode(lib, desc(), k=FAKE + 2) == 5                 # TMA needs 16-byte aligned caches
    assert call_decode(lib, desc(nb=1 << 30, hkv=8)) == 7            # row index overflows int32
    assert call_decode(lib, desc(), n=0, out=None) == 0              # nothing to do, nothing launched


def test_decode_append_argument_errors(lib):
    def call(d, key=FAKE, value=FAKE, m=1):
        return lib.pa_decode_append(FAKE, FAKE, FAKE, FAKE, key, value, FAKE, FAKE, 2, 4, m, ctypes.byref(d), 0.1, 0,
                                    None, 0, None, None, None)
    assert call(desc(dtype=pa.PA_F32)) == 2                          # no fused append over an fp32 cache
    assert call(desc(dtype=pa.PA_FP8_E4M3), key=None) == 1           # FP8 caches take it (arguments checked)
    assert call(desc(), key=None) == 1
    assert call(desc(), value=FAKE + 4) == 5                         # 16-byte rows
    assert call(desc(), m=100) == 4                                  # split partitions need a workspace


def test_partition_and_workspace_sizes(lib):
    d = desc(nb=16384, bs=16, hkv=8, d=128, dtype=pa.PA_BF16)
    assert pa.pa_decode_partition_size(2048, d, 0) == 1024            # library default
    assert pa.pa_decode_partition_size(2048, d, 512) == 512
    assert pa.pa_decode_partition_size(16, d, 0) == 256              # whole context fits: no split
    with pytest.raises(pa.PaError):
        pa.pa_decode_partition_size(2048, d, 100)
    # 8 seqs x 32 heads x 64 partitions x (128 + 2) floats
    rows = 8 * 32 * 64
    assert pa.pa_decode_workspace_size(8, 32, 2048, d, 512) == rows * 128 * 4 + rows * 2 * 4
    assert pa.pa_decode_workspace_size(8, 32, 16, d, 0) == 0


def test_workspace_size_with_half_partition_tail(lib):
    """The documented rule: with 2 <= P_max <= 8 on the 16-bit and FP8 caches, the last num_seqs // 12
    (fp16/bf16) or num_seqs // 24 (FP8) sequences take partitions of half the size and 2 P_max slots a row,
    when the half partition holds whole blocks and whole 32-token slabs; the outputs' part is padded to 256
    bytes, then (m, l) pairs follow."""
    def size(slots, d=128):
        return -(-slots * d * 4 // 256) * 256 + slots * 2 * 4

    def slots(n, hq, pmax, tail_n, cut=2):
        return ((n - tail_n) * pmax + tail_n * cut * pmax) * hq

    bf16 = desc(nb=16384, bs=32, hkv=8, d=128, dtype=pa.PA_BF16)
    fp8 = desc(nb=16384, bs=32, hkv=8, d=128, dtype=pa.PA_FP8_E4M3)
    f32 = desc(nb=16384, bs=32, hkv=8, d=128, dtype=pa.PA_F32)
    # 128 sequences x 64 query heads of up to 4096 tokens, 1024-token partitions: P_max = 4
    assert pa.pa_decode_workspace_size(128, 64, 128, bf16, 0) == size(slots(128, 64, 4, 128 // 12))
    assert pa.pa_decode_workspace_size(128, 64, 128, fp8, 0) == size(slots(128, 64, 4, 128 // 24))
    assert pa.pa_decode_workspace_size(128, 64, 128, f32, 0) == size(slots(128, 64, 4, 0))
    # P_max = 16 (256-token partitions): uniform
    assert pa.pa_decode_workspace_size(128, 64, 128, bf16, 256) == size(slots(128, 64, 16, 0))
    # fewer than twelve sequences: no tail
    assert pa.pa_decode_workspace_size(11, 64, 128, bf16, 0) == size(slots(11, 64, 4, 0))
    # a half partition of 128 tokens is not a whole 256-token block: uniform
    big_blocks = desc(nb=4096, bs=256, hkv=8, d=128, dtype=pa.PA_BF16)
    assert pa.pa_decode_workspace_size(128, 64, 4, big_blocks, 256) == size(slots(128, 64, 4, 0))


def call_prefill(lib, d, out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, sl=FAKE, qs=FAKE, n=2, tq=64, hq=4, m=4, mql=32,
                 scale=0.1):
    return lib.pa_prefill(out, q, k, v, bt, sl, qs, n, tq, hq, m, mql, ctypes.byref(d), scale, None, None)


def test_prefill_argument_errors(lib):
    assert call_prefill(lib, desc(d=64)) == 2                         # only head_size 128 is built
    assert call_prefill(lib, desc(dtype=pa.PA_F32, bs=16)) == 2      # no fp32 tensor-core path
    assert call_prefill(lib, desc(bs=256)) == 2                      # a key tile holds whole blocks
    assert call_prefill(lib, desc(), n=-1) == 3
    assert call_prefill(lib, desc(), tq=-1) == 3
    assert call_prefill(lib, desc(), hq=3) == 3                      # Hq % Hkv != 0
    assert call_prefill(lib, desc(), mql=-5) == 3
    assert call_prefill(lib, desc(), scale=float("nan")) == 3
    assert call_prefill(lib, desc(), scale=-0.1) == 3                 # softmax scale must be positive
    assert call_prefill(lib, desc(), scale=0.0) == 3
    assert call_prefill(lib, desc(), q=None) == 1
    assert call_prefill(lib, desc(), qs=None) == 1
    assert call_prefill(lib, desc(), out=FAKE + 8) == 5               # 16-byte alignment
    assert call_prefill(lib, desc(), n=0) == 0                        # nothing to do: no launch
    assert call_prefill(lib, desc(), tq=0) == 0
    assert call_prefill(lib, desc(), mql=0) == 0


def test_fp8_argument_errors(lib):
    f8 = desc(dtype=pa.PA_FP8_E4M3)
    assert call_decode(lib, desc(dtype=pa.PA_FP8_E4M3, d=64)) == 2   # FP8 is built for head_size 128
    opts = pa.pa_decode_options(None, -1.0, 1.0)                     # negative scale
    assert lib.pa_decode_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 4, ctypes.byref(f8), 0.1, 0, None, 0, None,
                            None, ctypes.byref(opts)) == 3
    assert lib.pa_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, 4, ctypes.byref(f8), None, None) == 2
    fp8_append = lib.pa_reshape_and_cache_fp8
    assert fp8_append(FAKE, FAKE, FAKE, FAKE, FAKE, 4, ctypes.byref(desc()), 1.0, 1.0, None, None) == 2
    assert fp8_append(FAKE, FAKE, FAKE, FAKE, FAKE, 4, ctypes.byref(f8), 0.0, 1.0, None, None) == 3
    assert fp8_append(FAKE, FAKE, FAKE, FAKE, FAKE, 4, ctypes.byref(f8), 1.0, float("inf"), None, None) == 3
    assert fp8_append(FAKE, FAKE, None, FAKE, FAKE, 4, ctypes.byref(f8), 1.0, 1.0, None, None) == 1
    assert fp8_append(FAKE + 8, FAKE, FAKE, FAKE, FAKE, 4, ctypes.byref(f8), 1.0, 1.0, None, None) == 5
    assert fp8_append(FAKE, FAKE, FAKE, FAKE, FAKE, 0, ctypes.byref(f8), 1.0, 1.0, None, None) == 0
    assert call_prefill(lib, f8) == 2                                   # no FP8 prefill


def test_write_argument_errors(lib):
    d = desc()
    assert lib.pa_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, -1, ctypes.byref(d), None, None) == 3
    assert lib.pa_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, 0, ctypes.byref(d), None, None) == 0
    assert lib.pa_reshape_and_cache(FAKE, FAKE, None, FAKE, FAKE, 4, ctypes.byref(d), None, None) == 1
    assert lib.pa_reshape_and_cache(FAKE, FAKE, FAKE + 8, FAKE, FAKE, 4, ctypes.byref(d), None, None) == 5
    assert lib.pa_copy_blocks(FAKE, FAKE, None, 3, ctypes.byref(d), None, None) == 1
    assert lib.pa_copy_blocks(FAKE, FAKE, FAKE, 0, ctypes.byref(d), None, None) == 0
    assert lib.pa_copy_blocks(FAKE, FAKE, FAKE, -2, ctypes.byref(d), None, None) == 3
    assert lib.pa_copy_blocks(FAKE, FAKE, FAKE, 3, None, None, None) == 1


def test_binding_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(pa._build, "LIB", "/nonexistent/libpa.so")
    monkeypatch.setattr(pa, "_lib", None)
    with pytest.raises(ImportError):
        pa.lib()


def test_product_package_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "paged_kv_cache_32_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "oracle" not in text.lower(), fn
                assert "pa_oracle" not in text and "pao_" not in text, fn

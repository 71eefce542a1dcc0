/*
 * pa.h - C ABI of the paged decode-attention library (libpa.so) for GB300 (sm_103a).
 *
 * The library implements the decode hot path of PagedAttention: single-query
 * attention over a KV cache held in fixed-size physical blocks reached through
 * per-sequence block tables, the slot-mapping append that writes new K/V into
 * the cache, and the whole-block copy used by copy-on-write.
 *
 * Sources (page title, section):
 *  [P1] "PagedAttention 详解：缓存的存储结构" - "Block Table", "软件地址翻译"
 *       (software address translation), "写入新 K/V" (writing new K/V).
 *  [P2] "PagedAttention 笔记" - "写时复制是正确性的边界" (copy-on-write).
 *  [P3] "vLLM 核心工程深度剖析" - "3.1 Kernel 签名与分块策略" (kernel signature),
 *       "4.1 Beam Search 中的 CoW" (block-level copy).
 *  [P4] "PagedAttention是什麼？" - "PagedAttention Kernel在做什麼？" (grid over
 *       sequence, head and partition; partition reduction for long contexts).
 *
 * Conventions shared by every call
 *  - All data pointers are DEVICE-ACCESSIBLE addresses owned by the caller.  No
 *    call allocates memory.  Between calls the library keeps only a lazily
 *    resolved driver entry point, per-kernel launch attributes and, for
 *    pa_decode_noalloc alone, one fixed scratch array per device (see there).
 *  - The K/V caches, the workspace and err_flag must be device memory (the
 *    caches are read by tensor-map copies).  For the decode calls, the appends
 *    and pa_copy_blocks, the small per-step arrays (q, out, block_tables,
 *    seq_lens, slot_mapping, new key/value, block_pairs, ALiBi slopes) may
 *    instead be pinned host memory mapped into the device's address space, as
 *    every cudaHostAlloc / cudaMallocHost allocation is under unified
 *    addressing: the kernels then read and write them in place over the host
 *    link (NVLink-C2C on GB300), with no copy in between, and the results are
 *    the same bytes as with device buffers.  pa_prefill moves q and out by
 *    tensor-map copies: those two must be device memory there.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Every call is asynchronous on that stream.
 *  - Cache layout (both K and V): [num_blocks][num_kv_heads][block_size][head_size],
 *    dense, element type `dtype`.  One (block, kv head) is one contiguous run of
 *    block_size * head_size elements.
 *  - Return value: PA_OK, or a PA_ERR_* code for an argument error detected on
 *    the host, in which case NOTHING is launched; PA_ERR_CUDA if a launch failed.
 *  - Data errors (a bad block ID or slot inside device arrays) are detected on
 *    the device, always: there is no switch that turns the checks off (each is
 *    one integer compare per block or slot, next to a memory access).  The
 *    offending item is skipped (never read or written out of bounds); if
 *    `err_flag` is non-NULL the first error code (PA_DEVERR_*) is stored there
 *    with an atomic compare-and-swap from 0.  `err_flag` is a device int32 the
 *    caller zeroes.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2, PA_FP8_E4M3 = 3 } pa_dtype;

/* Shape of one layer's KV cache pair. */
typedef struct {
  int32_t num_blocks;   /* physical blocks in the pool */
  int32_t block_size;   /* tokens per block B: f16/bf16 8 or a multiple of 16 (<= 256); fp8 a multiple of 16
                           (<= 256); f32 any B >= 1 */
  int32_t num_kv_heads; /* Hkv */
  int32_t head_size;    /* D: 64 or 128 (fp8: 128) */
  int32_t dtype;        /* pa_dtype of the cache, and of q/out and new key/value except for fp8 (see below) */
} pa_cache_desc;

/*
 * FP8 caches (dtype PA_FP8_E4M3).  ["PagedAttention 详解：缓存的存储结构"
 * "软件地址翻译": cache_t may be FP8, x = 16 / sizeof(cache_t) = 16 elements per
 * 16-byte access.]  The pages define nothing further; the reading implemented:
 *   - elements are OCP E4M3 codes (1 sign, 4 exponent bits with bias 7, 3
 *     mantissa bits; S.1111.111 is NaN; no infinities);
 *   - one fp32 scale per cache: a key code c stands for k_scale * e4m3(c), a
 *     value code for v_scale * e4m3(c) (scales > 0, passed per call);
 *   - keys   [num_blocks][num_kv_heads][block_size][head_size] bytes,
 *     values [num_blocks][num_kv_heads][block_size/16][head_size][16] bytes:
 *     the pages' value layout ([head_size][block_size], a dimension's tokens
 *     contiguous) tiled in 16-token groups, identical to it for block_size 16,
 *     so that the values of every 16 tokens of one head are contiguous;
 *   - q, out and the key/value rows written by pa_reshape_and_cache_fp8 are fp16;
 *   - written codes are the E4M3 code nearest to x / scale (fp32 division,
 *     ties to even; magnitudes past 448, infinities included, saturate to 448).
 */

/* Host-side status codes. */
enum {
  PA_OK = 0,
  PA_ERR_NULL_POINTER = 1, /* a required pointer is NULL */
  PA_ERR_UNSUPPORTED = 2,  /* dtype / head_size / block_size combination not built */
  PA_ERR_INVALID_ARG = 3,  /* negative size, Hq % Hkv != 0, bad partition size, ... */
  PA_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than pa_decode_workspace_size() */
  PA_ERR_MISALIGNED = 5,   /* a pointer is not aligned as documented */
  PA_ERR_CUDA = 6,         /* a CUDA runtime call or kernel launch failed */
  PA_ERR_TOO_LARGE = 7     /* sizes exceed the index ranges the kernels use */
};

/* Device-side data error codes written to *err_flag. */
enum {
  PA_DEVERR_NONE = 0,
  PA_DEVERR_BLOCK_ID = 1, /* a block_tables entry outside [0, num_blocks) */
  PA_DEVERR_SLOT = 2,     /* a slot_mapping entry >= num_blocks * block_size */
  PA_DEVERR_PAIR = 3,     /* a copy pair with an ID outside [0, num_blocks) */
  PA_DEVERR_TIMEOUT = 4,  /* a bounded wait on an asynchronous copy expired */
  PA_DEVERR_QUERY = 5     /* pa_prefill: a chunk outside [0, num_query_tokens), longer than
                             max_query_len or than its sequence, or a sequence past its table */
};

/*
 * pa_decode - one decode step of paged attention for one layer.
 *   [P3 "3.1"] signature: out/q [num_seqs, num_heads, head_size], block_tables
 *   [num_seqs, max_blocks_per_seq], context lengths, scale.
 *   [P1 "软件地址翻译"] token i of sequence s lives at offset i % B of block
 *   block_tables[s][i / B].
 *
 *   out[s][h][:] = sum_i softmax_i(scale * q[s][h] . k_i) * v_i over the
 *   seq_lens[s] tokens of sequence s, where k_i, v_i are the K/V rows of kv head
 *   h / (num_q_heads / num_kv_heads) (consecutive query heads share a kv head).
 *   Accumulation is in fp32; out is rounded to `dtype` round-to-nearest-even.
 *   seq_lens[s] == 0 writes a zero row.  Table entries at or beyond
 *   ceil(seq_lens[s] / B) are never read.
 *
 *   out          [num_seqs][num_q_heads][head_size] of dtype (written)
 *   q            [num_seqs][num_q_heads][head_size] of dtype, 16-byte aligned (f32: 4)
 *   k_cache, v_cache  cache pair (layout above), 16-byte aligned
 *   block_tables int32 [num_seqs][max_blocks_per_seq], row-major
 *   seq_lens     int32 [num_seqs]; each <= max_blocks_per_seq * block_size (not checked
 *                on the device beyond the table width: longer values are clamped)
 *   scale        softmax scale (usually 1/sqrt(head_size))
 *   partition_size  0 = library default (1024 tokens); else tokens per partition, a
 *                multiple of block_size and, for f16/bf16/fp8 caches, of 16 (the
 *                kernels' 16-token slabs never straddle a partition).  Sequences longer
 *                than one partition are split across CTAs and merged with a
 *                log-sum-exp reduction [P4 "PagedAttention Kernel在做什麼？"].
 *   workspace    device scratch of at least pa_decode_workspace_size(...) bytes,
 *                256-byte aligned; may be NULL when that size is 0.  Its
 *                contents on entry do not matter.
 *   err_flag     nullable device int32 (see above).
 *   Launches: the decode kernel, then (when a sequence spans two partitions) the
 *   merge kernel, both with programmatic stream serialization.  Their CTAs may be
 *   scheduled while the kernel before them on `stream` finishes.  They read
 *   seq_lens and block_tables at once, and execute griddepcontrol.wait before
 *   they read anything else (q, the caches, key/value, the workspace) or write
 *   anything, so stream order holds as for a plain launch provided that those
 *   two inputs are not written by a kernel that lets its dependents start
 *   early (no kernel of this library writes them; copies, and kernels that do
 *   not execute griddepcontrol.launch_dependents, complete first).  Stream
 *   capture records the dependencies as programmatic edges.
 */
int pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
              const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq,
              const pa_cache_desc* cache, float scale, int32_t partition_size, void* workspace,
              size_t workspace_bytes, int32_t* err_flag, void* stream);

/*
 * pa_decode_ex - pa_decode with optional extensions (options may be NULL, which
 * is exactly pa_decode).
 *   alibi_slopes  nullable device fp32 [num_q_heads], 4-byte aligned.  The kernel
 *                 signature of [P3 "3.1"] carries per-head ALiBi slopes without
 *                 defining them; the reading implemented is the standard linear
 *                 bias towards the query's own position: score_i of head h gains
 *                 alibi_slopes[h] * (i - (seq_lens[s] - 1)).
 *   k_scale, v_scale  the dequantisation scales of an FP8 cache (pa_decode uses 1).
 *   test_flags    0 in normal use.  PA_DECODE_TEST_EXPIRE_FIRST_WAIT exists for
 *                 tests of the kernels' hang protection (every wait on an
 *                 asynchronous copy is bounded, and an expired wait ends the
 *                 work item with PA_DEVERR_TIMEOUT once the copies already in
 *                 flight have landed): the f16/bf16/fp8 kernels then never
 *                 request the first slab of each warp's ring and bound the wait
 *                 for it at 20000 cycles, so it expires.  The call reports
 *                 PA_DEVERR_TIMEOUT in *err_flag and its output is undefined;
 *                 later calls are unaffected.  Ignored for fp32 caches, which
 *                 do not wait.
 */
#define PA_DECODE_TEST_EXPIRE_FIRST_WAIT 1u
typedef struct {
  const float* alibi_slopes;
  float k_scale; /* FP8 caches only (> 0); 0 means 1.  Ignored for other dtypes. */
  float v_scale; /* FP8 caches only (> 0); 0 means 1.  Ignored for other dtypes. */
  uint32_t test_flags; /* 0, or PA_DECODE_TEST_EXPIRE_FIRST_WAIT (tests only) */
} pa_decode_options;

int pa_decode_ex(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                 const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq,
                 const pa_cache_desc* cache, float scale, int32_t partition_size, void* workspace,
                 size_t workspace_bytes, int32_t* err_flag, void* stream, const pa_decode_options* options);

/*
 * pa_decode_append - one decode step with its append fused in: for every
 *   sequence s with seq_lens[s] = L > 0, the new token's key[s][h][:] and
 *   value[s][h][:] are stored at position L - 1 of both caches, i.e. at
 *   offset (L - 1) % B of block block_tables[s][(L - 1) / B]
 *   [P1 "写入新 K/V": slot = block * B + offset], and out is pa_decode's over
 *   positions 0 .. L - 1, the new token included.  The result and the cache
 *   contents equal pa_reshape_and_cache with those slots followed by pa_decode,
 *   in one launch (plus the merge when a sequence spans two partitions): the
 *   CTA that streams the new token's slab takes the token's rows from key and
 *   value, and the first query-head group of each kv head stores them.
 *
 *   key, value   [num_seqs][num_kv_heads][head_size] of dtype (fp16 for an FP8 cache),
 *                16-byte aligned
 *   options      nullable, as for pa_decode_ex (ALiBi slopes, FP8 scales)
 *   other arguments as for pa_decode; f16, bf16 and FP8 caches (fp32: use
 *   pa_reshape_and_cache and pa_decode).  Over an FP8 cache the rows are
 *   quantised as pa_reshape_and_cache_fp8 does (code of x / scale, fp32
 *   division, ties to even, saturating at +-448), bit for bit.  The slot at
 *   position L - 1 must belong to this sequence alone (the block manager copies
 *   a shared partial block on write first); a sequence's other slots are not
 *   written.
 */
int pa_decode_append(void* out, const void* q, void* k_cache, void* v_cache, const void* key, const void* value,
                     const int32_t* block_tables, const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads,
                     int32_t max_blocks_per_seq, const pa_cache_desc* cache, float scale, int32_t partition_size,
                     void* workspace, size_t workspace_bytes, int32_t* err_flag, void* stream,
                     const pa_decode_options* options);

/* Partition size pa_decode uses for these arguments (resolves 0 to the default);
 * returns a value >= max_blocks_per_seq * block_size when no split happens, or a
 * negative PA_ERR_* code for invalid arguments. */
int32_t pa_decode_partition_size(int32_t max_blocks_per_seq, const pa_cache_desc* cache, int32_t partition_size);

/* Bytes of workspace pa_decode needs: (head_size + 2) * 4 bytes (fp32 partial output,
 * maximum and sum) per row (sequence, query head) and partition slot, each part padded
 * to 256 bytes.  A row has P_max = ceil(max_blocks_per_seq * block_size / partition)
 * slots; on the fp16/bf16/FP8 kernels, when 2 <= P_max <= 8, the last num_seqs / 12
 * (fp16/bf16) or num_seqs / 24 (FP8) sequences (the grid's last items) are split into
 * partitions of half the size, if that half is a multiple of block_size and of 32,
 * and their rows have 2 P_max slots.  0 when no sequence can span two partitions.  Returns
 * 0 for invalid arguments as well (pa_decode then reports the argument error). */
size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq,
                                const pa_cache_desc* cache, int32_t partition_size);

/*
 * pa_prefill - chunked prefill attention over the paged cache.
 *   ["PagedAttention 详解：缓存的存储结构" "使用流程": prompt blocks that hit the
 *   prefix cache take part in attention directly, only missed blocks are
 *   computed and written through slot_mapping; "vLLM 核心工程深度剖析" "6.1":
 *   long prompts are prefilled in chunks.]
 *   Sequence s holds seq_lens[s] = L tokens in the cache (the chunk's own K/V
 *   already written, e.g. by pa_reshape_and_cache), the last
 *   n = query_start[s+1] - query_start[s] of which are this chunk's queries.
 *   Query j of head h (position L - n + j) attends causally to cache positions
 *   0 .. L - n + j: out = softmax_i(scale * q . k_i) v_i, fp32 accumulation,
 *   out rounded to dtype.
 *
 *   out, q           [num_query_tokens][num_q_heads][head_size], 16-byte aligned;
 *                    out rows outside every chunk are not written
 *   query_start      int32 [num_seqs + 1] on the device: chunk s is rows
 *                    query_start[s] .. query_start[s+1] - 1
 *   seq_lens         int32 [num_seqs], n <= L <= max_blocks_per_seq * block_size
 *   max_query_len    upper bound on n over the sequences (sizes the grid)
 *   scale            finite and > 0 (the softmax scale, e.g. 1/sqrt(head_size))
 *   A sequence whose chunk breaks these rules is skipped and PA_DEVERR_QUERY is
 *   reported; a bad block ID gives PA_DEVERR_BLOCK_ID and that sequence's
 *   output is undefined.
 *   Supported: dtype f16 / bf16, head_size 128, block_size 8, 16, 32, 64 or 128.
 *   Runs on the tcgen05 tensor cores: a persistent kernel, one CTA per SM,
 *   whose CTAs walk the work items (sequence, query head, tile of 128 queries).
 */
int pa_prefill(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
               const int32_t* seq_lens, const int32_t* query_start, int32_t num_seqs, int32_t num_query_tokens,
               int32_t num_q_heads, int32_t max_blocks_per_seq, int32_t max_query_len, const pa_cache_desc* cache,
               float scale, int32_t* err_flag, void* stream);

/*
 * pa_reshape_and_cache - append new tokens' K/V through slot_mapping.
 *   [P1 "写入新 K/V"] slot = block_id * B + offset; the kernel decodes
 *   block_id = slot / B, offset = slot % B and stores key[t][h][:] and
 *   value[t][h][:] at (block_id, h, offset) of k_cache / v_cache.
 *   A negative slot marks a padding token and is skipped.
 *
 *   key, value   [num_tokens][num_kv_heads][head_size] of dtype, dense, 16-byte aligned
 *   slot_mapping int64 [num_tokens]
 *   Slots must be distinct (two tokens with one slot race; either may win).
 */
int pa_reshape_and_cache(void* k_cache, void* v_cache, const void* key, const void* value,
                         const int64_t* slot_mapping, int32_t num_tokens, const pa_cache_desc* cache,
                         int32_t* err_flag, void* stream);

/*
 * pa_reshape_and_cache_fp8 - the append for an FP8 cache (dtype PA_FP8_E4M3):
 *   fp16 key/value [num_tokens][num_kv_heads][head_size] (16-byte aligned) are
 *   written as E4M3 codes of x / k_scale and x / v_scale (see "FP8 caches"
 *   above): key[t][h][d] at (block, h, offset, d), value[t][h][d] at (block, h,
 *   offset / 16, d, offset % 16).  Slots as for pa_reshape_and_cache.
 *   k_scale, v_scale > 0.
 */
int pa_reshape_and_cache_fp8(void* k_cache, void* v_cache, const void* key, const void* value,
                             const int64_t* slot_mapping, int32_t num_tokens, const pa_cache_desc* cache,
                             float k_scale, float v_scale, int32_t* err_flag, void* stream);

/*
 * pa_copy_blocks - the copy step of copy-on-write [P2 "写时复制是正确性的边界";
 *   P3 "4.1"]: for every pair, the whole physical block dst of both caches
 *   (all kv heads, all slots) becomes a copy of block src.
 *
 *   block_pairs  int32 [num_pairs][2] = (src, dst)
 *   Precondition: no dst appears twice and no dst is also a src (the pairs are
 *   copied concurrently).  A pair with src == dst is a no-op.
 */
int pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_pairs, int32_t num_pairs,
                   const pa_cache_desc* cache, int32_t* err_flag, void* stream);

/*
 * pa_decode_noalloc - pa_decode for callers that cannot allocate device memory
 *   while they decode (for example a serving plugin whose host engine owns all
 *   device memory, or a decode loop that must stay out of the CUDA allocator).
 *   The pages have no counterpart: this is a deployment convenience.
 *
 *   Same arguments and results as pa_decode, without workspace: the split-KV
 *   scratch is a library-owned device array of PA_NOALLOC_MAX_WORKSPACE_BYTES
 *   bytes.  Sizes whose pa_decode_workspace_size() exceeds that limit return
 *   PA_ERR_WORKSPACE and launch nothing.  The call itself allocates nothing.
 *   - Which sizes fit: the workspace is about num_seqs * num_q_heads * P_max *
 *     (head_size + 2) * 4 bytes (pa_decode_workspace_size gives it exactly).
 *     At the default 1024-token partition, 64 sequences x 32 heads of up to
 *     2048 tokens need 2.3 MB and 128 x 32 heads of up to 1280 tokens 4.6 MB;
 *     8 sequences x 32 heads of 32768 tokens in 512-token partitions need
 *     8.5 MB.  128 sequences x 64 query heads of up to 4096 tokens need 18.4 MB,
 *     over the limit: pass partition_size 2048 (9.2 MB) for them.  Sequences
 *     that fit one partition need none.
 *   - The first call on a device, whatever its sizes, looks up the array's
 *     device address with that device current and caches it.  Under CUDA's lazy
 *     module loading (the default) that lookup is also when the array is
 *     committed on the device, where it then stays until the process exits.
 *     Make that first call before any stream capture and outside any
 *     latency-critical loop.  It returns PA_ERR_CUDA if the lookup fails.
 *   - All calls share the one array and it keeps the previous call's contents;
 *     nothing in it needs clearing, but calls that overlap on the GPU (other
 *     streams, other host threads) race on it: order them on one stream.
 */
#define PA_NOALLOC_MAX_WORKSPACE_BYTES ((size_t)16 << 20)
int pa_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads,
                      int32_t max_blocks_per_seq, const pa_cache_desc* cache, float scale, int32_t partition_size,
                      int32_t* err_flag, void* stream);

/* Static description of a status code (never NULL). */
const char* pa_status_string(int status);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */

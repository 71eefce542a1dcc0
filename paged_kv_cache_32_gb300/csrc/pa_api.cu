// pa_api.cu - the C ABI of libpa: argument validation, tensor-map set-up and
// dispatch to the kernels.  Every host-side check runs before any CUDA call,
// so an argument error launches nothing (and needs no GPU to be reported).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <math.h>
#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace pa {
namespace host {

constexpr int32_t kDefaultPartition = 1024;  // tokens per partition when the caller passes 0 (measured best)
constexpr int32_t kTcSlab = 16;              // tokens per slab of the f16/bf16/fp8 decode kernels

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int elem_bytes(int32_t dtype) { return dtype == PA_F32 ? 4 : dtype == PA_FP8_E4M3 ? 1 : 2; }

// Shape checks common to every call.
int check_cache(const pa_cache_desc* c) {
  if (c == nullptr) return PA_ERR_NULL_POINTER;
  if (c->dtype != PA_F32 && c->dtype != PA_F16 && c->dtype != PA_BF16 && c->dtype != PA_FP8_E4M3)
    return PA_ERR_UNSUPPORTED;
  if (c->num_blocks < 0 || c->block_size <= 0 || c->num_kv_heads <= 0 || c->head_size <= 0)
    return PA_ERR_INVALID_ARG;
  if (c->head_size != 64 && c->head_size != 128) return PA_ERR_UNSUPPORTED;
  if (c->dtype == PA_FP8_E4M3 && c->head_size != 128) return PA_ERR_UNSUPPORTED;
  // fp8: whole 16-token value tiles; f16/bf16: 16-token slabs of one block, or of two 8-token blocks
  if (c->dtype == PA_FP8_E4M3 && (c->block_size % 16 != 0 || c->block_size > 256)) return PA_ERR_UNSUPPORTED;
  if ((c->dtype == PA_F16 || c->dtype == PA_BF16) &&
      !(c->block_size == 8 || (c->block_size % 16 == 0 && c->block_size <= 256)))
    return PA_ERR_UNSUPPORTED;
  // row index (block * Hkv + head) * B + slot must fit the kernels' int32 arithmetic
  if ((int64_t)c->num_blocks * c->num_kv_heads * c->block_size > kInt32Max) return PA_ERR_TOO_LARGE;
  return PA_OK;
}

// Resolved partition size, or a negative status.
int32_t resolve_partition(int32_t max_blocks_per_seq, const pa_cache_desc* c, int32_t requested) {
  const int rc = check_cache(c);
  if (rc != PA_OK) return -rc;
  if (max_blocks_per_seq < 0 || requested < 0) return -PA_ERR_INVALID_ARG;
  const int64_t max_len = (int64_t)max_blocks_per_seq * c->block_size;
  if (max_len > kInt32Max) return -PA_ERR_TOO_LARGE;
  int64_t part = requested;
  if (part == 0) {
    part = kDefaultPartition;
    if (part % c->block_size != 0) part = ((part + c->block_size - 1) / c->block_size) * c->block_size;
  } else if (part % c->block_size != 0) {
    return -PA_ERR_INVALID_ARG;
  }
  // the f16/bf16 kernel's 16-token slabs never straddle a partition boundary
  if (c->dtype != PA_F32 && part % kTcSlab != 0) return -PA_ERR_INVALID_ARG;
  if (part >= max_len) part = max_len > 0 ? max_len : c->block_size;  // no split needed
  return (int32_t)part;
}

int32_t num_partitions(int32_t max_blocks_per_seq, int32_t block_size, int32_t part) {
  const int64_t max_len = (int64_t)max_blocks_per_seq * block_size;
  return max_len <= part ? 1 : (int32_t)((max_len + part - 1) / part);
}

// The last twelfth of the sequences (fp16/bf16 caches) or twenty-fourth (FP8), the last items of the grid,
// are cut into partitions of half the size, so that the grid ends on shorter items.  Only for calls with a
// few partitions a sequence (longer splits are uniform already) on the tensor-core kernels, and when the
// half partition still holds whole blocks and whole 32-token slabs.  Measured against other shares (an
// eighth to a twenty-fourth) and quarter partitions on the GQA and FP8 steps: the 16-bit kernel, whose
// items take longer, gains most from a longer tail of short items.
struct TailPlan {
  int32_t seq0, ps, pmax;  // first tail sequence (num_seqs: none), its partition size, partition slots a row
};
constexpr int32_t kTailMaxPartitions = 8;
constexpr int32_t kTailShare16 = 12;  // 1 / kTailShare16 of the sequences over fp16/bf16 caches
constexpr int32_t kTailShareFp8 = 24; // 1 / kTailShareFp8 over FP8 caches
constexpr int32_t kTailCut = 2;       // partitions cut into kTailCut
TailPlan tail_plan(int32_t num_seqs, int32_t pmax, int32_t part, const pa_cache_desc* c) {
  const TailPlan none = {num_seqs, part, pmax};
  const int32_t n = num_seqs / (c->dtype == PA_FP8_E4M3 ? kTailShareFp8 : kTailShare16), ps = part / kTailCut;
  if (c->dtype == PA_F32 || pmax < 2 || pmax > kTailMaxPartitions || n == 0) return none;
  if (part % kTailCut != 0 || ps % c->block_size != 0 || ps % 32 != 0) return none;
  return {num_seqs - n, ps, kTailCut * pmax};
}

// Partition slots of a split call's workspace (one per row and partition slot).
size_t workspace_slots(int32_t num_seqs, int32_t num_q_heads, int32_t pmax, const TailPlan& t) {
  return ((size_t)t.seq0 * pmax + (size_t)(num_seqs - t.seq0) * t.pmax) * num_q_heads;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D view of a cache: rows = num_blocks * Hkv * B, columns = D elements;
// box = 64 columns (128 bytes, swizzled) x `slab` rows.
bool encode_cache_map(CUtensorMap* map, const void* base, const pa_cache_desc* c, int slab) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)c->head_size, (cuuint64_t)c->num_blocks * c->num_kv_heads * c->block_size};
  cuuint64_t strides[1] = {(cuuint64_t)c->head_size * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)slab};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      c->dtype == PA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// FP8 keys as rows of D bytes (box `rows` rows x 128 bytes, 128-byte swizzle); FP8 values need no map
// (every 16 tokens of one head are one contiguous run, read by 1-D bulk copies)
bool encode_fp8_key_map(CUtensorMap* tk, const void* k_cache, const pa_cache_desc* c, int rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint32_t estr[2] = {1, 1};
  const cuuint64_t heads = (cuuint64_t)c->num_blocks * c->num_kv_heads;
  cuuint64_t kdims[2] = {(cuuint64_t)c->head_size, heads * c->block_size};
  cuuint64_t kstrides[1] = {(cuuint64_t)c->head_size};
  cuuint32_t kbox[2] = {(cuuint32_t)c->head_size, (cuuint32_t)rows};
  CUresult r = enc(tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(k_cache), kdims, kstrides, kbox, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace host
}  // namespace pa

using namespace pa::host;

extern "C" {

int pa_version(void) { return 10100; }

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_NULL_POINTER: return "a required pointer is NULL";
    case PA_ERR_UNSUPPORTED: return "unsupported dtype / head_size / block_size";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_MISALIGNED: return "pointer misaligned";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_TOO_LARGE: return "sizes exceed the supported index range";
    default: return "unknown status";
  }
}

int32_t pa_decode_partition_size(int32_t max_blocks_per_seq, const pa_cache_desc* cache, int32_t partition_size) {
  return resolve_partition(max_blocks_per_seq, cache, partition_size);
}

size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq,
                                const pa_cache_desc* cache, int32_t partition_size) {
  const int32_t part = resolve_partition(max_blocks_per_seq, cache, partition_size);
  if (part <= 0 || num_seqs < 0 || num_q_heads <= 0) return 0;
  const int32_t pmax = num_partitions(max_blocks_per_seq, cache->block_size, part);
  if (pmax <= 1) return 0;
  const size_t slots = workspace_slots(num_seqs, num_q_heads, pmax, tail_plan(num_seqs, pmax, part, cache));
  const size_t o_bytes = slots * cache->head_size * sizeof(float);
  const size_t o_padded = (o_bytes + 255) / 256 * 256;
  return o_padded + slots * 2 * sizeof(float);
}

int pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
              const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq,
              const pa_cache_desc* cache, float scale, int32_t partition_size, void* workspace,
              size_t workspace_bytes, int32_t* err_flag, void* stream) {
  return pa_decode_ex(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_q_heads, max_blocks_per_seq,
                      cache, scale, partition_size, workspace, workspace_bytes, err_flag, stream, nullptr);
}

}  // extern "C"

// pa_decode_ex, and pa_decode_append when new_key / new_value are given
static int decode_call(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                       const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq,
                       const pa_cache_desc* cache, float scale, int32_t partition_size, void* workspace,
                       size_t workspace_bytes, int32_t* err_flag, void* stream, const pa_decode_options* options,
                       const void* new_key, const void* new_value) {
  int rc = check_cache(cache);
  if (rc != PA_OK) return rc;
  if (num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq < 0) return PA_ERR_INVALID_ARG;
  if (num_q_heads % cache->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
  if (!(scale == scale) || isinf(scale)) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (out == nullptr || q == nullptr || k_cache == nullptr || v_cache == nullptr || seq_lens == nullptr)
    return PA_ERR_NULL_POINTER;
  if (block_tables == nullptr && max_blocks_per_seq > 0) return PA_ERR_NULL_POINTER;
  const int32_t part = resolve_partition(max_blocks_per_seq, cache, partition_size);
  if (part < 0) return -part;
  const int32_t pmax = num_partitions(max_blocks_per_seq, cache->block_size, part);
  const size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, max_blocks_per_seq, cache, partition_size);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return PA_ERR_WORKSPACE;
  if (need > 0 && !aligned(workspace, 256)) return PA_ERR_MISALIGNED;
  // f16/bf16: caches and q are read by bulk copies (16-byte aligned); fp32: 4-byte loads
  const uintptr_t qalign = cache->dtype == PA_F32 ? 4 : 16;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, qalign) || !aligned(out, 4))
    return PA_ERR_MISALIGNED;
  const float* alibi = options != nullptr ? options->alibi_slopes : nullptr;
  if (alibi != nullptr && !aligned(alibi, 4)) return PA_ERR_MISALIGNED;
  float k_scale = options != nullptr ? options->k_scale : 0.f, v_scale = options != nullptr ? options->v_scale : 0.f;
  if (k_scale == 0.f) k_scale = 1.f;
  if (v_scale == 0.f) v_scale = 1.f;
  if (cache->dtype == PA_FP8_E4M3 && (!(k_scale > 0.f) || isinf(k_scale) || !(v_scale > 0.f) || isinf(v_scale)))
    return PA_ERR_INVALID_ARG;
  const int G = num_q_heads / cache->num_kv_heads;
  const int head_groups = (G + 7) / 8;
  const TailPlan tail = tail_plan(num_seqs, pmax, part, cache);
  const long long grid = (long long)tail.seq0 * cache->num_kv_heads * head_groups * pmax +
                         (long long)(num_seqs - tail.seq0) * cache->num_kv_heads * head_groups * tail.pmax;
  if (grid > kInt32Max || (long long)num_seqs * num_q_heads > kInt32Max) return PA_ERR_TOO_LARGE;

  pa::DecodeParams p;
  p.out = out;
  p.q = q;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.ws_o = nullptr;
  p.ws_ml = nullptr;
  if (need > 0) {
    const size_t slots = workspace_slots(num_seqs, num_q_heads, pmax, tail);
    const size_t o_padded = (slots * cache->head_size * sizeof(float) + 255) / 256 * 256;
    p.ws_o = static_cast<float*>(workspace);
    p.ws_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + o_padded);
  }
  p.err_flag = err_flag;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = cache->num_kv_heads;
  p.head_groups = head_groups;
  p.max_blocks = max_blocks_per_seq;
  p.block_size = cache->block_size;
  p.num_blocks = cache->num_blocks;
  p.partition_size = part;
  p.pmax = pmax;
  p.tail_seq0 = tail.seq0;
  p.tail_ps = tail.ps;
  p.tail_pmax = tail.pmax;
  p.scale_log2 = scale * 1.4426950408889634f;  // log2(e)
  p.alibi = alibi;
  p.test_expire_first_wait =
      (options != nullptr && (options->test_flags & PA_DECODE_TEST_EXPIRE_FIRST_WAIT) != 0u) ? 1 : 0;
  p.new_k = new_key;
  p.new_v = new_value;
  p.k_cache_out = const_cast<void*>(k_cache);
  p.v_cache_out = const_cast<void*>(v_cache);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (cache->dtype == PA_F32) {
    e = pa::launch_decode_f32(cache->head_size, static_cast<const float*>(k_cache),
                              static_cast<const float*>(v_cache), p, st);
  } else if (cache->dtype == PA_FP8_E4M3) {
    CUtensorMap tk, tk32;
    if (!encode_fp8_key_map(&tk, k_cache, cache, pa::kTcSlabTokens) ||
        !encode_fp8_key_map(&tk32, k_cache, cache, 2 * pa::kTcSlabTokens))
      return PA_ERR_CUDA;
    e = pa::launch_decode_fp8(cache->head_size, tk, tk32, v_cache, p, k_scale, v_scale, st);
  } else {
    CUtensorMap tk, tv;
    // a slab is one 16-row box, or (8-token blocks) two 8-row boxes from two blocks
    const int box_rows = cache->block_size < pa::kTcSlabTokens ? cache->block_size : pa::kTcSlabTokens;
    if (!encode_cache_map(&tk, k_cache, cache, box_rows) || !encode_cache_map(&tv, v_cache, cache, box_rows))
      return PA_ERR_CUDA;
    e = pa::launch_decode_tc(cache->dtype, cache->head_size, cache->block_size, tk, tv, p, st);
  }
  if (e != cudaSuccess) return PA_ERR_CUDA;
  if (pmax > 1) {  // partial outputs merge into the output dtype (fp16 for an FP8 cache)
    e = pa::launch_merge(cache->dtype == PA_FP8_E4M3 ? PA_F16 : cache->dtype, cache->head_size, p, st);
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

extern "C" {

int pa_decode_ex(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                 const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq,
                 const pa_cache_desc* cache, float scale, int32_t partition_size, void* workspace,
                 size_t workspace_bytes, int32_t* err_flag, void* stream, const pa_decode_options* options) {
  return decode_call(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_q_heads, max_blocks_per_seq,
                     cache, scale, partition_size, workspace, workspace_bytes, err_flag, stream, options, nullptr,
                     nullptr);
}

int pa_decode_append(void* out, const void* q, void* k_cache, void* v_cache, const void* key, const void* value,
                     const int32_t* block_tables, const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads,
                     int32_t max_blocks_per_seq, const pa_cache_desc* cache, float scale, int32_t partition_size,
                     void* workspace, size_t workspace_bytes, int32_t* err_flag, void* stream,
                     const pa_decode_options* options) {
  int rc = check_cache(cache);
  if (rc != PA_OK) return rc;
  if (cache->dtype == PA_F32) return PA_ERR_UNSUPPORTED;  // the tensor-core and FP8 kernels append
  if (num_seqs > 0 && (key == nullptr || value == nullptr)) return PA_ERR_NULL_POINTER;
  if (!aligned(key, 16) || !aligned(value, 16)) return PA_ERR_MISALIGNED;
  return decode_call(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_q_heads, max_blocks_per_seq,
                     cache, scale, partition_size, workspace, workspace_bytes, err_flag, stream, options, key, value);
}

int pa_reshape_and_cache(void* k_cache, void* v_cache, const void* key, const void* value,
                         const int64_t* slot_mapping, int32_t num_tokens, const pa_cache_desc* cache,
                         int32_t* err_flag, void* stream) {
  int rc = check_cache(cache);
  if (rc != PA_OK) return rc;
  if (cache->dtype == PA_FP8_E4M3) return PA_ERR_UNSUPPORTED;  // quantising append: pa_reshape_and_cache_fp8
  if (num_tokens < 0) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (k_cache == nullptr || v_cache == nullptr || key == nullptr || value == nullptr || slot_mapping == nullptr)
    return PA_ERR_NULL_POINTER;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(key, 16) || !aligned(value, 16) ||
      !aligned(slot_mapping, 8))
    return PA_ERR_MISALIGNED;
  const int32_t row_bytes = cache->head_size * elem_bytes(cache->dtype);
  cudaError_t e = pa::launch_reshape_and_cache(k_cache, v_cache, key, value, slot_mapping, num_tokens,
                                               cache->num_blocks, cache->block_size, cache->num_kv_heads, row_bytes,
                                               err_flag, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_reshape_and_cache_fp8(void* k_cache, void* v_cache, const void* key, const void* value,
                             const int64_t* slot_mapping, int32_t num_tokens, const pa_cache_desc* cache,
                             float k_scale, float v_scale, int32_t* err_flag, void* stream) {
  int rc = check_cache(cache);
  if (rc != PA_OK) return rc;
  if (cache->dtype != PA_FP8_E4M3) return PA_ERR_UNSUPPORTED;
  if (num_tokens < 0 || !(k_scale > 0.f) || isinf(k_scale) || !(v_scale > 0.f) || isinf(v_scale))
    return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (k_cache == nullptr || v_cache == nullptr || key == nullptr || value == nullptr || slot_mapping == nullptr)
    return PA_ERR_NULL_POINTER;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(key, 16) || !aligned(value, 16) ||
      !aligned(slot_mapping, 8))
    return PA_ERR_MISALIGNED;
  if ((int64_t)num_tokens * cache->num_kv_heads > kInt32Max) return PA_ERR_TOO_LARGE;
  cudaError_t e = pa::launch_reshape_and_cache_fp8(k_cache, v_cache, key, value, slot_mapping, num_tokens,
                                                   cache->num_blocks, cache->block_size, cache->num_kv_heads,
                                                   cache->head_size, k_scale, v_scale, err_flag,
                                                   static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_pairs, int32_t num_pairs,
                   const pa_cache_desc* cache, int32_t* err_flag, void* stream) {
  int rc = check_cache(cache);
  if (rc != PA_OK) return rc;
  if (num_pairs < 0) return PA_ERR_INVALID_ARG;
  if (num_pairs == 0) return PA_OK;
  if (k_cache == nullptr || v_cache == nullptr || block_pairs == nullptr) return PA_ERR_NULL_POINTER;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_pairs, 4)) return PA_ERR_MISALIGNED;
  const int64_t block_bytes =
      (int64_t)cache->num_kv_heads * cache->block_size * cache->head_size * elem_bytes(cache->dtype);
  const int64_t pieces = (block_bytes + 16383) / 16384;
  if (pieces * num_pairs > kInt32Max) return PA_ERR_TOO_LARGE;
  cudaError_t e = pa::launch_copy_blocks(k_cache, v_cache, block_pairs, num_pairs, cache->num_blocks, block_bytes,
                                         err_flag, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"

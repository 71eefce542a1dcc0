// pa_prefill_api.cu - the C-ABI entry point of chunked prefill attention:
// argument validation, the K/V tensor maps and the launch.  Every host-side
// check runs before any CUDA call, so an argument error launches nothing.
#include <cuda.h>
#include <cuda_runtime.h>

#include <math.h>

#include "pa.h"
#include "pa_internal.h"
#include "pa_prefill.h"

using namespace pa::host;

extern "C" {

int pa_prefill(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
               const int32_t* seq_lens, const int32_t* query_start, int32_t num_seqs, int32_t num_query_tokens,
               int32_t num_q_heads, int32_t max_blocks_per_seq, int32_t max_query_len, const pa_cache_desc* cache,
               float scale, int32_t* err_flag, void* stream) {
  int rc = check_cache(cache);
  if (rc != PA_OK) return rc;
  if ((cache->dtype != PA_F16 && cache->dtype != PA_BF16) || cache->head_size != 128) return PA_ERR_UNSUPPORTED;
  if (cache->block_size > 128 || 128 % cache->block_size != 0) return PA_ERR_UNSUPPORTED;
  if (num_seqs < 0 || num_query_tokens < 0 || num_q_heads <= 0 || max_blocks_per_seq < 0 || max_query_len < 0)
    return PA_ERR_INVALID_ARG;
  if (num_q_heads % cache->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || isinf(scale)) return PA_ERR_INVALID_ARG;  // the row max is taken on unscaled scores
  if (num_seqs == 0 || max_query_len == 0 || num_query_tokens == 0) return PA_OK;
  if (out == nullptr || q == nullptr || k_cache == nullptr || v_cache == nullptr || seq_lens == nullptr ||
      query_start == nullptr || block_tables == nullptr)
    return PA_ERR_NULL_POINTER;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) || !aligned(out, 16))
    return PA_ERR_MISALIGNED;
  const long long q_tiles = (max_query_len + 127) / 128;
  // work items (sequence, head, query tile) are counted in int32, with room for one grid stride past the end
  if ((long long)num_seqs * num_q_heads * q_tiles > kInt32Max - 4096) return PA_ERR_TOO_LARGE;
  if ((long long)max_blocks_per_seq * cache->block_size > kInt32Max) return PA_ERR_TOO_LARGE;
  if ((long long)num_query_tokens * num_q_heads * 128 > ((long long)1 << 40)) return PA_ERR_TOO_LARGE;

  auto enc = tensor_map_encoder();
  if (enc == nullptr) return PA_ERR_CUDA;
  CUtensorMap tk, tv, tq, to;
  if (!encode_cache_map(&tk, k_cache, cache, cache->block_size) ||
      !encode_cache_map(&tv, v_cache, cache, cache->block_size))
    return PA_ERR_CUDA;
  {
    // q and out [tokens][heads][D]: a 128-token tile of one head is one box of 64 columns x 1 x 128 per half
    cuuint64_t dims[3] = {(cuuint64_t)cache->head_size, (cuuint64_t)num_q_heads, (cuuint64_t)num_query_tokens};
    cuuint64_t strides[2] = {(cuuint64_t)cache->head_size * 2, (cuuint64_t)num_q_heads * cache->head_size * 2};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt =
        cache->dtype == PA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (enc(&tq, dt, 3, const_cast<void*>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&to, dt, 3, out, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PA_ERR_CUDA;
  }
  pa::PrefillParams p;
  p.out = out;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.query_start = query_start;
  p.err_flag = err_flag;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = cache->num_kv_heads;
  p.max_blocks = max_blocks_per_seq;
  p.block_size = cache->block_size;
  p.num_blocks = cache->num_blocks;
  p.q_tiles = (int32_t)q_tiles;
  p.num_query_tokens = num_query_tokens;
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaError_t e = pa::launch_prefill_tc(cache->dtype, tk, tv, tq, to, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"

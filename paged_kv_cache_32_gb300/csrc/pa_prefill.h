// pa_prefill.h - launch parameters of the tensor-core chunked prefill (not part
// of the public ABI).
#pragma once

#include "pa_internal.h"

namespace pa {

// Parameters of one chunked-prefill launch.
struct PrefillParams {
  void* out;                    // [total_q][Hq][D]
  const void* q;                // [total_q][Hq][D]
  const void* k_cache;          // [num_blocks][Hkv][B][D]
  const void* v_cache;
  const int32_t* block_tables;  // [N][M]
  const int32_t* seq_lens;      // [N] cached tokens including the chunk
  const int32_t* query_start;   // [N + 1]
  int32_t* err_flag;            // nullable
  int32_t num_seqs, num_q_heads, num_kv_heads;
  int32_t max_blocks, block_size, num_blocks;
  int32_t q_tiles;              // ceil(max_query_len / 128)
  int32_t num_query_tokens;     // rows of q and out
  float scale_log2;
};

// tk, tv: the caches as rows of D elements (box 64 columns x block_size rows, 128-byte swizzle);
// tq: q as [tokens][heads][D] (box 64 columns x 1 head x 128 tokens, 128-byte swizzle); to: out, the same
cudaError_t launch_prefill_tc(int dtype, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                              const CUtensorMap& to, const PrefillParams& p, cudaStream_t stream);

}  // namespace pa

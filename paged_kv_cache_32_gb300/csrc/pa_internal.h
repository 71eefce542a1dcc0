// pa_internal.h - launch parameters and kernel launchers shared by the
// translation units of libpa (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// Parameters of one decode launch (and of its partition merge).
struct DecodeParams {
  void* out;                  // [N][Hq][D] of the cache dtype
  const void* q;              // [N][Hq][D]
  const int32_t* block_tables;  // [N][M]
  const int32_t* seq_lens;    // [N]
  float* ws_o;                // [N][Hq][pmax][D] unnormalised partial outputs
  float* ws_ml;               // [N][Hq][pmax][2] (running max in log2 units, sum)
  int32_t* err_flag;          // nullable
  int32_t num_seqs, num_q_heads, num_kv_heads;
  int32_t head_groups;        // ceil(G / 8): CTAs per kv head, 8 query heads each
  int32_t max_blocks;         // M
  int32_t block_size;         // B
  int32_t num_blocks;
  int32_t partition_size;     // tokens per partition (multiple of B)
  int32_t pmax;               // partitions per sequence in the grid
  // Sequences tail_seq0 .. num_seqs - 1 (the last in the grid's order) are cut into partitions of tail_ps
  // tokens, tail_pmax per sequence in the grid, so that the grid ends on short items (tail_seq0 =
  // num_seqs: none).  Their partials follow the others' in the workspace, tail_pmax slots a row.
  int32_t tail_seq0, tail_ps, tail_pmax;
  float scale_log2;           // scale * log2(e)
  const float* alibi;         // nullable [Hq]: score_i += slope_h * (i - (L - 1))
  int32_t test_expire_first_wait;  // test hook: each ring's first slab is never requested (0 in normal use)
  // pa_decode_append (nullable otherwise): the new token of each sequence, [N][Hkv][D], stored at position
  // L - 1 of both caches and attended in the same launch
  const void* new_k;
  const void* new_v;
  void* k_cache_out;
  void* v_cache_out;
};

// Partition size of sequence s.
__host__ __device__ inline int seq_partition_size(const DecodeParams& p, int s) {
  return s >= p.tail_seq0 ? p.tail_ps : p.partition_size;
}
// Partition slots per row of sequence s in the workspace.
__host__ __device__ inline int seq_partition_slots(const DecodeParams& p, int s) {
  return s >= p.tail_seq0 ? p.tail_pmax : p.pmax;
}
// Workspace slot of partition 0 of row (sequence s, query head h); the row's partitions follow it.
__host__ __device__ inline size_t ws_row_slot(const DecodeParams& p, int s, int h) {
  if (s < p.tail_seq0) return ((size_t)s * p.num_q_heads + h) * p.pmax;
  return (size_t)p.tail_seq0 * p.num_q_heads * p.pmax + ((size_t)(s - p.tail_seq0) * p.num_q_heads + h) * p.tail_pmax;
}
// CTAs of a decode launch: one per (sequence, kv head, head group, partition slot).
__host__ __device__ inline long long decode_grid_size(const DecodeParams& p) {
  const long long per_seq = (long long)p.num_kv_heads * p.head_groups;
  return (long long)p.tail_seq0 * per_seq * p.pmax + (long long)(p.num_seqs - p.tail_seq0) * per_seq * p.tail_pmax;
}
// The work item of CTA id: sequence, kv-head group slot hh (kv head * head_groups + group) and partition.
// The host keeps the grid within int32, so the divisions are 32-bit.
__host__ __device__ inline void decode_item_ids(const DecodeParams& p, int id, int& s, int& hh, int& part) {
  const int per_seq = p.num_kv_heads * p.head_groups;
  const int grid_a = p.tail_seq0 * per_seq * p.pmax;
  if (id < grid_a) {
    part = id % p.pmax;
    hh = (id / p.pmax) % per_seq;
    s = id / (p.pmax * per_seq);
  } else {
    const int j = id - grid_a;
    part = j % p.tail_pmax;
    hh = (j / p.tail_pmax) % per_seq;
    s = p.tail_seq0 + j / (p.tail_pmax * per_seq);
  }
}

// Kernel launchers (return the cudaGetLastError of the launch).
cudaError_t launch_decode_tc(int dtype, int head_size, int block_size, const CUtensorMap& tk, const CUtensorMap& tv,
                             const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode_f32(int head_size, const float* k_cache, const float* v_cache, const DecodeParams& p,
                              cudaStream_t stream);
// tk: FP8 keys in 16-row boxes; tk32: the same in 32-row boxes (used when the block size is a multiple of 32)
cudaError_t launch_decode_fp8(int head_size, const CUtensorMap& tk, const CUtensorMap& tk32, const void* v_cache,
                              const DecodeParams& p, float k_scale, float v_scale, cudaStream_t stream);
cudaError_t launch_merge(int dtype, int head_size, const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_reshape_and_cache_fp8(void* k_cache, void* v_cache, const void* key, const void* value,
                                         const int64_t* slot_mapping, int32_t num_tokens, int32_t num_blocks,
                                         int32_t block_size, int32_t num_kv_heads, int32_t head_size,
                                         float k_scale, float v_scale, int32_t* err_flag, cudaStream_t stream);
cudaError_t launch_reshape_and_cache(void* k_cache, void* v_cache, const void* key, const void* value,
                                     const int64_t* slot_mapping, int32_t num_tokens, int32_t num_blocks,
                                     int32_t block_size, int32_t num_kv_heads, int32_t row_bytes,
                                     int32_t* err_flag, cudaStream_t stream);
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int32_t num_pairs,
                               int32_t num_blocks, int64_t block_bytes, int32_t* err_flag, cudaStream_t stream);

// Launch `kernel` as a programmatic dependent of the kernel before it on `stream`:
// its CTAs may be scheduled once every CTA of that kernel has executed
// griddepcontrol.launch_dependents (or exited), so the launch and CTA start-up
// overlap that kernel's end.  The kernel must execute griddepcontrol.wait before
// it reads anything the previous kernel writes or writes anything it reads.
template <typename... Params, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                    Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Host-side helpers of the C ABI (pa_api.cu), shared by the entry points in other files.
namespace host {
constexpr int64_t kInt32Max = 2147483647;
bool aligned(const void* p, uintptr_t a);
int elem_bytes(int32_t dtype);
int check_cache(const pa_cache_desc* c);  // shape checks common to every call
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
// 2-D tensor map over a cache pool viewed as rows of head_size elements, box of `slab` rows x 64 columns
bool encode_cache_map(CUtensorMap* map, const void* base, const pa_cache_desc* c, int slab);
// FP8 keys: rows of D bytes (boxes of `rows` rows, 128-byte swizzle)
bool encode_fp8_key_map(CUtensorMap* tk, const void* k_cache, const pa_cache_desc* c, int rows);
}  // namespace host

// Slab (TMA box height in tokens) of the tensor-core decode: 16 tokens of one
// block; the kernel's stage layout and transaction counts assume exactly this.
constexpr int kTcSlabTokens = 16;

}  // namespace pa

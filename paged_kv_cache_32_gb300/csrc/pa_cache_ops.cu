// pa_cache_ops.cu - the cache writes: the slot-mapping append and the
// copy-on-write block copy.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// ---------------------------------------------------------------------------
// Slot-mapping append ("PagedAttention 详解：缓存的存储结构", section "写入新
// K/V"): block = slot / B, offset = slot % B; the token's [Hkv][D] key and
// value rows go to (block, h, offset) of each cache.  Grid (token, chunk):
// every thread moves one 16-byte vector of K and one of V, so a step's few
// new tokens finish in one load-store round trip.  Negative slots are padding.
// ---------------------------------------------------------------------------
constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads)
    reshape_and_cache_kernel(uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                             const uint8_t* __restrict__ key, const uint8_t* __restrict__ value,
                             const int64_t* __restrict__ slot_mapping, int32_t num_blocks, int32_t block_size,
                             int32_t num_kv_heads, int32_t row_bytes, int32_t* err_flag) {
  griddep_launch_dependents();  // a decode launched as a dependent may be scheduled behind this grid
  const int t = blockIdx.x;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  const int64_t block = slot / block_size;
  const int64_t off = slot % block_size;
  if (block >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0) report_error(err_flag, PA_DEVERR_SLOT);
    return;
  }
  const int vec_per_row = row_bytes / 16;
  const int i = blockIdx.y * kAppendThreads + threadIdx.x;
  if (i >= num_kv_heads * vec_per_row) return;
  const int h = i / vec_per_row;
  const int c = i % vec_per_row;
  const size_t src = ((size_t)t * num_kv_heads + h) * row_bytes + (size_t)c * 16;
  const size_t dst = (((size_t)block * num_kv_heads + h) * block_size + off) * row_bytes + (size_t)c * 16;
  const uint4 kx = __ldg(reinterpret_cast<const uint4*>(key + src));
  const uint4 vx = __ldg(reinterpret_cast<const uint4*>(value + src));
  *reinterpret_cast<uint4*>(k_cache + dst) = kx;
  *reinterpret_cast<uint4*>(v_cache + dst) = vx;
}

cudaError_t launch_reshape_and_cache(void* k_cache, void* v_cache, const void* key, const void* value,
                                     const int64_t* slot_mapping, int32_t num_tokens, int32_t num_blocks,
                                     int32_t block_size, int32_t num_kv_heads, int32_t row_bytes,
                                     int32_t* err_flag, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int vectors = num_kv_heads * (row_bytes / 16);
  dim3 grid((unsigned)num_tokens, (unsigned)((vectors + kAppendThreads - 1) / kAppendThreads));
  reshape_and_cache_kernel<<<grid, kAppendThreads, 0, stream>>>(
      static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), static_cast<const uint8_t*>(key),
      static_cast<const uint8_t*>(value), slot_mapping, num_blocks, block_size, num_kv_heads, row_bytes, err_flag);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Block copy for copy-on-write ("PagedAttention 笔记", section "写时复制是
// 正确性的边界"; "vLLM 核心工程深度剖析", section "4.1 Beam Search 中的 CoW"):
// block dst of a cache becomes a copy of block src.  Grid: x = pair * pieces
// + piece, y = cache (K, V); each CTA moves one 16 KB piece with 16-byte
// vectors, four loads in flight per thread.
// ---------------------------------------------------------------------------
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;
constexpr int kCopyPiece = kCopyThreads * kCopyUnroll * 16;

__global__ void __launch_bounds__(kCopyThreads)
    copy_blocks_kernel(uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                       const int32_t* __restrict__ pairs, int32_t num_blocks, int64_t block_bytes,
                       int32_t pieces, int32_t* err_flag) {
  griddep_launch_dependents();  // a decode launched as a dependent may be scheduled behind this grid
  const int pair = blockIdx.x / pieces;
  const int piece = blockIdx.x % pieces;
  const int32_t src = pairs[2 * pair];
  const int32_t dst = pairs[2 * pair + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && piece == 0 && blockIdx.y == 0) report_error(err_flag, PA_DEVERR_PAIR);
    return;
  }
  if (src == dst) return;
  uint8_t* cache = blockIdx.y == 0 ? k_cache : v_cache;
  const uint8_t* from = cache + (size_t)src * block_bytes;
  uint8_t* to = cache + (size_t)dst * block_bytes;
  const int64_t begin = (int64_t)piece * kCopyPiece;
  uint4 r[kCopyUnroll];
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) {
    const int64_t off = begin + ((int64_t)u * kCopyThreads + threadIdx.x) * 16;
    if (off < block_bytes) r[u] = __ldg(reinterpret_cast<const uint4*>(from + off));
  }
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) {
    const int64_t off = begin + ((int64_t)u * kCopyThreads + threadIdx.x) * 16;
    if (off < block_bytes) *reinterpret_cast<uint4*>(to + off) = r[u];
  }
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int32_t num_pairs,
                               int32_t num_blocks, int64_t block_bytes, int32_t* err_flag, cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  const int32_t pieces = (int32_t)((block_bytes + kCopyPiece - 1) / kCopyPiece);
  dim3 grid((unsigned)((int64_t)pieces * num_pairs), 2);
  copy_blocks_kernel<<<grid, kCopyThreads, 0, stream>>>(static_cast<uint8_t*>(k_cache),
                                                        static_cast<uint8_t*>(v_cache), pairs, num_blocks,
                                                        block_bytes, pieces, err_flag);
  return cudaGetLastError();
}

}  // namespace pa

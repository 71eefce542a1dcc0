// pa_noalloc.cu - pa_decode_noalloc: paged decode attention whose split-KV
// scratch lives in a fixed device array owned by the library, so the call
// itself allocates nothing.
//
// Who needs it: callers that cannot allocate device memory when they decode.
// Examples are a serving plugin whose host engine owns and pre-plans every byte
// of device memory, or a latency-critical decode loop that must not enter the
// CUDA allocator (cudaMalloc can synchronise the device and stall for far
// longer than a decode step).  Such a caller passes its inputs and output
// buffers as usual and lets the library use the scratch array below.
//
// Cost: every GPU on which this call has run once holds kScratchBytes of
// device memory for the scratch array until the process exits.  With CUDA's
// lazy module loading (the default) the array is committed on a device when
// the first call there looks up its address, not when the library is loaded.
#include <cuda_runtime.h>

#include <mutex>

#include "pa.h"

namespace {

constexpr size_t kScratchBytes = PA_NOALLOC_MAX_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

// The scratch.  In host code this name is only a host-side stand-in for the
// device symbol: it must never be passed to a kernel.  Its device address
// comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, resolved on the first
// call per device (with that device current) and cached.  NULL on failure.
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = ptr;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" int pa_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_tables, const int32_t* seq_lens, int32_t num_seqs,
                                 int32_t num_q_heads, int32_t max_blocks_per_seq, const pa_cache_desc* cache,
                                 float scale, int32_t partition_size, int32_t* err_flag, void* stream) {
  // cache-shape and partition errors are reported before any CUDA call, as pa_decode does
  const int32_t part = pa_decode_partition_size(max_blocks_per_seq, cache, partition_size);
  if (part < 0) return -part;
  const size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, max_blocks_per_seq, cache, partition_size);
  if (need > kScratchBytes) return PA_ERR_WORKSPACE;  // these sizes need more scratch than the array holds
  // Resolved on every call, also when this call needs no scratch: the first
  // call on a device (a warm-up with short sequences, say) then does the
  // one-time lookup, never a later call that may sit inside a stream capture.
  // After the first call per device this is a cached read.
  void* scratch = scratch_address();
  if (scratch == nullptr) return PA_ERR_CUDA;
  // The decode kernels write every scratch slot they later read, so nothing
  // has to be cleared between calls.
  return pa_decode(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_q_heads, max_blocks_per_seq,
                   cache, scale, partition_size, scratch, need > 0 ? kScratchBytes : 0, err_flag, stream);
}

// pa_decode_tc.cu - paged decode attention for fp16 / bf16 caches on sm_103a.
//
// What it computes ("vLLM 核心工程深度剖析", section "3.1 Kernel 签名与分块策略";
// "PagedAttention 详解：缓存的存储结构", section "软件地址翻译"): for every sequence
// s and query head h, out = softmax(scale * q K^T) V over the sequence's
// seq_lens[s] tokens, where token i's key/value row sits at offset i % B of
// physical block block_tables[s][i / B].  Long sequences are cut into
// partitions whose partial results a second kernel merges with a log-sum-exp
// reduction ("PagedAttention是什麼？", section "PagedAttention Kernel在做什麼？").
//
// How (GB300 design, not the pages' CUDA-core kernel):
//  * One CTA per work item = (sequence, kv head, group of <= 8 query heads,
//    partition); all query heads of a GQA group share one pass over the K/V
//    bytes.  Several CTAs share an SM, and the hardware hands a finished
//    CTA's slot to the next item, which balances uneven sequence lengths.
//  * The item's tokens are cut into "slabs" of 16 tokens of one block; the
//    CTA's NW warps take the slabs round-robin.  Every warp is its own
//    producer and consumer: it keeps a private ring of NS shared-memory slab
//    buffers filled with 2-D tensor-map copies (cp.async.bulk.tensor, 128-byte
//    swizzle, completion counted in bytes on a per-buffer mbarrier), reading
//    the block IDs from the table 32 slabs at a time across its lanes.  Each
//    SM therefore has many independent copy issuers and NS - 1 slabs in flight
//    per warp; a ring's buffers are refilled and drained by the same warp in
//    order, so the parity-based barrier waits cannot alias.
//  * Per slab a warp computes S^T[16 tokens x 8 heads] = K Q^T and
//    O^T[D x 8 heads] += V^T P^T on the tensor cores (mma.m16n8k16, fp32
//    accumulate) from ldmatrix reads of the swizzled tiles, with movmatrix
//    turning the probability tile from accumulator into operand layout, and an
//    online softmax (running max and sum per head, fp32; the max moves only when
//    a score exceeds it by more than 8 in log2 units).  The warps' partial
//    results are merged through shared memory once, at the end of the item.
//  The path is bound by HBM bandwidth (1 to 8 flop per byte); the tensor cores
//  only keep the instruction count per byte low.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "pa.h"
#include "pa_decode_epilogue.cuh"
#include "pa_decode_slab.cuh"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

constexpr long long kWaitCycles = 500ll * 1000 * 1000;  // bound on one wait: ~0.25 s at 2 GHz
constexpr long long kTestWaitCycles = 20000;              // the test hook's bound on a ring's first wait

template <int D, int NW, int NS>
struct Shape {
  static constexpr int SB = kTcSlabTokens;                 // tokens per slab (= TMA box rows)
  static constexpr int KSTEPS = D / 16;                    // k-steps of Q K^T = m-tiles of V^T P^T
  static constexpr int NBOX = D / 64;                      // 128-byte (64-element) TMA boxes per row
  static constexpr int BOX_BYTES = SB * 128;               // one box: 16 rows x 128 bytes
  static constexpr int SLAB_BYTES = 2 * NBOX * BOX_BYTES;  // K boxes, then V boxes
  static constexpr int RING_BYTES = NS * SLAB_BYTES;       // per warp
  static constexpr int OROW = D + 4;                       // merge row stride (floats): conflict-free stores
  static constexpr int WARP_MERGE = 8 * OROW + 16;         // per warp: O[8][OROW], (m, l)[8]
  static constexpr int BAR_OFF = NW * RING_BYTES;
  static constexpr int FLAG_OFF = BAR_OFF + NW * NS * 8;   // the CTA's abort flag
  static constexpr int STAGE_OFF = FLAG_OFF + 16;         // the appended token's K and V rows (16-bit)
  static constexpr int SMEM_BYTES = STAGE_OFF + 2 * D * 2 + 1024;  // + alignment slack
  static constexpr int THREADS = NW * 32;
  static_assert(D % 64 == 0, "head_size must be a multiple of 64");
  static_assert(NS >= 2, "a ring needs at least two buffers");
  static_assert(RING_BYTES >= WARP_MERGE * 4, "a warp's ring holds its partial result at the end");
};

// One work item.
struct Item {
  int s, hkv, hq0, gcount, part;
  int L;           // tokens of the sequence
  int t_end;       // end of this partition
  int j0;          // first slab (16 tokens) of the partition
  int nslabs;
  bool final_out;  // the sequence has a single partition: write the normalised output
};

__device__ __forceinline__ bool decode_item(const DecodeParams& p, int id, Item& it) {
  int hh;
  decode_item_ids(p, id, it.s, hh, it.part);
  const int ps = seq_partition_size(p, it.s);
  it.hkv = hh / p.head_groups;
  const int hg = hh % p.head_groups;
  const int G = p.num_q_heads / p.num_kv_heads;
  it.hq0 = it.hkv * G + hg * 8;
  it.gcount = min(8, G - hg * 8);
  int L = __ldg(p.seq_lens + it.s);
  L = max(0, min(L, p.max_blocks * p.block_size));
  it.L = L;
  const int t_begin = it.part * ps;
  if (L == 0) {  // an empty sequence: partition 0 writes a zero row
    it.t_end = 0;
    it.j0 = 0;
    it.nslabs = 0;
    it.final_out = true;
    return it.part == 0;
  }
  if (t_begin >= L) return false;
  it.t_end = min(L, t_begin + ps);
  it.j0 = t_begin / kTcSlabTokens;
  it.nslabs = (it.t_end - t_begin + kTcSlabTokens - 1) / kTcSlabTokens;
  it.final_out = L <= ps;
  return true;
}

// Wait for a barrier phase; gives up (returning false) when the CTA's abort
// flag is set or after `limit` SM cycles, in which case it raises the flag.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int32_t* abort_flag,
                                           long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long start = clock64();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((i & 15u) == 15u && clock64() - start > limit) {
      *abort_flag = 1;
      return false;
    }
  }
}

// The decode step's append (pa_decode_append): the sequence's new token sits at position L - 1,
// in this slab's row r.  Its key and value rows replace that row of the slab's shared-memory tiles
// (the copy brought whatever the slot held before), and the CTA of the first head group also stores
// them into the cache at the slot the block table gives, for later steps; no other CTA of this
// launch reads that slot ("PagedAttention 详解：缓存的存储结构", section "写入新 K/V": the new token's K/V
// goes to slot block * B + offset).  Lane l moves 16-byte chunk l % CH of the key (l < CH) or the
// value row, which it copied into stage_rows at the start of the kernel (so the global load's latency
// is not paid here); the async proxy refills the buffer later, so the lanes fence their generic writes.
template <typename T, int D>
__device__ __forceinline__ void append_token(const DecodeParams& p, const Item& it, uint8_t* kst, int r, int lane,
                                             const uint8_t* stage_rows) {
  constexpr int CH = D * (int)sizeof(T) / 16;  // 16-byte chunks per row
  constexpr int BOX_BYTES = kTcSlabTokens * 128;
  const int G = p.num_q_heads / p.num_kv_heads;
  if (lane < 2 * CH) {
    const bool is_v = lane >= CH;
    const int c = lane % CH;
    asm volatile("cp.async.wait_all;" ::: "memory");
    const uint4 x = *reinterpret_cast<const uint4*>(stage_rows + 16 * lane);
    uint8_t* tile = kst + (is_v ? (D / 64) * BOX_BYTES : 0);
    *reinterpret_cast<uint4*>(tile + (c / 8) * BOX_BYTES + swz128(r, c % 8)) = x;
    if (it.hq0 == it.hkv * G) {  // the first head group of the kv head writes the cache
      const int pos = it.L - 1;
      const int pb = __ldg(p.block_tables + (size_t)it.s * p.max_blocks + pos / p.block_size);
      if (pb >= 0 && pb < p.num_blocks) {
        const size_t dst = (((size_t)pb * p.num_kv_heads + it.hkv) * p.block_size + pos % p.block_size) * CH + c;
        reinterpret_cast<uint4*>(is_v ? p.v_cache_out : p.k_cache_out)[dst] = x;
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncwarp();
}

template <typename T, int D, int NW, int NS>
__global__ void __launch_bounds__(Shape<D, NW, NS>::THREADS)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                     const DecodeParams p) {
  using S = Shape<D, NW, NS>;
  griddep_launch_dependents();  // the partition merge may be scheduled behind this grid's last CTAs
  // seq_lens and block_tables are read before griddepcontrol.wait: no kernel of this library writes them.
  // q and the ALiBi slopes, which a GEMM before this kernel may produce, are read after it; the CTA's q
  // rows are only prefetched into L2 before it (a later load of them sees the final data).
  Item it;
  if (!decode_item(p, blockIdx.x, it)) return;  // partition past the end of its sequence

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;   // fragment row group
  const int q4 = lane & 3;   // fragment column pair
  uint8_t* ring = smem + warp * S::RING_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BAR_OFF) + warp * NS;
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + S::FLAG_OFF);
  // ---- this warp's slabs: j = warp + k * NW, k < n_my
  const int n_my = it.nslabs > warp ? (it.nslabs - warp + NW - 1) / NW : 0;
  const int B = p.block_size;
  const bool split = B < S::SB;  // 8-token blocks: a slab is two 8-row halves from two blocks
  const int32_t* table = p.block_tables + (size_t)it.s * p.max_blocks;
  // lane l holds the table entries of this warp's slab 32 b + l: its (first) block, and with 8-token
  // blocks that of its second half (-1 when the half lies past the partition)
  auto fetch = [&](int kk, int& e0, int& e1) {
    e0 = e1 = -1;
    if (kk < n_my) {
      const int tok0 = (it.j0 + warp + kk * NW) * S::SB;
      e0 = __ldg(table + tok0 / B);
      if (split && tok0 + B < it.t_end) e1 = __ldg(table + tok0 / B + 1);
    }
  };
  int pb_batch = 0, pb_reg, pb_reg2;
  fetch(lane, pb_reg, pb_reg2);

  if (warp == 0)
    prefetch_l2(reinterpret_cast<const T*>(p.q) + ((size_t)it.s * p.num_q_heads + it.hq0) * D,
                it.gcount * D * (int)sizeof(T), lane);
  if (threadIdx.x == 0) {
    abort_flag[0] = 0;
    tma_prefetch_descriptor(&tmap_k);
    tma_prefetch_descriptor(&tmap_v);
  }
  if (lane == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
  }
  __syncthreads();

  griddep_wait();  // launched as a dependent: the previous kernel's writes (cache, output) are visible from here
  // ---- query fragments (B operand of S^T = K Q^T): head g, dims 16j + 2q4 (+8)
  uint32_t qf[S::KSTEPS][2];
  {
    const bool real = g < it.gcount;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(reinterpret_cast<const T*>(p.q) +
                                                             ((size_t)it.s * p.num_q_heads + it.hq0 + g) * D);
#pragma unroll
    for (int j = 0; j < S::KSTEPS; ++j) {
      qf[j][0] = real ? __ldg(qrow + (16 * j + 2 * q4) / 2) : 0u;
      qf[j][1] = real ? __ldg(qrow + (16 * j + 2 * q4 + 8) / 2) : 0u;
    }
  }

  // ALiBi slopes of this lane's two heads, in log2 units (0: no bias)
  float bias_a = 0.f, bias_b = 0.f;
  if (p.alibi != nullptr) {
    constexpr float kLog2e = 1.4426950408889634f;
    if (2 * q4 < it.gcount) bias_a = __ldg(p.alibi + it.hq0 + 2 * q4) * kLog2e;
    if (2 * q4 + 1 < it.gcount) bias_b = __ldg(p.alibi + it.hq0 + 2 * q4 + 1) * kLog2e;
  }

  // the appended token's rows: the warp whose slab holds position L - 1 starts copying them now,
  // so that they are in shared memory when that slab is processed
  uint8_t* stage_rows = smem + S::STAGE_OFF;
  {
    constexpr int CH = D * 2 / 16;
    const int apos = it.L - 1;
    if (p.new_k != nullptr && apos >= it.j0 * S::SB && apos < it.t_end && ((apos / S::SB - it.j0) % NW) == warp &&
        lane < 2 * CH) {
      const size_t row = (size_t)it.s * p.num_kv_heads + it.hkv;
      const void* src = reinterpret_cast<const uint4*>(lane >= CH ? p.new_v : p.new_k) + row * CH + lane % CH;
      const uint32_t dst = (uint32_t)__cvta_generic_to_shared(stage_rows + 16 * lane);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n\tcp.async.commit_group;" ::"r"(dst), "l"(src)
                   : "memory");
    }
  }

  uint32_t valid_mask = 0;  // bit `stage`: the slab in that buffer was loaded
  auto issue = [&](int k) {  // called by the whole warp, k increasing
    if ((k >> 5) != pb_batch) {
      pb_batch = k >> 5;
      fetch(k + lane, pb_reg, pb_reg2);
    }
    const int pb = __shfl_sync(0xffffffffu, pb_reg, k & 31);
    const int pb2 = __shfl_sync(0xffffffffu, pb_reg2, k & 31);
    const int tok0 = (it.j0 + warp + k * NW) * S::SB;
    const bool has2 = split && tok0 + B < it.t_end;  // the second 8-token half holds tokens of the item
    const bool valid = pb >= 0 && pb < p.num_blocks && (!has2 || (pb2 >= 0 && pb2 < p.num_blocks));
    const int stage = k % NS;
    valid_mask = valid ? (valid_mask | (1u << stage)) : (valid_mask & ~(1u << stage));
    if (lane == 0) {
      uint64_t* bar = &bars[stage];
      uint8_t* dst = ring + stage * S::SLAB_BYTES;
      if (valid && !split) {
        const int y = (pb * p.num_kv_heads + it.hkv) * B + tok0 % B;  // first row
        mbar_arrive_expect_tx(bar, S::SLAB_BYTES);
#pragma unroll
        for (int b = 0; b < S::NBOX; ++b) tma_load_2d(dst + b * S::BOX_BYTES, &tmap_k, b * 64, y, bar);
#pragma unroll
        for (int b = 0; b < S::NBOX; ++b) tma_load_2d(dst + (S::NBOX + b) * S::BOX_BYTES, &tmap_v, b * 64, y, bar);
      } else if (valid) {
        // 8-row boxes: rows 8u .. 8u + 7 of each 16-row box region come from block pb (u = 0) or pb2 (u = 1),
        // 1024 bytes apart, which keeps the 128-byte swizzle of a 16-row box.  Rows of an absent second half
        // are left as they are: the slab step masks tokens past the item.
        mbar_arrive_expect_tx(bar, has2 ? S::SLAB_BYTES : S::SLAB_BYTES / 2);
        for (int u = 0; u < (has2 ? 2 : 1); ++u) {
          const int y = ((u ? pb2 : pb) * p.num_kv_heads + it.hkv) * B;
#pragma unroll
          for (int b = 0; b < S::NBOX; ++b)
            tma_load_2d(dst + b * S::BOX_BYTES + u * (S::BOX_BYTES / 2), &tmap_k, b * 64, y, bar);
#pragma unroll
          for (int b = 0; b < S::NBOX; ++b)
            tma_load_2d(dst + (S::NBOX + b) * S::BOX_BYTES + u * (S::BOX_BYTES / 2), &tmap_v, b * 64, y, bar);
        }
      } else {
        report_error(p.err_flag, PA_DEVERR_BLOCK_ID);
        mbar_arrive(bar);  // complete the phase without data; the slab is skipped
      }
    }
  };

  float o[S::KSTEPS][4];
#pragma unroll
  for (int i = 0; i < S::KSTEPS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY;  // running max (log2 units) of heads 2q4, 2q4+1
  float l_a = 0.f, l_b = 0.f;              // this lane's share of the running sums

  // test hook (pa_decode_options.test_flags): slab 0 of each ring is never requested and the
  // first wait has a short bound, so that wait expires and the abort path below runs
  const int first_issued = p.test_expire_first_wait ? 1 : 0;
  const int prologue = n_my < NS ? n_my : NS;
  for (int k = first_issued; k < prologue; ++k) issue(k);
  int k = 0;
  for (; k < n_my; ++k) {
    const int stage = k % NS;
    const long long limit = (k == 0 && p.test_expire_first_wait) ? kTestWaitCycles : kWaitCycles;
    if (!__all_sync(0xffffffffu, wait_phase(&bars[stage], (k / NS) & 1, abort_flag, limit))) break;
    if ((valid_mask >> stage) & 1u) {
      const int tok0 = (it.j0 + warp + k * NW) * S::SB;
      const int nvalid = min(S::SB, it.t_end - tok0);
      uint8_t* kst = ring + stage * S::SLAB_BYTES;
      if (p.new_k != nullptr && it.L - 1 < tok0 + S::SB && it.L - 1 >= tok0) append_token<T, D>(p, it, kst, it.L - 1 - tok0, lane, stage_rows);
      process_slab<T, D>(kst, kst + S::NBOX * S::BOX_BYTES, nvalid, qf, o, m_a, m_b, l_a, l_b, lane, p.scale_log2,
                         bias_a, bias_b, (float)(tok0 - (it.L - 1)));
    }
    __syncwarp();
    if (k + NS < n_my) issue(k + NS);
  }
  asm volatile("cp.async.wait_all;" ::: "memory");  // the staged rows' copy, if its slab was skipped
  if (k < n_my) {  // timed out: let this warp's copies already in flight land first
    report_error(p.err_flag, PA_DEVERR_TIMEOUT);
    const int issued = n_my < k + NS ? n_my : k + NS;
    if (lane == 0)
      for (int kk = k > first_issued ? k : first_issued; kk < issued; ++kk) drain_phase(&bars[kk % NS], (kk / NS) & 1);
    __syncwarp();
  }

  // ---- per-warp totals into the warp's (now idle) ring, then merge the warps
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l_a += __shfl_xor_sync(0xffffffffu, l_a, off);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, off);
  }
  float* wo = reinterpret_cast<float*>(ring);  // [8 heads][OROW], then [8 heads][2]
  float* wml = wo + 8 * S::OROW;
#pragma unroll
  for (int i = 0; i < S::KSTEPS; ++i) {
    wo[(2 * q4) * S::OROW + 16 * i + g] = o[i][0];
    wo[(2 * q4 + 1) * S::OROW + 16 * i + g] = o[i][1];
    wo[(2 * q4) * S::OROW + 16 * i + g + 8] = o[i][2];
    wo[(2 * q4 + 1) * S::OROW + 16 * i + g + 8] = o[i][3];
  }
  if (g == 0) {
    wml[(2 * q4) * 2] = m_a;
    wml[(2 * q4) * 2 + 1] = l_a;
    wml[(2 * q4 + 1) * 2] = m_b;
    wml[(2 * q4 + 1) * 2 + 1] = l_b;
  }
  __syncthreads();

  finish_item<T, D, NW, S::OROW, S::RING_BYTES>(smem, p, (size_t)it.s * p.num_q_heads + it.hq0, it.gcount,
                                                it.final_out, ws_row_slot(p, it.s, it.hq0) + it.part,
                                                seq_partition_slots(p, it.s));
}

// ------------------------------------------------------------------ launch
template <typename T, int D, int NW, int NS>
static cudaError_t launch_tc(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                             cudaStream_t stream) {
  using S = Shape<D, NW, NS>;
  auto kernel = decode_tc_kernel<T, D, NW, NS>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long items = decode_grid_size(p);
  if (items == 0) return cudaSuccess;
  return launch_dependent(kernel, dim3((unsigned)items), dim3(S::THREADS), S::SMEM_BYTES, stream, tk, tv, p);
}

// Four warps per CTA, two slab buffers per warp (64 KB per CTA at D = 128):
// three CTAs, i.e. twelve copy-issuing warps, per SM.  Measured best among
// 1-8 warps x 2-4 buffers on the MHA, GQA and long-context workloads.
template <typename T>
static cudaError_t dispatch_tc(int head_size, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                               cudaStream_t stream) {
  if (head_size == 128) return launch_tc<T, 128, 4, 2>(tk, tv, p, stream);
  if (head_size == 64) return launch_tc<T, 64, 4, 4>(tk, tv, p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_tc(int dtype, int head_size, int block_size, const CUtensorMap& tk, const CUtensorMap& tv,
                             const DecodeParams& p, cudaStream_t stream) {
  (void)block_size;
  if (dtype == PA_F16) return dispatch_tc<__half>(head_size, tk, tv, p, stream);
  if (dtype == PA_BF16) return dispatch_tc<__nv_bfloat16>(head_size, tk, tv, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa

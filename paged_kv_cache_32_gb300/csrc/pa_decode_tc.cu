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
//  * Work item = (sequence, kv head, group of <= 8 query heads, partition).
//    All query heads of a GQA group share one pass over the K/V bytes.
//  * Persistent CTAs (one per SM) walk a static round-robin list of items.
//    Inside a CTA one producer warp streams "slabs" (16 tokens of one block,
//    K and V) through a deep ring of shared-memory stages with 2-D tensor-map
//    copies (cp.async.bulk.tensor, 128-byte swizzle), completion counted on
//    per-stage mbarriers.  It reads the block IDs from the table a batch of 32
//    ahead and never waits for compute except when the ring is full, and it
//    runs on into the next item while the consumers finish the current one,
//    so HBM sees one continuous stream per SM.
//  * NC consumer warps take the slabs round-robin (slab kk -> warp kk % NC).
//    Stage s = kk % NS is filled only by producer s % NP and drained only by
//    consumer s % NC, so each stage's uses are issued and consumed in order
//    and parity-based barrier waits never alias.  Per 16-token
//    slab a warp computes S^T[16 tokens x 8 heads] = K Q^T and
//    O^T[D x 8 heads] += V^T P^T on the tensor cores (mma.m16n8k16, fp32
//    accumulate) from ldmatrix reads of the swizzled tiles, with movmatrix
//    turning the probability tile from accumulator into operand layout, and an
//    online softmax (running max and sum per head, fp32).  At the end of an
//    item the consumers merge their partial results through shared memory.
//  The path is bound by HBM bandwidth (1 to 8 flop per byte); the tensor cores
//  only keep the instruction count per byte low.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

constexpr long long kWaitCycles = 500ll * 1000 * 1000;  // bound on one wait: ~0.25 s at 2 GHz

// bf16 probabilities are split into a rounded part and its residual (see the value MMA)
template <typename T>
constexpr bool kSplitP = false;
template <>
constexpr bool kSplitP<__nv_bfloat16> = true;

template <int D, int NC, int NP, int NS>
struct Pipe {
  static constexpr int SB = kTcSlabTokens;                 // tokens per slab (= TMA box rows)
  static constexpr int KSTEPS = D / 16;                    // k-steps of Q K^T = m-tiles of V^T P^T
  static constexpr int NBOX = D / 64;                      // 128-byte (64-element) TMA boxes per row
  static constexpr int BOX_BYTES = SB * 128;               // one box: 16 rows x 128 bytes
  static constexpr int SLAB_BYTES = 2 * NBOX * BOX_BYTES;  // K boxes, then V boxes
  static constexpr int RING_BYTES = NS * SLAB_BYTES;
  static constexpr int OROW = D + 4;                       // merge row stride (floats): conflict-free stores
  static constexpr int WARP_MERGE = 8 * OROW + 16;         // per consumer warp: O[8][OROW], (m, l)[8]
  static constexpr int MERGE_OFF = RING_BYTES;
  static constexpr int Q_OFF = MERGE_OFF + NC * WARP_MERGE * 4;
  static constexpr int Q_BYTES = 8 * D * 2;                // one item's query rows (<= 8 heads)
  static constexpr int FULL_OFF = Q_OFF + 2 * Q_BYTES;
  static constexpr int EMPTY_OFF = FULL_OFF + NS * 8;
  static constexpr int QFULL_OFF = EMPTY_OFF + NS * 8;
  static constexpr int QEMPTY_OFF = QFULL_OFF + 2 * 8;
  static constexpr int VALID_OFF = QEMPTY_OFF + 2 * 8;
  static constexpr int ABORT_OFF = VALID_OFF + NS * 4;     // abort flag, then a word that stays 0
  static constexpr int SMEM_BYTES = ABORT_OFF + 16 + 1024;  // + alignment slack
  static constexpr int THREADS = (NC + NP) * 32;
  static_assert(D % 64 == 0, "head_size must be a multiple of 64");
  static_assert(NS % NP == 0 && NS % NC == 0, "each stage has one producer and one consumer warp");
  static_assert(Q_OFF % 16 == 0 && FULL_OFF % 8 == 0, "alignment of the q buffers and barriers");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// One work item, decoded identically by the producer and the consumers.
struct Item {
  int s, hkv, hq0, gcount, part;
  int t_end;      // end of this partition
  int j0;         // first slab (16 tokens) of the partition
  int nslabs;
  bool final_out;  // the sequence has a single partition: write the normalised output
};

__device__ __forceinline__ bool decode_item(const DecodeParams& p, int id, Item& it) {
  const int per_seq = p.num_kv_heads * p.head_groups;
  it.part = id % p.pmax;
  const int hh = (id / p.pmax) % per_seq;
  it.s = id / (p.pmax * per_seq);
  it.hkv = hh / p.head_groups;
  const int hg = hh % p.head_groups;
  const int G = p.num_q_heads / p.num_kv_heads;
  it.hq0 = it.hkv * G + hg * 8;
  it.gcount = min(8, G - hg * 8);
  int L = __ldg(p.seq_lens + it.s);
  L = max(0, min(L, p.max_blocks * p.block_size));
  const int t_begin = it.part * p.partition_size;
  if (L == 0) {  // an empty sequence: partition 0 writes a zero row
    it.t_end = 0;
    it.j0 = 0;
    it.nslabs = 0;
    it.final_out = true;
    return it.part == 0;
  }
  if (t_begin >= L) return false;
  it.t_end = min(L, t_begin + p.partition_size);
  it.j0 = t_begin / kTcSlabTokens;
  it.nslabs = (it.t_end - t_begin + kTcSlabTokens - 1) / kTcSlabTokens;
  it.final_out = L <= p.partition_size;
  return true;
}

// First item id >= `id` (stepping by `stride`) that has work; `total` if none.
__device__ __forceinline__ int next_active(const DecodeParams& p, int id, int stride, int total, Item& it) {
  while (id < total && !decode_item(p, id, it)) id += stride;
  return id;
}

// Wait for a barrier phase; gives up (returning false) when the CTA's abort
// flag is set or after kWaitCycles SM cycles, in which case it raises the flag.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int32_t* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long start = clock64();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((i & 15u) == 15u && clock64() - start > kWaitCycles) {
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

template <typename T, int D, int NC, int NP, int NS>
__global__ void __launch_bounds__(Pipe<D, NC, NP, NS>::THREADS, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                     const DecodeParams p) {
  using S = Pipe<D, NC, NP, NS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  float* merge = reinterpret_cast<float*>(smem + S::MERGE_OFF);
  uint8_t* qbuf = smem + S::Q_OFF;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::FULL_OFF);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + S::EMPTY_OFF);
  uint64_t* qfull = reinterpret_cast<uint64_t*>(smem + S::QFULL_OFF);
  uint64_t* qempty = reinterpret_cast<uint64_t*>(smem + S::QEMPTY_OFF);
  volatile int32_t* stage_valid = reinterpret_cast<volatile int32_t*>(smem + S::VALID_OFF);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + S::ABORT_OFF);
  volatile int32_t* never_flag = abort_flag + 1;  // stays 0: waits that must not be cut short

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int total_items = p.num_seqs * p.num_kv_heads * p.head_groups * p.pmax;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], NC);
    }
    abort_flag[0] = 0;
    never_flag[0] = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp >= NC) {
    // ======================= producer warps =======================
    // A tensor copy takes a producer thread a few hundred cycles to issue, so NP
    // warps issue in parallel.  Producer pw owns the stages s with s % NP == pw
    // (NS is a multiple of NP) and issues exactly the slabs kk with
    // kk % NP == pw, in order, so every use of a stage is issued by one warp
    // right after the previous use was released (no phase aliasing).  All
    // producers walk the same item sequence; producer 0 also copies each item's
    // query rows.  Lane 0 issues; the other lanes fetch block-table entries
    // (32 slabs per batch), the next item's first batch while the current item
    // streams, so no dependent global load sits between items.
    const int pw = warp - NC;
    tma_prefetch_descriptor(&tmap_k);
    tma_prefetch_descriptor(&tmap_v);
    const int B = p.block_size;
    auto table_batch = [&](const Item& it, int j) -> int {
      const int jj = j + lane;
      return jj < it.nslabs ? __ldg(p.block_tables + (size_t)it.s * p.max_blocks + ((it.j0 + jj) * S::SB) / B) : -1;
    };
    Item cur, nxt;
    int cur_id = next_active(p, blockIdx.x, gridDim.x, total_items, cur);
    int nxt_id = cur_id < total_items ? next_active(p, cur_id + gridDim.x, gridDim.x, total_items, nxt) : total_items;
    int pb_cur = cur_id < total_items ? table_batch(cur, 0) : -1;
    int pb_nxt = nxt_id < total_items ? table_batch(nxt, 0) : -1;
    uint32_t kk = 0;      // slabs issued by this CTA so far
    uint32_t n_item = 0;  // items started by this CTA so far
    bool ok = true;
    while (ok && cur_id < total_items) {
      // ---- the item's query rows -> q buffer (n_item & 1)
      if (lane == 0 && pw == 0) {
        const int qb = n_item & 1;
        if (n_item >= 2) ok = wait_phase(&qempty[qb], ((n_item >> 1) - 1) & 1, abort_flag);
        if (ok) {
          const uint32_t bytes = cur.gcount * D * 2;
          mbar_arrive_expect_tx(&qfull[qb], bytes);
          bulk_load_1d(qbuf + qb * S::Q_BYTES,
                       reinterpret_cast<const T*>(p.q) + ((size_t)cur.s * p.num_q_heads + cur.hq0) * D, bytes,
                       &qfull[qb]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      // ---- the item's K/V slabs
      for (int j = 0; ok && j < cur.nslabs; ++j, ++kk) {
        if (j > 0 && (j & 31) == 0) pb_cur = table_batch(cur, j);
        const int pb = __shfl_sync(0xffffffffu, pb_cur, j & 31);
        if ((int)(kk % NP) != pw) continue;  // another producer's slab
        const int stage = kk % NS;
        if (lane == 0 && kk >= (uint32_t)NS) ok = wait_phase(&empty[stage], ((kk / NS) - 1) & 1, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          uint64_t* bar = &full[stage];
          const bool valid = pb >= 0 && pb < p.num_blocks;
          stage_valid[stage] = valid;
          if (valid) {
            const int y = (pb * p.num_kv_heads + cur.hkv) * B + ((cur.j0 + j) * S::SB) % B;  // first row
            uint8_t* dst = ring + stage * S::SLAB_BYTES;
            mbar_arrive_expect_tx(bar, S::SLAB_BYTES);
#pragma unroll
            for (int b = 0; b < S::NBOX; ++b) tma_load_2d(dst + b * S::BOX_BYTES, &tmap_k, b * 64, y, bar);
#pragma unroll
            for (int b = 0; b < S::NBOX; ++b)
              tma_load_2d(dst + (S::NBOX + b) * S::BOX_BYTES, &tmap_v, b * 64, y, bar);
          } else {
            report_error(p.err_flag, PA_DEVERR_BLOCK_ID);
            mbar_arrive(bar);  // complete the phase without data; consumers skip the slab
          }
        }
        __syncwarp();
      }
      // ---- advance: the prefetched next item becomes current
      ++n_item;
      cur = nxt;
      cur_id = nxt_id;
      pb_cur = pb_nxt;
      if (cur_id < total_items) {
        nxt_id = next_active(p, cur_id + gridDim.x, gridDim.x, total_items, nxt);
        pb_nxt = nxt_id < total_items ? table_batch(nxt, 0) : -1;
      }
    }
    if (!ok) {
      report_error(p.err_flag, PA_DEVERR_TIMEOUT);
      // let copies already in flight land before the CTA's shared memory is released
      if (lane == 0) {
        const uint32_t first = kk > (uint32_t)NS ? kk - NS : 0;
        for (uint32_t k = first; k < kk; ++k)
          if ((int)(k % NP) == pw) wait_phase(&full[k % NS], (k / NS) & 1, never_flag);
        if (pw == 0 && n_item >= 1) wait_phase(&qfull[(n_item - 1) & 1], ((n_item - 1) >> 1) & 1, never_flag);
        if (pw == 0 && n_item >= 2) wait_phase(&qfull[n_item & 1], ((n_item - 2) >> 1) & 1, never_flag);
      }
    }
    return;
  }

  // ======================= consumer warps =======================
  const int g = lane >> 2;   // fragment row group
  const int q4 = lane & 3;   // fragment column pair
  const float sl2 = p.scale_log2;
  uint32_t kk_base = 0;
  uint32_t n_item = 0;
  for (int id = blockIdx.x; id < total_items; id += gridDim.x) {
    Item it;
    if (!decode_item(p, id, it)) continue;
    // (no early exit: every consumer warp must reach both barriers of every
    // item; after an abort the waits below return at once instead)

    // query fragments (B operand of S^T = K Q^T): head g, dims 16j + 2q4 (+8)
    uint32_t qf[S::KSTEPS][2];
    {
      const int qb = n_item & 1;
      __all_sync(0xffffffffu, wait_phase(&qfull[qb], (n_item >> 1) & 1, abort_flag));
      const bool real = g < it.gcount;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(qbuf + qb * S::Q_BYTES + g * D * 2);
#pragma unroll
      for (int j = 0; j < S::KSTEPS; ++j) {
        qf[j][0] = real ? qrow[(16 * j + 2 * q4) / 2] : 0u;
        qf[j][1] = real ? qrow[(16 * j + 2 * q4 + 8) / 2] : 0u;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&qempty[qb]);
    }
    ++n_item;
    float o[S::KSTEPS][4];
#pragma unroll
    for (int i = 0; i < S::KSTEPS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY;  // running max (log2 units) of heads 2q4, 2q4+1
    float l_a = 0.f, l_b = 0.f;              // this lane's share of the running sums

    // slab kk goes to consumer kk % NC: with NS a multiple of NC every stage is
    // consumed by one warp, which therefore waits for its uses strictly in order
    // (a warp never tests a stage's barrier two phases ahead).
    for (int j = (int)((warp + NC - kk_base % NC) % NC); j < it.nslabs; j += NC) {
      const uint32_t kk = kk_base + j;
      const int stage = kk % NS;
      if (!__all_sync(0xffffffffu, wait_phase(&full[stage], (kk / NS) & 1, abort_flag))) break;
      if (stage_valid[stage]) {
        const int nvalid = min(S::SB, it.t_end - (it.j0 + j) * S::SB);
        const uint8_t* kst = ring + stage * S::SLAB_BYTES;
        const uint8_t* vst = kst + S::NBOX * S::BOX_BYTES;
        // ---- S^T[16 tokens x 8 heads] = K_slab Q^T (two accumulators: shorter dependency chain)
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        float sd[4] = {0.f, 0.f, 0.f, 0.f};
        {
          const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
          const int khalf = lane >> 4;
#pragma unroll
          for (int jj = 0; jj < S::KSTEPS; ++jj) {
            const uint32_t addr = smem_u32(kst + (jj >> 2) * S::BOX_BYTES) + swz128(row, (jj & 3) * 2 + khalf);
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4(addr, a0, a1, a2, a3);
            if (jj & 1)
              Mma<T>::run(sd, a0, a1, a2, a3, qf[jj][0], qf[jj][1]);
            else
              Mma<T>::run(sc, a0, a1, a2, a3, qf[jj][0], qf[jj][1]);
          }
        }
        // scores: (token g, head 2q4), (token g, head 2q4+1), (token g+8, head 2q4), (token g+8, head 2q4+1)
        float s0 = (sc[0] + sd[0]) * sl2, s1 = (sc[1] + sd[1]) * sl2;
        float s2 = (sc[2] + sd[2]) * sl2, s3 = (sc[3] + sd[3]) * sl2;
        if (nvalid < 16) {
          if (g >= nvalid) s0 = s1 = -INFINITY;
          if (g + 8 >= nvalid) s2 = s3 = -INFINITY;
        }
        float mx_a = fmaxf(s0, s2), mx_b = fmaxf(s1, s3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, off));
          mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, off));
        }
        const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
        const float al_a = fast_exp2(m_a - mn_a), al_b = fast_exp2(m_b - mn_b);
        m_a = mn_a;
        m_b = mn_b;
        const float p0 = fast_exp2(s0 - mn_a), p1 = fast_exp2(s1 - mn_b);
        const float p2 = fast_exp2(s2 - mn_a), p3 = fast_exp2(s3 - mn_b);
        const uint32_t x0 = Mma<T>::pack(p0, p1);
        const uint32_t x1 = Mma<T>::pack(p2, p3);
        // bf16 keeps only 8 significant bits of P; its rounding residual goes
        // through a second MMA so P enters the value sum with ~16 bits.
        uint32_t y0 = 0, y1 = 0;
        if constexpr (kSplitP<T>) {
          y0 = Mma<T>::pack(p0 - Mma<T>::lo(x0), p1 - Mma<T>::hi(x0));
          y1 = Mma<T>::pack(p2 - Mma<T>::lo(x1), p3 - Mma<T>::hi(x1));
          l_a = l_a * al_a + (p0 + p2);
          l_b = l_b * al_b + (p1 + p3);
        } else {  // fp16: the sums use the rounded probabilities the value MMA multiplies with
          l_a = l_a * al_a + (Mma<T>::lo(x0) + Mma<T>::lo(x1));
          l_b = l_b * al_b + (Mma<T>::hi(x0) + Mma<T>::hi(x1));
        }
#pragma unroll
        for (int i = 0; i < S::KSTEPS; ++i) {
          o[i][0] *= al_a;
          o[i][1] *= al_b;
          o[i][2] *= al_a;
          o[i][3] *= al_b;
        }
        // P^T fragments: (tokens 2q4, 2q4+1 | +8, +9 ; head g)
        const uint32_t pb0 = movmatrix_trans(x0);
        const uint32_t pb1 = movmatrix_trans(x1);
        uint32_t pc0 = 0, pc1 = 0;
        if constexpr (kSplitP<T>) {
          pc0 = movmatrix_trans(y0);
          pc1 = movmatrix_trans(y1);
        }
        // ---- O^T[D x 8 heads] += V_slab^T P^T
        {
          const int row = (lane & 7) + (lane >> 4) * 8;
          const int dhalf = (lane >> 3) & 1;
#pragma unroll
          for (int i = 0; i < S::KSTEPS; ++i) {
            const uint32_t addr = smem_u32(vst + (i >> 2) * S::BOX_BYTES) + swz128(row, (i & 3) * 2 + dhalf);
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4_trans(addr, a0, a1, a2, a3);
            if (nvalid < 16) {  // zero values of tokens past the end (they may hold NaN)
              const int t0 = 2 * q4, t1 = 2 * q4 + 8;
              const uint32_t mlo = (t0 < nvalid ? 0x0000ffffu : 0u) | (t0 + 1 < nvalid ? 0xffff0000u : 0u);
              const uint32_t mhi = (t1 < nvalid ? 0x0000ffffu : 0u) | (t1 + 1 < nvalid ? 0xffff0000u : 0u);
              a0 &= mlo;
              a1 &= mlo;
              a2 &= mhi;
              a3 &= mhi;
            }
            Mma<T>::run(o[i], a0, a1, a2, a3, pb0, pb1);
            if constexpr (kSplitP<T>) Mma<T>::run(o[i], a0, a1, a2, a3, pc0, pc1);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);  // stage free for the producer
    }
    kk_base += it.nslabs;

    // ---- per-warp totals into shared memory, then merge the warps
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l_a += __shfl_xor_sync(0xffffffffu, l_a, off);
      l_b += __shfl_xor_sync(0xffffffffu, l_b, off);
    }
    float* wo = merge + warp * S::WARP_MERGE;  // [8 heads][OROW], then [8 heads][2]
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
    consumer_sync(NC * 32);

    const size_t row0 = (size_t)it.s * p.num_q_heads + it.hq0;
    for (int idx = threadIdx.x; idx < it.gcount * D; idx += NC * 32) {
      const int gh = idx / D, d = idx % D;
      float mstar = -INFINITY;
#pragma unroll
      for (int w = 0; w < NC; ++w) mstar = fmaxf(mstar, merge[w * S::WARP_MERGE + 8 * S::OROW + gh * 2]);
      float lsum = 0.f, acc = 0.f;
      if (mstar != -INFINITY) {
#pragma unroll
        for (int w = 0; w < NC; ++w) {
          const float* wb = merge + w * S::WARP_MERGE;
          const float wt = fast_exp2(wb[8 * S::OROW + gh * 2] - mstar);
          lsum += wt * wb[8 * S::OROW + gh * 2 + 1];
          acc += wt * wb[gh * S::OROW + d];
        }
      }
      if (it.final_out) {
        T* out = reinterpret_cast<T*>(p.out);
        out[(row0 + gh) * D + d] = from_float<T>(lsum > 0.f ? acc / lsum : 0.f);
      } else {
        const size_t slot = (row0 + gh) * p.pmax + it.part;
        p.ws_o[slot * D + d] = acc;
        if (d == 0) {
          p.ws_ml[slot * 2] = mstar;
          p.ws_ml[slot * 2 + 1] = lsum;
        }
      }
    }
    consumer_sync(NC * 32);  // merge buffer free again
  }
}

// ------------------------------------------------------------------ launch
static int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

template <typename T, int D, int NC, int NP, int NS>
static cudaError_t launch_tc(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                             cudaStream_t stream) {
  using S = Pipe<D, NC, NP, NS>;
  auto kernel = decode_tc_kernel<T, D, NC, NP, NS>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long items = (long long)p.num_seqs * p.num_kv_heads * p.head_groups * p.pmax;
  if (items == 0) return cudaSuccess;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const unsigned grid = (unsigned)(items < sms ? items : sms);
  kernel<<<grid, S::THREADS, S::SMEM_BYTES, stream>>>(tk, tv, p);
  return cudaGetLastError();
}

// One persistent CTA per SM: 8 consumer warps + 4 producer warps; the ring
// takes the shared memory left after the consumers' merge buffers.
template <typename T>
static cudaError_t dispatch_tc(int head_size, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                               cudaStream_t stream) {
  if (head_size == 128) return launch_tc<T, 128, 8, 4, 16>(tk, tv, p, stream);
  if (head_size == 64) return launch_tc<T, 64, 8, 4, 48>(tk, tv, p, stream);
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

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
//  * One CTA per (sequence, kv head, group of <= 8 query heads, partition).
//    All query heads of a GQA group share one pass over the K/V bytes.
//  * Cache layout [blocks][kv_heads][B][D]: one (block, kv head) is one
//    contiguous B x D tile.  Each "slab" (16 or 32 tokens of one block) of K
//    and of V is fetched by the tensor-memory-access engine
//    (cp.async.bulk.tensor.2d, 128-byte swizzle) straight into shared memory,
//    completion tracked by an mbarrier; the block ID comes from the table.
//  * Every warp owns a private ring of NS slab buffers and a private subset of
//    the partition's slabs (round-robin), so there is no inter-warp
//    synchronisation until the final merge of the warps' partial results.
//  * Scores S^T[16 tokens x 8 heads] = K Q^T and the value sum
//    O^T[D x 8 heads] += V^T P^T run on the tensor cores (mma.m16n8k16, fp32
//    accumulate), operands read with ldmatrix from the swizzled tiles; the
//    probability tile is moved from accumulator layout to operand layout with
//    movmatrix.  Softmax is online (running max and sum per head, fp32).
//  The path is bound by HBM bandwidth (1 to 8 flop per byte), so the tensor
//  cores only keep instruction issue low; the design goal is to keep enough
//  bulk copies in flight to saturate HBM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

constexpr uint64_t kWaitLimit = 250ull * 1000 * 1000;  // 250 ms per wait

// bf16 probabilities are split into a rounded part and its residual (see the value MMA)
template <typename T>
constexpr bool kSplitP = false;
template <>
constexpr bool kSplitP<__nv_bfloat16> = true;

template <int D, int SB, int NW, int NS>
struct TcShape {
  static constexpr int KSTEPS = D / 16;             // k-steps of Q K^T = m-tiles of V^T P^T
  static constexpr int NBOX = D / 64;               // 128-byte (64-element) TMA boxes per row
  static constexpr int BOX_BYTES = SB * 128;        // one box: SB rows x 128 bytes
  static constexpr int SLAB_BYTES = 2 * NBOX * BOX_BYTES;  // K boxes, then V boxes
  static constexpr int UNITS = SB / 16;             // 16-token MMA units per slab
  static constexpr int RING_BYTES = NS * SLAB_BYTES;  // per warp
  static constexpr int SMEM_BYTES = NW * RING_BYTES + NW * NS * 8 + 1024;  // + barriers + alignment slack
  static_assert(D % 64 == 0, "head_size must be a multiple of 64");
  static_assert(SB == 16 || SB == 32, "slab is 16 or 32 tokens");
  static_assert(RING_BYTES >= 8 * D * 4 + 8 * 2 * 4, "ring must hold a warp's partial result");
};

template <typename T, int D, int SB, int NW, int NS>
__global__ void __launch_bounds__(NW * 32)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                     const DecodeParams p) {
  using S = TcShape<D, SB, NW, NS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;   // fragment row group
  const int q4 = lane & 3;   // fragment column pair
  uint8_t* ring = smem + warp * S::RING_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NW * S::RING_BYTES) + warp * NS;

  // ---- work item: (sequence, kv head, head group, partition)
  const int per_seq = p.num_kv_heads * p.head_groups;
  const int part = blockIdx.x % p.pmax;
  const int hh = (blockIdx.x / p.pmax) % per_seq;
  const int s = blockIdx.x / (p.pmax * per_seq);
  const int hkv = hh / p.head_groups;
  const int hg = hh % p.head_groups;
  const int G = p.num_q_heads / p.num_kv_heads;
  const int hq0 = hkv * G + hg * 8;
  const int gcount = min(8, G - hg * 8);
  const int B = p.block_size;
  const int P = p.partition_size;

  int L = p.seq_lens[s];
  L = max(0, min(L, p.max_blocks * B));
  const int t_begin = part * P;
  if (L == 0) {
    if (part == 0) {  // an empty sequence has a zero output
      T* out = reinterpret_cast<T*>(p.out) + ((size_t)s * p.num_q_heads + hq0) * D;
      for (int i = threadIdx.x; i < gcount * D; i += NW * 32) out[i] = from_float<T>(0.f);
    }
    return;
  }
  if (t_begin >= L) return;  // partition past the end of this sequence
  // after a timed-out copy anywhere in this launch, the remaining CTAs stop early
  if (p.err_flag != nullptr && *reinterpret_cast<volatile int32_t*>(p.err_flag) == PA_DEVERR_TIMEOUT) return;
  const int t_end = min(L, t_begin + P);
  const bool final_out = L <= P;  // single partition: write the normalised output directly

  // ---- slabs of this partition owned by this warp: j = j0 + warp + k * NW
  const int j0 = t_begin / SB;
  const int j1 = (t_end + SB - 1) / SB;
  const int n_my = (j1 - j0 - warp + NW - 1) / NW > 0 ? (j1 - j0 - warp + NW - 1) / NW : 0;
  const int32_t* table = p.block_tables + (size_t)s * p.max_blocks;

  if (lane == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
  }
  __syncwarp();

  // ---- query fragments (B operand of S^T = K Q^T): head g, dims 16j + 2q4 (+8)
  uint32_t qf[S::KSTEPS][2];
  {
    const bool real = g < gcount;
    const uint32_t* qrow =
        reinterpret_cast<const uint32_t*>(reinterpret_cast<const T*>(p.q) + ((size_t)s * p.num_q_heads + hq0 + g) * D);
#pragma unroll
    for (int j = 0; j < S::KSTEPS; ++j) {
      qf[j][0] = real ? __ldg(qrow + (16 * j + 2 * q4) / 2) : 0u;
      qf[j][1] = real ? __ldg(qrow + (16 * j + 2 * q4 + 8) / 2) : 0u;
    }
  }

  // ---- block-table entries, fetched 32 slabs at a time across the lanes
  int pb_batch = -1;
  int pb_reg = -1;
  uint32_t valid_mask = 0;  // bit stage: the slab in that stage was loaded
  auto issue = [&](int k) {
    const int batch = k >> 5;
    if (batch != pb_batch) {
      const int kk = batch * 32 + lane;
      pb_reg = kk < n_my ? __ldg(table + ((j0 + warp + kk * NW) * SB) / B) : -1;
      pb_batch = batch;
    }
    const int pb = __shfl_sync(0xffffffffu, pb_reg, k & 31);
    const bool ok = pb >= 0 && pb < p.num_blocks;
    const int stage = k % NS;
    valid_mask = ok ? (valid_mask | (1u << stage)) : (valid_mask & ~(1u << stage));
    if (lane == 0) {
      uint64_t* bar = &bars[stage];
      if (ok) {
        const int j = j0 + warp + k * NW;
        const int y = (pb * p.num_kv_heads + hkv) * B + (j * SB) % B;  // first row of the slab
        uint8_t* dst = ring + stage * S::SLAB_BYTES;
        mbar_arrive_expect_tx(bar, S::SLAB_BYTES);
#pragma unroll
        for (int b = 0; b < S::NBOX; ++b) tma_load_2d(dst + b * S::BOX_BYTES, &tmap_k, b * 64, y, bar);
#pragma unroll
        for (int b = 0; b < S::NBOX; ++b) tma_load_2d(dst + (S::NBOX + b) * S::BOX_BYTES, &tmap_v, b * 64, y, bar);
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
  const float sl2 = p.scale_log2;

  const int prologue = n_my < NS ? n_my : NS;
  for (int k = 0; k < prologue; ++k) issue(k);

  int consumed = 0;
  bool timed_out = false;
  for (int k = 0; k < n_my; ++k) {
    const int stage = k % NS;
    if (!mbar_wait_bounded(&bars[stage], (k / NS) & 1, kWaitLimit)) {
      timed_out = true;
      break;
    }
    consumed = k + 1;
    if ((valid_mask >> stage) & 1u) {
      const int j = j0 + warp + k * NW;
      const int valid = min(SB, t_end - j * SB);
      const uint8_t* kst = ring + stage * S::SLAB_BYTES;
      const uint8_t* vst = kst + S::NBOX * S::BOX_BYTES;
#pragma unroll
      for (int u = 0; u < S::UNITS; ++u) {
        const int nvalid = valid - u * 16;
        if (nvalid <= 0) break;
        // ---- S^T[16 tokens x 8 heads] = K_unit Q^T
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        {
          const int row = u * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int khalf = lane >> 4;
#pragma unroll
          for (int jj = 0; jj < S::KSTEPS; ++jj) {
            const uint32_t addr = smem_u32(kst + (jj >> 2) * S::BOX_BYTES) + swz128(row, (jj & 3) * 2 + khalf);
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4(addr, a0, a1, a2, a3);
            Mma<T>::run(sc, a0, a1, a2, a3, qf[jj][0], qf[jj][1]);
          }
        }
        // sc: (token g, head 2q4), (token g, head 2q4+1), (token g+8, head 2q4), (token g+8, head 2q4+1)
        float s0 = sc[0] * sl2, s1 = sc[1] * sl2, s2 = sc[2] * sl2, s3 = sc[3] * sl2;
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
        const T* h0 = reinterpret_cast<const T*>(&x0);
        const T* h1 = reinterpret_cast<const T*>(&x1);
        if constexpr (kSplitP<T>) {
          y0 = Mma<T>::pack(p0 - float(h0[0]), p1 - float(h0[1]));
          y1 = Mma<T>::pack(p2 - float(h1[0]), p3 - float(h1[1]));
          l_a = l_a * al_a + (p0 + p2);
          l_b = l_b * al_b + (p1 + p3);
        } else {  // fp16: the sums use the rounded probabilities the value MMA multiplies with
          l_a = l_a * al_a + (float(h0[0]) + float(h1[0]));
          l_b = l_b * al_b + (float(h0[1]) + float(h1[1]));
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
        // ---- O^T[D x 8 heads] += V_unit^T P^T
        {
          const int row = u * 16 + (lane & 7) + (lane >> 4) * 8;
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
    }
    __syncwarp();
    if (k + NS < n_my) issue(k + NS);
  }

  if (timed_out) {
    report_error(p.err_flag, PA_DEVERR_TIMEOUT);
    // let copies already in flight land before this warp's buffers are reused
    const int issued = n_my < consumed + NS ? n_my : consumed + NS;
    for (int k = consumed; k < issued; ++k) mbar_wait_bounded(&bars[k % NS], (k / NS) & 1, kWaitLimit);
  }

  // ---- per-warp totals, then merge the warps through shared memory
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l_a += __shfl_xor_sync(0xffffffffu, l_a, off);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, off);
  }
  __syncwarp();
  float* wo = reinterpret_cast<float*>(ring);  // [8 heads][D]
  float* wml = wo + 8 * D;                     // [8 heads][2]
#pragma unroll
  for (int i = 0; i < S::KSTEPS; ++i) {
    wo[(2 * q4) * D + 16 * i + g] = o[i][0];
    wo[(2 * q4 + 1) * D + 16 * i + g] = o[i][1];
    wo[(2 * q4) * D + 16 * i + g + 8] = o[i][2];
    wo[(2 * q4 + 1) * D + 16 * i + g + 8] = o[i][3];
  }
  if (g == 0) {
    wml[(2 * q4) * 2] = m_a;
    wml[(2 * q4) * 2 + 1] = l_a;
    wml[(2 * q4 + 1) * 2] = m_b;
    wml[(2 * q4 + 1) * 2 + 1] = l_b;
  }
  __syncthreads();

  const size_t row0 = (size_t)s * p.num_q_heads + hq0;
  for (int idx = threadIdx.x; idx < gcount * D; idx += NW * 32) {
    const int gh = idx / D, d = idx % D;
    float mstar = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* wm = reinterpret_cast<const float*>(smem + w * S::RING_BYTES) + 8 * D;
      mstar = fmaxf(mstar, wm[gh * 2]);
    }
    float lsum = 0.f, acc = 0.f;
    if (mstar != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float* wb = reinterpret_cast<const float*>(smem + w * S::RING_BYTES);
        const float wt = fast_exp2(wb[8 * D + gh * 2] - mstar);
        lsum += wt * wb[8 * D + gh * 2 + 1];
        acc += wt * wb[gh * D + d];
      }
    }
    if (final_out) {
      T* out = reinterpret_cast<T*>(p.out);
      out[(row0 + gh) * D + d] = from_float<T>(lsum > 0.f ? acc / lsum : 0.f);
    } else {
      const size_t slot = (row0 + gh) * p.pmax + part;
      p.ws_o[slot * D + d] = acc;
      if (d == 0) {
        p.ws_ml[slot * 2] = mstar;
        p.ws_ml[slot * 2 + 1] = lsum;
      }
    }
  }
}

// ------------------------------------------------------------------ launch
template <typename T, int D, int SB, int NW, int NS>
static cudaError_t launch_tc(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                             cudaStream_t stream) {
  using S = TcShape<D, SB, NW, NS>;
  auto kernel = decode_tc_kernel<T, D, SB, NW, NS>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)p.num_seqs * p.num_kv_heads * p.head_groups * p.pmax;
  if (grid == 0) return cudaSuccess;
  kernel<<<(unsigned)grid, NW * 32, S::SMEM_BYTES, stream>>>(tk, tv, p);
  return cudaGetLastError();
}

// Per-warp ring depth and warps per CTA chosen so a CTA holds about 96 KB of
// slabs (two CTAs per SM) with every warp keeping NS - 1 slabs in flight.
template <typename T>
static cudaError_t dispatch_tc(int head_size, int block_size, const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeParams& p, cudaStream_t stream) {
  const int sb = tc_slab_tokens(block_size);
  if (head_size == 128 && sb == 16) return launch_tc<T, 128, 16, 4, 3>(tk, tv, p, stream);
  if (head_size == 128 && sb == 32) return launch_tc<T, 128, 32, 2, 3>(tk, tv, p, stream);
  if (head_size == 64 && sb == 16) return launch_tc<T, 64, 16, 4, 4>(tk, tv, p, stream);
  if (head_size == 64 && sb == 32) return launch_tc<T, 64, 32, 4, 3>(tk, tv, p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_tc(int dtype, int head_size, int block_size, const CUtensorMap& tk, const CUtensorMap& tv,
                             const DecodeParams& p, cudaStream_t stream) {
  if (dtype == PA_F16) return dispatch_tc<__half>(head_size, block_size, tk, tv, p, stream);
  if (dtype == PA_BF16) return dispatch_tc<__nv_bfloat16>(head_size, block_size, tk, tv, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa

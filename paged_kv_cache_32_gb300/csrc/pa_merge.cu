// pa_merge.cu - the partition merge of long-context decode.
//
// What it computes ("PagedAttention是什麼？", section "PagedAttention Kernel在做
// 什麼？": long contexts are cut into partitions whose results a log-sum-exp
// reduction combines).  Partition p of a sequence left, per query head, m_p
// (the max score, log2 units), l_p = sum 2^(s_i - m_p) and the unnormalised
// o_p = sum 2^(s_i - m_p) v_i.  With m* = max_p m_p and w_p = 2^(m_p - m*):
//   out = sum_p w_p o_p / sum_p w_p l_p.
//
// How: the merge is a short, latency-bound pass over partials that sit in L2,
// so it is sized to finish in one wave and to start early.
//  * WPR warps per (sequence, query head) row, 8 warps per CTA: each lane owns
//    D / 32 consecutive output elements, so one partition's o_p is one
//    coalesced 512-byte (D = 128) warp load; warp k of a row takes partitions
//    k, k + WPR, ...  and the row's warps add up through shared memory.  The
//    host picks WPR from the partition count (1 for a few partitions, up to 8
//    for long contexts) so the per-warp chain of dependent loads stays short.
//  * It is launched as a programmatic dependent of the decode kernel: the
//    decode CTAs allow the launch as they start, so the merge CTAs are resident
//    and have read their sequence lengths by the time the last decode CTA
//    ends; griddepcontrol.wait then holds them until the decode grid has
//    finished and its partial stores are visible.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int kMergeThreads = 256;
constexpr int kMergePreload = 4;  // partitions per warp whose outputs are loaded before the weights are known

template <int V>
__device__ __forceinline__ void load_vec(const float* src, float (&v)[V]) {
  if constexpr (V == 4) {
    const float4 x = *reinterpret_cast<const float4*>(src);
    v[0] = x.x, v[1] = x.y, v[2] = x.z, v[3] = x.w;
  } else if constexpr (V == 2) {
    const float2 x = *reinterpret_cast<const float2*>(src);
    v[0] = x.x, v[1] = x.y;
  } else {
#pragma unroll
    for (int e = 0; e < V; ++e) v[e] = src[e];
  }
}

// w_i = 2^(m_i - m*) of partition i (the same i in every lane of the warp): lane i
// holds it for the first 32 partitions, later ones are read again.
__device__ __forceinline__ float partition_weight(int i, float w_own, const float2* ml, float mx) {
  if (i < 32) return __shfl_sync(0xffffffffu, w_own, i);
  const float m = ml[i].x;
  return (m == -INFINITY || mx == -INFINITY) ? 0.f : fast_exp2(m - mx);
}

template <typename T, int D, int WPR>
__global__ void __launch_bounds__(kMergeThreads, 5) merge_kernel(const DecodeParams p) {
  constexpr int NWARP = kMergeThreads / 32;
  constexpr int ROWS = NWARP / WPR;  // rows per CTA
  constexpr int V = D / 32;          // output elements per lane
  __shared__ float s_acc[WPR > 1 ? NWARP : 1][WPR > 1 ? D : 1];

  griddep_launch_dependents();  // the next decode, launched as a dependent, may be scheduled behind this grid
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = warp % WPR;
  const long long row = (long long)blockIdx.x * ROWS + warp / WPR;
  int nparts = 0;
  size_t slot0 = 0;  // the row's first partition slot in the workspace
  if (row < (long long)p.num_seqs * p.num_q_heads) {  // seq_lens is an input of the step, not a decode output
    const int s = (int)(row / p.num_q_heads);
    int L = p.seq_lens[s];
    L = max(0, min(L, p.max_blocks * p.block_size));
    const int ps = seq_partition_size(p, s);
    nparts = (L + ps - 1) / ps;
    slot0 = ws_row_slot(p, s, (int)(row % p.num_q_heads));
  }
  griddep_wait();  // the decode grid has finished; its partials are visible

  float acc[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  float lsum = 0.f;
  if (nparts > 1) {  // a single partition was written out by the decode kernel
    const float2* ml = reinterpret_cast<const float2*>(p.ws_ml) + slot0;  // (m_p, l_p)
    const float* os = p.ws_o + slot0 * D + lane * V;
    // One round trip: this warp's first kMergePreload partial outputs and lane i's pair (m_i, l_i).
    float pre[kMergePreload][V];
#pragma unroll
    for (int k = 0; k < kMergePreload; ++k)
      if (sub + k * WPR < nparts) load_vec<V>(os + (size_t)(sub + k * WPR) * D, pre[k]);
    const float2 own = lane < nparts ? ml[lane] : make_float2(-INFINITY, 0.f);
    float mx = own.x;
    for (int i = lane + 32; i < nparts; i += 32) mx = fmaxf(mx, ml[i].x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float w_own = (own.x == -INFINITY || mx == -INFINITY) ? 0.f : fast_exp2(own.x - mx);  // w_lane
    if (sub == 0) {
      lsum = w_own * own.y;
      for (int i = lane + 32; i < nparts; i += 32) {
        const float2 v = ml[i];
        if (v.x != -INFINITY && mx != -INFINITY) lsum += fast_exp2(v.x - mx) * v.y;
      }
    }
#pragma unroll
    for (int k = 0; k < kMergePreload; ++k) {
      if (sub + k * WPR < nparts) {
        const float w = partition_weight(sub + k * WPR, w_own, ml, mx);
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = fmaf(w, pre[k][e], acc[e]);
      }
    }
#pragma unroll 4
    for (int i = sub + kMergePreload * WPR; i < nparts; i += WPR) {
      const float w = partition_weight(i, w_own, ml, mx);
      float o[V];
      load_vec<V>(os + (size_t)i * D, o);
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] = fmaf(w, o[e], acc[e]);
    }
  }
  if constexpr (WPR > 1) {  // the row's warps add their partition subsets
#pragma unroll
    for (int e = 0; e < V; ++e) s_acc[warp][lane * V + e] = acc[e];
    __syncthreads();
    if (sub == 0) {
#pragma unroll
      for (int k = 1; k < WPR; ++k)
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] += s_acc[warp + k][lane * V + e];
    }
  }
  if (sub != 0 || nparts <= 1) return;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
  T* out = reinterpret_cast<T*>(p.out) + (size_t)row * D + lane * V;
#pragma unroll
  for (int e = 0; e < V; ++e) out[e] = from_float<T>(lsum > 0.f ? acc[e] / lsum : 0.f);
}

template <typename T, int D>
static cudaError_t launch_merge_t(const DecodeParams& p, cudaStream_t stream) {
  const long long rows = (long long)p.num_seqs * p.num_q_heads;
  // warps per row from the main partitions (rows of tail sequences, with up to twice as many, loop over the rest)
  const int wpr = p.pmax <= 4 ? 1 : p.pmax <= 8 ? 2 : p.pmax <= 16 ? 4 : 8;
  const long long per_cta = (kMergeThreads / 32) / wpr;
  const dim3 grid((unsigned)((rows + per_cta - 1) / per_cta)), block(kMergeThreads);
  switch (wpr) {
    case 1: return launch_dependent(merge_kernel<T, D, 1>, grid, block, 0, stream, p);
    case 2: return launch_dependent(merge_kernel<T, D, 2>, grid, block, 0, stream, p);
    case 4: return launch_dependent(merge_kernel<T, D, 4>, grid, block, 0, stream, p);
    default: return launch_dependent(merge_kernel<T, D, 8>, grid, block, 0, stream, p);
  }
}

cudaError_t launch_merge(int dtype, int head_size, const DecodeParams& p, cudaStream_t stream) {
  if ((long long)p.num_seqs * p.num_q_heads == 0) return cudaSuccess;
  if (dtype == PA_F32 && head_size == 64) return launch_merge_t<float, 64>(p, stream);
  if (dtype == PA_F32 && head_size == 128) return launch_merge_t<float, 128>(p, stream);
  if (dtype == PA_F16 && head_size == 64) return launch_merge_t<__half, 64>(p, stream);
  if (dtype == PA_F16 && head_size == 128) return launch_merge_t<__half, 128>(p, stream);
  if (dtype == PA_BF16 && head_size == 64) return launch_merge_t<__nv_bfloat16, 64>(p, stream);
  if (dtype == PA_BF16 && head_size == 128) return launch_merge_t<__nv_bfloat16, 128>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa

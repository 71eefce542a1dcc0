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

template <typename T, int D, int WPR>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const DecodeParams p) {
  constexpr int NWARP = kMergeThreads / 32;
  constexpr int ROWS = NWARP / WPR;  // rows per CTA
  constexpr int V = D / 32;          // output elements per lane
  __shared__ float s_acc[WPR > 1 ? NWARP : 1][WPR > 1 ? D : 1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = warp % WPR;
  const long long row = (long long)blockIdx.x * ROWS + warp / WPR;
  int nparts = 0;
  if (row < (long long)p.num_seqs * p.num_q_heads) {  // seq_lens is an input of the step, not a decode output
    int L = p.seq_lens[row / p.num_q_heads];
    L = max(0, min(L, p.max_blocks * p.block_size));
    nparts = (L + p.partition_size - 1) / p.partition_size;
  }
  griddep_wait();  // the decode grid has finished; its partials are visible

  float acc[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  float lsum = 0.f;
  if (nparts > 1) {  // a single partition was written out by the decode kernel
    const float* ml = p.ws_ml + (size_t)row * p.pmax * 2;
    const float* os = p.ws_o + (size_t)row * p.pmax * D + lane * V;
    float mx = -INFINITY;
    for (int i = lane; i < nparts; i += 32) mx = fmaxf(mx, ml[2 * i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (sub == 0 && mx != -INFINITY) {
      for (int i = lane; i < nparts; i += 32) {
        const float2 v = *reinterpret_cast<const float2*>(ml + 2 * i);
        if (v.x != -INFINITY) lsum += fast_exp2(v.x - mx) * v.y;
      }
    }
    if (mx != -INFINITY) {
#pragma unroll 4
      for (int i = sub; i < nparts; i += WPR) {
        const float m = ml[2 * i];  // the same word for every lane: one broadcast load
        const float w = m == -INFINITY ? 0.f : fast_exp2(m - mx);
        if constexpr (V == 4) {
          const float4 o = *reinterpret_cast<const float4*>(os + (size_t)i * D);
          acc[0] = fmaf(w, o.x, acc[0]);
          acc[1] = fmaf(w, o.y, acc[1]);
          acc[2] = fmaf(w, o.z, acc[2]);
          acc[3] = fmaf(w, o.w, acc[3]);
        } else {
#pragma unroll
          for (int e = 0; e < V; ++e) acc[e] = fmaf(w, os[(size_t)i * D + e], acc[e]);
        }
      }
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
  const int wpr = p.pmax <= 4 ? 1 : p.pmax <= 8 ? 2 : p.pmax <= 16 ? 4 : 8;
  const long long per_cta = (kMergeThreads / 32) / wpr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((rows + per_cta - 1) / per_cta));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (wpr) {
    case 1: return cudaLaunchKernelEx(&cfg, merge_kernel<T, D, 1>, p);
    case 2: return cudaLaunchKernelEx(&cfg, merge_kernel<T, D, 2>, p);
    case 4: return cudaLaunchKernelEx(&cfg, merge_kernel<T, D, 4>, p);
    default: return cudaLaunchKernelEx(&cfg, merge_kernel<T, D, 8>, p);
  }
}

cudaError_t launch_merge(int dtype, int head_size, const DecodeParams& p, cudaStream_t stream) {
  if ((long long)p.num_seqs * p.num_q_heads == 0) return cudaSuccess;
  cudaError_t e;
  if (dtype == PA_F32 && head_size == 64) e = launch_merge_t<float, 64>(p, stream);
  else if (dtype == PA_F32 && head_size == 128) e = launch_merge_t<float, 128>(p, stream);
  else if (dtype == PA_F16 && head_size == 64) e = launch_merge_t<__half, 64>(p, stream);
  else if (dtype == PA_F16 && head_size == 128) e = launch_merge_t<__half, 128>(p, stream);
  else if (dtype == PA_BF16 && head_size == 64) e = launch_merge_t<__nv_bfloat16, 64>(p, stream);
  else if (dtype == PA_BF16 && head_size == 128) e = launch_merge_t<__nv_bfloat16, 128>(p, stream);
  else return cudaErrorInvalidValue;
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace pa

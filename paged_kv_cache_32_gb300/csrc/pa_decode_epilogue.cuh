// pa_decode_epilogue.cuh - the end of a decode work item, shared by the fp16/bf16
// and FP8 decode kernels: the merge of the CTA's warps and the item's output.
//
// Each warp streamed its own subset of the item's slabs with an online softmax
// and left, at the start of its ring buffer, its unnormalised O[8 heads][OROW]
// followed by (m, l)[8 heads] (max score in log2 units and the sum of 2^(s - m)
// over its tokens).  The warps combine like partitions do ("PagedAttention是什
// 麼？", section "PagedAttention Kernel在做什麼？"): with m* = max_w m_w and
// weights 2^(m_w - m*), O = sum_w weight_w O_w and l = sum_w weight_w l_w.
// The per-head weights are computed once; every output element is then an
// independent NW-term sum, so the epilogue is a short burst of parallel work
// rather than a chain of dependent loads per element.
#pragma once

#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// Called by all NW * 32 threads after the CTA barrier that follows the warps'
// partial stores.  Writes the normalised rows of out (TOut) when the item is a
// whole sequence, else the unnormalised partial (o, m*, l) of the item's
// partition: workspace slot slot0 for the first of its rows, slot0 + g * stride
// for row g.
template <typename TOut, int D, int NW, int OROW, int RING_BYTES>
__device__ __forceinline__ void finish_item(const uint8_t* smem, const DecodeParams& p, size_t row0, int gcount,
                                            bool final_out, size_t slot0, int stride) {
  constexpr int WARP_MERGE = 8 * OROW + 16;  // floats of one warp's partial
  static_assert(RING_BYTES >= (WARP_MERGE + 8 * NW + 16) * 4, "warp 0's ring also holds the head weights");
  const float* rings = reinterpret_cast<const float*>(smem);
  constexpr int RF = RING_BYTES / 4;  // ring stride in floats
  float* wt = const_cast<float*>(rings) + WARP_MERGE;  // [8][NW] weights, then m*[8], l[8]
  float* mst = wt + 8 * NW;
  float* lsum = mst + 8;

  if (threadIdx.x < 8) {
    const int gh = threadIdx.x;
    float mw[NW];
    float ms = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      mw[w] = rings[w * RF + 8 * OROW + gh * 2];
      ms = fmaxf(ms, mw[w]);
    }
    float l = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float x = ms == -INFINITY ? 0.f : fast_exp2(mw[w] - ms);
      l += x * rings[w * RF + 8 * OROW + gh * 2 + 1];
      wt[gh * NW + w] = x;
    }
    mst[gh] = ms;
    lsum[gh] = l;
  }
  __syncthreads();

#pragma unroll 4
  for (int idx = threadIdx.x; idx < gcount * D; idx += NW * 32) {
    const int gh = idx / D, d = idx % D;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) acc += wt[gh * NW + w] * rings[w * RF + gh * OROW + d];
    if (final_out) {
      const float l = lsum[gh];
      reinterpret_cast<TOut*>(p.out)[(row0 + gh) * D + d] = from_float<TOut>(l > 0.f ? acc / l : 0.f);
    } else {
      const size_t slot = slot0 + (size_t)gh * stride;
      p.ws_o[slot * D + d] = acc;
      if (d == 0) {
        p.ws_ml[slot * 2] = mst[gh];
        p.ws_ml[slot * 2 + 1] = lsum[gh];
      }
    }
  }
}

}  // namespace pa

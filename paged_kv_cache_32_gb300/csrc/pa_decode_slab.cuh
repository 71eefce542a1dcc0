// pa_decode_slab.cuh - the per-slab step of the fp16/bf16 decode kernels: one
// 16-token slab of one kv head against up to eight query heads, on mma.sync
// tensor-core tiles, with the online softmax of "vLLM 核心工程深度剖析", section
// "3.1 Kernel 签名与分块策略" (running max and sum, rescaled when the max grows;
// here the max grows only by more than 8 in log2 units at a time).
#pragma once

#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// bf16 probabilities are split into a rounded part and its residual (see the value MMA)
template <typename T>
constexpr bool kSplitP = false;
template <>
constexpr bool kSplitP<__nv_bfloat16> = true;

// One 16-token slab: S^T = K Q^T, online softmax update, O^T += V^T P^T.
// kst / vst: the slab's swizzled K and V tiles; nvalid: tokens of the slab
// inside the partition (1..16).  ALiBi: bias_a / bias_b are the slopes of
// heads 2q4 / 2q4+1 in log2 units (0 without ALiBi) and rel0 is the position
// of the slab's first token relative to the query, i.e. first token - (L - 1).
template <typename T, int D>
__device__ __forceinline__ void process_slab(const uint8_t* kst, const uint8_t* vst, int nvalid,
                                             const uint32_t (&qf)[D / 16][2], float (&o)[D / 16][4], float& m_a,
                                             float& m_b, float& l_a, float& l_b, int lane, float sl2, float bias_a,
                                             float bias_b, float rel0) {
  constexpr int KSTEPS = D / 16;
  constexpr int BOX_BYTES = kTcSlabTokens * 128;
  const int g = lane >> 2, q4 = lane & 3;
  // ---- S^T[16 tokens x 8 heads] (two accumulators: shorter dependency chain)
  float sc[4] = {0.f, 0.f, 0.f, 0.f};
  float sd[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int khalf = lane >> 4;
#pragma unroll
    for (int jj = 0; jj < KSTEPS; ++jj) {
      const uint32_t addr = smem_u32(kst + (jj >> 2) * BOX_BYTES) + swz128(row, (jj & 3) * 2 + khalf);
      uint32_t a0, a1, a2, a3;
      ldmatrix_x4(addr, a0, a1, a2, a3);
      if (jj & 1)
        Mma<T>::run(sd, a0, a1, a2, a3, qf[jj][0], qf[jj][1]);
      else
        Mma<T>::run(sc, a0, a1, a2, a3, qf[jj][0], qf[jj][1]);
    }
  }
  // scores: (token g, head 2q4), (token g, head 2q4+1), (token g+8, head 2q4), (token g+8, head 2q4+1)
  const float r_lo = rel0 + (float)g, r_hi = r_lo + 8.f;  // tokens g and g + 8 of the slab
  float s0 = fmaf(bias_a, r_lo, (sc[0] + sd[0]) * sl2), s1 = fmaf(bias_b, r_lo, (sc[1] + sd[1]) * sl2);
  float s2 = fmaf(bias_a, r_hi, (sc[2] + sd[2]) * sl2), s3 = fmaf(bias_b, r_hi, (sc[3] + sd[3]) * sl2);
  if (nvalid < 16) {
    if (g >= nvalid) s0 = s1 = -INFINITY;
    if (g + 8 >= nvalid) s2 = s3 = -INFINITY;
  }
  // The running maxima stay while no score of the slab exceeds them by more than kSlabSlack (log2 units):
  // the weights are then at most 2^kSlabSlack, and the slab's maxima, their shuffles and the rescale of O
  // are skipped.  Otherwise the maxima move to the slab's (the first slab always: they start at -inf).
  if (__any_sync(0xffffffffu, s0 - m_a > kSlabSlack || s1 - m_b > kSlabSlack || s2 - m_a > kSlabSlack ||
                                  s3 - m_b > kSlabSlack)) {
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
    l_a *= al_a;
    l_b *= al_b;
#pragma unroll
    for (int i = 0; i < KSTEPS; ++i) {
      o[i][0] *= al_a;
      o[i][1] *= al_b;
      o[i][2] *= al_a;
      o[i][3] *= al_b;
    }
  }
  const float p0 = fast_exp2(s0 - m_a), p1 = fast_exp2(s1 - m_b);
  const float p2 = fast_exp2(s2 - m_a), p3 = fast_exp2(s3 - m_b);
  const uint32_t x0 = Mma<T>::pack(p0, p1);
  const uint32_t x1 = Mma<T>::pack(p2, p3);
  // bf16 keeps only 8 significant bits of P; its rounding residual goes
  // through a second MMA so P enters the value sum with ~16 bits.
  uint32_t y0 = 0, y1 = 0;
  if constexpr (kSplitP<T>) {
    y0 = Mma<T>::pack(p0 - Mma<T>::lo(x0), p1 - Mma<T>::hi(x0));
    y1 = Mma<T>::pack(p2 - Mma<T>::lo(x1), p3 - Mma<T>::hi(x1));
    l_a += p0 + p2;
    l_b += p1 + p3;
  } else {  // fp16: the sums use the rounded probabilities the value MMA multiplies with
    l_a += Mma<T>::lo(x0) + Mma<T>::lo(x1);
    l_b += Mma<T>::hi(x0) + Mma<T>::hi(x1);
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
  const int row = (lane & 7) + (lane >> 4) * 8;
  const int dhalf = (lane >> 3) & 1;
#pragma unroll
  for (int i = 0; i < KSTEPS; ++i) {
    const uint32_t addr = smem_u32(vst + (i >> 2) * BOX_BYTES) + swz128(row, (i & 3) * 2 + dhalf);
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

}  // namespace pa

// pa_decode_f32.cu - paged decode attention for fp32 caches (CUDA cores).
//
// Same definition as the fp16/bf16 kernel ("vLLM 核心工程深度剖析", section
// "3.1 Kernel 签名与分块策略"; address translation per "PagedAttention 详解：
// 缓存的存储结构", section "软件地址翻译"), same grid of (sequence, kv head,
// head group, partition) CTAs and same partial-result format, so one merge
// kernel serves all decode kernels.  fp32 needs exact fp32 products, so no tensor-core path:
// each warp walks a strided subset of the partition's tokens, every lane holds
// D/32 consecutive elements of each row (coalesced 256/512-byte row loads),
// dot products are reduced with warp shuffles, and the softmax is online.
#include <cuda.h>
#include <math.h>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

template <int D, int NW>
__global__ void __launch_bounds__(NW * 32)
    decode_f32_kernel(const float* __restrict__ k_cache, const float* __restrict__ v_cache, const DecodeParams p) {
  constexpr int VEC = D / 32;
  __shared__ float s_o[NW][8][D];
  __shared__ float s_ml[NW][8][2];

  griddep_launch_dependents();  // the partition merge may be scheduled behind this grid's last CTAs
  griddep_wait();               // launched as a dependent: the previous kernel's writes are visible from here
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
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
    if (part == 0) {
      float* out = reinterpret_cast<float*>(p.out) + ((size_t)s * p.num_q_heads + hq0) * D;
      for (int i = threadIdx.x; i < gcount * D; i += NW * 32) out[i] = 0.f;
    }
    return;
  }
  if (t_begin >= L) return;
  const int t_end = min(L, t_begin + P);
  const bool final_out = L <= P;
  const int32_t* table = p.block_tables + (size_t)s * p.max_blocks;

  float qv[8][VEC];
#pragma unroll
  for (int gh = 0; gh < 8; ++gh) {
#pragma unroll
    for (int e = 0; e < VEC; ++e)
      qv[gh][e] = gh < gcount ? reinterpret_cast<const float*>(p.q)[((size_t)s * p.num_q_heads + hq0 + gh) * D +
                                                                  lane * VEC + e]
                              : 0.f;
  }
  float bias[8];  // ALiBi slopes in log2 units (0: no bias)
#pragma unroll
  for (int gh = 0; gh < 8; ++gh)
    bias[gh] = (p.alibi != nullptr && gh < gcount) ? __ldg(p.alibi + hq0 + gh) * 1.4426950408889634f : 0.f;
  float m[8], l[8], o[8][VEC];
#pragma unroll
  for (int gh = 0; gh < 8; ++gh) {
    m[gh] = -INFINITY;
    l[gh] = 0.f;
#pragma unroll
    for (int e = 0; e < VEC; ++e) o[gh][e] = 0.f;
  }

  for (int t = t_begin + warp; t < t_end; t += NW) {
    const int pb = __ldg(table + t / B);
    if (pb < 0 || pb >= p.num_blocks) {
      if (lane == 0) report_error(p.err_flag, PA_DEVERR_BLOCK_ID);
      continue;
    }
    const size_t row = (((size_t)pb * p.num_kv_heads + hkv) * B + t % B) * D + lane * VEC;
    float kv[VEC], vv[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      kv[e] = __ldg(k_cache + row + e);
      vv[e] = __ldg(v_cache + row + e);
    }
#pragma unroll
    for (int gh = 0; gh < 8; ++gh) {
      if (gh >= gcount) break;
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < VEC; ++e) dot = fmaf(qv[gh][e], kv[e], dot);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      const float sc = fmaf(bias[gh], (float)(t - (L - 1)), dot * p.scale_log2);
      const float mn = fmaxf(m[gh], sc);
      const float al = fast_exp2(m[gh] - mn);
      const float pe = fast_exp2(sc - mn);
      m[gh] = mn;
      l[gh] = l[gh] * al + pe;
#pragma unroll
      for (int e = 0; e < VEC; ++e) o[gh][e] = fmaf(pe, vv[e], o[gh][e] * al);
    }
  }

#pragma unroll
  for (int gh = 0; gh < 8; ++gh) {
#pragma unroll
    for (int e = 0; e < VEC; ++e) s_o[warp][gh][lane * VEC + e] = o[gh][e];
    if (lane == 0) {
      s_ml[warp][gh][0] = m[gh];
      s_ml[warp][gh][1] = l[gh];
    }
  }
  __syncthreads();

  const size_t row0 = (size_t)s * p.num_q_heads + hq0;
  for (int idx = threadIdx.x; idx < gcount * D; idx += NW * 32) {
    const int gh = idx / D, d = idx % D;
    float mstar = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) mstar = fmaxf(mstar, s_ml[w][gh][0]);
    float lsum = 0.f, acc = 0.f;
    if (mstar != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float wt = fast_exp2(s_ml[w][gh][0] - mstar);
        lsum += wt * s_ml[w][gh][1];
        acc += wt * s_o[w][gh][d];
      }
    }
    if (final_out) {
      reinterpret_cast<float*>(p.out)[(row0 + gh) * D + d] = lsum > 0.f ? acc / lsum : 0.f;
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

cudaError_t launch_decode_f32(int head_size, const float* k_cache, const float* v_cache, const DecodeParams& p,
                              cudaStream_t stream) {
  const long long grid = (long long)p.num_seqs * p.num_kv_heads * p.head_groups * p.pmax;
  if (grid == 0) return cudaSuccess;
  if (head_size == 64) return launch_dependent(decode_f32_kernel<64, 4>, dim3((unsigned)grid), dim3(128), 0, stream,
                                               k_cache, v_cache, p);
  if (head_size == 128)
    return launch_dependent(decode_f32_kernel<128, 4>, dim3((unsigned)grid), dim3(128), 0, stream, k_cache, v_cache, p);
  return cudaErrorInvalidValue;
}

}  // namespace pa

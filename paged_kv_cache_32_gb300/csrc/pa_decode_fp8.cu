// pa_decode_fp8.cu - paged decode attention over an FP8 (E4M3) KV cache, and
// the quantising append that fills it, on sm_103a.
//
// What it computes: the decode attention of "vLLM 核心工程深度剖析", section
// "3.1 Kernel 签名与分块策略", over a cache whose elements are FP8 ("PagedAttention
// 详解：缓存的存储结构", section "软件地址翻译": cache_t may be FP8, x = 16 /
// sizeof(cache_t) = 16 elements per 16-byte access).  Reading of the scale:
// every stored key code c stands for k_scale * e4m3(c) and every value code
// for v_scale * e4m3(c), one fp32 scale per cache; queries and outputs are
// fp16.  The append writes the E4M3 code nearest to x / scale (fp32 division,
// ties to even, saturating at +-448).
//
// Layout: keys [blocks][kv_heads][B][D] (a token's key is one D-byte row),
// values [blocks][kv_heads][B/16][D][16]: the value layout of "软件地址翻译"
// ([D][B], a dimension's tokens contiguous) tiled in groups of 16 tokens, the
// same thing for B = 16, so that the values of every 16 tokens of one head are
// one contiguous 2 KB run for any block size.
//
// How: the structure of the fp16/bf16 kernel (one CTA per (sequence, kv head,
// head group, partition), four warps each streaming slabs through a private
// ring filled by asynchronous bulk copies).  A slab is 32 tokens: two 16-token
// sub-slabs, each inside one block, each one 2 KB tensor-map box of keys (16
// rows x 128 bytes, 128-byte swizzle) and one 2 KB 1-D bulk copy of values
// (D rows of 16 bytes; a tensor-map box of 128 rows x 16 bytes moves the same
// bytes measurably slower).  When B is a multiple of 32 both sub-slabs lie in
// one block, and a slab is one 32-row key box and one 4 KB run of values: two
// copies instead of four, the same shared-memory image;
// 32 tokens per slab halve the fixed per-slab work (barrier wait, block-table
// shuffle, row-max shuffles) per byte against 16.  A head's running max moves
// only when a score exceeds it by more than 8 (log2 units); on the other slabs
// the row maxima, their shuffles and the output rescale are skipped.  E4M3 values convert exactly to fp16 (cvt e4m3x2 -> f16x2), so
// both contractions run on mma.m16n8k16 in fp16 with fp32 accumulation.  One
// 32-bit ldmatrix element holds four FP8 codes, which fixes the k order inside
// an MMA: slot 2c <- element 4c, 2c+1 <- 4c+1, 2c+8 <- 4c+2, 2c+9 <- 4c+3.
//  * S^T = K Q^T: k runs over head dimensions; the query fragments are loaded
//    in the same order, so each k-step still covers 16 dimensions exactly once.
//  * O^T += V^T P^T: k runs over the slab's tokens.  The key rows of the S MMA
//    are read in the order tau(r) = (r < 8 ? 4(r/2) + r%2 : 4((r-8)/2) + 2 +
//    r%2), so that after the movmatrix transpose of P every probability lands
//    in the k slot of its token.
// k_scale is folded into the softmax scale and v_scale into the output.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "pa.h"
#include "pa_decode_epilogue.cuh"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr long long kWaitCyclesFp8 = 500ll * 1000 * 1000;  // bound on one wait: ~0.25 s at 2 GHz
constexpr long long kTestWaitCyclesFp8 = 20000;              // the test hook's bound on a ring's first wait

template <int D, int NW, int NS>
struct Fp8Shape {
  static constexpr int SUB = kTcSlabTokens;               // tokens per sub-slab (one box, inside one block)
  static constexpr int NSUB = 2;                          // sub-slabs per slab
  static constexpr int SB = SUB * NSUB;                   // tokens per slab
  static constexpr int KBOX = SUB * D;                    // key box: 16 rows x D bytes
  static constexpr int VBOX = D * SUB;                    // value run: D rows x 16 bytes, contiguous
  static constexpr int SLAB_BYTES = NSUB * (KBOX + VBOX); // keys of both sub-slabs, then their values
  static constexpr int RING_BYTES = NS * SLAB_BYTES;      // per warp
  static constexpr int OROW = D + 4;                      // merge row stride (floats)
  static constexpr int WARP_MERGE = 8 * OROW + 16;
  static constexpr int BAR_OFF = NW * RING_BYTES;
  static constexpr int FLAG_OFF = BAR_OFF + NW * NS * 8;
  static constexpr int STAGE_OFF = FLAG_OFF + 16;  // pa_decode_append: the new token's fp16 K and V rows
  static constexpr int SMEM_BYTES = STAGE_OFF + 2 * D * 2 + 1024;
  static constexpr int THREADS = NW * 32;
  static_assert(D == 128, "the FP8 key box is one 128-byte swizzle row per token");
  static_assert(RING_BYTES >= WARP_MERGE * 4, "a warp's ring holds its partial result at the end");
};

struct Fp8Item {
  int s, hkv, hq0, gcount, part, L, t_end, j0, nslabs;
  bool final_out;
};

__device__ __forceinline__ bool fp8_item(const DecodeParams& p, int id, Fp8Item& it) {
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
  if (L == 0) {
    it.t_end = it.j0 = it.nslabs = 0;
    it.final_out = true;
    return it.part == 0;
  }
  if (t_begin >= L) return false;
  it.t_end = min(L, t_begin + ps);
  it.j0 = t_begin;  // slabs of 2 x 16 tokens are counted from the partition's first token
  it.nslabs = (it.t_end - t_begin + 2 * kTcSlabTokens - 1) / (2 * kTcSlabTokens);
  it.final_out = L <= ps;
  return true;
}

// try_wait that lets the hardware park the thread (up to ~20 us) until the phase completes, so
// waiting warps take no issue slots from the warps that compute
__device__ __forceinline__ bool fp8_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool fp8_wait(uint64_t* bar, uint32_t parity, volatile int32_t* abort_flag,
                                         long long limit) {
  if (fp8_try_wait(bar, parity)) return true;
  const long long start = clock64();
  for (uint32_t i = 0;; ++i) {
    if (fp8_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((i & 15u) == 15u && clock64() - start > limit) {
      *abort_flag = 1;
      return false;
    }
  }
}

// four E4M3 codes (bytes 0..3 of r) -> two f16x2: lo = (byte 0, byte 1), hi = (byte 2, byte 3), exact;
// the 16-bit halves of r feed the conversions directly
__device__ __forceinline__ void e4m3x4_to_h2x2(uint32_t r, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(r));
}

// The decode step's append over an FP8 cache (pa_decode_append): the sequence's new token sits at
// position L - 1, in row r (0..31) of this slab.  Its fp16 key and value rows, copied into stage_rows
// when the CTA started, are quantised exactly as the quantising append does (code of x / scale, fp32
// division, ties to even, saturating), replace that token's codes in the slab's shared-memory tiles (the
// copy brought whatever the slot held), and the CTA of the first head group also stores them into the
// caches at the slot the block table gives ("PagedAttention 详解：缓存的存储结构", section "写入新
// K/V").  Lane l handles dimensions 4l .. 4l + 3: one 32-bit word of the key row, four bytes of the value
// tile.  The async proxy refills the buffer later, so the lanes fence their generic writes.
template <int D>
__device__ __forceinline__ void append_token_fp8(const DecodeParams& p, const Fp8Item& it, uint8_t* kst, int r,
                                                 int lane, const uint8_t* stage_rows, float k_scale, float v_scale) {
  static_assert(D == 128, "one 32-bit word of key codes per lane");
  constexpr int KBOX = 16 * D, VBOX = D * 16;
  asm volatile("cp.async.wait_all;" ::: "memory");
  const uint2 kh = *reinterpret_cast<const uint2*>(stage_rows + 8 * lane);
  const uint2 vh = *reinterpret_cast<const uint2*>(stage_rows + 2 * D + 8 * lane);
  auto quant4 = [](uint2 h, float scale) -> uint32_t {
    const __half2 a = *reinterpret_cast<const __half2*>(&h.x), b = *reinterpret_cast<const __half2*>(&h.y);
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(__low2float(a), scale), __fdiv_rn(__high2float(a), scale)), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(__low2float(b), scale), __fdiv_rn(__high2float(b), scale)), __NV_SATFINITE, __NV_E4M3);
    return (uint32_t)lo | ((uint32_t)hi << 16);
  };
  const uint32_t kc = quant4(kh, k_scale), vc = quant4(vh, v_scale);
  const int u = r >> 4, rr = r & 15;
  *reinterpret_cast<uint32_t*>(kst + u * KBOX + swz128(rr, lane >> 2) + 4 * (lane & 3)) = kc;
  uint8_t* vt = kst + 2 * KBOX + u * VBOX + rr;  // value tile of sub-slab u: byte d * 16 + token
#pragma unroll
  for (int i = 0; i < 4; ++i) vt[(4 * lane + i) * 16] = (uint8_t)(vc >> (8 * i));
  const int G = p.num_q_heads / p.num_kv_heads;
  if (it.hq0 == it.hkv * G) {  // the first head group of the kv head writes the caches
    const int pos = it.L - 1;
    const int pb = __ldg(p.block_tables + (size_t)it.s * p.max_blocks + pos / p.block_size);
    if (pb >= 0 && pb < p.num_blocks) {
      const int off = pos % p.block_size;
      const size_t head_base = ((size_t)pb * p.num_kv_heads + it.hkv) * (size_t)p.block_size * D;
      *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(p.k_cache_out) + head_base + (size_t)off * D + 4 * lane) = kc;
      uint8_t* vg = static_cast<uint8_t*>(p.v_cache_out) + head_base + (size_t)(off / 16) * D * 16 + off % 16;
#pragma unroll
      for (int i = 0; i < 4; ++i) vg[(size_t)(4 * lane + i) * 16] = (uint8_t)(vc >> (8 * i));
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
}

// key row of the S MMA's A row r: tau(r) (see the file comment)
__device__ __forceinline__ int tau(int r) { return r < 8 ? 4 * (r >> 1) + (r & 1) : 4 * ((r - 8) >> 1) + 2 + (r & 1); }

// One slab of 32 tokens (two 16-token sub-slabs).  kst: keys of sub-slab u at
// kst + u * 16 * 128 (16 rows x 128 bytes, 128-byte swizzle); vst: values of
// sub-slab u at vst + u * 128 * 16 (128 rows = dimensions x 16 bytes = tokens).
// nvalid: tokens of the slab inside the partition (1..32).  qf: query
// fragments in the k order of the file comment.
template <int D>
__device__ __forceinline__ void fp8_slab(const uint8_t* kst, const uint8_t* vst, int nvalid,
                                         const uint32_t (&qf)[D / 16][2], float (&o)[D / 16][4], float& m_a,
                                         float& m_b, float& l_a, float& l_b, int lane, float sl2, float bias_a,
                                         float bias_b, float rel0) {
  constexpr int KBOX = 16 * D, VBOX = D * 16;
  const int g = lane >> 2, c = lane & 3;
  // ---- S^T[32 token rows x 8 heads]: per sub-slab u, rows in tau order
  float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  float sd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  {
    const int mi = lane >> 3, r = (lane & 7) + 8 * (mi & 1);
    const int krow = tau(r);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
#pragma unroll
      for (int j = 0; j < D / 32; ++j) {  // 32 dimensions = two k-steps per ldmatrix.x4
        uint32_t r0, r1, r2, r3;
        ldmatrix_x4(smem_u32(kst + u * KBOX) + swz128(krow, 2 * j + (mi >> 1)), r0, r1, r2, r3);
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        e4m3x4_to_h2x2(r0, a0, a2);
        e4m3x4_to_h2x2(r1, a1, a3);
        e4m3x4_to_h2x2(r2, b0, b2);
        e4m3x4_to_h2x2(r3, b1, b3);
        Mma<__half>::run(sc[u], a0, a1, a2, a3, qf[2 * j][0], qf[2 * j][1]);
        Mma<__half>::run(sd[u], b0, b1, b2, b3, qf[2 * j + 1][0], qf[2 * j + 1][1]);
      }
    }
  }
  // scores of sub-slab u: (token 16u + tau(g), heads 2c, 2c+1), (token 16u + tau(g+8), heads 2c, 2c+1)
  const int tok_lo = tau(g), tok_hi = tau(g + 8);
  float s[2][4];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const float r_lo = rel0 + (float)(16 * u + tok_lo), r_hi = rel0 + (float)(16 * u + tok_hi);
    s[u][0] = fmaf(bias_a, r_lo, (sc[u][0] + sd[u][0]) * sl2);
    s[u][1] = fmaf(bias_b, r_lo, (sc[u][1] + sd[u][1]) * sl2);
    s[u][2] = fmaf(bias_a, r_hi, (sc[u][2] + sd[u][2]) * sl2);
    s[u][3] = fmaf(bias_b, r_hi, (sc[u][3] + sd[u][3]) * sl2);
    if (nvalid < 16 * u + 16) {
      if (16 * u + tok_lo >= nvalid) s[u][0] = s[u][1] = -INFINITY;
      if (16 * u + tok_hi >= nvalid) s[u][2] = s[u][3] = -INFINITY;
    }
  }
  // the running maxima stay while no score exceeds them by more than kSlabSlack (log2 units), as in the
  // fp16/bf16 slab: then the slab's maxima and their shuffles are skipped
  bool over = false;
#pragma unroll
  for (int u = 0; u < 2; ++u)
    over = over || s[u][0] - m_a > kSlabSlack || s[u][1] - m_b > kSlabSlack || s[u][2] - m_a > kSlabSlack ||
           s[u][3] - m_b > kSlabSlack;
  float mn_a = m_a, mn_b = m_b;
  if (__any_sync(0xffffffffu, over)) {
    float mx_a = fmaxf(fmaxf(s[0][0], s[0][2]), fmaxf(s[1][0], s[1][2]));
    float mx_b = fmaxf(fmaxf(s[0][1], s[0][3]), fmaxf(s[1][1], s[1][3]));
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, off));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, off));
    }
    mn_a = fmaxf(m_a, mx_a);
    mn_b = fmaxf(m_b, mx_b);
  }
  if (__any_sync(0xffffffffu, mn_a != m_a || mn_b != m_b)) {  // a running max moved: rescale (rare after a while)
    const float al_a = fast_exp2(m_a - mn_a), al_b = fast_exp2(m_b - mn_b);
    l_a *= al_a;
    l_b *= al_b;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      o[i][0] *= al_a;
      o[i][1] *= al_b;
      o[i][2] *= al_a;
      o[i][3] *= al_b;
    }
    m_a = mn_a;
    m_b = mn_b;
  }
  uint32_t pb[2][2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const uint32_t x0 = Mma<__half>::pack(fast_exp2(s[u][0] - m_a), fast_exp2(s[u][1] - m_b));
    const uint32_t x1 = Mma<__half>::pack(fast_exp2(s[u][2] - m_a), fast_exp2(s[u][3] - m_b));
    // the sums use the rounded probabilities the value MMA multiplies with
    l_a += Mma<__half>::lo(x0) + Mma<__half>::lo(x1);
    l_b += Mma<__half>::hi(x0) + Mma<__half>::hi(x1);
    // P^T fragments: rows 2c, 2c+1 (tokens 4c, 4c+1) and rows 2c+8, 2c+9 (tokens 4c+2, 4c+3); head g
    pb[u][0] = movmatrix_trans(x0);
    pb[u][1] = movmatrix_trans(x1);
  }
  // ---- O^T[D x 8 heads] += V^T P^T; this lane's value elements are tokens 16u + 4c .. 16u + 4c+3
  uint32_t m_lo[2], m_hi[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int t0 = 16 * u + 4 * c;
    m_lo[u] = (t0 < nvalid ? 0x0000ffffu : 0u) | (t0 + 1 < nvalid ? 0xffff0000u : 0u);
    m_hi[u] = (t0 + 2 < nvalid ? 0x0000ffffu : 0u) | (t0 + 3 < nvalid ? 0xffff0000u : 0u);
  }
#pragma unroll
  for (int i = 0; i < D / 32; ++i) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      uint32_t r0, r1, r2, r3;
      ldmatrix_x4(smem_u32(vst + u * VBOX) + (32 * i + lane) * 16, r0, r1, r2, r3);
      // m-tile 2i: dimensions 32i + g (r0) and 32i + 8 + g (r1); m-tile 2i+1: r2, r3
      uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
      e4m3x4_to_h2x2(r0, a0, a2);
      e4m3x4_to_h2x2(r1, a1, a3);
      e4m3x4_to_h2x2(r2, b0, b2);
      e4m3x4_to_h2x2(r3, b1, b3);
      if (nvalid < 16 * u + 16) {  // values of tokens past the end may be NaN codes: zero them
        a0 &= m_lo[u], a1 &= m_lo[u], b0 &= m_lo[u], b1 &= m_lo[u];
        a2 &= m_hi[u], a3 &= m_hi[u], b2 &= m_hi[u], b3 &= m_hi[u];
      }
      Mma<__half>::run(o[2 * i], a0, a1, a2, a3, pb[u][0], pb[u][1]);
      Mma<__half>::run(o[2 * i + 1], b0, b1, b2, b3, pb[u][0], pb[u][1]);
    }
  }
}

template <int D, int NW, int NS>
__global__ void __launch_bounds__(Fp8Shape<D, NW, NS>::THREADS)
    decode_fp8_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_k32,
                      const uint8_t* __restrict__ v_cache, const DecodeParams p, const float k_scale,
                      const float v_scale) {
  using S = Fp8Shape<D, NW, NS>;
  griddep_launch_dependents();  // the partition merge may be scheduled behind this grid's last CTAs
  // seq_lens and block_tables are read before griddepcontrol.wait: no kernel of this library writes them.
  // q and the ALiBi slopes, which a GEMM before this kernel may produce, are read after it; the CTA's q
  // rows are only prefetched into L2 before it (a later load of them sees the final data).
  Fp8Item it;
  if (!fp8_item(p, blockIdx.x, it)) return;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  uint8_t* ring = smem + warp * S::RING_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BAR_OFF) + warp * NS;
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + S::FLAG_OFF);
  const int n_my = it.nslabs > warp ? (it.nslabs - warp + NW - 1) / NW : 0;
  const int B = p.block_size;
  // B a multiple of 32: a slab (32 tokens from a multiple of 32; partitions start on block boundaries)
  // lies in one block, so one 32-row key box and one 4 KB value run fetch it
  const bool whole_slabs = B % S::SB == 0;
  const int32_t* table = p.block_tables + (size_t)it.s * p.max_blocks;
  // first token of sub-slab u of this warp's k-th slab
  auto sub_tok = [&](int k, int u) { return it.j0 + (warp + k * NW) * S::SB + u * S::SUB; };
  // lane l holds the table entries of both sub-slabs of slab (batch * 32 + l); -1 past the item
  auto fetch = [&](int k, int u) -> int {
    const int t = sub_tok(k, u);
    return (k < n_my && t < it.t_end) ? __ldg(table + t / B) : -1;
  };
  int pb_batch = 0;
  int pb_reg0 = fetch(lane, 0), pb_reg1 = fetch(lane, 1);

  if (warp == 0)
    prefetch_l2(reinterpret_cast<const __half*>(p.q) + ((size_t)it.s * p.num_q_heads + it.hq0) * D,
                it.gcount * D * (int)sizeof(__half), lane);
  if (threadIdx.x == 0) {
    abort_flag[0] = 0;
    tma_prefetch_descriptor(whole_slabs ? &tmap_k32 : &tmap_k);
  }
  if (lane == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
  }
  __syncthreads();

  griddep_wait();  // launched as a dependent: the previous kernel's writes (cache, output) are visible from here
  // ---- query fragments (B operand of S^T = K Q^T): head g; k-step j covers dimensions
  //      16j .. 16j+15 in the order of the key fragments: slots (2c, 2c+1 | 2c+8, 2c+9) <- 4c .. 4c+3
  uint32_t qf[D / 16][2];
  {
    const bool real = g < it.gcount;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(reinterpret_cast<const __half*>(p.q) +
                                                             ((size_t)it.s * p.num_q_heads + it.hq0 + g) * D);
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
      qf[j][0] = real ? __ldg(qrow + (16 * j + 4 * c) / 2) : 0u;
      qf[j][1] = real ? __ldg(qrow + (16 * j + 4 * c + 2) / 2) : 0u;
    }
  }
  float bias_a = 0.f, bias_b = 0.f;
  if (p.alibi != nullptr) {
    constexpr float kLog2e = 1.4426950408889634f;
    if (2 * c < it.gcount) bias_a = __ldg(p.alibi + it.hq0 + 2 * c) * kLog2e;
    if (2 * c + 1 < it.gcount) bias_b = __ldg(p.alibi + it.hq0 + 2 * c + 1) * kLog2e;
  }
  const float sl2 = p.scale_log2 * k_scale;  // scores of the stored codes, in log2 units

  // pa_decode_append: the warp whose slab holds position L - 1 starts copying the new token's fp16 rows
  // (lanes 0..15 the key, 16..31 the value, 16 bytes each) into the stage
  uint8_t* stage_rows = smem + S::STAGE_OFF;
  {
    const int apos = it.L - 1;
    if (p.new_k != nullptr && apos >= it.j0 && apos < it.t_end && ((apos - it.j0) / S::SB) % NW == warp) {
      constexpr int CH = D * 2 / 16;
      const size_t row = (size_t)it.s * p.num_kv_heads + it.hkv;
      const void* src = reinterpret_cast<const uint4*>(lane >= CH ? p.new_v : p.new_k) + row * CH + lane % CH;
      const uint32_t dst = smem_u32(stage_rows + 16 * lane);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n\tcp.async.commit_group;" ::"r"(dst), "l"(src)
                   : "memory");
    }
  }

  uint32_t valid_mask = 0;
  auto issue = [&](int k) {  // the whole warp, k increasing
    if ((k >> 5) != pb_batch) {
      pb_batch = k >> 5;
      pb_reg0 = fetch(k + lane, 0);
      pb_reg1 = fetch(k + lane, 1);
    }
    const int pb0 = __shfl_sync(0xffffffffu, pb_reg0, k & 31), pb1 = __shfl_sync(0xffffffffu, pb_reg1, k & 31);
    // sub-slab 1 may lie past the item's end (pb1 = -1, nothing to load); any other bad ID skips the slab
    const bool has1 = sub_tok(k, 1) < it.t_end;
    const bool valid = pb0 >= 0 && pb0 < p.num_blocks && (!has1 || (pb1 >= 0 && pb1 < p.num_blocks));
    const int stage = k % NS;
    valid_mask = valid ? (valid_mask | (1u << stage)) : (valid_mask & ~(1u << stage));
    if (lane == 0) {
      uint64_t* bar = &bars[stage];
      if (valid && whole_slabs) {
        // both sub-slabs in block pb0 (rows past the item inside that block are masked, or zeroed for values)
        uint8_t* dst = ring + stage * S::SLAB_BYTES;
        const int slot0 = sub_tok(k, 0) % B;
        const int head_row = pb0 * p.num_kv_heads + it.hkv;
        mbar_arrive_expect_tx(bar, S::NSUB * (S::KBOX + S::VBOX));
        tma_load_2d(dst, &tmap_k32, 0, head_row * B + slot0, bar);
        bulk_load_1d(dst + S::NSUB * S::KBOX, v_cache + (size_t)(head_row * B + slot0) * D, S::NSUB * S::VBOX, bar);
      } else if (valid) {
        uint8_t* dst = ring + stage * S::SLAB_BYTES;
        mbar_arrive_expect_tx(bar, (has1 ? 2 : 1) * (S::KBOX + S::VBOX));
#pragma unroll
        for (int u = 0; u < S::NSUB; ++u) {
          if (u == 1 && !has1) break;
          const int pb = u ? pb1 : pb0;
          const int slot0 = sub_tok(k, u) % B;  // first token of the sub-slab in its block
          const int head_row = pb * p.num_kv_heads + it.hkv;
          tma_load_2d(dst + u * S::KBOX, &tmap_k, 0, head_row * B + slot0, bar);
          // values of tokens slot0 .. slot0 + 15 (slot0 a multiple of 16): [D][16] at (head_row * B + slot0) * D
          bulk_load_1d(dst + S::NSUB * S::KBOX + u * S::VBOX, v_cache + (size_t)(head_row * B + slot0) * D, S::VBOX,
                       bar);
        }
      } else {
        report_error(p.err_flag, PA_DEVERR_BLOCK_ID);
        mbar_arrive(bar);
      }
    }
  };

  float o[D / 16][4];
#pragma unroll
  for (int i = 0; i < D / 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY;
  float l_a = 0.f, l_b = 0.f;

  // test hook (pa_decode_options.test_flags): slab 0 of each ring is never requested and the
  // first wait has a short bound, so that wait expires and the abort path below runs
  const int first_issued = p.test_expire_first_wait ? 1 : 0;
  const int prologue = n_my < NS ? n_my : NS;
  for (int k = first_issued; k < prologue; ++k) issue(k);
  int k = 0;
  for (; k < n_my; ++k) {
    const int stage = k % NS;
    const long long limit = (k == 0 && p.test_expire_first_wait) ? kTestWaitCyclesFp8 : kWaitCyclesFp8;
    if (!__all_sync(0xffffffffu, fp8_wait(&bars[stage], (k / NS) & 1, abort_flag, limit))) break;
    if ((valid_mask >> stage) & 1u) {
      const int tok0 = sub_tok(k, 0);
      const int nvalid = min(S::SB, it.t_end - tok0);
      uint8_t* kst = ring + stage * S::SLAB_BYTES;
      // (a 16-token partition ends inside its last slab: the token must lie in this partition's part of it)
      if (p.new_k != nullptr && it.L - 1 >= tok0 && it.L - 1 < tok0 + nvalid)
        append_token_fp8<D>(p, it, kst, it.L - 1 - tok0, lane, stage_rows, k_scale, v_scale);
      fp8_slab<D>(kst, kst + S::NSUB * S::KBOX, nvalid, qf, o, m_a, m_b, l_a, l_b, lane, sl2, bias_a, bias_b,
                  (float)(tok0 - (it.L - 1)));
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

  // ---- per-warp totals into the warp's ring, then merge the warps (o scaled by v_scale)
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l_a += __shfl_xor_sync(0xffffffffu, l_a, off);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, off);
  }
  float* wo = reinterpret_cast<float*>(ring);
  float* wml = wo + 8 * S::OROW;
#pragma unroll
  for (int i = 0; i < D / 16; ++i) {
    wo[(2 * c) * S::OROW + 16 * i + g] = o[i][0] * v_scale;
    wo[(2 * c + 1) * S::OROW + 16 * i + g] = o[i][1] * v_scale;
    wo[(2 * c) * S::OROW + 16 * i + g + 8] = o[i][2] * v_scale;
    wo[(2 * c + 1) * S::OROW + 16 * i + g + 8] = o[i][3] * v_scale;
  }
  if (g == 0) {
    wml[(2 * c) * 2] = m_a;
    wml[(2 * c) * 2 + 1] = l_a;
    wml[(2 * c + 1) * 2] = m_b;
    wml[(2 * c + 1) * 2 + 1] = l_b;
  }
  __syncthreads();

  finish_item<__half, D, NW, S::OROW, S::RING_BYTES>(smem, p, (size_t)it.s * p.num_q_heads + it.hq0, it.gcount,
                                                     it.final_out, ws_row_slot(p, it.s, it.hq0) + it.part,
                                                     seq_partition_slots(p, it.s));
}

// The quantising append: block (token, kv head); thread d handles element d.
// Keys go to [block][head][offset][d] (one coalesced row), values to
// [block][head][offset / 16][d][offset % 16].
__global__ void __launch_bounds__(128)
    reshape_and_cache_fp8_kernel(uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                                 const __half* __restrict__ key, const __half* __restrict__ value,
                                 const int64_t* __restrict__ slot_mapping, int32_t num_blocks, int32_t block_size,
                                 int32_t num_kv_heads, int32_t head_size, float k_scale, float v_scale,
                                 int32_t* err_flag) {
  griddep_launch_dependents();  // a decode launched as a dependent may be scheduled behind this grid
  const int t = blockIdx.x, h = blockIdx.y;
  const int64_t slot = __ldg(slot_mapping + t);
  if (slot < 0) return;  // padding token
  const int64_t blk = slot / block_size, off = slot % block_size;
  if (blk >= num_blocks) {
    if (threadIdx.x == 0 && h == 0) report_error(err_flag, PA_DEVERR_SLOT);
    return;
  }
  const size_t src = ((size_t)t * num_kv_heads + h) * head_size;
  const size_t head_base = ((size_t)blk * num_kv_heads + h) * (size_t)block_size * head_size;
  const size_t vtile = head_base + (size_t)(off / 16) * head_size * 16 + off % 16;  // + 16 d
  for (int d = 2 * threadIdx.x; d < head_size; d += 2 * blockDim.x) {
    const __half2 kx = *reinterpret_cast<const __half2*>(key + src + d);
    const __half2 vx = *reinterpret_cast<const __half2*>(value + src + d);
    const float2 kr = make_float2(__fdiv_rn(__low2float(kx), k_scale), __fdiv_rn(__high2float(kx), k_scale));
    const float2 vr = make_float2(__fdiv_rn(__low2float(vx), v_scale), __fdiv_rn(__high2float(vx), v_scale));
    const __nv_fp8x2_storage_t kc = __nv_cvt_float2_to_fp8x2(kr, __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t vc = __nv_cvt_float2_to_fp8x2(vr, __NV_SATFINITE, __NV_E4M3);
    *reinterpret_cast<__nv_fp8x2_storage_t*>(k_cache + head_base + (size_t)off * head_size + d) = kc;
    v_cache[vtile + (size_t)d * 16] = (uint8_t)(vc & 0xff);  // element d: the low byte
    v_cache[vtile + (size_t)(d + 1) * 16] = (uint8_t)(vc >> 8);
  }
}

}  // namespace

cudaError_t launch_decode_fp8(int head_size, const CUtensorMap& tk, const CUtensorMap& tk32, const void* v_cache,
                              const DecodeParams& p, float k_scale, float v_scale, cudaStream_t stream) {
  if (head_size != 128) return cudaErrorInvalidValue;
  using S = Fp8Shape<128, 4, 2>;
  auto kernel = decode_fp8_kernel<128, 4, 2>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long items = decode_grid_size(p);
  if (items == 0) return cudaSuccess;
  return launch_dependent(kernel, dim3((unsigned)items), dim3(S::THREADS), S::SMEM_BYTES, stream, tk, tk32,
                          static_cast<const uint8_t*>(v_cache), p, k_scale, v_scale);
}

cudaError_t launch_reshape_and_cache_fp8(void* k_cache, void* v_cache, const void* key, const void* value,
                                         const int64_t* slot_mapping, int32_t num_tokens, int32_t num_blocks,
                                         int32_t block_size, int32_t num_kv_heads, int32_t head_size,
                                         float k_scale, float v_scale, int32_t* err_flag, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  dim3 grid((unsigned)num_tokens, (unsigned)num_kv_heads);
  reshape_and_cache_fp8_kernel<<<grid, 64, 0, stream>>>(
      static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), static_cast<const __half*>(key),
      static_cast<const __half*>(value), slot_mapping, num_blocks, block_size, num_kv_heads, head_size, k_scale,
      v_scale, err_flag);
  return cudaGetLastError();
}

}  // namespace pa

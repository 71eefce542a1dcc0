// pa_prefill_tc.cu - chunked prefill attention over the paged KV cache, on the
// fifth-generation tensor cores (tcgen05 + TMEM) of sm_103a.
//
// What it computes ("PagedAttention 详解：缓存的存储结构", section "使用流程": cached
// prompt blocks take part in attention directly, only missed blocks are
// computed and written through slot_mapping; "vLLM 核心工程深度剖析", section "6.1":
// long prompts are prefilled in chunks): sequence s holds seq_lens[s] = L
// tokens in the cache, the last n of which are this chunk's queries.  Query j
// (position p = L - n + j) of head h attends causally to cache positions
// 0..p: out = softmax_i(scale * q . k_i) v_i.  Keys and values of token i come
// from offset i % B of block block_tables[s][i / B] (section "软件地址翻译").
//
// How (one CTA per sequence, query head and tile of 128 queries; 9 warps):
//  * Data: the query tile is fetched once by a 3-D tensor-map copy; key and
//    value tiles of 128 tokens are gathered block by block through the block
//    table with 2-D tensor-map copies (128-byte swizzle) into two-stage K and
//    V rings.  Each copy (one block, one 64-column half) is issued by its own
//    thread, which arrives on the stage barrier with the bytes it copies.
//  * Tensor memory (512 columns): two S buffers (0..127, 128..255) and two
//    output accumulators O0, O1 (256..383, 384..511).
//  * Warp 8 (one thread) issues every MMA: S = Q K^T (M = 128 queries,
//    N = 128 keys, K = D; A and B from shared memory) and O_g += P_g V_g
//    (A = P from tensor memory, B = V from shared memory), kind::f16 with fp32
//    accumulation.  S of tile kt + 2 goes into the buffer of tile kt once
//    P V of tile kt has finished, so the softmax of tile kt + 1 overlaps both.
//  * Warps 0..7 run the softmax as two groups: group g owns keys
//    64g .. 64g + 63 of every key tile (columns of S), with its own running
//    max m_g, sum l_g and accumulator O_g for every query row (thread = row
//    in the 32x32b tensor-memory layout, no cross-thread reduction).  P is
//    written back into the S columns it came from (tcgen05.st) and consumed
//    there by the P V MMA; bf16 P is written as two terms hi + lo (two MMAs),
//    since 8 significant bits alone would cost up to 2^-8 of each weight.
//  * Rescaling: a row's reference max moves only when the tile max exceeds it
//    by more than 8 (log2 units), so P <= 2^8 and O_g is rescaled in place
//    (tcgen05.ld / st) on few tiles.  The epilogue merges the two groups:
//    out = (O0 2^(m0-M) + O1 2^(m1-M)) / (l0 2^(m0-M) + l1 2^(m1-M)).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <type_traits>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kTile = 128;            // queries per CTA = keys per key tile
constexpr int kD = 128;               // head size of this kernel
constexpr int kHalf = kTile * 128;    // one 128-row x 128-byte swizzled region (16 KB)
constexpr int kQOff = 0;              // Q: 2 regions (dims 0-63, 64-127)
constexpr int kKOff = 2 * kHalf;      // K stages: 2 x 2 regions
constexpr int kVOff = 6 * kHalf;      // V stages: 2 x 2 regions
constexpr int kBarOff = 10 * kHalf;   // barriers, flags, the (m, l) exchange
constexpr int kSmemBytes = kBarOff + 128 + 2 * kTile * 8 + 1024;
constexpr int kSoftmaxWarps = 8;
constexpr int kThreads = (kSoftmaxWarps + 1) * 32;
constexpr int kControlWarp = kSoftmaxWarps;
constexpr float kRescaleThreshold = 8.f;  // log2 units: P <= 2^8 between rescales
constexpr long long kWaitCyclesPf = 500ll * 1000 * 1000;

// bf16 keeps 8 significant bits, so P is fed to the tensor cores as two bf16
// terms (P = hi + lo, two MMAs); fp16's 11 bits need one
template <typename T>
constexpr bool split_p() {
  return std::is_same<T, __nv_bfloat16>::value;
}

// bounded wait; gives up at once when another thread has recorded a failure
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCyclesPf) {
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

// drain wait: bounded, ignores the abort flag
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitCyclesPf) return;
}

// shared-memory matrix descriptor, 128-byte swizzle (version 1)
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// instruction descriptor, kind::f16: fp32 accumulate, A/B element type (0 f16, 1 bf16), B major (0 K, 1 MN),
// M = N = 128
template <typename T>
__device__ __forceinline__ constexpr uint32_t idesc(uint32_t b_mn) {
  constexpr uint32_t ab = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | (b_mn << 16) | ((uint32_t)(kTile >> 3) << 17) |
         ((uint32_t)(kTile >> 4) << 24);
}

// D (tensor memory) (+)= A (shared memory) x B (shared memory)
__device__ __forceinline__ void mma_ss(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t id, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(id), "r"((uint32_t)accumulate)
      : "memory");
}

// D (tensor memory) (+)= A (tensor memory, row m in lane m, 2 elements per column) x B (shared memory)
__device__ __forceinline__ void mma_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t id, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(b), "r"(id), "r"((uint32_t)accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 consecutive columns of this warp's 32 lanes; completes with tmem_wait_ld()
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// wait for outstanding tensor-memory loads, then tie each loaded register to the wait so that
// no use of it is scheduled before the data has arrived
template <int N>
__device__ __forceinline__ void tmem_wait_ld(float* v) {
  tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+f"(v[i]));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// packed fp32 pair arithmetic (one instruction for two lanes of work)
__device__ __forceinline__ unsigned long long f2_bits(float2 a) {
  return (unsigned long long)__float_as_uint(a.x) | ((unsigned long long)__float_as_uint(a.y) << 32);
}
__device__ __forceinline__ float2 bits_f2(unsigned long long d) {
  return make_float2(__uint_as_float((uint32_t)d), __uint_as_float((uint32_t)(d >> 32)));
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)), "l"(f2_bits(c)));
  return bits_f2(d);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(d);
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  unsigned long long d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(d);
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap, int32_t x, int32_t y, int32_t z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
          "r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// P of one row's 64 keys (two per 32-bit column, lower key in the low half) from
// the scores v (raw q . k), the scale in log2 units and the reference max; keys
// i > lim are masked.  Writes hi (and for bf16 lo) words; returns the row sum
// of the unrounded weights.
template <typename T, bool kMasked>
__device__ __forceinline__ float make_p(const float* v, float sl2, float m_ref, int lim, uint32_t* hi,
                                        uint32_t* lo) {
  float2 acc = make_float2(0.f, 0.f);
  const float2 s2 = make_float2(sl2, sl2), nm2 = make_float2(-m_ref, -m_ref);
#pragma unroll
  for (int i = 0; i < 64; i += 2) {
    const float2 x = fma2(make_float2(v[i], v[i + 1]), s2, nm2);
    float e0 = fast_exp2(x.x), e1 = fast_exp2(x.y);
    if (kMasked) {
      e0 = i <= lim ? e0 : 0.f;
      e1 = i + 1 <= lim ? e1 : 0.f;
    }
    acc = add2(acc, make_float2(e0, e1));
    if constexpr (split_p<T>()) {
      // hi = e truncated to bf16 (exact as a float), lo = the remainder rounded to bf16
      const uint32_t b0 = __float_as_uint(e0), b1 = __float_as_uint(e1);
      hi[i / 2] = __byte_perm(b0, b1, 0x7632);
      const float2 r = sub2(make_float2(e0, e1), make_float2(__uint_as_float(b0 & 0xffff0000u),
                                                            __uint_as_float(b1 & 0xffff0000u)));
      lo[i / 2] = Mma<T>::pack(r.x, r.y);
    } else {
      hi[i / 2] = Mma<T>::pack(e0, e1);
    }
  }
  return acc.x + acc.y;
}

}  // namespace

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const PrefillParams p) {
  // ---- work item
  const int tiles = p.q_tiles;
  const int qt = tiles - 1 - (int)(blockIdx.x % tiles);  // the longest (last) query tiles start first
  const int h = (blockIdx.x / tiles) % p.num_q_heads;
  const int s = blockIdx.x / (tiles * p.num_q_heads);
  const int q0 = __ldg(p.query_start + s);
  const int n = __ldg(p.query_start + s + 1) - q0;
  const int B = p.block_size;
  const int L = __ldg(p.seq_lens + s);
  // a chunk must lie inside q / out, fit the grid, and be part of its sequence's cached tokens
  if (q0 < 0 || n < 0 || (long long)q0 + n > p.num_query_tokens || n > tiles * kTile || L < n ||
      (long long)L > (long long)p.max_blocks * B) {
    if (threadIdx.x == 0 && qt == 0 && h == 0) report_error(p.err_flag, PA_DEVERR_QUERY);
    return;
  }
  const int tile0 = qt * kTile;
  if (tile0 >= n) return;
  const int hkv = h / (p.num_q_heads / p.num_kv_heads);
  const int rows = min(kTile, n - tile0);               // valid query rows of this tile
  const int pos0 = L - n + tile0;                       // position of query row 0
  const int key_tiles = (pos0 + rows - 1) / kTile + 1;  // key tiles reaching the last row's position
  const int blocks_per_tile = kTile / B;
  const int slots = 2 * blocks_per_tile;                // copies per K (or V) tile: one per block and half
  const int32_t* table = p.block_tables + (size_t)s * p.max_blocks;
  const int nblocks_seq = (L + B - 1) / B;              // <= max_blocks (checked above)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_q = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* bar_k = bar_q + 1;  // [2] K stage landed
  uint64_t* bar_v = bar_q + 3;  // [2] V stage landed
  uint64_t* bar_s = bar_q + 5;  // [2] S buffer computed
  uint64_t* bar_p = bar_q + 7;  // [2] P of the buffer written by all softmax warps
  uint64_t* bar_o = bar_q + 9;  // O += P V done
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kBarOff + 96);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + 104);
  float2* ml = reinterpret_cast<float2*>(smem + kBarOff + 128);  // [2][128] (m, l) per group and row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int n_s = 0, n_o = 0;  // S / P V commits (control thread)
  int n_k = 0, n_v = 0;  // K / V tiles requested (uniform over the softmax warps)

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_k[b], slots);  // every copy slot arrives once per tile (with its bytes, or none)
      mbar_init(&bar_v[b], slots);
      mbar_init(&bar_s[b], 1);
      mbar_init(&bar_p[b], kSoftmaxWarps);
    }
    mbar_init(bar_o, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(512u)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // physical block of block i of key tile kt: -1 past the sequence, -2 for an ID outside the pool
  auto block_id = [&](int kt, int i) -> int {
    const int bi = kt * blocks_per_tile + i;
    if (bi >= nblocks_seq) return -1;
    const int pb = __ldg(table + bi);
    return (pb >= 0 && pb < p.num_blocks) ? pb : -2;
  };
  // copy slot c = lane * 8 + warp (block c / 2, column half c % 2), softmax warps only: each slot's
  // thread arrives on the stage barrier with the bytes it is about to copy
  auto load_tile = [&](bool is_v, int kt) {
    const int c = lane * kSoftmaxWarps + warp;
    if (c >= slots) return;
    uint64_t* bar = is_v ? &bar_v[kt & 1] : &bar_k[kt & 1];
    const int i = c >> 1, half = c & 1;
    const int pb = block_id(kt, i);
    if (pb < 0) {
      if (pb == -2 && !is_v && half == 0) report_error(p.err_flag, PA_DEVERR_BLOCK_ID);
      mbar_arrive(bar);
      return;
    }
    mbar_arrive_expect_tx(bar, (uint32_t)B * 128);
    uint8_t* dst = smem + (is_v ? kVOff : kKOff) + (kt & 1) * 2 * kHalf + half * kHalf + i * B * 128;
    tma_load_2d(dst, is_v ? (const void*)&tmap_v : (const void*)&tmap_k, half * 64, (pb * p.num_kv_heads + hkv) * B,
                bar);
  };

  if (warp == kControlWarp) {
    // =================================================================== control warp: every MMA
    if (lane == 0) {
      const uint32_t id_s = idesc<T>(0), id_o = idesc<T>(1);
      auto issue_s = [&](int kt) {  // S buffer kt % 2 = Q K^T of key tile kt
        const uint32_t qb = smem_u32(smem + kQOff), kb = smem_u32(smem + kKOff + (kt & 1) * 2 * kHalf);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          mma_ss(tmem + (kt & 1) * 128, sw128_desc(qb + off, 16, 1024), sw128_desc(kb + off, 16, 1024), id_s, kk > 0);
        }
        mma_commit(&bar_s[kt & 1]);
        ++n_s;
      };
      tma_prefetch_descriptor(&tmap_q);
      mbar_arrive_expect_tx(bar_q, 2 * kHalf);
      for (int half = 0; half < 2; ++half)
        tma_load_3d(smem + kQOff + half * kHalf, &tmap_q, half * 64, h, q0 + tile0, bar_q);
      bool ok = wait_bar(bar_q, 0, abort_flag);
      for (int t = 0; ok && t < 2 && t < key_tiles; ++t) {
        ok = wait_bar(&bar_k[t], 0, abort_flag);
        if (ok) {
          tc_fence_after();
          issue_s(t);
        }
      }
      for (int kt = 0; ok && kt < key_tiles; ++kt) {
        const int buf = kt & 1;
        // O_g += P_g V_g once every softmax warp has written P of tile kt and V of tile kt has landed
        ok = wait_bar(&bar_p[buf], (kt >> 1) & 1, abort_flag) && wait_bar(&bar_v[buf], (kt >> 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t vb = smem_u32(smem + kVOff + buf * 2 * kHalf);
#pragma unroll
        for (int g = 0; g < 2; ++g) {
#pragma unroll
          for (int part = 0; part < (split_p<T>() ? 2 : 1); ++part) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts(tmem + 256 + 128 * g, tmem + buf * 128 + 64 * g + part * 32 + kk * 8,
                     sw128_desc(vb + g * 8192 + kk * 2048, kHalf, 1024), id_o, kt > 0 || part > 0 || kk > 0);
          }
        }
        mma_commit(bar_o);
        ++n_o;
        if (kt + 2 < key_tiles) {
          // S of tile kt + 2 overwrites this buffer (P of tile kt): after that P V has finished
          ok = wait_bar(bar_o, kt & 1, abort_flag) && wait_bar(&bar_k[buf], ((kt + 2) >> 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          issue_s(kt + 2);
        }
      }
    }
    __syncwarp();
  } else {
    // =================================================================== softmax warps
    const int g = warp >> 2;                         // key columns 64g .. 64g + 63 of every tile
    const int row = (warp & 3) * 32 + lane;          // query row = tensor-memory lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t o_addr = tmem + lane_base + 256 + 128 * g;
    const float sl2 = p.scale_log2;
    const int lim_base = min(pos0 + row, L - 1);     // last key position this row sees
    float m_ref = -INFINITY, l_run = 0.f;
    // a wait whose outcome every lane of the warp shares (warp-collective tensor-memory ops follow)
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag));
    };
    for (int t = 0; t < 2 && t < key_tiles; ++t) {
      load_tile(false, t);
      load_tile(true, t);
      ++n_k;
      ++n_v;
    }
    bool ok = true;
    for (int kt = 0; kt < key_tiles; ++kt) {
      const int buf = kt & 1;
      ok = warp_wait(&bar_s[buf], (kt >> 1) & 1);
      if (!ok) break;
      tc_fence_after();
      if (kt + 2 < key_tiles) {  // S(kt) done: its K stage takes key tile kt + 2
        load_tile(false, kt + 2);
        ++n_k;
      }
      const uint32_t s_addr = tmem + lane_base + buf * 128 + 64 * g;
      float v[64];
      tmem_ld32(s_addr, v);
      tmem_ld32(s_addr + 32, v + 32);
      tmem_wait_ld<64>(v);
      const int lim = lim_base - (kt * kTile + 64 * g);  // keys 0..lim of these 64 are visible
      const bool unmasked = __all_sync(0xffffffffu, lim >= 63);
      // ---- the tile's row max, and the reference max it implies
      float mx = -INFINITY;
      if (unmasked) {
#pragma unroll
        for (int i = 0; i < 64; i += 2) mx = max3(mx, v[i], v[i + 1]);
      } else {
#pragma unroll
        for (int i = 0; i < 64; i += 2)
          mx = max3(mx, i <= lim ? v[i] : -INFINITY, i + 1 <= lim ? v[i + 1] : -INFINITY);
      }
      const float mx_s = mx * sl2;  // scale > 0
      const bool upd = mx_s > m_ref + kRescaleThreshold;
      const float alpha = upd ? fast_exp2(m_ref - mx_s) : 1.f;
      // P V of tile kt - 1 is confirmed once per tile, in order (phase kt - 1 of bar_o; phase kt cannot
      // complete before this warp's P arrival below): first here if O must be rescaled, else before the arrival
      bool o_prev_done = kt == 0;
      if (__any_sync(0xffffffffu, upd) && kt > 0) {
        // O_g of these rows is rescaled between P V of tile kt - 1 (done) and that of tile kt
        ok = warp_wait(bar_o, (kt - 1) & 1);
        if (!ok) break;
        o_prev_done = true;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32(o_addr + c * 32, o);
          tmem_wait_ld<32>(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(o_addr + c * 32, reinterpret_cast<const uint32_t*>(o));
        }
        tmem_wait_st();
      }
      if (upd) m_ref = mx_s;
      // ---- P into the S columns it came from
      uint32_t hi[32], lo[32];
      const float lsum = unmasked ? make_p<T, false>(v, sl2, m_ref, lim, hi, lo)
                                  : make_p<T, true>(v, sl2, m_ref, lim, hi, lo);
      l_run = l_run * alpha + lsum;
      tmem_st32(s_addr, hi);
      if constexpr (split_p<T>()) tmem_st32(s_addr + 32, lo);
      tmem_wait_st();
      // ---- values of key rows past the sequence (or of blocks not loaded) may hold NaN: zero them
      if (kt * kTile + kTile > L || (kt + 1) * blocks_per_tile > nblocks_seq) {
        ok = warp_wait(&bar_v[buf], (kt >> 1) & 1);
        if (!ok) break;
        uint8_t* vst = smem + kVOff + buf * 2 * kHalf;
        for (int idx = threadIdx.x; idx < kTile * 16; idx += kSoftmaxWarps * 32) {  // 128 rows x 16 chunks
          const int r = idx >> 4, chunk = idx & 15;
          if (kt * kTile + r >= L || block_id(kt, r / B) < 0)
            *reinterpret_cast<uint4*>(vst + (chunk >> 3) * kHalf + swz128(r, chunk & 7)) = make_uint4(0, 0, 0, 0);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> tensor-core reads
      }
      // ---- V stage (kt + 1) % 2 held tile kt - 1, whose P V is done: fetch value tile kt + 1 there
      if (!o_prev_done) {
        ok = warp_wait(bar_o, (kt - 1) & 1);
        if (!ok) break;
      }
      if (kt >= 1 && kt + 1 < key_tiles) {
        load_tile(true, kt + 1);
        ++n_v;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p[buf]);
    }
    // ---- epilogue: merge the two groups' (m, l, O) per row and write out (P V of every tile before
    //      the last was confirmed inside the loop, so this parity wait cannot pass early)
    if (ok) ok = warp_wait(bar_o, (key_tiles - 1) & 1);
    ml[g * kTile + row] = make_float2(m_ref, l_run);
    asm volatile("bar.sync 1, %0;" ::"n"(kSoftmaxWarps * 32) : "memory");
    if (!__any_sync(0xffffffffu, *abort_flag != 0)) {
      tc_fence_after();
      const float2 a = ml[row], b = ml[kTile + row];
      const float M = fmaxf(a.x, b.x);
      const float w0 = a.x == -INFINITY ? 0.f : fast_exp2(a.x - M), w1 = b.x == -INFINITY ? 0.f : fast_exp2(b.x - M);
      const float den = a.y * w0 + b.y * w1;
      const float inv = den > 0.f ? 1.f / den : 0.f;
      const float c0 = w0 * inv, c1 = w1 * inv;
      T* out = reinterpret_cast<T*>(p.out) + ((size_t)(q0 + tile0 + row) * p.num_q_heads + h) * kD + 64 * g;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {  // this group writes output columns 64g .. 64g + 63
        float o0[32], o1[32];
        tmem_ld32(tmem + lane_base + 256 + 64 * g + 32 * c, o0);
        tmem_ld32(tmem + lane_base + 384 + 64 * g + 32 * c, o1);
        tmem_wait_ld<32>(o0);
        tmem_wait_ld<32>(o1);
        if (row < rows) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 val;
            val.x = Mma<T>::pack(o0[i] * c0 + o1[i] * c1, o0[i + 1] * c0 + o1[i + 1] * c1);
            val.y = Mma<T>::pack(o0[i + 2] * c0 + o1[i + 2] * c1, o0[i + 3] * c0 + o1[i + 3] * c1);
            val.z = Mma<T>::pack(o0[i + 4] * c0 + o1[i + 4] * c1, o0[i + 5] * c0 + o1[i + 5] * c1);
            val.w = Mma<T>::pack(o0[i + 6] * c0 + o1[i + 6] * c1, o0[i + 7] * c0 + o1[i + 7] * c1);
            *reinterpret_cast<uint4*>(out + 32 * c + i) = val;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // a wait expired (the flag is stable: every thread has left its loop): record it, and let the
    // copies and MMAs this CTA started finish, each wait bounded, before its memory is released
    if (threadIdx.x == 0) {
      report_error(p.err_flag, PA_DEVERR_TIMEOUT);
      for (int t = max(0, n_k - 2); t < n_k; ++t) drain_wait(&bar_k[t & 1], (t >> 1) & 1);
      for (int t = max(0, n_v - 2); t < n_v; ++t) drain_wait(&bar_v[t & 1], (t >> 1) & 1);
    }
    if (warp == kControlWarp && lane == 0) {
      for (int t = max(0, n_s - 2); t < n_s; ++t) drain_wait(&bar_s[t & 1], (t >> 1) & 1);
      if (n_o > 0) drain_wait(bar_o, (n_o - 1) & 1);
    }
    __syncthreads();
  }
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512u) : "memory");
}

cudaError_t launch_prefill_tc(int dtype, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const PrefillParams& p, cudaStream_t stream) {
  const long long grid = (long long)p.num_seqs * p.num_q_heads * p.q_tiles;
  if (grid == 0) return cudaSuccess;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  if (dtype == PA_F16) {
    cudaError_t e =
        cudaFuncSetAttribute(prefill_tc_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    prefill_tc_kernel<__half><<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, p);
  } else if (dtype == PA_BF16) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<__nv_bfloat16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    prefill_tc_kernel<__nv_bfloat16><<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace pa

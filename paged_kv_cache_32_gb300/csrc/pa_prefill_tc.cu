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
// How:
//  * One CTA (4 warps) per (sequence, query head, tile of 128 queries).  The
//    query tile is fetched once by a 3-D tensor-map copy; key/value tiles of
//    128 tokens are gathered block by block through the block table with 2-D
//    tensor-map copies (128-byte swizzle) into a two-stage ring; the four
//    warps issue the copies of a tile together.
//  * S = Q K^T (M = 128 queries, N = 128 keys, K = D) and O_t = P V
//    (M = 128, N = D, K = 128 keys) are tcgen05.mma (kind::f16, fp32
//    accumulate) issued by one thread from shared-memory descriptors; the
//    accumulators live in tensor memory (S in columns 0..127, O in 128..255).
//  * With the 32x32b tensor-memory layout thread t owns query row t, so the
//    online softmax (row max, exp2, row sum) needs no cross-thread reduction.
//    P is written to shared memory in the 128-byte-swizzled K-major layout the
//    second MMA reads (bf16 P as hi + lo terms, two MMAs, since 8 significant
//    bits alone would cost up to 2^-9 of each weight).  O accumulates in tensor memory across key tiles; when
//    a row's running max grows, its warp rescales its 32 rows of O in place
//    (tcgen05.ld / st) after the previous P V has finished and before the next
//    one is issued, so the rescale is skipped on most tiles.
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

constexpr int kTile = 128;           // queries per CTA = keys per key tile
constexpr int kD = 128;              // head size of this kernel
constexpr int kHalf = kTile * 128;   // one 128-row x 128-byte swizzled region (16 KB)
constexpr int kQOff = 0;             // Q: 2 regions (dims 0-63, 64-127)
constexpr int kKOff = 2 * kHalf;     // K stages: 2 x 2 regions
constexpr int kVOff = 6 * kHalf;     // V stages: 2 x 2 regions
constexpr int kPOff = 10 * kHalf;    // P: 2 regions (keys 0-63, 64-127)
constexpr int kPLoOff = 12 * kHalf;  // bf16 only: P - bf16(P), the same layout

// bf16 keeps 8 significant bits, so P is fed to the tensor cores as two bf16
// terms (P = hi + lo, two MMAs); fp16's 11 bits need one
template <typename T>
constexpr bool split_p() {
  return std::is_same<T, __nv_bfloat16>::value;
}
template <typename T>
constexpr int bar_off() {  // barriers: q, kv[2], s, o; then the tensor-memory address
  return split_p<T>() ? 14 * kHalf : 12 * kHalf;
}
template <typename T>
constexpr int smem_bytes() {
  return bar_off<T>() + 64 + 16 + 1024;
}
constexpr long long kWaitCyclesPf = 500ll * 1000 * 1000;

__device__ __forceinline__ bool wait_cycles(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitCyclesPf) return false;
  return true;
}

// shared-memory matrix descriptor, 128-byte swizzle (version 1)
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// instruction descriptor, kind::f16: fp32 accumulate, A/B element type (0 f16, 1 bf16), B major (0 K, 1 MN)
template <typename T>
__device__ __forceinline__ constexpr uint32_t idesc(uint32_t b_mn) {
  constexpr uint32_t ab = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | (b_mn << 16) | ((uint32_t)(kTile >> 3) << 17) |
         ((uint32_t)(kTile >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t id, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(id), "r"((uint32_t)accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
      "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
      "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])),
      "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap, int32_t x, int32_t y, int32_t z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
          "r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace

template <typename T>
__global__ void __launch_bounds__(128, 1)
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
  const int rows = min(kTile, n - tile0);             // valid query rows of this tile
  const int pos0 = L - n + tile0;                     // position of query row 0
  const int key_tiles = (pos0 + rows - 1) / kTile + 1;  // key tiles reaching the last row's position
  const int blocks_per_tile = kTile / B;
  const int32_t* table = p.block_tables + (size_t)s * p.max_blocks;
  const int nblocks_seq = min((L + B - 1) / B, p.max_blocks);  // never read past the table row

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kBarOff = bar_off<T>();
  uint64_t* bar_q = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* bar_kv = bar_q + 1;  // [2]
  uint64_t* bar_s = bar_q + 3;
  uint64_t* bar_o = bar_q + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + 64);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = threadIdx.x;  // query row owned by this thread (TMEM lane)

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    mbar_init(&bar_kv[0], 1);
    mbar_init(&bar_kv[1], 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(256u)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_s = tmem, tmem_o = tmem + 128;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

  // valid (loadable) blocks of key tile kt: in the sequence and with an in-range ID
  auto block_id = [&](int kt, int i) -> int {
    const int bi = kt * blocks_per_tile + i;
    if (bi >= nblocks_seq) return -1;
    const int pb = __ldg(table + bi);
    return (pb >= 0 && pb < p.num_blocks) ? pb : -2;
  };
  // expect the bytes of tile kt on stage kt % 2 (thread 0), then every warp issues its share of the copies
  auto expect_tile = [&](int kt) {
    int nvalid = 0;
    for (int i = 0; i < blocks_per_tile; ++i) {
      const int pb = block_id(kt, i);
      if (pb >= 0) ++nvalid;
      else if (pb == -2) report_error(p.err_flag, PA_DEVERR_BLOCK_ID);
    }
    mbar_arrive_expect_tx(&bar_kv[kt & 1], (uint32_t)nvalid * B * 128 * 4);
  };
  auto issue_tile = [&](int kt) {
    if (lane != 0) return;
    uint8_t* kst = smem + kKOff + (kt & 1) * 2 * kHalf;
    uint8_t* vst = smem + kVOff + (kt & 1) * 2 * kHalf;
    for (int i = warp; i < blocks_per_tile; i += 4) {
      const int pb = block_id(kt, i);
      if (pb < 0) continue;
      const int y = (pb * p.num_kv_heads + hkv) * B;
      for (int half = 0; half < 2; ++half) {
        tma_load_2d(kst + half * kHalf + i * B * 128, &tmap_k, half * 64, y, &bar_kv[kt & 1]);
        tma_load_2d(vst + half * kHalf + i * B * 128, &tmap_v, half * 64, y, &bar_kv[kt & 1]);
      }
    }
  };

  // ---- prologue: the query tile and the first two key tiles
  if (threadIdx.x == 0) {
    tma_prefetch_descriptor(&tmap_q);
    mbar_arrive_expect_tx(bar_q, 2 * kHalf);
    for (int half = 0; half < 2; ++half)
      tma_load_3d(smem + kQOff + half * kHalf, &tmap_q, half * 64, h, q0 + tile0, bar_q);
    expect_tile(0);
    if (key_tiles > 1) expect_tile(1);
  }
  __syncthreads();
  issue_tile(0);
  if (key_tiles > 1) issue_tile(1);

  const float sl2 = p.scale_log2;
  const int my_pos = pos0 + row;  // causal limit of this thread's row (row >= rows: unused)
  float m_run = -INFINITY, l_run = 0.f;
  bool ok = true;

  int n_s = 0, n_o = 0, n_kv = key_tiles > 1 ? 2 : 1;  // S / PV commits and key tiles expected (thread 0)
  const uint32_t id_s = idesc<T>(0), id_o = idesc<T>(1);
  auto issue_s = [&](int kt) {  // S = Q K^T for key tile kt (thread 0)
    const uint32_t qb = smem_u32(smem + kQOff), kb = smem_u32(smem + kKOff + (kt & 1) * 2 * kHalf);
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
      mma_f16(tmem_s, sw128_desc(qb + off, 16, 1024), sw128_desc(kb + off, 16, 1024), id_s, kk > 0);
    }
    mma_commit(bar_s);
    ++n_s;
  };
  if (threadIdx.x == 0) {
    ok = wait_cycles(bar_q, 0) && wait_cycles(&bar_kv[0], 0);
    if (ok) {
      tc_fence_after();
      issue_s(0);
    }
  }
  ok = __syncthreads_and(ok);

  for (int kt = 0; kt < key_tiles; ++kt) {
    // ---- pass 1 over the scores of tile kt: the row max (masked: causal and past the sequence)
    ok = ok && wait_cycles(bar_s, kt & 1) && wait_cycles(&bar_kv[kt & 1], (kt >> 1) & 1);
    ok = __syncthreads_and(ok);
    if (!ok) break;
    tc_fence_after();
    const int kpos0 = kt * kTile;
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float v[32];
      tmem_ld32(tmem_s + lane_base + c * 32, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int kp = kpos0 + c * 32 + i;
        if (kp <= my_pos && kp < L) mx = fmaxf(mx, v[i] * sl2);
      }
    }
    const float m_new = fmaxf(m_run, mx);
    const float alpha = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run - m_new);
    if (kt > 0) {
      // the previous tile's O += P V is done: P, that tile's K/V stage and O may be touched
      ok = wait_cycles(bar_o, (kt - 1) & 1);
      tc_fence_after();
      if (__any_sync(0xffffffffu, alpha != 1.f)) {  // rescale this warp's rows of O in tensor memory
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float v[32];
          tmem_ld32(tmem_o + lane_base + c * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= alpha;
          tmem_st32(tmem_o + lane_base + c * 32, v);
        }
      }
    }
    // ---- stage (kt + 1) & 1 held tile kt - 1, now consumed: fetch tile kt + 1's successor there
    //      (tiles 0 and 1 were fetched up front; tile kt + 1 >= 2 goes into stage (kt + 1) & 1)
    tc_fence_before();
    if (threadIdx.x == 0 && kt >= 1 && kt + 1 < key_tiles) {
      expect_tile(kt + 1);
      ++n_kv;
    }
    ok = __syncthreads_and(ok);
    if (!ok) break;
    tc_fence_after();
    if (kt >= 1 && kt + 1 < key_tiles) issue_tile(kt + 1);
    // ---- pass 2: P = exp2(s - m) (f16/bf16, swizzled K-major; bf16 also the residual) and its row sum
    float lsum = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float v[32];
      tmem_ld32(tmem_s + lane_base + c * 32, v);
      // keys c*32 .. c*32+31 of this row: region c / 2, 16-byte chunks (c % 2) * 4 .. +3
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          const int kp = kpos0 + c * 32 + j * 8 + i;
          const float x0 = v[j * 8 + i] * sl2 - m_new, x1 = v[j * 8 + i + 1] * sl2 - m_new;
          const float e0 = (kp <= my_pos && kp < L) ? fast_exp2(x0) : 0.f;
          const float e1 = (kp + 1 <= my_pos && kp + 1 < L) ? fast_exp2(x1) : 0.f;
          hi[i / 2] = Mma<T>::pack(e0, e1);
          if constexpr (split_p<T>()) {
            lo[i / 2] = Mma<T>::pack(e0 - Mma<T>::lo(hi[i / 2]), e1 - Mma<T>::hi(hi[i / 2]));
            lsum += e0 + e1;
          } else {
            lsum += Mma<T>::lo(hi[i / 2]) + Mma<T>::hi(hi[i / 2]);  // the values the MMA multiplies with
          }
        }
        const int off = (c >> 1) * kHalf + swz128(row, (c & 1) * 4 + j);
        *reinterpret_cast<uint4*>(smem + kPOff + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        if constexpr (split_p<T>())
          *reinterpret_cast<uint4*>(smem + kPLoOff + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
    m_run = m_new;
    l_run = l_run * alpha + lsum;
    // values of key rows past the sequence (or of skipped blocks) may hold NaN: zero them
    if (kpos0 + kTile > L || kt * blocks_per_tile + blocks_per_tile > nblocks_seq) {
      uint8_t* vst = smem + kVOff + (kt & 1) * 2 * kHalf;
      for (int idx = threadIdx.x; idx < kTile * 16; idx += 128) {  // 128 rows x 16 chunks of 16 bytes
        const int r = idx >> 4, chunk = idx & 15;
        const int kp = kpos0 + r;
        if (kp >= L || block_id(kt, r / B) < 0)
          *reinterpret_cast<uint4*>(vst + (chunk >> 3) * kHalf + swz128(r, chunk & 7)) = make_uint4(0, 0, 0, 0);
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // P and V writes -> tensor-core reads
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // ---- the next tile's scores, then O += P V (thread 0): P V runs while pass 1 of the next tile reads S
    if (threadIdx.x == 0) {
      if (kt + 1 < key_tiles) {
        ok = wait_cycles(&bar_kv[(kt + 1) & 1], ((kt + 1) >> 1) & 1);
        if (ok) {
          tc_fence_after();
          issue_s(kt + 1);
        }
      }
      const uint32_t vb = smem_u32(smem + kVOff + (kt & 1) * 2 * kHalf);
#pragma unroll
      for (int part = 0; part < (split_p<T>() ? 2 : 1); ++part) {
        const uint32_t pb = smem_u32(smem + (part ? kPLoOff : kPOff));
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_f16(tmem_o, sw128_desc(pb + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024),
                  sw128_desc(vb + kk * 2048, kHalf, 1024), id_o, kt > 0 || part > 0 || kk > 0);
      }
      mma_commit(bar_o);
      ++n_o;
    }
  }
  // ---- out = O / l for this thread's query row
  if (ok) ok = wait_cycles(bar_o, (key_tiles - 1) & 1);
  ok = __syncthreads_and(ok);
  if (!ok) {
    // a wait expired: record it, then let the copies and MMAs this CTA started finish (each wait
    // bounded) before the tensor memory is freed and the CTA's shared memory is released
    if (threadIdx.x == 0) {
      report_error(p.err_flag, PA_DEVERR_TIMEOUT);
      if (n_s > 0) wait_cycles(bar_s, (n_s - 1) & 1);
      if (n_o > 0) wait_cycles(bar_o, (n_o - 1) & 1);
      for (int t = max(0, n_kv - 2); t < n_kv; ++t) wait_cycles(&bar_kv[t & 1], (t >> 1) & 1);
    }
  } else {
    tc_fence_after();
    T* out = reinterpret_cast<T*>(p.out) + ((size_t)(q0 + tile0 + row) * p.num_q_heads + h) * kD;
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float v[32];
      tmem_ld32(tmem_o + lane_base + c * 32, v);  // warp-collective: every lane loads
      if (row < rows) {
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
          uint4 val = make_uint4(Mma<T>::pack(v[i] * inv, v[i + 1] * inv), Mma<T>::pack(v[i + 2] * inv, v[i + 3] * inv),
                                 Mma<T>::pack(v[i + 4] * inv, v[i + 5] * inv),
                                 Mma<T>::pack(v[i + 6] * inv, v[i + 7] * inv));
          *reinterpret_cast<uint4*>(out + c * 32 + i) = val;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(256u) : "memory");
}

cudaError_t launch_prefill_tc(int dtype, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const PrefillParams& p, cudaStream_t stream) {
  const long long grid = (long long)p.num_seqs * p.num_q_heads * p.q_tiles;
  if (grid == 0) return cudaSuccess;
  if (dtype == PA_F16) {
    constexpr int smem = smem_bytes<__half>();
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    prefill_tc_kernel<__half><<<(unsigned)grid, 128, smem, stream>>>(tq, tk, tv, p);
  } else if (dtype == PA_BF16) {
    constexpr int smem = smem_bytes<__nv_bfloat16>();
    static_assert(smem <= 227 * 1024, "shared memory per CTA");
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<__nv_bfloat16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    prefill_tc_kernel<__nv_bfloat16><<<(unsigned)grid, 128, smem, stream>>>(tq, tk, tv, p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace pa

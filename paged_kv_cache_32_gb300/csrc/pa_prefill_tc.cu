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
// How (persistent: one CTA of 14 warps per SM walks work items = (sequence,
// query head, tile of 128 queries); see pf_item for the order):
//  * Tensor memory (512 columns): three S buffers (0..127, 128..255,
//    256..383) and the output accumulator O (384..511).  Q stays in shared
//    memory: each item's Q tile is copied there by a tensor-map copy (two
//    buffers, so the next item's copy overlaps the current item), and the S
//    MMA reads both operands from shared memory (measured about as fast as
//    with A in tensor memory, alongside the P V MMAs, the copies and the
//    softmax's tensor-memory traffic).  Three S buffers let S of tile kt + 3
//    wait for P V of tile kt instead of S of tile kt + 2.
//  * Data: key and value tiles of 128 tokens are gathered block by block
//    through the block table by four producer warps (K and V, one warp per
//    64-column half: a single thread issues a copy in about 200 cycles and
//    the lanes of one warp largely serialise, so the copies of a tile are
//    spread over warps) with 2-D tensor-map copies (one per block and half,
//    128-byte swizzle) into two-stage rings; each copy's lane arrives on the
//    stage barrier with its bytes.  A producer refills a stage as soon as the
//    MMA that read it has finished.  Value rows past the sequence must read as
//    zeros (P is 0 there, but 0 * NaN is not): each V producer copies its half
//    of the last, partial block row by row with cp.async and zero-fills the
//    rest, then fences those generic-proxy writes before its extra arrival.
//  * Two threads in different warps issue the MMAs (kind::f16, fp32
//    accumulation): warp 9 S = Q K^T (M = 128 queries, N = 128 keys, K = D),
//    warp 8 O += P V (M = 128, N = D, K = 128 keys; P from tensor memory).
//    S of tile kt + 3 goes into the buffer of tile kt once P V of tile kt has
//    finished; with separate issuers that wait never delays the next P V, and
//    the softmax of tile kt + 1 overlaps P V of tile kt and S of tile kt + 3.
//  * Items: the S-issuing thread also publishes each item in shared memory
//    and starts its Q copy; item k + 1 is published once every softmax warp
//    has read item k.  The softmax warps process the next item's first tile
//    right after the current item's last one (it writes no O), then run the
//    current item's epilogue while its last P V finishes.
//  * Warps 0..7 run the softmax.  Each owns 16 query rows (tensor-memory
//    lanes) and all 128 keys of a tile, read with the 16-lane 16x256b shape:
//    a thread holds two rows, 32 keys of each, so a row's maximum and sum
//    take two shuffles among its four threads and no warp waits for another.
//    P is written back into the S buffer it came from (16x128b shape, two
//    keys per 32-bit column: hi words in columns 0..63, lo words in
//    64..127); bf16 P is written as two terms hi + lo (two MMAs), since 8
//    significant bits alone would cost up to 2^-8 of a weight.
//  * Rescaling: a row's reference max moves only when the tile max exceeds it
//    by more than 8 (log2 units), so P <= 2^8 and O is rescaled in place
//    (tcgen05.ld / st of the warp's 16 rows) on few tiles.  fp16 takes an
//    unmasked tile's weights with the current reference maxima first and
//    computes the tile maxima only when a weight could exceed 2^8 (same bits).
//  * Epilogue: each warp reads its 16 rows of O (16x256b layout), releases O
//    to the next item's first P V and normalises them (out = O / l).  bf16
//    stores them from registers.  fp16, whose softmax warps set the pace,
//    writes them into a 32 KB shared-memory stage in the output tensor map's
//    swizzled layout; the P V issuer then stores a full tile with two
//    tensor-map stores, and a ragged tile (rows past the chunk belong to
//    another sequence) is copied out row by row by its warps.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <climits>
#include <math.h>

#include <type_traits>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_prefill.h"

namespace pa {
namespace {

constexpr int kTile = 128;            // queries per CTA = keys per key tile
constexpr int kD = 128;               // head size of this kernel
constexpr int kHalf = kTile * 128;    // one 128-row x 128-byte swizzled region (16 KB)
constexpr int kKOff = 0;              // K stages: 2 x 2 regions (dims 0-63, 64-127)
constexpr int kVOff = 4 * kHalf;      // V stages: 2 x 2 regions
constexpr int kQOff = 8 * kHalf;      // Q tiles of two items (item k in buffer k % 2): 2 x 2 regions
constexpr int kOutOff = 12 * kHalf;   // one item's output tile, staged for a tensor-map store: 2 regions
constexpr int kBarOff = 14 * kHalf;   // barriers, flags, the published work items
constexpr int kSmemBytes = kBarOff + 512 + 1024;
constexpr int kSBufs = 3;             // S buffers in tensor memory (columns 128 b .. 128 b + 127)
constexpr uint32_t kOCol = 384;       // tensor-memory column of O
constexpr int kSoftmaxWarps = 8;
constexpr int kPVWarp = kSoftmaxWarps;         // issues O += P V
constexpr int kSWarp = kSoftmaxWarps + 1;      // issues S = Q K^T
constexpr int kLoadWarp0 = kSoftmaxWarps + 2;  // four producers: K half 0, K half 1, V half 0, V half 1
constexpr int kThreads = (kSoftmaxWarps + 6) * 32;
constexpr float kRescaleThreshold = 8.f;  // log2 units: P <= 2^8 between rescales
// A tile's weights taken with the current reference maxima stand when no thread's share of a row's tile
// sum exceeds this (so no weight does): then no weight is above 2^(threshold) - 1, no reference max would
// move, and the tile's maxima are not needed.
constexpr float kLazyBound = 255.f;
constexpr long long kWaitCyclesPf = 500ll * 1000 * 1000;

// bf16 keeps 8 significant bits, so P is fed to the tensor cores as two bf16
// terms (P = hi + lo, two MMAs); fp16's 11 bits need one
template <typename T>
constexpr bool split_p() {
  return std::is_same<T, __nv_bfloat16>::value;
}

// Where the epilogue writes the output tile.  fp16 (softmax-bound): to a shared-memory stage that the P V
// issuer sends out with two tensor-map stores, which takes the global stores off the softmax warps.  bf16
// (tensor-bound): straight from registers; its copies keep the tensor-memory-access unit busy, and the
// stores through it cost more than the softmax time they save (measured 3.9% slower).
template <typename T>
constexpr bool kStagedOut = !split_p<T>();

// try_wait that lets the hardware park the thread (up to ~20 us) until the phase completes,
// instead of spinning on the barrier and taking issue slots from the softmax warps
__device__ __forceinline__ bool mbar_try_wait_parked(uint64_t* bar, uint32_t parity) {
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

// bounded wait; gives up at once when another thread has recorded a failure
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait_parked(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_parked(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCyclesPf) {
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

// the same, spinning: for the waits on the critical path (the MMA issuers, and the softmax waiting
// for S), where waking a parked thread costs a few hundred cycles
__device__ __forceinline__ bool wait_bar_spin(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
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

// D (tensor memory) (+)= A (tensor memory, row m in lane m, 2 elements per column) x B (shared memory)
__device__ __forceinline__ void mma_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t id, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(b), "r"(id), "r"((uint32_t)accumulate)
      : "memory");
}

// D (tensor memory) (+)= A (shared memory) x B (shared memory)
__device__ __forceinline__ void mma_ss(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t id, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(id), "r"((uint32_t)accumulate)
      : "memory");
}

// shared -> global tensor-map store, tracked as a bulk group of the issuing thread.  The threads that
// wrote the source must have made their writes visible to the async proxy (fence.proxy.async) first.
__device__ __forceinline__ void tma_store_3d(const void* tmap, int32_t x, int32_t y, int32_t z, const void* smem_src) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(smem_u32(smem_src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// every committed bulk store of this thread has finished reading its shared-memory source
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// every committed bulk store of this thread has completed its writes
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// non-blocking: has the phase of the given parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
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

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// The 16-lane shapes: a warp addresses one half (16 lanes) of its lane quarter.  Thread t holds
// lanes t / 4 and t / 4 + 8 of that half.
//  16x256b.x8 (64 columns): v[4j], v[4j + 1] = lane t / 4, columns 8j + 2 (t % 4) and + 1;
//                           v[4j + 2], v[4j + 3] = lane t / 4 + 8, the same columns.
//  16x128b.x8 (32 columns): r[2j] = lane t / 4, column 4j + t % 4; r[2j + 1] = lane t / 4 + 8.
__device__ __forceinline__ void tmem_ld16x256_x8(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16x256_x8(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16x128_x8(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x128b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

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

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
// all of this thread's cp.async copies have landed (commits the pending ones first)
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// P of 8 of the 16 key pairs this thread holds in each of its two rows, pairs j0 .. j0 + 7 (v in
// the 16x256b layout over the tile's 128 columns: pair j = keys 8j + 2c, 8j + 2c + 1, c = thread % 4;
// v[4j], v[4j + 1] row 0, v[4j + 2], v[4j + 3] row 1) from the raw scores, the scale in log2 units
// and the rows' reference maxima; a pair's keys past e0 (e1) of row 0 (1), counted from key 2c, are
// masked.  Writes the packed words of those pairs in the 16x128b layout (hi[2i] row 0, hi[2i + 1]
// row 1 for pair j0 + i; for bf16 also lo) and adds the rows' sums of the unrounded weights to s0, s1.
template <typename T, bool kMasked>
__device__ __forceinline__ void make_p(const float* v, int j0, float sl2, float mr0, float mr1, int e0, int e1,
                                       uint32_t* hi, uint32_t* lo, float& s0, float& s1) {
  float2 acc0[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  float2 acc1[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  const float2 sc2 = make_float2(sl2, sl2), n0 = make_float2(-mr0, -mr0), n1 = make_float2(-mr1, -mr1);
#pragma unroll
  for (int j = j0; j < j0 + 8; ++j) {
    const float2 x = fma2(make_float2(v[4 * j], v[4 * j + 1]), sc2, n0);
    const float2 y = fma2(make_float2(v[4 * j + 2], v[4 * j + 3]), sc2, n1);
    float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y), p2 = fast_exp2(y.x), p3 = fast_exp2(y.y);
    if (kMasked) {
      p0 = 8 * j <= e0 ? p0 : 0.f;
      p1 = 8 * j + 1 <= e0 ? p1 : 0.f;
      p2 = 8 * j <= e1 ? p2 : 0.f;
      p3 = 8 * j + 1 <= e1 ? p3 : 0.f;
    }
    acc0[j & 1] = add2(acc0[j & 1], make_float2(p0, p1));
    acc1[j & 1] = add2(acc1[j & 1], make_float2(p2, p3));
    if constexpr (split_p<T>()) {
      // hi = p truncated to bf16 (exact as a float), lo = the remainder rounded to bf16
      const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
      const uint32_t b2 = __float_as_uint(p2), b3 = __float_as_uint(p3);
      hi[2 * (j - j0)] = __byte_perm(b0, b1, 0x7632);
      hi[2 * (j - j0) + 1] = __byte_perm(b2, b3, 0x7632);
      const float2 r0 = sub2(make_float2(p0, p1), make_float2(__uint_as_float(b0 & 0xffff0000u),
                                                              __uint_as_float(b1 & 0xffff0000u)));
      const float2 r1 = sub2(make_float2(p2, p3), make_float2(__uint_as_float(b2 & 0xffff0000u),
                                                              __uint_as_float(b3 & 0xffff0000u)));
      lo[2 * (j - j0)] = Mma<T>::pack(r0.x, r0.y);
      lo[2 * (j - j0) + 1] = Mma<T>::pack(r1.x, r1.y);
    } else {
      hi[2 * (j - j0)] = Mma<T>::pack(p0, p1);
      hi[2 * (j - j0) + 1] = Mma<T>::pack(p2, p3);
    }
  }
  const float2 t0 = add2(acc0[0], acc0[1]), t1 = add2(acc1[0], acc1[1]);
  s0 += t0.x + t0.y;
  s1 += t1.x + t1.y;
}

}  // namespace

// One work item: query tile qt of (sequence s, query head h).
struct PfItem {
  int s, h, hkv, q0, n, L, tile0, rows, pos0, key_tiles, nblocks_seq;
};

// The idx-th work item in schedule order: sequence by sequence; within a sequence its last query
// tile (the one that sees the most keys) first, then the next-to-last, each over all query heads
// (heads sharing a kv head side by side).  The CTAs at work at any time then share one sequence's
// K/V, which stays in L2, and the schedule ends on short items.  False when the item has no queries,
// or when its sequence's chunk is inconsistent (reported once per sequence, by the item of its first
// tile and head, when `report`).
__device__ __forceinline__ bool pf_item(const PrefillParams& p, int idx, PfItem& it, bool report) {
  const int per_seq = p.q_tiles * p.num_q_heads;
  it.s = idx / per_seq;
  const int rem = idx % per_seq;
  const int qt = p.q_tiles - 1 - rem / p.num_q_heads;
  it.h = rem % p.num_q_heads;
  it.q0 = __ldg(p.query_start + it.s);
  it.n = __ldg(p.query_start + it.s + 1) - it.q0;
  it.L = __ldg(p.seq_lens + it.s);
  const int B = p.block_size;
  // a chunk must lie inside q / out, fit the tiles, and be part of its sequence's cached tokens
  if (it.q0 < 0 || it.n < 0 || (long long)it.q0 + it.n > p.num_query_tokens || it.n > p.q_tiles * kTile ||
      it.L < it.n || (long long)it.L > (long long)p.max_blocks * B) {
    if (report && qt == 0 && it.h == 0) report_error(p.err_flag, PA_DEVERR_QUERY);
    return false;
  }
  it.tile0 = qt * kTile;
  if (it.tile0 >= it.n) return false;
  it.hkv = it.h / (p.num_q_heads / p.num_kv_heads);
  it.rows = min(kTile, it.n - it.tile0);               // valid query rows of this tile
  it.pos0 = it.L - it.n + it.tile0;                    // position of query row 0
  it.key_tiles = (it.pos0 + it.rows - 1) / kTile + 1;  // key tiles reaching the last row's position
  it.nblocks_seq = (it.L + B - 1) / B;                 // <= max_blocks (checked above)
  return true;
}

// Persistent: each CTA takes items blockIdx.x, blockIdx.x + gridDim.x, ...  Every role walks the same
// items; the K/V rings, the S buffers and their barriers run on across items (tg counts this CTA's
// key tiles so far), so the next item's Q, K/V copies and first S MMAs overlap this item's last
// P V and epilogue.
template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                      const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_out,
                      const PrefillParams p) {
  const int n_items = p.num_seqs * p.num_q_heads * p.q_tiles;
  const int B = p.block_size;
  const int blocks_per_tile = kTile / B;
  const int slots = 2 * blocks_per_tile;  // tensor-map copies per tile: one per block and half

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // every softmax warp has read item k's publication (phase k; item k + 1 is published only after it, so
  // no softmax warp can find bar_qs two phases on)
  uint64_t* bar_q = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* bar_k = bar_q + 1;      // [2] K stage filled
  uint64_t* bar_v = bar_q + 3;      // [2] V stage filled
  uint64_t* bar_s = bar_q + 5;      // [3] S buffer computed (one phase per tile held)
  uint64_t* bar_p = bar_q + 8;      // [3] P in the S buffer written by all softmax warps
  uint64_t* bar_o = bar_q + 11;     // [3] O += P V of the tile in S buffer b done (one phase per tile held)
  uint64_t* bar_done = bar_q + 14;  // every P V of the item done (one phase per item)
  uint64_t* bar_ofree = bar_q + 15; // the item's epilogue has read O (one phase per item)
  uint64_t* bar_qs = bar_q + 16;    // item k published and its Q tile in shared memory (phase k)
  uint64_t* bar_staged = bar_q + 17; // the item's output tile written to the stage (or stored) (phase per item)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kBarOff + 192);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + 200);
  PfItem* items = reinterpret_cast<PfItem*>(smem + kBarOff + 256);  // [2] published items (s < 0: none left)
  uint8_t* qbuf = smem + kQOff;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int n_s = 0, n_o = 0;  // S / P V commits (control thread)
  int n_pub = 0;         // items published, i.e. phases of bar_qs started (scheduling thread)
  int n_issued = 0;      // tiles whose copies this producer warp has issued

  if (threadIdx.x == 0) {
    mbar_init(bar_q, kSoftmaxWarps);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_k[b], slots);      // each copy slot arrives once per tile (with its bytes, or none)
      mbar_init(&bar_v[b], slots + 2);  // + each V producer's partial-block / zero-fill arrival
    }
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(&bar_s[b], 1);
      mbar_init(&bar_p[b], kSoftmaxWarps);
      mbar_init(&bar_o[b], 1);
    }
    mbar_init(bar_done, 1);
    mbar_init(bar_ofree, kSoftmaxWarps);
    mbar_init(bar_qs, 1);
    mbar_init(bar_staged, kSoftmaxWarps);
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
  // a wait whose outcome every lane of the warp shares (warp-collective instructions follow)
  auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag));
  };

  if (warp >= kLoadWarp0) {
    // =================================================================== producers: one half of K or V tiles
    const bool is_v = warp >= kLoadWarp0 + 2;
    const int half = (warp - kLoadWarp0) & 1;  // columns 64 half .. 64 half + 63
    const T* cache = static_cast<const T*>(is_v ? p.v_cache : p.k_cache);
    const CUtensorMap* tmap = is_v ? &tmap_v : &tmap_k;
    uint8_t* ring = smem + (is_v ? kVOff : kKOff);
    constexpr int kPastEnd = INT_MIN;
    const int blk = lane;  // lane b < blocks_per_tile copies this half of block b of every tile
    if (lane == 0) tma_prefetch_descriptor(tmap);
    bool ok = true;
    int tg = 0;
    for (int idx = blockIdx.x; ok && idx < n_items; idx += gridDim.x) {
      PfItem it;
      if (!pf_item(p, idx, it, false)) continue;
      const int32_t* table = p.block_tables + (size_t)it.s * p.max_blocks;
      // the table entry of this lane's block, read one tile ahead
      auto fetch = [&](int kt) -> int {
        const int bi = kt * blocks_per_tile + blk;
        return (blk < blocks_per_tile && kt < it.key_tiles && bi < it.nblocks_seq) ? __ldg(table + bi) : kPastEnd;
      };
      int entry_next = fetch(0);
      for (int t = 0; t < it.key_tiles; ++t, ++tg) {
        // the stage of tile tg held tile tg - 2: wait until the MMA that read it has finished.  The
        // barrier of its S buffer has one phase per tile held; this producer waits them in order and
        // their next phase (tile tg + 1) needs this producer's copies, so the wait is exact.
        if (tg >= 2 && !warp_wait(is_v ? &bar_o[(tg - 2) % kSBufs] : &bar_s[(tg - 2) % kSBufs],
                                  ((tg - 2) / kSBufs) & 1)) {
          ok = false;
          break;
        }
        const int entry = entry_next;
        entry_next = fetch(t + 1);
        uint64_t* bar = is_v ? &bar_v[tg & 1] : &bar_k[tg & 1];
        uint8_t* st = ring + (tg & 1) * 2 * kHalf + half * kHalf;
        const bool in_pool = entry >= 0 && entry < p.num_blocks;
        if (!is_v && half == 0 && entry != kPastEnd && !in_pool) report_error(p.err_flag, PA_DEVERR_BLOCK_ID);
        // V: only blocks entirely inside the sequence go by tensor-map copy
        const bool whole = in_pool && (!is_v || (t * blocks_per_tile + blk + 1) * B <= it.L);
        if (blk < blocks_per_tile) {
          if (whole) {
            mbar_arrive_expect_tx(bar, (uint32_t)B * 128);
            tma_load_2d(st + blk * B * 128, tmap, half * 64, (entry * p.num_kv_heads + it.hkv) * B, bar);
          } else {
            mbar_arrive(bar);
          }
        }
        if (is_v) {
          // this half of the blocks not copied above: rows inside the sequence of an in-pool block by
          // cp.async, the rest zeros.  Four rows of eight 16-byte chunks per step; the four rows lie in
          // one block (B is a multiple of 16), so every branch below is uniform across the warp.
          const unsigned partial = __ballot_sync(0xffffffffu, blk < blocks_per_tile && !whole);
          if (partial) {
            const int first = (__ffs(partial) - 1) * B;  // rows before the first such block are all copied
            for (int r0 = first; r0 < kTile; r0 += 4) {
              const int b = r0 / B;
              const int e = __shfl_sync(0xffffffffu, entry, b);
              if (!((partial >> b) & 1)) continue;
              const int r = r0 + (lane >> 3), chunk = lane & 7;
              const int pos = t * kTile + r;
              uint8_t* dst = st + swz128(r, chunk);
              if (pos < it.L && e >= 0 && e < p.num_blocks)
                cp_async16(dst, cache + (((size_t)e * p.num_kv_heads + it.hkv) * B + (pos % B)) * kD + half * 64 +
                                    chunk * 8);
              else
                *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
            }
            cp_async_wait_all();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> tensor-core reads
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar);
        }
        ++n_issued;
      }
    }
  } else if (warp == kSWarp) {
    // =================================================================== S = Q K^T issuer
    if (lane == 0) {
      const uint32_t id_s = idesc<T>(0);
      tma_prefetch_descriptor(&tmap_q);
      // This thread also schedules: it publishes item k (the first one with queries at or after index
      // idx) in items[k % 2] and starts the copy of its Q tile into Q buffer k % 2, both completing
      // phase k of bar_qs.  Item k + 1 is published once every softmax warp has read item k (bar_q
      // phase k), which also means the S MMAs of item k - 1, the last readers of that Q buffer, have
      // finished.  It reports inconsistent chunks: every item of this CTA passes through here once.
      auto publish = [&](int idx, int k, PfItem& it) {
        for (; idx < n_items; idx += gridDim.x)
          if (pf_item(p, idx, it, true)) break;
        if (idx >= n_items) it.s = -1;
        items[k & 1] = it;
        ++n_pub;
        if (idx < n_items) {
          uint8_t* qb = qbuf + (k & 1) * 2 * kHalf;
          mbar_arrive_expect_tx(bar_qs, 2 * kHalf);
          tma_load_3d(qb, &tmap_q, 0, it.h, it.q0 + it.tile0, bar_qs);
          tma_load_3d(qb + kHalf, &tmap_q, 64, it.h, it.q0 + it.tile0, bar_qs);
        } else {
          mbar_arrive(bar_qs);
        }
        return idx;
      };
      bool ok = true;
      int tg = 0, item_no = 0;
      PfItem it;
      int idx = publish(blockIdx.x, 0, it);
      while (ok && idx < n_items) {
        // Q of this item in its buffer (this thread publishes the barrier's next phase: exact)
        ok = wait_bar_spin(bar_qs, item_no & 1, abort_flag);
        if (!ok) break;
        PfItem nx;
        int idx_next = n_items;
        bool published = false;
        // publish the next item once every softmax warp has read this one (checked between tiles, and
        // waited for at the end of the item; the barrier's next phase needs that publication: exact)
        auto try_publish = [&](bool block) {
          if (published) return;
          if (block ? wait_bar_spin(bar_q, item_no & 1, abort_flag) : mbar_test_wait(bar_q, item_no & 1)) {
            idx_next = publish(idx + gridDim.x, item_no + 1, nx);
            published = true;
          } else if (block) {
            ok = false;
          }
        };
        const uint32_t qa = smem_u32(qbuf + (item_no & 1) * 2 * kHalf);
        for (int t = 0; ok && t < it.key_tiles; ++t, ++tg) {
          try_publish(false);
          const int buf = tg % kSBufs;
          // buffer tg % 3 held P of tile tg - 3 (its P V must have finished; the barrier's next phase,
          // tile tg, needs this S, so the wait is exact) and K stage tg % 2 must hold key tile tg
          if (tg >= kSBufs) ok = wait_bar_spin(&bar_o[buf], ((tg - kSBufs) / kSBufs) & 1, abort_flag);
          ok = ok && wait_bar_spin(&bar_k[tg & 1], (tg >> 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t kb = smem_u32(smem + kKOff + (tg & 1) * 2 * kHalf);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            mma_ss(tmem + buf * 128, sw128_desc(qa + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024),
                   sw128_desc(kb + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024), id_s, kk > 0);
          mma_commit(&bar_s[buf]);
          ++n_s;
        }
        if (ok) try_publish(true);
        ++item_no;
        idx = idx_next;
        it = nx;
      }
    }
    __syncwarp();
  } else if (warp == kPVWarp) {
    // =================================================================== O += P V issuer
    if (lane == 0) {
      const uint32_t id_o = idesc<T>(1);
      bool ok = true;
      int tg = 0, item_no = 0;
      int prev_row0 = 0, prev_h = 0;  // the previous item's output tile
      bool prev_full = false;
      // The previous item's output, once every softmax warp has staged (or, ragged, written) its rows:
      // two tensor-map stores of a full tile (the barrier's next phase needs this item's bar_done, which
      // this thread arrives on later, so the wait is exact).
      auto store_prev = [&]() {
        if constexpr (!kStagedOut<T>) return;
        ok = wait_bar_spin(bar_staged, (item_no - 1) & 1, abort_flag);
        if (ok && prev_full) {
          tma_store_3d(&tmap_out, 0, prev_h, prev_row0, smem + kOutOff);
          tma_store_3d(&tmap_out, 64, prev_h, prev_row0, smem + kOutOff + kHalf);
          bulk_commit_group();
        }
      };
      for (int idx = blockIdx.x; ok && idx < n_items; idx += gridDim.x) {
        PfItem it;
        if (!pf_item(p, idx, it, false)) continue;
        // the first P V overwrites O: the previous item's epilogue must have read it (the barrier's
        // next phase is this item's epilogue, which needs these MMAs, so the wait is exact)
        if (item_no > 0) ok = wait_bar_spin(bar_ofree, (item_no - 1) & 1, abort_flag);
        for (int kt = 0; ok && kt < it.key_tiles; ++kt, ++tg) {
          const int buf = tg % kSBufs;
          // once every softmax warp has written P of tile tg and V of tile tg is in place
          ok = wait_bar_spin(&bar_p[buf], (tg / kSBufs) & 1, abort_flag) &&
               wait_bar_spin(&bar_v[tg & 1], (tg >> 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t vb = smem_u32(smem + kVOff + (tg & 1) * 2 * kHalf);
          // keys 16kk .. 16kk + 15 of the tile: P hi (lo) in columns 8kk (64 + 8kk) of the buffer
#pragma unroll
          for (int part = 0; part < (split_p<T>() ? 2 : 1); ++part) {
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_ts(tmem + kOCol, tmem + buf * 128 + part * 64 + kk * 8, sw128_desc(vb + kk * 2048, kHalf, 1024),
                     id_o, kt > 0 || part > 0 || kk > 0);
          }
          mma_commit(&bar_o[buf]);
          ++n_o;
          // the previous item's store, a few tiles into this item: clear of the copies that start an item
          if (kt == min(2, it.key_tiles - 1) && item_no > 0) store_prev();
        }
        // the item's last P V has finished: O is complete (the buffer barrier's previous phase finished
        // before the S that fed this P; its next phase needs a P V not yet issued, so the wait is exact)
        if (ok) ok = wait_bar_spin(&bar_o[(tg - 1) % kSBufs], ((tg - 1) / kSBufs) & 1, abort_flag);
        // the stage may take this item's output once the previous item's store has read it
        if constexpr (kStagedOut<T>) bulk_wait_group_read0();
        if (ok) mbar_arrive(bar_done);
        prev_row0 = it.q0 + it.tile0;
        prev_h = it.h;
        prev_full = it.rows == kTile;
        ++item_no;
      }
      if (ok && item_no > 0) store_prev();
      if constexpr (kStagedOut<T>) bulk_wait_group0();  // the output is written before the CTA ends
    }
    __syncwarp();
  } else {
    // =================================================================== softmax warps
    // Warp w owns the 16 query rows (tensor-memory lanes) 32 (w % 4) + 16 (w / 4) .. + 15 of the tile,
    // all 128 key columns: thread t holds rows r0 = base + t / 4 and r1 = r0 + 8, keys 8j + 2 (t % 4)
    // and + 1 (j = 0..15), so a row's maximum and sum take two shuffles among its four threads.
    const int q4 = warp & 3, hh = warp >> 2, c4 = lane & 3;
    const uint32_t half_base = (uint32_t)(q4 * 32 + hh * 16) << 16;  // first lane of this warp's rows
    const int r0 = q4 * 32 + hh * 16 + (lane >> 2), r1 = r0 + 8;
    const float sl2 = p.scale_log2;
    // every warp arrives on bar_q once it has read the published item
    auto take_item = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_q);
    };
    bool ok = true;
    int tg = 0, item_no = 0;
    int lim0 = 0, lim1 = 0;                                    // last key position each row sees
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // reference maxima (log2 units), partial sums
    // key tile kt of the current item (this CTA's tile tg)
    auto tile = [&](int kt) {
      const int buf = tg % kSBufs;
      ok = __all_sync(0xffffffffu, wait_bar_spin(&bar_s[buf], (tg / kSBufs) & 1, abort_flag)) && ok;
      tc_fence_after();
      const uint32_t s_addr = tmem + half_base + buf * 128;
      float v[64];
      tmem_ld16x256_x8(s_addr, v);
      tmem_ld16x256_x8(s_addr + 64, v + 32);
      tmem_wait_ld<64>(v);
      const int key0 = kt * kTile + 2 * c4;          // key of this thread's pair 0
      const int e0 = lim0 - key0, e1 = lim1 - key0;  // pair j's keys 8j, 8j + 1 are visible up to e
      const bool unmasked = __all_sync(0xffffffffu, min(lim0, lim1) >= kt * kTile + kTile - 1);
      // ---- fp16, an unmasked tile after the item's first: P with the current reference maxima, kept
      //      when no weight can exceed 2^threshold (each thread's share of a row's tile sum is at most
      //      kLazyBound).  The exact path below would then move no reference max and compute the same
      //      words and sums, so the result is the same bit for bit; otherwise it runs and stores P again.
      //      (bf16, whose P has two terms, would hold both paths' words and spill.)
      bool lazy = !split_p<T>() && unmasked && kt > 0;
      if (lazy) {
        float n0 = l0, n1 = l1;
#pragma unroll
        for (int j0 = 0; j0 < 16; j0 += 8) {
          uint32_t hi[16], lo[16];
          make_p<T, false>(v, j0, sl2, m0, m1, e0, e1, hi, lo, n0, n1);
          tmem_st16x128_x8(s_addr + 4 * j0, hi);
          if constexpr (split_p<T>()) tmem_st16x128_x8(s_addr + 64 + 4 * j0, lo);
        }
        lazy = !__any_sync(0xffffffffu, n0 - l0 > kLazyBound || n1 - l1 > kLazyBound);
        if (lazy) {
          l0 = n0;
          l1 = n1;
        } else {
          tmem_wait_st();  // the words stored above land before the exact path's stores
        }
      }
      if (!lazy) {
        // ---- the rows' tile maxima, and the reference maxima they imply
        float a0 = -INFINITY, b0 = -INFINITY, a1 = -INFINITY, b1 = -INFINITY;  // two chains per row
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          a0 = max3(a0, v[4 * j], v[4 * j + 1]);
          a1 = max3(a1, v[4 * j + 2], v[4 * j + 3]);
          b0 = max3(b0, v[4 * j + 4], v[4 * j + 5]);
          b1 = max3(b1, v[4 * j + 6], v[4 * j + 7]);
        }
        if (!unmasked) {
          // The maxima over all 128 keys bound the visible keys' maxima from above.  A bound that moves
          // no row's reference max decides as the visible maxima would, so those are taken only when
          // the bound would move one (rare after an item's first tiles).
          float u0 = fmaxf(a0, b0), u1 = fmaxf(a1, b1);
          u0 = fmaxf(u0, __shfl_xor_sync(0xffffffffu, u0, 1));
          u1 = fmaxf(u1, __shfl_xor_sync(0xffffffffu, u1, 1));
          u0 = fmaxf(u0, __shfl_xor_sync(0xffffffffu, u0, 2));
          u1 = fmaxf(u1, __shfl_xor_sync(0xffffffffu, u1, 2));
          if (__any_sync(0xffffffffu, u0 * sl2 > m0 + kRescaleThreshold || u1 * sl2 > m1 + kRescaleThreshold)) {
            a0 = b0 = a1 = b1 = -INFINITY;
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
              a0 = max3(a0, 8 * j <= e0 ? v[4 * j] : -INFINITY, 8 * j + 1 <= e0 ? v[4 * j + 1] : -INFINITY);
              a1 = max3(a1, 8 * j <= e1 ? v[4 * j + 2] : -INFINITY, 8 * j + 1 <= e1 ? v[4 * j + 3] : -INFINITY);
              b0 = max3(b0, 8 * j + 8 <= e0 ? v[4 * j + 4] : -INFINITY, 8 * j + 9 <= e0 ? v[4 * j + 5] : -INFINITY);
              b1 = max3(b1, 8 * j + 8 <= e1 ? v[4 * j + 6] : -INFINITY, 8 * j + 9 <= e1 ? v[4 * j + 7] : -INFINITY);
            }
          }
        }
        a0 = fmaxf(a0, b0);
        a1 = fmaxf(a1, b1);
        a0 = fmaxf(a0, __shfl_xor_sync(0xffffffffu, a0, 1));
        a1 = fmaxf(a1, __shfl_xor_sync(0xffffffffu, a1, 1));
        a0 = fmaxf(a0, __shfl_xor_sync(0xffffffffu, a0, 2));
        a1 = fmaxf(a1, __shfl_xor_sync(0xffffffffu, a1, 2));
        const float mx0 = a0 * sl2, mx1 = a1 * sl2;  // scale > 0
        const bool upd0 = mx0 > m0 + kRescaleThreshold, upd1 = mx1 > m1 + kRescaleThreshold;
        const float al0 = upd0 ? fast_exp2(m0 - mx0) : 1.f, al1 = upd1 ? fast_exp2(m1 - mx1) : 1.f;
        if (__any_sync(0xffffffffu, upd0 || upd1) && kt > 0 && ok) {
          // O of these rows is rescaled between P V of tile tg - 1 and that of tile tg.  The barrier
          // of its S buffer finished tile tg - 4 before S(tg - 1) was issued and its next phase (tile
          // tg + 2) needs this warp's P, so the parity wait below is exact.
          ok = warp_wait(&bar_o[(tg - 1) % kSBufs], ((tg - 1) / kSBufs) & 1);
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            float o[32];
            tmem_ld16x256_x8(tmem + half_base + kOCol + 64 * c, o);
            tmem_wait_ld<32>(o);
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              o[i] *= al0, o[i + 1] *= al0;
              o[i + 2] *= al1, o[i + 3] *= al1;
            }
            tmem_st16x256_x8(tmem + half_base + kOCol + 64 * c, reinterpret_cast<const uint32_t*>(o));
          }
          tmem_wait_st();
        }
        if (upd0) m0 = mx0;
        if (upd1) m1 = mx1;
        // ---- P into the buffer, 8 pairs (32 columns of packed words) at a time: hi words in columns
        //      0..63, lo words in 64..127
        l0 *= al0;
        l1 *= al1;
#pragma unroll
        for (int j0 = 0; j0 < 16; j0 += 8) {
          uint32_t hi[16], lo[16];
          if (unmasked)
            make_p<T, false>(v, j0, sl2, m0, m1, e0, e1, hi, lo, l0, l1);
          else
            make_p<T, true>(v, j0, sl2, m0, m1, e0, e1, hi, lo, l0, l1);
          tmem_st16x128_x8(s_addr + 4 * j0, hi);
          if constexpr (split_p<T>()) tmem_st16x128_x8(s_addr + 64 + 4 * j0, lo);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p[buf]);
      ++tg;
    };
    auto start_item = [&](const PfItem& x) {
      take_item();
      lim0 = min(x.pos0 + r0, x.L - 1);
      lim1 = min(x.pos0 + r1, x.L - 1);
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
      tile(0);
    };
    // the first item and its first tile
    ok = warp_wait(bar_qs, 0);
    PfItem it = items[0];
    if (ok && it.s >= 0) start_item(it);
    // After a failure (a wait gave up) every warp leaves at the next wait: no warp waits for another
    // softmax warp, and the other roles stop at their next wait too.
    while (ok && it.s >= 0) {
      for (int kt = 1; kt < it.key_tiles; ++kt) tile(kt);
      if (!ok) break;
      // ---- row sums of this item over each row's four threads
      float s0 = l0, s1 = l1;
      s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
      s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
      // ---- the next item and its first tile.  That tile writes no O (no rescale on a first tile) and its
      //      P V waits for this item's epilogue to have read O, so it runs before the epilogue, beside
      //      this item's last P V.
      // (what the epilogue needs of this item is kept apart, and the next item becomes the current one)
      const int orow0 = it.q0 + it.tile0, oh = it.h;  // the tile's first output row, and its head
      T* out0 = reinterpret_cast<T*>(p.out) + ((size_t)(orow0 + r0) * p.num_q_heads + oh) * kD;  // row r0
      const int rows = it.rows;
      ok = warp_wait(bar_qs, (item_no + 1) & 1);
      it = items[(item_no + 1) & 1];
      if (ok && it.s >= 0) start_item(it);
      // ---- epilogue: out = O / l for this warp's 16 rows, from the 16x256b layout (thread: rows r0, r1,
      //      columns 8j + 2 (t % 4) and + 1)
      if (ok) ok = warp_wait(bar_done, item_no & 1);
      if (!ok) break;
      tc_fence_after();
      float o[64];
      tmem_ld16x256_x8(tmem + half_base + kOCol, o);
      tmem_ld16x256_x8(tmem + half_base + kOCol + 64, o + 32);
      tmem_wait_ld<64>(o);
      // O may take the next item's first P V
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ofree);
      const float inv0 = s0 > 0.f ? 1.f / s0 : 0.f, inv1 = s1 > 0.f ? 1.f / s1 : 0.f;
      if constexpr (kStagedOut<T>) {
        // The tile goes to the stage, in the 128-byte-swizzled layout of the output's tensor map (row r's
        // 16-byte chunk k of column half h at h * kHalf + swz128(r, k)).  Thread c of a quad writes bytes
        // 4c .. 4c + 3 of each chunk, so the eight rows and four threads of a store fall in 32 banks.
        uint8_t* stage = smem + kOutOff;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          uint8_t* col = stage + (j >> 3) * kHalf + 4 * c4;
          *reinterpret_cast<uint32_t*>(col + swz128(r0, j & 7)) =
              Mma<T>::pack(o[4 * j] * inv0, o[4 * j + 1] * inv0);
          *reinterpret_cast<uint32_t*>(col + swz128(r1, j & 7)) =
              Mma<T>::pack(o[4 * j + 2] * inv1, o[4 * j + 3] * inv1);
        }
        if (rows == kTile) {
          // a full tile: the P V issuer stores it once every softmax warp has written its rows
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> the tensor-map store
        } else {
          // a ragged tile (the last of a chunk): its rows past the chunk belong to another sequence, so this
          // warp copies its own rows inside the chunk out, 16 lanes per 256-byte row
          __syncwarp();
          const int row_base = r0 - (lane >> 2);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rl = 2 * i + (lane >> 4), chunk = lane & 15;  // row row_base + rl, bytes 16 chunk ..
            const int r = row_base + rl;
            if (r < rows) {
              const uint4 v = *reinterpret_cast<const uint4*>(stage + (chunk >> 3) * kHalf + swz128(r, chunk & 7));
              T* dst = reinterpret_cast<T*>(p.out) + ((size_t)(orow0 + r) * p.num_q_heads + oh) * kD + 8 * chunk;
              *reinterpret_cast<uint4*>(dst) = v;
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_staged);
      } else {
        // Thread c of a quad holds packed word j of a row for columns 8j + 2c, 8j + 2c + 1.  A 4 x 4 word
        // transpose within the quad (two xor-shuffle steps per group of 4 j) gives thread c the 16 bytes
        // of columns 8j .. 8j + 7 for j = 4g + c, so a store writes 16 bytes per thread and 64
        // contiguous bytes per row and quad.
        T* out1 = out0 + (size_t)8 * p.num_q_heads * kD;  // row r1 = r0 + 8
        const bool hi2 = (c4 >> 1) != 0, odd = (c4 & 1) != 0;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const float inv = rr ? inv1 : inv0;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
              w[i] = Mma<T>::pack(o[4 * (4 * g + i) + 2 * rr] * inv, o[4 * (4 * g + i) + 2 * rr + 1] * inv);
            // step 1 (lanes c, c ^ 2): the upper pair of words of threads 0, 1 swaps with the lower pair of 2, 3
            const uint32_t x0 = __shfl_xor_sync(0xffffffffu, hi2 ? w[0] : w[2], 2);
            const uint32_t x1 = __shfl_xor_sync(0xffffffffu, hi2 ? w[1] : w[3], 2);
            if (hi2) w[0] = x0, w[1] = x1;
            else w[2] = x0, w[3] = x1;
            // step 2 (lanes c, c ^ 1): within each pair of words, an odd word of an even thread swaps with an
            // even word of an odd thread
            const uint32_t y0 = __shfl_xor_sync(0xffffffffu, odd ? w[0] : w[1], 1);
            const uint32_t y1 = __shfl_xor_sync(0xffffffffu, odd ? w[2] : w[3], 1);
            if (odd) w[0] = y0, w[2] = y1;
            else w[1] = y0, w[3] = y1;
            if ((rr ? r1 : r0) < rows)
              *reinterpret_cast<uint4*>((rr ? out1 : out0) + 8 * (4 * g + c4)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      ++item_no;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // a wait expired (the flag is stable: every thread has left its loop): record it, and let the
    // copies and MMAs this CTA started finish, each wait bounded, before its memory is released
    if (threadIdx.x == 0) report_error(p.err_flag, PA_DEVERR_TIMEOUT);
    if (warp >= kLoadWarp0 && lane == 0) {  // copies still landing
      uint64_t* ring_bar = warp >= kLoadWarp0 + 2 ? bar_v : bar_k;
      for (int t = max(0, n_issued - 2); t < n_issued; ++t) drain_wait(&ring_bar[t & 1], (t >> 1) & 1);
    }
    if (warp == kSWarp && lane == 0) {
      for (int t = max(0, n_s - kSBufs); t < n_s; ++t) drain_wait(&bar_s[t % kSBufs], (t / kSBufs) & 1);
      // the Q copy of the last item published (at most one phase of bar_qs is outstanding: an item is
      // published only after the previous one's Q has been waited for; a completed phase returns at once)
      if (n_pub > 0) drain_wait(bar_qs, (n_pub - 1) & 1);
    }
    if (warp == kPVWarp && lane == 0)
      for (int t = max(0, n_o - kSBufs); t < n_o; ++t) drain_wait(&bar_o[t % kSBufs], (t / kSBufs) & 1);
    __syncthreads();
  }
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512u) : "memory");
}

// one CTA per SM (the kernel holds all of tensor memory and most of shared memory), at most one per item
cudaError_t launch_prefill_tc(int dtype, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                              const CUtensorMap& to, const PrefillParams& p, cudaStream_t stream) {
  const long long items = (long long)p.num_seqs * p.num_q_heads * p.q_tiles;
  if (items == 0) return cudaSuccess;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(items < sms ? items : sms);
  if (dtype == PA_F16) {
    e = cudaFuncSetAttribute(prefill_tc_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    prefill_tc_kernel<__half><<<grid, kThreads, kSmemBytes, stream>>>(tk, tv, tq, to, p);
  } else if (dtype == PA_BF16) {
    e = cudaFuncSetAttribute(prefill_tc_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    prefill_tc_kernel<__nv_bfloat16><<<grid, kThreads, kSmemBytes, stream>>>(tk, tv, tq, to, p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace pa

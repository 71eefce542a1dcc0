/*
 * pa_oracle.c - plain CPU fp64 oracle for paged decode attention and its two
 * companion write operations (slot-mapping append, whole-block copy).
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
 * CPU-baseline leg are the only callers.  The CUDA library never calls this
 * code, and the two share no source, header, table or helper.
 *
 * Every step is the plain definition, written out with no blocking, fusion or
 * reordering: gather each token's key/value through the block table, score it
 * against the query, take an exact max-subtracted softmax in two passes, and
 * sum the values with the softmax weights.  All arithmetic is in double.
 *
 * Sources (page title, then section):
 *  [P1] "PagedAttention 详解：缓存的存储结构" (kefan.life)
 *       - "Block Table": block_idx indexes the table, the entry is the block ID,
 *         token_idx = block_idx * B + offset; the 35-token example [7, 3, 12].
 *       - "软件地址翻译" (software address translation): block_idx = i / B,
 *         offset = i % B, block = block_tables[seq][block_idx]; the prior-art
 *         key layout [blocks, kv_heads, head_size/x, B, x] and value layout
 *         [blocks, kv_heads, head_size, B]; the strides.
 *       - "一个具体的例子" (worked example): element offset 206880.
 *       - "写入新 K/V" (writing new K/V): slot = block * B + offset and back.
 *  [P2] "PagedAttention 笔记" (imreese.github.io)
 *       - "写时复制是正确性的边界" (copy-on-write): copy the shared block to a
 *         fresh one, remap, then write.
 *  [P3] "vLLM 核心工程深度剖析" (ybb.press)
 *       - "3.1 Kernel 签名与分块策略": out/q [num_seqs, num_heads, head_size],
 *         block_tables [num_seqs, max_blocks], context lengths, scale;
 *         max-subtracted softmax, then the value-weighted sum.
 *  [P4] "PagedAttention是什麼？" (yololab.net)
 *       - "常見問題" (FAQ): paging changes only where K/V are stored, never
 *         the attention result.
 *
 * Optional ALiBi: the kernel signature of [P3 "3.1"] carries per-head
 * `alibi_slopes` without defining their use.  The reading taken is the
 * standard linear bias of the query (at position L-1) towards key i:
 * s_i += slope_h * (i - (L - 1)), i.e. zero for the newest token and
 * increasingly negative for older ones (positive slopes).
 *
 * Layout codes: PAO_LAYOUT_OURS is [blocks][kv_heads][B][head_size], dense.
 * PAO_LAYOUT_PRIOR is the [P1] prior-art pair above, kept to pin the address
 * arithmetic against the page's worked example.  PAO_LAYOUT_FP8 pairs our key
 * layout with the [P1] value layout [blocks][kv_heads][head_size][B] tiled in
 * 16-token groups: [blocks][kv_heads][B/16][head_size][16] (the same thing for
 * B = 16), so that every 16 tokens of one head's values are contiguous.
 *
 * FP8 KV cache: [P1 "软件地址翻译"] allows cache_t to be FP8 (x = 16 /
 * sizeof(cache_t) = 16 elements per 16-byte access) and says nothing more.
 * Reading taken: OCP E4M3 codes (1 sign, 4 exponent bits with bias 7, 3
 * mantissa bits; S.1111.111 is NaN, no infinities), one fp32 scale for all of
 * K and one for all of V; a stored code c stands for scale * e4m3(c), and a
 * value x is written as the code nearest to x / scale (fp32 division, ties to
 * the even code, overflow saturating to +-448).  Queries and outputs stay fp16.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { PAO_F32 = 0, PAO_F16 = 1, PAO_BF16 = 2, PAO_FP8_E4M3 = 3 };
enum { PAO_LAYOUT_OURS = 0, PAO_LAYOUT_PRIOR = 1, PAO_LAYOUT_FP8 = 2 };
enum {
  PAO_OK = 0,
  PAO_BAD_ARG = -1,
  PAO_BAD_BLOCK = -2,
  PAO_BAD_SLOT = -3,
  PAO_NO_MEMORY = -4
};

/* ---------- element access: exact conversion of stored bits to double ---------- */

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double pao_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  } else if (e == 31) {
    v = (m == 0) ? INFINITY : NAN;
  } else {
    v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
double pao_bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0
 * holds the subnormals m * 2^-9; S.1111.111 is NaN; there is no infinity. */
double pao_e4m3_to_f64(uint8_t c) {
  int sign = (c >> 7) & 1;
  int e = (c >> 3) & 0xf;
  int m = c & 7;
  double v;
  if (e == 15 && m == 7) {
    v = NAN;
  } else if (e == 0) {
    v = ldexp((double)m, -9);
  } else {
    v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
  }
  return sign ? -v : v;
}

/* The E4M3 code nearest to r, ties to the even code; a magnitude that rounds
 * above the largest finite value 448 (infinity included) saturates to it; NaN
 * gives S.1111.111.
 * The grid spacing is 2^-9 below 2^-6 (subnormals) and 2^(e-3) in the binade
 * [2^e, 2^(e+1)); a / spacing is exact in double, and nearbyint rounds half to
 * even in the default rounding mode. */
uint8_t pao_f32_to_e4m3_sat(float r) {
  if (isnan(r)) return 0x7F;
  const uint8_t sign = signbit(r) ? 0x80 : 0;
  const double a = fabs((double)r);
  if (isinf(a)) return sign | 0x7E; /* an infinite input saturates like any other overflow */
  int e = a > 0.0 ? ilogb(a) : -6;
  if (e < -6) e = -6;
  const double v = nearbyint(a / ldexp(1.0, e - 3)) * ldexp(1.0, e - 3);
  if (v > 448.0) return sign | 0x7E;
  if (v == 0.0) return sign;
  const int ev = ilogb(v);
  if (ev < -6) return sign | (uint8_t)(v * 512.0); /* subnormal: m = v / 2^-9 */
  const int m = (int)(v / ldexp(1.0, ev - 3)) - 8;
  return sign | (uint8_t)((ev + 7) << 3) | (uint8_t)m;
}

/* pao_f32_to_e4m3_sat over an array (OpenMP): the codes of a whole pool. */
void pao_f32_to_e4m3_array(const float* r, uint8_t* codes, int64_t n) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
  for (int64_t i = 0; i < n; ++i) codes[i] = pao_f32_to_e4m3_sat(r[i]);
}

static size_t elem_size(int dtype) { return dtype == PAO_F32 ? 4 : dtype == PAO_FP8_E4M3 ? 1 : 2; }

double pao_load(const void* base, int64_t i, int dtype) {
  if (dtype == PAO_F32) return (double)((const float*)base)[i];
  if (dtype == PAO_FP8_E4M3) return pao_e4m3_to_f64(((const uint8_t*)base)[i]);
  uint16_t bits = ((const uint16_t*)base)[i];
  return dtype == PAO_F16 ? pao_f16_to_f64(bits) : pao_bf16_to_f64(bits);
}

/* ---------- address translation ---------- */

/* [P1 "软件地址翻译"]: block_idx = i / B, offset = i % B,
 * physical block = block_tables[seq][block_idx]. */
void pao_locate(const int32_t* table_row, int B, int64_t i, int32_t* block, int32_t* offset) {
  int64_t block_idx = i / B;
  *offset = (int32_t)(i % B);
  *block = table_row[block_idx];
}

/* Our layout [blocks][kv_heads][B][D]: element index of (block, head, slot, d). */
int64_t pao_offset_ours(int64_t block, int64_t head, int64_t slot, int64_t d, int Hkv, int B, int D) {
  return ((block * Hkv + head) * B + slot) * D + d;
}

/* [P1 "软件地址翻译"] prior-art key layout [blocks, Hkv, D/x, B, x] with
 * kv_block_stride = Hkv*D*B and kv_head_stride = D*B.  The page prints the
 * inner term garbled; the reading used is (d/x)*B*x + slot*x + d%x, the only
 * one consistent with that shape. */
int64_t pao_key_offset_prior(int64_t block, int64_t head, int64_t slot, int64_t d, int Hkv, int B, int D, int x) {
  int64_t kv_block_stride = (int64_t)Hkv * D * B;
  int64_t kv_head_stride = (int64_t)D * B;
  return block * kv_block_stride + head * kv_head_stride + (d / x) * B * x + slot * x + d % x;
}

/* [P1 "软件地址翻译"] prior-art value layout [blocks, Hkv, D, B]:
 * v_ptr + head_dim_idx * B + slot. */
int64_t pao_value_offset_prior(int64_t block, int64_t head, int64_t slot, int64_t d, int Hkv, int B, int D) {
  int64_t kv_block_stride = (int64_t)Hkv * D * B;
  int64_t kv_head_stride = (int64_t)D * B;
  return block * kv_block_stride + head * kv_head_stride + d * B + slot;
}

/* FP8 value layout: [P1] value layout tiled in 16-token groups,
 * [blocks][Hkv][B/16][D][16]; B is a multiple of 16. */
int64_t pao_value_offset_fp8(int64_t block, int64_t head, int64_t slot, int64_t d, int Hkv, int B, int D) {
  int64_t kv_block_stride = (int64_t)Hkv * D * B;
  int64_t kv_head_stride = (int64_t)D * B;
  return block * kv_block_stride + head * kv_head_stride + (slot / 16) * D * 16 + d * 16 + slot % 16;
}

static int64_t key_index(int layout, int64_t block, int64_t head, int64_t slot, int64_t d, int Hkv, int B, int D,
                         int dtype) {
  if (layout == PAO_LAYOUT_PRIOR) return pao_key_offset_prior(block, head, slot, d, Hkv, B, D, (int)(16 / elem_size(dtype)));
  return pao_offset_ours(block, head, slot, d, Hkv, B, D);
}

static int64_t value_index(int layout, int64_t block, int64_t head, int64_t slot, int64_t d, int Hkv, int B, int D) {
  if (layout == PAO_LAYOUT_PRIOR) return pao_value_offset_prior(block, head, slot, d, Hkv, B, D);
  if (layout == PAO_LAYOUT_FP8) return pao_value_offset_fp8(block, head, slot, d, Hkv, B, D);
  return pao_offset_ours(block, head, slot, d, Hkv, B, D);
}

/* ---------- attention ---------- */

typedef struct {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  int dtype, layout;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  int N, Hq, Hkv, D, B, M, num_blocks;
  double scale;
  const double* alibi; /* nullable: one slope per query head */
  int q_dtype;         /* element type of q (the cache's, except fp16 queries with an FP8 cache) */
  double k_scale, v_scale; /* a stored key (value) element stands for k_scale (v_scale) times its decoded value */
} pao_problem;

/* Scores s_i = scale * <q, k_i> for tokens [t0, t1) of one (seq, query head),
 * gathering k_i through the block table.  Also returns each token's location. */
static int gather_scores(const pao_problem* p, int s, int h, int64_t t0, int64_t t1, double* scores,
                         int32_t* blocks, int32_t* slots) {
  int G = p->Hq / p->Hkv;
  int hkv = h / G; /* consecutive query heads share one KV head */
  const int32_t* row = p->block_tables + (int64_t)s * p->M;
  for (int64_t i = t0; i < t1; ++i) {
    int32_t blk, off;
    pao_locate(row, p->B, i, &blk, &off);
    if (blk < 0 || blk >= p->num_blocks) return PAO_BAD_BLOCK;
    double dot = 0.0;
    for (int d = 0; d < p->D; ++d) {
      double qd = pao_load(p->q, ((int64_t)s * p->Hq + h) * p->D + d, p->q_dtype);
      double kd = p->k_scale *
                  pao_load(p->k_cache, key_index(p->layout, blk, hkv, off, d, p->Hkv, p->B, p->D, p->dtype), p->dtype);
      dot += qd * kd;
    }
    scores[i - t0] = p->scale * dot;
    if (p->alibi) scores[i - t0] += p->alibi[h] * (double)(i - (p->seq_lens[s] - 1));
    blocks[i - t0] = blk;
    slots[i - t0] = off;
  }
  return PAO_OK;
}

static double value_at(const pao_problem* p, int32_t blk, int hkv, int32_t off, int d) {
  return p->v_scale * pao_load(p->v_cache, value_index(p->layout, blk, hkv, off, d, p->Hkv, p->B, p->D), p->dtype);
}

/* One (seq, query head): out = softmax(scale * q K^T) V over the seq_len tokens.
 * A zero-length sequence gives a zero output. */
static int attend_one(const pao_problem* p, int s, int h, double* out) {
  int64_t L = p->seq_lens[s];
  int hkv = h / (p->Hq / p->Hkv);
  for (int d = 0; d < p->D; ++d) out[d] = 0.0;
  if (L <= 0) return PAO_OK;
  double* scores = (double*)malloc(sizeof(double) * L);
  int32_t* blocks = (int32_t*)malloc(sizeof(int32_t) * L);
  int32_t* slots = (int32_t*)malloc(sizeof(int32_t) * L);
  if (!scores || !blocks || !slots) {
    free(scores); free(blocks); free(slots);
    return PAO_NO_MEMORY;
  }
  int rc = gather_scores(p, s, h, 0, L, scores, blocks, slots);
  if (rc == PAO_OK) {
    /* pass 1: max; pass 2: normaliser */
    double mx = -INFINITY;
    for (int64_t i = 0; i < L; ++i) mx = scores[i] > mx ? scores[i] : mx;
    double den = 0.0;
    for (int64_t i = 0; i < L; ++i) den += exp(scores[i] - mx);
    for (int64_t i = 0; i < L; ++i) {
      double w = exp(scores[i] - mx) / den;
      for (int d = 0; d < p->D; ++d) out[d] += w * value_at(p, blocks[i], hkv, slots[i], d);
    }
  }
  free(scores); free(blocks); free(slots);
  return rc;
}

/* Partitioned form: each partition of `P` tokens keeps its own max m_p, sum
 * l_p = sum exp(s_i - m_p) and unnormalised o_p = sum exp(s_i - m_p) v_i; the
 * partitions are then merged with weights exp(m_p - max_p m_p).  Mathematically
 * equal to attend_one; used to pin the merge step of the long-context path. */
static int attend_one_split(const pao_problem* p, int s, int h, int64_t P, double* out) {
  int64_t L = p->seq_lens[s];
  int hkv = h / (p->Hq / p->Hkv);
  for (int d = 0; d < p->D; ++d) out[d] = 0.0;
  if (L <= 0) return PAO_OK;
  int64_t nparts = (L + P - 1) / P;
  double* m = (double*)malloc(sizeof(double) * nparts);
  double* l = (double*)malloc(sizeof(double) * nparts);
  double* o = (double*)calloc((size_t)(nparts * p->D), sizeof(double));
  double* scores = (double*)malloc(sizeof(double) * P);
  int32_t* blocks = (int32_t*)malloc(sizeof(int32_t) * P);
  int32_t* slots = (int32_t*)malloc(sizeof(int32_t) * P);
  int rc = PAO_OK;
  if (!m || !l || !o || !scores || !blocks || !slots) rc = PAO_NO_MEMORY;
  for (int64_t part = 0; rc == PAO_OK && part < nparts; ++part) {
    int64_t t0 = part * P, t1 = (part + 1) * P < L ? (part + 1) * P : L;
    rc = gather_scores(p, s, h, t0, t1, scores, blocks, slots);
    if (rc != PAO_OK) break;
    double mx = -INFINITY;
    for (int64_t i = 0; i < t1 - t0; ++i) mx = scores[i] > mx ? scores[i] : mx;
    double sum = 0.0;
    for (int64_t i = 0; i < t1 - t0; ++i) {
      double e = exp(scores[i] - mx);
      sum += e;
      for (int d = 0; d < p->D; ++d) o[part * p->D + d] += e * value_at(p, blocks[i], hkv, slots[i], d);
    }
    m[part] = mx;
    l[part] = sum;
  }
  if (rc == PAO_OK) {
    double mstar = -INFINITY;
    for (int64_t part = 0; part < nparts; ++part) mstar = m[part] > mstar ? m[part] : mstar;
    double den = 0.0;
    for (int64_t part = 0; part < nparts; ++part) den += exp(m[part] - mstar) * l[part];
    for (int64_t part = 0; part < nparts; ++part) {
      double w = exp(m[part] - mstar);
      for (int d = 0; d < p->D; ++d) out[d] += w * o[part * p->D + d];
    }
    for (int d = 0; d < p->D; ++d) out[d] /= den;
  }
  free(m); free(l); free(o); free(scores); free(blocks); free(slots);
  return rc;
}

static int check_problem(const pao_problem* p) {
  if (!p->q || !p->k_cache || !p->v_cache || !p->block_tables || !p->seq_lens) return PAO_BAD_ARG;
  if (p->N < 0 || p->Hq <= 0 || p->Hkv <= 0 || p->D <= 0 || p->B <= 0 || p->M < 0 || p->num_blocks < 0) return PAO_BAD_ARG;
  if (p->Hq % p->Hkv != 0) return PAO_BAD_ARG;
  if (p->dtype < PAO_F32 || p->dtype > PAO_FP8_E4M3) return PAO_BAD_ARG;
  if ((p->dtype == PAO_FP8_E4M3) != (p->layout == PAO_LAYOUT_FP8)) return PAO_BAD_ARG;
  if (p->layout == PAO_LAYOUT_FP8 && p->B % 16 != 0) return PAO_BAD_ARG;
  if (p->layout == PAO_LAYOUT_PRIOR && p->D % (int)(16 / elem_size(p->dtype)) != 0) return PAO_BAD_ARG;
  for (int s = 0; s < p->N; ++s) {
    if (p->seq_lens[s] < 0) return PAO_BAD_ARG;
    if ((int64_t)p->seq_lens[s] > (int64_t)p->M * p->B) return PAO_BAD_ARG;
  }
  return PAO_OK;
}

/* partition_size <= 0: unsplit definition; > 0: partitioned form + merge. */
int pao_attention(double* out, const void* q, const void* k_cache, const void* v_cache, int dtype, int layout,
                  const int32_t* block_tables, const int32_t* seq_lens, int N, int Hq, int Hkv, int D, int B, int M,
                  int num_blocks, double scale, int partition_size, int threads, const double* alibi_slopes) {
  pao_problem p = {q, k_cache, v_cache, dtype, layout, block_tables, seq_lens, N,
                   Hq, Hkv, D, B, M, num_blocks, scale, alibi_slopes, dtype, 1.0, 1.0};
  int rc = check_problem(&p);
  if (rc != PAO_OK || !out) return rc != PAO_OK ? rc : PAO_BAD_ARG;
  int64_t total = (int64_t)N * Hq;
  int err = PAO_OK;
#ifdef _OPENMP
  if (threads <= 0) threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads)
#endif
  for (int64_t sh = 0; sh < total; ++sh) {
    int s = (int)(sh / Hq), h = (int)(sh % Hq);
    int r = partition_size > 0 ? attend_one_split(&p, s, h, partition_size, out + sh * D)
                               : attend_one(&p, s, h, out + sh * D);
    if (r != PAO_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
      err = r;
    }
  }
  (void)threads;
  return err;
}

/* FP8 (E4M3) cache: keys [blocks][kv_heads][B][D] and values [blocks][kv_heads][B/16][D][16]
 * of E4M3 codes, fp16 queries; the definition above with k = k_scale * e4m3(code),
 * v = v_scale * e4m3(code). */
int pao_attention_fp8(double* out, const void* q_f16, const uint8_t* k_cache, const uint8_t* v_cache,
                      const int32_t* block_tables, const int32_t* seq_lens, int N, int Hq, int Hkv, int D, int B,
                      int M, int num_blocks, double scale, double k_scale, double v_scale, int partition_size,
                      int threads, const double* alibi_slopes) {
  if (!(k_scale > 0.0) || !(v_scale > 0.0)) return PAO_BAD_ARG;
  pao_problem p = {q_f16, k_cache, v_cache, PAO_FP8_E4M3, PAO_LAYOUT_FP8, block_tables, seq_lens, N,
                   Hq, Hkv, D, B, M, num_blocks, scale, alibi_slopes, PAO_F16, k_scale, v_scale};
  int rc = check_problem(&p);
  if (rc != PAO_OK || !out) return rc != PAO_OK ? rc : PAO_BAD_ARG;
  int64_t total = (int64_t)N * Hq;
  int err = PAO_OK;
#ifdef _OPENMP
  if (threads <= 0) threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads)
#endif
  for (int64_t sh = 0; sh < total; ++sh) {
    int s = (int)(sh / Hq), h = (int)(sh % Hq);
    int r = partition_size > 0 ? attend_one_split(&p, s, h, partition_size, out + sh * D)
                               : attend_one(&p, s, h, out + sh * D);
    if (r != PAO_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
      err = r;
    }
  }
  (void)threads;
  return err;
}

/* ---------- prefill (chunked) attention ---------- */

/* The prefill step reads the same paged cache as decode ("PagedAttention 详解：
 * 缓存的存储结构", section "使用流程": prompt blocks that hit the prefix cache
 * "directly take part in the attention computation" and only the missed
 * blocks' K/V are computed and written through slot_mapping; "vLLM 核心工程深度
 * 剖析", section "6.1": long prompts are prefilled in chunks).  Sequence s holds
 * seq_lens[s] tokens in the cache, the last n_s = query_start[s+1] -
 * query_start[s] of which are this chunk's queries.  Query j of the chunk sits
 * at position p = seq_lens[s] - n_s + j and attends causally to the cached
 * tokens 0..p:  out = softmax_i(scale * q . k_i) v_i, i in [0, p].
 * q and out are packed [total_query_tokens][Hq][D]. */
int pao_prefill_attention(double* out, const void* q, const void* k_cache, const void* v_cache, int dtype,
                          const int32_t* block_tables, const int32_t* seq_lens, const int32_t* query_start, int N,
                          int Hq, int Hkv, int D, int B, int M, int num_blocks, double scale, int threads) {
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !query_start) return PAO_BAD_ARG;
  if (N < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || B <= 0 || M < 0) return PAO_BAD_ARG;
  for (int s = 0; s < N; ++s) {
    int32_t n = query_start[s + 1] - query_start[s];
    if (n < 0 || n > seq_lens[s] || (int64_t)seq_lens[s] > (int64_t)M * B) return PAO_BAD_ARG;
  }
  const int64_t total_q = query_start[N];
  int err = PAO_OK;
#ifdef _OPENMP
  if (threads <= 0) threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads)
#endif
  for (int64_t th = 0; th < total_q * Hq; ++th) {
    const int64_t t = th / Hq;
    const int h = (int)(th % Hq);
    int s = 0;
    while (query_start[s + 1] <= t) ++s; /* the sequence that owns query token t */
    const int64_t n = query_start[s + 1] - query_start[s];
    const int64_t pos = seq_lens[s] - n + (t - query_start[s]);
    /* a one-sequence problem over the cache prefix [0, pos]: the decode definition with L = pos + 1 */
    const int32_t len = (int32_t)(pos + 1);
    pao_problem p = {(const char*)q + (size_t)t * Hq * D * elem_size(dtype) - (size_t)0,
                     k_cache, v_cache, dtype, PAO_LAYOUT_OURS, block_tables + (int64_t)s * M, &len,
                     1, Hq, Hkv, D, B, M, num_blocks, scale, NULL, dtype, 1.0, 1.0};
    double* o = out + (size_t)th * D;
    int r = attend_one(&p, 0, h, o);
    if (r != PAO_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
      err = r;
    }
  }
  (void)threads;
  return err;
}

/* ---------- write operations ---------- */

/* [P1 "写入新 K/V"]: block = slot / B, offset = slot % B; token t's key and
 * value rows [Hkv][D] are stored at (block, head, offset).  A negative slot
 * marks a padding token and is skipped. */
int pao_reshape_and_cache(void* k_cache, void* v_cache, const void* key, const void* value,
                          const int64_t* slot_mapping, int T, int dtype, int Hkv, int D, int B, int num_blocks) {
  if (!k_cache || !v_cache || !key || !value || !slot_mapping || T < 0) return PAO_BAD_ARG;
  size_t es = elem_size(dtype);
  for (int t = 0; t < T; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    int64_t block = slot / B, off = slot % B;
    if (block >= num_blocks) return PAO_BAD_SLOT;
    for (int h = 0; h < Hkv; ++h) {
      size_t src = ((size_t)t * Hkv + h) * D * es;
      size_t dst = (size_t)pao_offset_ours(block, h, off, 0, Hkv, B, D) * es;
      memcpy((char*)k_cache + dst, (const char*)key + src, D * es);
      memcpy((char*)v_cache + dst, (const char*)value + src, D * es);
    }
  }
  return PAO_OK;
}

/* The FP8 append: as above, but each element of the fp16 key (value) row is
 * written as the E4M3 code of x / k_scale (x / v_scale), the division in fp32;
 * keys go to [block][head][offset][d], values to [block][head][offset/16][d][offset%16]. */
int pao_reshape_and_cache_fp8(uint8_t* k_cache, uint8_t* v_cache, const uint16_t* key_f16, const uint16_t* value_f16,
                              const int64_t* slot_mapping, int T, int Hkv, int D, int B, int num_blocks,
                              float k_scale, float v_scale) {
  if (!k_cache || !v_cache || !key_f16 || !value_f16 || !slot_mapping || T < 0) return PAO_BAD_ARG;
  if (!(k_scale > 0.0f) || !(v_scale > 0.0f) || B % 16 != 0) return PAO_BAD_ARG;
  for (int t = 0; t < T; ++t) {
    int64_t sl = slot_mapping[t];
    if (sl < 0) continue; /* padding token */
    const int64_t blk = sl / B, off = sl % B;
    if (blk >= num_blocks) return PAO_BAD_SLOT;
    for (int h = 0; h < Hkv; ++h) {
      for (int d = 0; d < D; ++d) {
        const size_t src = ((size_t)t * Hkv + h) * D + d;
        const float xk = (float)pao_f16_to_f64(key_f16[src]); /* exact: every fp16 value is a float */
        const float xv = (float)pao_f16_to_f64(value_f16[src]);
        const float rk = xk / k_scale, rv = xv / v_scale;
        k_cache[pao_offset_ours(blk, h, off, d, Hkv, B, D)] = pao_f32_to_e4m3_sat(rk);
        v_cache[pao_value_offset_fp8(blk, h, off, d, Hkv, B, D)] = pao_f32_to_e4m3_sat(rv);
      }
    }
  }
  return PAO_OK;
}

/* [P2 "写时复制是正确性的边界"]: the copy step of copy-on-write.  For each
 * (src, dst) pair, in order, the whole physical block dst of both caches
 * becomes a byte copy of block src. */
int pao_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int n, int dtype, int Hkv, int D, int B,
                    int num_blocks) {
  if (!k_cache || !v_cache || (!pairs && n > 0) || n < 0) return PAO_BAD_ARG;
  size_t block_bytes = (size_t)Hkv * B * D * elem_size(dtype);
  for (int i = 0; i < n; ++i) {
    int32_t src = pairs[2 * i], dst = pairs[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return PAO_BAD_BLOCK;
    memmove((char*)k_cache + (size_t)dst * block_bytes, (const char*)k_cache + (size_t)src * block_bytes, block_bytes);
    memmove((char*)v_cache + (size_t)dst * block_bytes, (const char*)v_cache + (size_t)src * block_bytes, block_bytes);
  }
  return PAO_OK;
}

int pao_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

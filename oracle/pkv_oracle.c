/*
 * pkv_oracle.c - plain, slow CPU oracle for paged KV-cache attention.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the package's smoke() check and the bench's
 * CPU-baseline leg load this file; the product path never does. It shares no code, header,
 * table or constant generator with the CUDA library: every formula here is restated from
 * the pages and written the plain way (explicit loops, explicit block-table gathers, no
 * tiling, no fusion).
 *
 * Sources (page title, then the part of the page):
 *   [P109] HyperQwen PR #109 "int64 cast in the int8 prefill attention": description items
 *          1-2 (the three kernels _k_stats_kernel, _k_quant_kernel, _prefill_attn_kernel, the
 *          block-table load blk = table[req][pos // BLOCK_SIZE] and the cast of blk to int64),
 *          and the review (exact-QK and int8-QK arms, top == bottom placement test).
 *   [P91]  HyperQwen PR #91 "int64 cast in _spec_attn_partial": description and review (the
 *          kernel excerpt: blk from the table, slot = pos % BLOCK_SIZE, K pointer
 *          blk * stride_kb + ..., int8 per-token-head scales via the same blk; split-KV).
 *   [P3360] vllm.cpp PR #3360 "serve fp8 KV prefill through the bf16 dense dequant": "What
 *          changed" (dequantize once per layer into a dense bf16 scratch with an identity
 *          block table and block_size = max_seq).
 *   [P91r] the same PR #91 page, the tester's report of the int8 route (a cache stored as
 *          int8 per token and head with its scales, "--kv-cache-dtype int8_per_token_head")
 *          and the fp8 store with a per-tensor descale (k_descale); these are the formats the
 *          cache write below produces.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - cache layout [num_blocks][block_size][num_kv_heads][head_dim] with explicit strides;
 *   - query head h reads KV head h / (num_q_heads / num_kv_heads);
 *   - request r's queries are its last q_len positions: position seq_len - q_len + i, and a
 *     query at position p attends keys 0..p;
 *   - symmetric int8 quantizer per (token, head) row: scale = absmax / 127 (fp32 divide),
 *     code = clamp(rint(x * (127 / absmax)), -127, 127) with one fp32 divide per row and one
 *     fp32 multiply per element, ties to even; an all-zero row gives scale 0 and codes 0;
 *   - e4m3 is the OCP FP8 E4M3 format (bias 7, subnormals, no infinities, S.1111.111 = NaN);
 *   - split s of a verify request covers key positions [s*split_tokens, (s+1)*split_tokens).
 *   - a cache write stores request r's new rows (its last q_len positions, as above) through the
 *     block table; the int8 cache uses the quantizer above per (token, head) row, the fp8 cache
 *     stores e4m3_rn_satfinite(x / scale) with one fp32 divide per element.
 *
 * Precision: attention is computed with double accumulators from the stored bf16 / int8 /
 * e4m3 values (at least as precise as the pages' fp32 reference); the quantizers and the fp8
 * dequantizer use exactly the fp32 operations named above (build with -ffp-contract=off).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_BOUNDS 4

/* ---------------------------------------------------------------------------------------- */
/* scalar formats                                                                           */
/* ---------------------------------------------------------------------------------------- */

float orc_bf16_to_f32(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* IEEE round-to-nearest-even of an fp32 value to bf16 (8 significand bits). */
uint16_t orc_f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0) /* NaN stays NaN */
    return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lower = u & 0xFFFFu;
  uint32_t upper = u >> 16;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u; /* ties to even */
  return (uint16_t)upper;
}

/* OCP FP8 E4M3: value = (-1)^s * 2^(e-7) * (1 + m/8) for e > 0, (-1)^s * 2^-6 * (m/8) for e == 0,
 * and the single pattern e == 15, m == 7 is NaN (no infinities; largest finite 448). */
float orc_e4m3_to_f32(uint8_t code) {
  int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  float mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexpf((float)m, -9);
  else
    mag = ldexpf((float)(8 + m), e - 10);
  return s ? -mag : mag;
}

/* fp32 -> OCP E4M3, round to nearest with ties to even, saturating: every finite or infinite
 * magnitude above the largest finite value 448 becomes +-448, NaN becomes 0x7F. Written from the
 * format: normal numbers have a quantum of 2^(e-3) for 2^e <= |x| < 2^(e+1) (e >= -6), subnormals
 * a quantum of 2^-9; the scaled magnitude |x| / quantum is exact, so rintf (ties to even in the
 * default rounding mode) rounds it once. */
uint8_t orc_f32_to_e4m3_sat(float x) {
  if (isnan(x)) return 0x7Fu;
  uint8_t sign = signbit(x) ? 0x80u : 0x00u;
  float a = fabsf(x);
  if (a >= 448.0f) return sign | 0x7Eu; /* includes infinity */
  if (a < ldexpf(1.0f, -6)) {          /* subnormal range: code = multiple of 2^-9 */
    int m = (int)rintf(ldexpf(a, 9));  /* 0..8; 8 is the smallest normal, code 0x08 */
    return sign | (uint8_t)m;
  }
  int e2;
  frexpf(a, &e2); /* a = f * 2^e2, f in [0.5, 1) -> 2^(e2-1) <= a < 2^e2 */
  int e = e2 - 1;
  int m = (int)rintf(ldexpf(a, 3 - e)); /* 8..16 */
  if (m == 16) { m = 8; e += 1; }
  int code = ((e + 7) << 3) | (m - 8);
  if (code > 0x7E) code = 0x7E; /* 480 does not exist: saturate */
  return sign | (uint8_t)code;
}

/* ---------------------------------------------------------------------------------------- */
/* block addressing [P109 item 1, P91 kernel excerpt]                                       */
/* ---------------------------------------------------------------------------------------- */

/* 0: block id widened to int64 before the stride product (the method).
 * 1: the product taken in 32-bit two's complement, the pre-fix behaviour the pages describe;
 *    a planted mistake for the tests that prove the placement test can tell the two apart. */
static int g_offset_mode = 0;
void orc_set_offset_mode_for_testing(int mode) { g_offset_mode = mode; }

static int64_t block_base(int64_t blk, int64_t stride_blk) {
  if (g_offset_mode == 1) {
    uint32_t w = (uint32_t)blk * (uint32_t)stride_blk;
    return (int64_t)(int32_t)w;
  }
  return blk * stride_blk;
}

typedef struct {
  const void* base;
  int64_t num_blocks, stride_blk, stride_tok, stride_head;
  int64_t pool_elems;
  const int32_t* table;
  int64_t bt_stride;
  int32_t block_size;
} paged_view;

static paged_view make_view(const void* base, int64_t nb, int64_t sb, int64_t st, int64_t sh,
                            const int32_t* table, int64_t bts, int32_t bs) {
  paged_view v;
  v.base = base; v.num_blocks = nb; v.stride_blk = sb; v.stride_tok = st; v.stride_head = sh;
  v.pool_elems = nb * sb; v.table = table; v.bt_stride = bts; v.block_size = bs;
  return v;
}

/* Element offset of (request r, key position pos, kv head h, element 0); -1 when the resulting
 * address falls outside the pool (only possible with the planted 32-bit product). *bad is set
 * when the table holds a block id outside [0, num_blocks). */
static int64_t paged_offset(const paged_view* v, int r, int64_t pos, int h, int* bad) {
  int64_t blk = (int64_t)v->table[(int64_t)r * v->bt_stride + pos / v->block_size];
  int64_t slot = pos % v->block_size;
  if (blk < 0 || blk >= v->num_blocks) { *bad = 1; return -1; }
  int64_t off = block_base(blk, v->stride_blk) + slot * v->stride_tok + (int64_t)h * v->stride_head;
  if (off < 0 || off >= v->pool_elems) return -1;
  return off;
}

/* ---------------------------------------------------------------------------------------- */
/* A1 / A2: symmetric int8 quantizer per (token, head) row [P109 _k_stats_kernel /           */
/* _k_quant_kernel; the int8-QK arm quantizes Q rows the same way]                           */
/* ---------------------------------------------------------------------------------------- */

void orc_quant_row_i8(const uint16_t* x, int n, int8_t* codes, float* scale) {
  float absmax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float a = fabsf(orc_bf16_to_f32(x[i]));
    if (isnan(a)) { /* a NaN row has no defined codes: report it through a NaN scale */
      *scale = NAN;
      for (int k = 0; k < n; ++k) codes[k] = 0;
      return;
    }
    if (a > absmax) absmax = a;
  }
  if (absmax == 0.0f) {
    *scale = 0.0f;
    for (int i = 0; i < n; ++i) codes[i] = 0;
    return;
  }
  *scale = absmax / 127.0f;
  float inv = 127.0f / absmax;
  for (int i = 0; i < n; ++i) {
    float t = rintf(orc_bf16_to_f32(x[i]) * inv);
    if (t > 127.0f) t = 127.0f;
    if (t < -127.0f) t = -127.0f;
    codes[i] = (int8_t)t;
  }
}

/* For each request r and key position pos in [pos_begin[r], pos_end[r]) and each kv head h:
 * gather the bf16 K row through the block table and quantize it into the dense scratch
 * k8[r][pos][h][:] with scale k8_scale[r][pos][h]. */
int orc_kv_int8_stats_quant(const uint16_t* k_cache, int64_t num_blocks, int64_t stride_blk,
                            int64_t stride_tok, int64_t stride_head, const int32_t* block_table,
                            int64_t bt_stride, const int32_t* pos_begin, const int32_t* pos_end,
                            int32_t num_reqs, int32_t block_size, int32_t num_kv_heads,
                            int32_t head_dim, int8_t* k8, float* k8_scale, int64_t max_ctx) {
  paged_view v = make_view(k_cache, num_blocks, stride_blk, stride_tok, stride_head, block_table,
                           bt_stride, block_size);
  int bad = 0;
  uint16_t* nanrow = (uint16_t*)malloc(sizeof(uint16_t) * head_dim);
  for (int d = 0; d < head_dim; ++d) nanrow[d] = 0x7FC0u;
  for (int r = 0; r < num_reqs; ++r) {
    if (pos_begin[r] < 0 || pos_end[r] > max_ctx || pos_begin[r] > pos_end[r]) { free(nanrow); return ORC_ERR_ARG; }
    for (int64_t pos = pos_begin[r]; pos < pos_end[r]; ++pos) {
      for (int h = 0; h < num_kv_heads; ++h) {
        int64_t off = paged_offset(&v, r, pos, h, &bad);
        const uint16_t* row = off < 0 ? nanrow : k_cache + off;
        int64_t o = ((int64_t)r * max_ctx + pos) * num_kv_heads + h;
        orc_quant_row_i8(row, head_dim, k8 + o * head_dim, k8_scale + o);
      }
    }
  }
  free(nanrow);
  return bad ? ORC_ERR_BOUNDS : ORC_OK;
}

/* ---------------------------------------------------------------------------------------- */
/* A4: per-tensor fp8 e4m3 cache -> dense bf16 scratch, once per layer [P3360]              */
/* dense[r][pos][h][d] = bf16_rn(fp32(e4m3(byte)) * scale), for pos < seq_len[r].           */
/* ---------------------------------------------------------------------------------------- */

int orc_kv_fp8_dequant_dense(const uint8_t* k_fp8, const uint8_t* v_fp8, int64_t num_blocks,
                             int64_t stride_blk, int64_t stride_tok, int64_t stride_head,
                             const int32_t* block_table, int64_t bt_stride,
                             const int32_t* seq_lens, int32_t num_reqs, int32_t max_seq,
                             int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                             float k_scale, float v_scale, uint16_t* k_dense, uint16_t* v_dense) {
  int bad = 0;
  for (int which = 0; which < 2; ++which) {
    const uint8_t* src = which == 0 ? k_fp8 : v_fp8;
    uint16_t* dst = which == 0 ? k_dense : v_dense;
    float scale = which == 0 ? k_scale : v_scale;
    paged_view v = make_view(src, num_blocks, stride_blk, stride_tok, stride_head, block_table,
                             bt_stride, block_size);
    for (int r = 0; r < num_reqs; ++r) {
      if (seq_lens[r] > max_seq) return ORC_ERR_ARG;
      for (int64_t pos = 0; pos < seq_lens[r]; ++pos) {
        for (int h = 0; h < num_kv_heads; ++h) {
          int64_t off = paged_offset(&v, r, pos, h, &bad);
          uint16_t* out = dst + (((int64_t)r * max_seq + pos) * num_kv_heads + h) * head_dim;
          for (int d = 0; d < head_dim; ++d) {
            float x = off < 0 ? NAN : orc_e4m3_to_f32(src[off + d]);
            out[d] = orc_f32_to_bf16_rne(x * scale);
          }
        }
      }
    }
  }
  return bad ? ORC_ERR_BOUNDS : ORC_OK;
}

/* ---------------------------------------------------------------------------------------- */
/* cache write: a chunk's new K/V rows stored into the paged pool through the block table    */
/* [P109 item 1 addressing; P91r cache formats]                                              */
/* ---------------------------------------------------------------------------------------- */

/* kv_dtype 0: bf16 copy. 1: int8 per (token, head) row with the quantizer above; the scale goes to
 * scale_cache[blk * scale_stride_blk + slot * scale_stride_tok + h]. 2: e4m3 per tensor,
 * code = orc_f32_to_e4m3_sat(x / scale). Row t of k_new / v_new ([total_tokens][hkv][D]) belongs
 * to the request r with qsl[r] <= t < qsl[r+1] and lands at position seq_len[r] - q_len[r] +
 * (t - qsl[r]). Rows whose table entry is outside [0, num_blocks) are not written (bounds status).
 */
int orc_kv_cache_write(int kv_dtype, const uint16_t* k_new, const uint16_t* v_new,
                       const int32_t* block_table, int64_t bt_stride, const int32_t* seq_lens,
                       const int32_t* qsl, int32_t num_reqs, int64_t num_blocks, int64_t stride_blk,
                       int64_t stride_tok, int64_t stride_head, int32_t block_size,
                       int32_t num_kv_heads, int32_t head_dim, void* k_cache, void* v_cache,
                       float* k_scale_cache, float* v_scale_cache, int64_t scale_stride_blk,
                       int64_t scale_stride_tok, float k_scale, float v_scale) {
  if (kv_dtype < 0 || kv_dtype > 2) return ORC_ERR_ARG;
  int bad = 0;
  for (int which = 0; which < 2; ++which) {
    const uint16_t* src = which == 0 ? k_new : v_new;
    void* dst = which == 0 ? k_cache : v_cache;
    float* sdst = which == 0 ? k_scale_cache : v_scale_cache;
    float tscale = which == 0 ? k_scale : v_scale;
    paged_view v = make_view(dst, num_blocks, stride_blk, stride_tok, stride_head, block_table,
                             bt_stride, block_size);
    for (int r = 0; r < num_reqs; ++r) {
      int64_t q_len = (int64_t)qsl[r + 1] - qsl[r];
      if (q_len < 0 || q_len > seq_lens[r]) return ORC_ERR_ARG;
      for (int64_t i = 0; i < q_len; ++i) {
        int64_t pos = seq_lens[r] - q_len + i;
        int64_t t = qsl[r] + i;
        for (int h = 0; h < num_kv_heads; ++h) {
          const uint16_t* row = src + (t * num_kv_heads + h) * head_dim;
          int row_bad = 0;
          int64_t off = paged_offset(&v, r, pos, h, &row_bad);
          if (row_bad) { bad = 1; continue; }
          if (off < 0) continue; /* planted 32-bit product left the pool: nothing written */
          if (kv_dtype == 0) {
            memcpy((uint16_t*)dst + off, row, sizeof(uint16_t) * head_dim);
          } else if (kv_dtype == 1) {
            int64_t blk = (int64_t)block_table[(int64_t)r * bt_stride + pos / block_size];
            int64_t soff = block_base(blk, scale_stride_blk) + (pos % block_size) * scale_stride_tok + h;
            float sc;
            orc_quant_row_i8(row, head_dim, (int8_t*)dst + off, &sc);
            if (soff >= 0 && soff < num_blocks * scale_stride_blk) sdst[soff] = sc;
          } else {
            for (int d = 0; d < head_dim; ++d)
              ((uint8_t*)dst)[off + d] = orc_f32_to_e4m3_sat(orc_bf16_to_f32(row[d]) / tscale);
          }
        }
      }
    }
  }
  return bad ? ORC_ERR_BOUNDS : ORC_OK;
}

/* ---------------------------------------------------------------------------------------- */
/* A3: chunked causal prefill attention over a paged cache [P109]                           */
/* ---------------------------------------------------------------------------------------- */

static int find_request(const int32_t* qsl, int num_reqs, int64_t t) {
  for (int r = 0; r < num_reqs; ++r)
    if (t >= qsl[r] && t < qsl[r + 1]) return r;
  return -1;
}

/* Softmax-weighted sum for one query row, given its scores s[0..n) and a fetcher that gathers the
 * value row of key j (through the block table) into a buffer of head_dim doubles.
 * o = sum_j exp(s_j - m) v_j / sum_j exp(s_j - m), m = max_j s_j; two passes, ascending j. */
typedef void (*row_fn)(void* ctx, int64_t j, double* row, int head_dim);

static void softmax_pv(const double* s, int64_t n, int head_dim, row_fn fetch, void* ctx,
                       float* out, double* lse_out) {
  double m = -INFINITY;
  int any_nan = 0;
  for (int64_t j = 0; j < n; ++j) {
    if (isnan(s[j])) any_nan = 1;
    if (s[j] > m) m = s[j];
  }
  if (any_nan) { /* a NaN score poisons the row, as it would in any softmax */
    for (int d = 0; d < head_dim; ++d) out[d] = NAN;
    if (lse_out) *lse_out = NAN;
    return;
  }
  double* acc = (double*)calloc((size_t)head_dim, sizeof(double));
  double* v = (double*)malloc(sizeof(double) * (size_t)head_dim);
  double l = 0.0;
  if (n > 0 && m != -INFINITY) {
    for (int64_t j = 0; j < n; ++j) {
      double w = exp(s[j] - m);
      l += w;
      fetch(ctx, j, v, head_dim);
      for (int d = 0; d < head_dim; ++d) acc[d] += w * v[d];
    }
  }
  for (int d = 0; d < head_dim; ++d) out[d] = l > 0.0 ? (float)(acc[d] / l) : 0.0f;
  if (lse_out) *lse_out = l > 0.0 ? m + log(l) : -INFINITY;
  free(v);
  free(acc);
}

typedef struct {
  const paged_view* v;
  int r, h;
  int64_t base_pos;
  const uint16_t* bf16;      /* bf16 V pool */
  const int8_t* i8;          /* int8 V pool */
  const float* vscale;       /* per-token-head V scales (int8 pool) */
  int64_t sc_blk, sc_tok;
  int* bad;
  uint16_t nan_bits;
} vctx;

static void v_bf16(void* c, int64_t j, double* row, int head_dim) {
  vctx* x = (vctx*)c;
  int64_t off = paged_offset(x->v, x->r, x->base_pos + j, x->h, x->bad);
  for (int d = 0; d < head_dim; ++d)
    row[d] = off < 0 ? NAN : (double)orc_bf16_to_f32(x->bf16[off + d]);
}

/* Int8 per-token-head value: v8 * vs, the scale read through the same block id [P91]. */
static double scale_of(const paged_view* v, const float* sc, int64_t sc_blk, int64_t sc_tok,
                       int r, int64_t pos, int h, int* bad) {
  int64_t blk = (int64_t)v->table[(int64_t)r * v->bt_stride + pos / v->block_size];
  if (blk < 0 || blk >= v->num_blocks) { *bad = 1; return NAN; }
  int64_t off = block_base(blk, sc_blk) + (pos % v->block_size) * sc_tok + h;
  if (off < 0 || off >= v->num_blocks * sc_blk) return NAN;
  return (double)sc[off];
}

static void v_int8(void* c, int64_t j, double* row, int head_dim) {
  vctx* x = (vctx*)c;
  int64_t pos = x->base_pos + j;
  int64_t off = paged_offset(x->v, x->r, pos, x->h, x->bad);
  double sc = off < 0 ? NAN : scale_of(x->v, x->vscale, x->sc_blk, x->sc_tok, x->r, pos, x->h, x->bad);
  for (int d = 0; d < head_dim; ++d) row[d] = off < 0 ? NAN : (double)x->i8[off + d] * sc;
}

/* Prefill attention for global query tokens [tok_begin, tok_end), all query heads.
 * qk_mode 0 (exact QK): s_j = scale * sum_d q_d k_jd on the bf16 values.
 * qk_mode 1 (int8 QK): q is quantized per (token, head) row with the int8 quantizer above, and
 *   s_j = scale * q_scale * k8_scale[r][j][kvh] * (sum_d q8_d k8[r][j][kvh][d]) with the integer
 *   dot product accumulated in int32. V is the bf16 cache in both modes.
 * out is fp32 [tok_end - tok_begin][num_q_heads][head_dim]. */
int orc_paged_prefill_attn(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                           int64_t num_blocks, int64_t stride_blk, int64_t stride_tok,
                           int64_t stride_head, const int32_t* block_table, int64_t bt_stride,
                           const int32_t* seq_lens, const int32_t* query_start_loc,
                           int32_t num_reqs, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_dim, int32_t block_size, float softmax_scale,
                           int32_t qk_mode, const int8_t* k8, const float* k8_scale,
                           int64_t max_ctx, int64_t tok_begin, int64_t tok_end, float* out) {
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return ORC_ERR_ARG;
  int group = num_q_heads / num_kv_heads;
  paged_view kv = make_view(k_cache, num_blocks, stride_blk, stride_tok, stride_head, block_table,
                            bt_stride, block_size);
  paged_view vv = make_view(v_cache, num_blocks, stride_blk, stride_tok, stride_head, block_table,
                            bt_stride, block_size);
  int bad = 0;
  int8_t* q8 = (int8_t*)malloc((size_t)head_dim);
  for (int64_t t = tok_begin; t < tok_end; ++t) {
    int r = find_request(query_start_loc, num_reqs, t);
    if (r < 0) { free(q8); return ORC_ERR_ARG; }
    int64_t q_len = query_start_loc[r + 1] - query_start_loc[r];
    int64_t p = (int64_t)seq_lens[r] - q_len + (t - query_start_loc[r]);
    if (p < 0) { free(q8); return ORC_ERR_ARG; }
    int64_t n = p + 1;
    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    for (int h = 0; h < num_q_heads; ++h) {
      int kvh = h / group;
      const uint16_t* qrow = q + (t * num_q_heads + h) * (int64_t)head_dim;
      float qs = 0.0f;
      if (qk_mode == 1) orc_quant_row_i8(qrow, head_dim, q8, &qs);
      for (int64_t j = 0; j < n; ++j) {
        if (qk_mode == 1) {
          int64_t o = ((int64_t)r * max_ctx + j) * num_kv_heads + kvh;
          const int8_t* krow = k8 + o * head_dim;
          int32_t dot = 0;
          for (int d = 0; d < head_dim; ++d) dot += (int32_t)q8[d] * (int32_t)krow[d];
          s[j] = (double)softmax_scale * (double)qs * (double)k8_scale[o] * (double)dot;
        } else {
          int64_t off = paged_offset(&kv, r, j, kvh, &bad);
          double acc = 0.0;
          if (off < 0) {
            acc = NAN;
          } else {
            for (int d = 0; d < head_dim; ++d)
              acc += (double)orc_bf16_to_f32(qrow[d]) * (double)orc_bf16_to_f32(k_cache[off + d]);
          }
          s[j] = (double)softmax_scale * acc;
        }
      }
      vctx c = {&vv, r, kvh, 0, v_cache, NULL, NULL, 0, 0, &bad, 0x7FC0u};
      softmax_pv(s, n, head_dim, v_bf16, &c,
                 out + ((t - tok_begin) * num_q_heads + h) * (int64_t)head_dim, NULL);
    }
    free(s);
  }
  free(q8);
  return bad ? ORC_ERR_BOUNDS : ORC_OK;
}

/* Dense (non-paged) causal attention brute force: K/V given per position as [L][Hkv][D] bf16,
 * queries at positions qpos[i]. A pin for the paged gather above. out fp32 [nq][Hq][D]. */
int orc_dense_attn(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int64_t* qpos,
                   int64_t nq, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                   float softmax_scale, float* out) {
  int group = num_q_heads / num_kv_heads;
  for (int64_t i = 0; i < nq; ++i) {
    for (int h = 0; h < num_q_heads; ++h) {
      int kvh = h / group;
      int64_t n = qpos[i] + 1;
      double* w = (double*)malloc(sizeof(double) * (size_t)n);
      double m = -INFINITY, l = 0.0;
      for (int64_t j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int d = 0; d < head_dim; ++d)
          acc += (double)orc_bf16_to_f32(q[(i * num_q_heads + h) * head_dim + d]) *
                 (double)orc_bf16_to_f32(k[(j * num_kv_heads + kvh) * head_dim + d]);
        w[j] = softmax_scale * acc;
        if (w[j] > m) m = w[j];
      }
      for (int64_t j = 0; j < n; ++j) { w[j] = exp(w[j] - m); l += w[j]; }
      for (int d = 0; d < head_dim; ++d) {
        double acc = 0.0;
        for (int64_t j = 0; j < n; ++j)
          acc += w[j] * (double)orc_bf16_to_f32(v[(j * num_kv_heads + kvh) * head_dim + d]);
        out[(i * num_q_heads + h) * head_dim + d] = (float)(acc / l);
      }
      free(w);
    }
  }
  return ORC_OK;
}

/* ---------------------------------------------------------------------------------------- */
/* A5 / A6: speculative-verify attention over an int8 per-token-head cache [P91]            */
/* ---------------------------------------------------------------------------------------- */

/* Scores of query token t (0..T-1) of request r, head h, over keys [j0, j1) that it can see
 * (key position <= seq_len - T + t). k = k8 * ks, per token-head, scales read through the
 * same block id as the codes. Returns the number of visible keys written to s. */
static int64_t verify_scores(const uint16_t* q, const int8_t* k_cache, const float* k_scale,
                             const paged_view* kv, int64_t sc_blk, int64_t sc_tok, int r, int T,
                             int t, int h, int kvh, int num_q_heads, int head_dim, int64_t seq_len,
                             float softmax_scale, int64_t j0, int64_t j1, double* s, int* bad) {
  int64_t last = seq_len - T + t; /* causal limit */
  if (j1 > last + 1) j1 = last + 1;
  const uint16_t* qrow = q + (((int64_t)r * T + t) * num_q_heads + h) * head_dim;
  int64_t n = 0;
  for (int64_t j = j0; j < j1; ++j, ++n) {
    int64_t off = paged_offset(kv, r, j, kvh, bad);
    if (off < 0) { s[n] = NAN; continue; }
    double ks = scale_of(kv, k_scale, sc_blk, sc_tok, r, j, kvh, bad);
    double acc = 0.0;
    for (int d = 0; d < head_dim; ++d)
      acc += (double)orc_bf16_to_f32(qrow[d]) * ((double)k_cache[off + d] * ks);
    s[n] = (double)softmax_scale * acc;
  }
  return n;
}

/* Unsplit verify attention: out fp32 [num_reqs*T][Hq][D]. */
int orc_spec_verify_attn(const uint16_t* q, const int8_t* k_cache, const int8_t* v_cache,
                         const float* k_scale, const float* v_scale, int64_t num_blocks,
                         int64_t stride_blk, int64_t stride_tok, int64_t stride_head,
                         int64_t scale_stride_blk, int64_t scale_stride_tok,
                         const int32_t* block_table, int64_t bt_stride, const int32_t* seq_lens,
                         int32_t num_reqs, int32_t T, int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, float softmax_scale,
                         int32_t req_begin, int32_t req_end, float* out) {
  int group = num_q_heads / num_kv_heads;
  paged_view kv = make_view(k_cache, num_blocks, stride_blk, stride_tok, stride_head, block_table,
                            bt_stride, block_size);
  paged_view vv = make_view(v_cache, num_blocks, stride_blk, stride_tok, stride_head, block_table,
                            bt_stride, block_size);
  int bad = 0;
  for (int r = req_begin; r < req_end; ++r) {
    int64_t L = seq_lens[r];
    double* s = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    for (int t = 0; t < T; ++t) {
      for (int h = 0; h < num_q_heads; ++h) {
        int kvh = h / group;
        int64_t n = verify_scores(q, k_cache, k_scale, &kv, scale_stride_blk, scale_stride_tok, r, T,
                                  t, h, kvh, num_q_heads, head_dim, L, softmax_scale, 0, L, s, &bad);
        vctx c = {&vv, r, kvh, 0, NULL, v_cache, v_scale, scale_stride_blk, scale_stride_tok, &bad, 0};
        softmax_pv(s, n, head_dim, v_int8, &c,
                   out + (((int64_t)r * T + t) * num_q_heads + h) * (int64_t)head_dim, NULL);
      }
    }
    free(s);
  }
  return bad ? ORC_ERR_BOUNDS : ORC_OK;
}

/* Split-KV partials: for split s (keys [s*split_tokens, min((s+1)*split_tokens, seq_len))) and
 * each query row: o_s = normalised weighted sum over the split's visible keys and
 * lse_s = m_s + ln(l_s); a split with no visible key has lse = -inf and o = 0.
 * part_o fp32 [max_splits][num_reqs*T][Hq][D], part_lse fp32 [max_splits][num_reqs*T][Hq]. */
int orc_spec_verify_partial(const uint16_t* q, const int8_t* k_cache, const int8_t* v_cache,
                            const float* k_scale, const float* v_scale, int64_t num_blocks,
                            int64_t stride_blk, int64_t stride_tok, int64_t stride_head,
                            int64_t scale_stride_blk, int64_t scale_stride_tok,
                            const int32_t* block_table, int64_t bt_stride, const int32_t* seq_lens,
                            int32_t num_reqs, int32_t T, int32_t num_q_heads, int32_t num_kv_heads,
                            int32_t head_dim, int32_t block_size, float softmax_scale,
                            int32_t split_tokens, int32_t max_splits, int32_t req_begin,
                            int32_t req_end, float* part_o, float* part_lse) {
  int group = num_q_heads / num_kv_heads;
  int64_t rows = (int64_t)num_reqs * T * num_q_heads;
  paged_view kv = make_view(k_cache, num_blocks, stride_blk, stride_tok, stride_head, block_table,
                            bt_stride, block_size);
  paged_view vv = make_view(v_cache, num_blocks, stride_blk, stride_tok, stride_head, block_table,
                            bt_stride, block_size);
  int bad = 0;
  double* s = (double*)malloc(sizeof(double) * (size_t)split_tokens);
  for (int r = req_begin; r < req_end; ++r) {
    int64_t L = seq_lens[r];
    int64_t nsplit = (L + split_tokens - 1) / split_tokens;
    if (nsplit > max_splits) { free(s); return ORC_ERR_ARG; }
    for (int64_t sp = 0; sp < nsplit; ++sp) {
      int64_t j0 = sp * split_tokens, j1 = j0 + split_tokens < L ? j0 + split_tokens : L;
      for (int t = 0; t < T; ++t) {
        for (int h = 0; h < num_q_heads; ++h) {
          int kvh = h / group;
          int64_t row = ((int64_t)r * T + t) * num_q_heads + h;
          int64_t n = verify_scores(q, k_cache, k_scale, &kv, scale_stride_blk, scale_stride_tok, r,
                                    T, t, h, kvh, num_q_heads, head_dim, L, softmax_scale, j0, j1, s,
                                    &bad);
          vctx c = {&vv, r, kvh, j0, NULL, v_cache, v_scale, scale_stride_blk, scale_stride_tok, &bad, 0};
          double lse;
          softmax_pv(s, n, head_dim, v_int8, &c, part_o + (sp * rows + row) * head_dim, &lse);
          part_lse[sp * rows + row] = (float)lse;
        }
      }
    }
  }
  free(s);
  return bad ? ORC_ERR_BOUNDS : ORC_OK;
}

/* ---------------------------------------------------------------------------------------- */
/* Verify over a per-tensor fp8 e4m3 cache [P91 description and review: the fp8 arm of the    */
/* big-pool test, "k_descale"; the split-KV verify on the per-tensor fp8 KV cache]             */
/* k = e4m3(byte) * k_descale, v = e4m3(byte) * v_descale; otherwise as the int8 verify.      */
/* ---------------------------------------------------------------------------------------- */

static int64_t verify_scores_fp8(const uint16_t* q, const uint8_t* k_cache, double k_descale,
                                 const paged_view* kv, int r, int T, int t, int h, int kvh,
                                 int num_q_heads, int head_dim, int64_t seq_len, float softmax_scale,
                                 int64_t j0, int64_t j1, double* s, int* bad) {
  int64_t last = seq_len - T + t;
  if (j1 > last + 1) j1 = last + 1;
  const uint16_t* qrow = q + (((int64_t)r * T + t) * num_q_heads + h) * head_dim;
  int64_t n = 0;
  for (int64_t j = j0; j < j1; ++j, ++n) {
    int64_t off = paged_offset(kv, r, j, kvh, bad);
    if (off < 0) { s[n] = NAN; continue; }
    double acc = 0.0;
    for (int d = 0; d < head_dim; ++d)
      acc += (double)orc_bf16_to_f32(qrow[d]) * ((double)orc_e4m3_to_f32(k_cache[off + d]) * k_descale);
    s[n] = (double)softmax_scale * acc;
  }
  return n;
}

typedef struct {
  const paged_view* v;
  int r, h;
  int64_t base_pos;
  const uint8_t* codes;
  double descale;
  int* bad;
} vctx_fp8;

static void v_e4m3(void* c, int64_t j, double* row, int head_dim) {
  vctx_fp8* x = (vctx_fp8*)c;
  int64_t off = paged_offset(x->v, x->r, x->base_pos + j, x->h, x->bad);
  for (int d = 0; d < head_dim; ++d)
    row[d] = off < 0 ? NAN : (double)orc_e4m3_to_f32(x->codes[off + d]) * x->descale;
}

int orc_spec_verify_attn_fp8(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache,
                             float k_descale, float v_descale, int64_t num_blocks, int64_t stride_blk,
                             int64_t stride_tok, int64_t stride_head, const int32_t* block_table,
                             int64_t bt_stride, const int32_t* seq_lens, int32_t num_reqs, int32_t T,
                             int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t block_size, float softmax_scale, int32_t req_begin,
                             int32_t req_end, float* out) {
  int group = num_q_heads / num_kv_heads;
  paged_view kv = make_view(k_cache, num_blocks, stride_blk, stride_tok, stride_head, block_table,
                            bt_stride, block_size);
  paged_view vv = make_view(v_cache, num_blocks, stride_blk, stride_tok, stride_head, block_table,
                            bt_stride, block_size);
  int bad = 0;
  for (int r = req_begin; r < req_end; ++r) {
    int64_t L = seq_lens[r];
    double* s = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    for (int t = 0; t < T; ++t) {
      for (int h = 0; h < num_q_heads; ++h) {
        int kvh = h / group;
        int64_t n = verify_scores_fp8(q, k_cache, k_descale, &kv, r, T, t, h, kvh, num_q_heads,
                                      head_dim, L, softmax_scale, 0, L, s, &bad);
        vctx_fp8 c = {&vv, r, kvh, 0, v_cache, v_descale, &bad};
        softmax_pv(s, n, head_dim, v_e4m3, &c,
                   out + (((int64_t)r * T + t) * num_q_heads + h) * (int64_t)head_dim, NULL);
      }
    }
    free(s);
  }
  return bad ? ORC_ERR_BOUNDS : ORC_OK;
}

int orc_spec_verify_partial_fp8(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                float k_descale, float v_descale, int64_t num_blocks,
                                int64_t stride_blk, int64_t stride_tok, int64_t stride_head,
                                const int32_t* block_table, int64_t bt_stride,
                                const int32_t* seq_lens, int32_t num_reqs, int32_t T,
                                int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                int32_t block_size, float softmax_scale, int32_t split_tokens,
                                int32_t max_splits, int32_t req_begin, int32_t req_end,
                                float* part_o, float* part_lse) {
  int group = num_q_heads / num_kv_heads;
  int64_t rows = (int64_t)num_reqs * T * num_q_heads;
  paged_view kv = make_view(k_cache, num_blocks, stride_blk, stride_tok, stride_head, block_table,
                            bt_stride, block_size);
  paged_view vv = make_view(v_cache, num_blocks, stride_blk, stride_tok, stride_head, block_table,
                            bt_stride, block_size);
  int bad = 0;
  double* s = (double*)malloc(sizeof(double) * (size_t)split_tokens);
  for (int r = req_begin; r < req_end; ++r) {
    int64_t L = seq_lens[r];
    int64_t nsplit = (L + split_tokens - 1) / split_tokens;
    if (nsplit > max_splits) { free(s); return ORC_ERR_ARG; }
    for (int64_t sp = 0; sp < nsplit; ++sp) {
      int64_t j0 = sp * split_tokens, j1 = j0 + split_tokens < L ? j0 + split_tokens : L;
      for (int t = 0; t < T; ++t) {
        for (int h = 0; h < num_q_heads; ++h) {
          int kvh = h / group;
          int64_t row = ((int64_t)r * T + t) * num_q_heads + h;
          int64_t n = verify_scores_fp8(q, k_cache, k_descale, &kv, r, T, t, h, kvh, num_q_heads,
                                        head_dim, L, softmax_scale, j0, j1, s, &bad);
          vctx_fp8 c = {&vv, r, kvh, j0, v_cache, v_descale, &bad};
          double lse;
          softmax_pv(s, n, head_dim, v_e4m3, &c, part_o + (sp * rows + row) * head_dim, &lse);
          part_lse[sp * rows + row] = (float)lse;
        }
      }
    }
  }
  free(s);
  return bad ? ORC_ERR_BOUNDS : ORC_OK;
}

/* Log-sum-exp combine: LSE = ln sum_s exp(lse_s); out = sum_s exp(lse_s - LSE) o_s.
 * Splits beyond ceil(seq_len / split_tokens) are not read. out fp32 [num_reqs*T][Hq][D]. */
int orc_spec_verify_combine(const float* part_o, const float* part_lse, const int32_t* seq_lens,
                            int32_t num_reqs, int32_t T, int32_t num_q_heads, int32_t head_dim,
                            int32_t split_tokens, int32_t max_splits, float* out) {
  int64_t rows = (int64_t)num_reqs * T * num_q_heads;
  for (int r = 0; r < num_reqs; ++r) {
    int64_t nsplit = ((int64_t)seq_lens[r] + split_tokens - 1) / split_tokens;
    if (nsplit > max_splits) return ORC_ERR_ARG;
    for (int t = 0; t < T; ++t) {
      for (int h = 0; h < num_q_heads; ++h) {
        int64_t row = ((int64_t)r * T + t) * num_q_heads + h;
        double M = -INFINITY;
        for (int64_t sp = 0; sp < nsplit; ++sp)
          if (part_lse[sp * rows + row] > M) M = part_lse[sp * rows + row];
        double sum = 0.0;
        for (int64_t sp = 0; sp < nsplit; ++sp)
          if (part_lse[sp * rows + row] != -INFINITY) sum += exp((double)part_lse[sp * rows + row] - M);
        double LSE = M + log(sum);
        for (int d = 0; d < head_dim; ++d) {
          double acc = 0.0;
          for (int64_t sp = 0; sp < nsplit; ++sp) {
            float ls = part_lse[sp * rows + row];
            if (ls == -INFINITY) continue;
            acc += exp((double)ls - LSE) * (double)part_o[(sp * rows + row) * head_dim + d];
          }
          out[row * head_dim + d] = (float)acc;
        }
      }
    }
  }
  return ORC_OK;
}

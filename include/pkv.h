/*
 * pkv.h - C ABI of libpkv.so: attention over a paged KV cache addressed through an int32 block
 * table, for NVIDIA GB300 (sm_103a).
 *
 * Sources (page title, then the part of the page that defines the operation):
 *   [P109]  HyperQwen PR #109 - int64 cast in the int8 prefill attention (prefill_attn_hd256.py):
 *           description items 1-2 and the review (three kernels _k_stats_kernel,
 *           _k_quant_kernel, _prefill_attn_kernel; exact-QK and int8-QK arms; chunk 2048,
 *           head_dim 256, block 880; top-vs-bottom placement in a 2,600-block pool).
 *   [P91]   HyperQwen PR #91 - int64 cast in the speculative-decode verify kernel
 *           _spec_attn_partial: description and review (kernel excerpt: blk = table[req][pos //
 *           BLOCK_SIZE], slot = pos % BLOCK_SIZE, K address blk * stride_kb + ...; int8
 *           per-token-head scales addressed by the same blk; split-KV partials).
 *   [P3360] vllm.cpp PR #3360 - serve fp8 KV prefill through the bf16 dense dequant, "What
 *           changed": dequantize ONCE per layer into a dense bf16 scratch, one block per request
 *           with block_size = max_seq and an identity block table, then run the bf16 kernel.
 *
 * Conventions shared by every call
 *   - Caches are [num_blocks][block_size][num_kv_heads][head_dim] with explicit element strides
 *     (stride_blk, stride_tok, stride_head; the head_dim axis is contiguous). The element
 *     offset of (block blk, slot s, head h, d) is blk*stride_blk + s*stride_tok + h*stride_head + d,
 *     and every block-id x stride product is formed in 64-bit arithmetic, so pools of any size
 *     (past 2^31 elements) are addressed correctly [P109 item 1, P91 description].
 *   - Key position pos of request r lives in block block_table[r*bt_stride + pos/block_size],
 *     slot pos % block_size. Table entries past ceil(seq_len/block_size) are never read.
 *   - Query head qh reads KV head qh / (num_q_heads / num_kv_heads).
 *   - Request r's queries are its last q_len positions (seq_len - q_len .. seq_len - 1); a query
 *     at position p attends keys 0..p (causal).
 *   - head_dim must be 256 (the pages' geometry); other values return PKV_ERR_UNSUPPORTED.
 *   - Ownership: the caller allocates every buffer (caches, tables, scratch, partials, outputs).
 *     The library never allocates device memory (no cudaMalloc). Its state: a thread-local error
 *     message, per-device records of kernel attributes already set, and the fixed scratch array of
 *     pkv_spec_verify_attn_noalloc (part of the library's device image, with its address cached
 *     per device; see that call for its sharing rules). All pointers except `stream` are device
 *     pointers unless stated otherwise.
 *   - Streams: every call enqueues work on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and returns without synchronising. Results are ready when the stream is.
 *   - Errors: arguments are validated on the host before anything is launched; a failed check
 *     returns a non-zero pkv_status, launches nothing and leaves a message for pkv_last_error().
 *     `dev_err` (nullable, device int32, caller-zeroed) receives a device-side status when a
 *     kernel meets a block id outside [0, num_blocks) or a position past the table
 *     (PKV_ERR_DEVICE_BOUNDS; the access is skipped and reads as zero) or a bounded internal
 *     wait expires (PKV_ERR_TIMEOUT). Kernels never trap.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad stride or alignment */
  PKV_ERR_UNSUPPORTED = 2,   /* valid but outside what the kernels implement (e.g. head_dim) */
  PKV_ERR_CUDA = 3,          /* a CUDA runtime call or kernel launch failed */
  PKV_ERR_DEVICE_BOUNDS = 4, /* device-side: out-of-range block id or position (via dev_err) */
  PKV_ERR_TIMEOUT = 5        /* device-side: a bounded wait gave up (via dev_err) */
} pkv_status;

typedef enum pkv_qk_mode {
  PKV_QK_BF16 = 0, /* exact QK: bf16 q . bf16 k, fp32 accumulate [P109 review, int8_qk=False] */
  PKV_QK_INT8 = 1  /* int8 QK: per-row int8 q . per-token-head int8 k, exact integer dot,
                      scaled by q_scale * k_scale [P109 review, int8_qk=True] */
} pkv_qk_mode;

typedef enum pkv_kv_dtype {
  PKV_KV_BF16 = 0, /* bf16 rows */
  PKV_KV_INT8 = 1, /* int8 per (token, head) row with an fp32 scale per row [P91 review:
                      "int8_per_token_head"] */
  PKV_KV_FP8 = 2   /* OCP e4m3 bytes with one fp32 scale per tensor [P91 review: k_descale] */
} pkv_kv_dtype;

/* Message of the last failed call on this host thread ("" if none). Never NULL. */
PKV_API const char* pkv_last_error(void);

/* ABI version of this header (incremented on any signature change). */
#define PKV_ABI_VERSION 7
PKV_API int32_t pkv_abi_version(void);

/*
 * testing_set_wait_limit_ns - a testing hook with no counterpart on the pages: the next attention
 * kernel launched by the calling host thread (pkv_paged_prefill_attn, pkv_paged_prefill_attn_fp8,
 * pkv_spec_verify_attn_partial, pkv_spec_verify_attn_partial_fp8) bounds each of its internal
 * waits by ns nanoseconds instead of the default one second; later launches use the default
 * again. ns = 0 keeps the default. With a bound far below the time a copy or an MMA takes, the
 * launch's CTAs give up at their first wait that is not already satisfied: each records
 * PKV_ERR_TIMEOUT in dev_err, waits (with its own bound) for the copies and MMAs it has in flight,
 * frees its tensor memory and exits, so the context stays usable; the outputs of that launch are
 * undefined. This is how the give-up path is tested without a hung kernel.
 */
PKV_API void pkv_testing_set_wait_limit_ns(uint64_t ns);

/*
 * kv_int8_stats_quant - per-token-head symmetric int8 quantization of the bf16 K cache
 * [P109: _k_stats_kernel (per-token-head statistics read through blk = block_table[...]) and
 *  _k_quant_kernel (int8 K written to a dense scratch indexed by position, one scale per slot)].
 *
 * For every request r, key position pos in [pos_begin[r], pos_end[r]) and KV head h, with
 * x = the bf16 row k_cache[blk(r,pos)][pos % block_size][h][0..head_dim):
 *   absmax = max |x|;  scale = absmax / 127 (fp32, round to nearest);
 *   k8[r][pos][h][d] = clamp(rint(x[d] * (127 / absmax)), -127, 127)  (one fp32 divide per
 *   row, one fp32 multiply per element, ties to even); absmax == 0 gives scale 0, codes 0.
 * Output k8 int8 [num_reqs][max_ctx][num_kv_heads][head_dim] (contiguous),
 *        k8_scale fp32 [num_reqs][max_ctx][num_kv_heads]; other positions are not written.
 * pos_begin / pos_end: device int32 [num_reqs], 0 <= pos_begin <= pos_end <= max_ctx.
 * max_tokens: host upper bound on pos_end[r] - pos_begin[r] (sizes the grid).
 * max_blocks: columns of the block table (pos_end <= max_blocks * block_size).
 * k16 (nullable): fp16 [num_reqs][max_ctx][num_kv_heads][head_dim]; when given, the same codes are
 *   also written there as fp16 values (exact). GB300's tensor cores have no int8 MMA, so the
 *   int8-QK prefill multiplies the codes as fp16; passing k16 to pkv_paged_prefill_attn lets it
 *   read them with TMA instead of widening every K row in every query tile.
 */
PKV_API pkv_status pkv_kv_int8_stats_quant(const void* k_cache, int64_t num_blocks, int64_t stride_blk,
                                   int64_t stride_tok, int64_t stride_head,
                                   const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                                   const int32_t* pos_begin, const int32_t* pos_end, int32_t num_reqs,
                                   int32_t max_tokens, int32_t block_size, int32_t num_kv_heads,
                                   int32_t head_dim, int8_t* k8, float* k8_scale, void* k16,
                                   int64_t max_ctx, int32_t* dev_err, void* stream);

/*
 * kv_fp8_dequant_dense - per-tensor fp8 e4m3 K/V cache to a dense bf16 scratch, once per layer
 * [P3360 "What changed"].
 *
 * For every request r, position pos < seq_lens[r], head h and d:
 *   k_dense[r][pos][h][d] = bf16_rn(float(e4m3(k_fp8[blk][slot][h][d])) * (*k_scale))
 * (one fp32 multiply rounded to nearest, then round-to-nearest-even to bf16), same for V.
 * e4m3 is the OCP FP8 E4M3 format. Dense outputs are [num_reqs][max_seq][num_kv_heads][head_dim]
 * contiguous bf16; positions >= seq_lens[r] are not written. The consumer then calls
 * pkv_paged_prefill_attn on the dense scratch with block_size = max_seq, num_blocks = num_reqs
 * and the identity table block_table[r] = r, so the paged address is the dense address.
 * k_scale / v_scale: device pointers to one fp32 each. max_seq: host, >= every seq_lens[r].
 */
PKV_API pkv_status pkv_kv_fp8_dequant_dense(const uint8_t* k_fp8, const uint8_t* v_fp8, int64_t num_blocks,
                                    int64_t stride_blk, int64_t stride_tok, int64_t stride_head,
                                    const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                                    const int32_t* seq_lens, int32_t num_reqs, int32_t max_seq,
                                    int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                    const float* k_scale, const float* v_scale, void* k_dense,
                                    void* v_dense, int32_t* dev_err, void* stream);

/*
 * paged_prefill_attn - chunked causal prefill attention over a paged bf16 cache
 * [P109: _prefill_attn_kernel; exact-QK and int8-QK arms].
 *
 * q:   bf16 [total_q][num_q_heads][head_dim], contiguous; request r owns rows
 *      query_start_loc[r] .. query_start_loc[r+1]-1 (device int32 [num_reqs+1]).
 * out: bf16, same layout as q.
 * For query row i of request r (position p = seq_lens[r] - q_len + i) and query head qh:
 *   s_j = softmax_scale * q . k_j              (PKV_QK_BF16; fp32 accumulation)
 *   s_j = softmax_scale * q_scale * k8_scale[r][j][kvh] * (q8 . k8[r][j][kvh])   (PKV_QK_INT8;
 *         q8 / q_scale = the kv_int8_stats_quant quantizer applied to the bf16 q row; the
 *         integer dot product is exact)
 *   out = sum_{j<=p} exp(s_j - m) v_j / sum_{j<=p} exp(s_j - m),   v_j from the bf16 V cache.
 * PKV_QK_INT8 reads k8 / k8_scale ([num_reqs][max_ctx][num_kv_heads][head_dim] / [...][kvh], as
 * written by pkv_kv_int8_stats_quant, covering positions 0..seq_len-1) instead of the K cache;
 * k_cache may then be NULL. When k16 (the fp16 copy of the codes that pkv_kv_int8_stats_quant
 * writes on request) is given it is read instead of k8 (same result, faster); k8 may then be NULL.
 * PKV_QK_BF16 ignores k8, k8_scale, k16 and max_ctx.
 * max_q_len: host upper bound on any request's q_len. total_q: host, = query_start_loc[num_reqs].
 * workspace (nullable, caller-owned device memory, 16-byte aligned, workspace_bytes long): NULL
 *   launches one CTA per (128-row query tile, head, request). Given, the call launches a
 *   persistent grid of P = min(SM count, workspace_bytes / pkv_paged_prefill_workspace_bytes(1),
 *   1024) CTAs: the query tiles in full waves of P, then the tiles of the last partial wave cut
 *   into up to 4 equal key ranges so that every CTA has work, plus a merge kernel for the cut
 *   tiles. Uncut tiles give the same bytes as the NULL launch; the rows of cut tiles are merged in
 *   fp32 and rounded to bf16 once. Size it with pkv_paged_prefill_workspace_bytes(SM count); its
 *   contents are scratch, overwritten per call.
 * Requirements: head_dim == 256; block_size a multiple of 8; q, caches and strides 16-byte
 * aligned; num_q_heads a multiple of num_kv_heads.
 */
PKV_API pkv_status pkv_paged_prefill_attn(const void* q, const void* k_cache, const void* v_cache,
                                  int64_t num_blocks, int64_t stride_blk, int64_t stride_tok,
                                  int64_t stride_head, const int32_t* block_table, int64_t bt_stride,
                                  int32_t max_blocks, const int32_t* seq_lens,
                                  const int32_t* query_start_loc, int32_t num_reqs, int32_t total_q,
                                  int32_t max_q_len, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t block_size, float softmax_scale,
                                  int32_t qk_mode, const int8_t* k8, const float* k8_scale,
                                  const void* k16, int64_t max_ctx, void* out, void* workspace,
                                  int64_t workspace_bytes, int32_t* dev_err, void* stream);

/*
 * paged_prefill_workspace_bytes - bytes of the persistent prefill workspace for num_ctas CTAs
 * (four slots per CTA of 128 x 256 fp32 partial outputs and 128 fp32 log-sum-exps: 526,336 bytes
 * per CTA); 0 for num_ctas <= 0. Pass the device's SM count for a full persistent grid.
 */
PKV_API size_t pkv_paged_prefill_workspace_bytes(int32_t num_ctas);

/*
 * spec_verify_attn_partial - speculative-decode verify attention over an int8 per-token-head
 * cache, as split-KV partials [P91: _spec_attn_partial; scales read via the same blk].
 *
 * Every request has T query tokens (rows r*T .. r*T+T-1 of q, bf16 [num_reqs*T][num_q_heads]
 * [head_dim]); seq_lens[r] counts the cached prefix plus these T tokens, and query token t sits
 * at position seq_lens[r] - T + t. Keys and values are int8 codes times fp32 per-token-head
 * scales: k = k_cache[...] * k_scale[blk*scale_stride_blk + slot*scale_stride_tok + h], same for v.
 * Split s of request r covers key positions [s*split_tokens, min((s+1)*split_tokens, seq_len));
 * request r has ceil(seq_lens[r] / split_tokens) <= max_splits splits. For each split and row:
 *   part_o[s][row][qh][:] = sum_j w_j v_j / sum_j w_j,  part_lse[s][row][qh] = m + ln(sum_j w_j),
 *   w_j = exp(s_j - m) over the split's keys the row can see, s_j = softmax_scale * q . k_j;
 *   a split with no visible key gives part_lse = -inf and part_o = 0.
 * part_o fp32 [max_splits][num_reqs*T][num_q_heads][head_dim], part_lse fp32
 * [max_splits][num_reqs*T][num_q_heads]: caller-allocated, pkv_spec_verify_workspace_bytes()
 * bytes in total (part_o first, part_lse right after, each 256-byte aligned when carved from
 * one allocation). split_tokens must be a positive multiple of 128.
 * Requirements: head_dim == 256; group = num_q_heads / num_kv_heads <= 32. A CTA serves 32 query
 * columns: floor(32 / group) tokens x group heads (the pages' 8 tokens x 4 heads fill it exactly; a
 * one-token decode step runs with padding columns), or 48 when that needs fewer CTAs per key range
 * (e.g. 24/4 heads with T = 8: one CTA instead of two); otherwise the tokens are spread over
 * adjacent CTAs that read the same keys. block_size a multiple
 * of 8; q, caches and cache strides 16-byte aligned; scale pools 4-byte aligned with
 * scale_stride_tok >= num_kv_heads (head stride 1). Keys in a
 * block whose id is out of range read as zero (k = v = 0) and PKV_ERR_DEVICE_BOUNDS is recorded.
 */
PKV_API size_t pkv_spec_verify_workspace_bytes(int32_t num_tokens, int32_t num_q_heads, int32_t head_dim,
                                       int32_t max_splits);
/*
 * spec_verify_pick_split - host-side planning for pkv_spec_verify_attn_partial: the split_tokens (a
 * multiple of 512 from 1,024 to 16,384) for which a model of the launch predicts the shortest
 * time, given the batch's seq_lens in HOST memory (num_reqs of them), T, the head counts and the
 * device's SM count. The model: the CTAs run longest first, one per SM; each costs a fixed time
 * plus a time per 128-key tile, each CTA past a request's keys a small fixed time (constants
 * measured on GB300); the result is the makespan of that list schedule. Larger splits mean fewer
 * partials and empty CTAs, smaller ones a finer balance over the SMs. Reads nothing on the device.
 * Returns 0 on a bad argument (null pointer, non-positive count, num_q_heads not a multiple of
 * num_kv_heads, group above 32).
 */
PKV_API int32_t pkv_spec_verify_pick_split(const int32_t* seq_lens, int32_t num_reqs, int32_t T,
                                           int32_t num_q_heads, int32_t num_kv_heads, int32_t num_sms);
PKV_API pkv_status pkv_spec_verify_attn_partial(const void* q, const int8_t* k_cache, const int8_t* v_cache,
                                        const float* k_scale, const float* v_scale,
                                        int64_t num_blocks, int64_t stride_blk, int64_t stride_tok,
                                        int64_t stride_head, int64_t scale_stride_blk,
                                        int64_t scale_stride_tok, const int32_t* block_table,
                                        int64_t bt_stride, int32_t max_blocks,
                                        const int32_t* seq_lens, int32_t num_reqs, int32_t T,
                                        int32_t num_q_heads, int32_t num_kv_heads,
                                        int32_t head_dim, int32_t block_size,
                                        float softmax_scale, int32_t split_tokens,
                                        int32_t max_splits, float* part_o, float* part_lse,
                                        int32_t* dev_err, void* stream);

/*
 * spec_verify_attn_partial_fp8 - the same split-KV verify over a per-tensor fp8 e4m3 cache
 * [P91: the fp8 arm of the big-pool verify test ("k_descale" argument) and the split-KV verify on
 * the per-tensor fp8 KV cache that the review names].
 * k = float(e4m3(k_fp8[...])) * (*k_descale), v = float(e4m3(v_fp8[...])) * (*v_descale), one
 * descale per tensor (device scalars); everything else (layouts, splits, partials, requirements
 * other than the scale arrays) as pkv_spec_verify_attn_partial; merge with pkv_spec_verify_combine.
 */
PKV_API pkv_status pkv_spec_verify_attn_partial_fp8(const void* q, const uint8_t* k_fp8, const uint8_t* v_fp8,
                                                    const float* k_descale, const float* v_descale,
                                                    int64_t num_blocks, int64_t stride_blk, int64_t stride_tok,
                                                    int64_t stride_head, const int32_t* block_table,
                                                    int64_t bt_stride, int32_t max_blocks,
                                                    const int32_t* seq_lens, int32_t num_reqs, int32_t T,
                                                    int32_t num_q_heads, int32_t num_kv_heads,
                                                    int32_t head_dim, int32_t block_size, float softmax_scale,
                                                    int32_t split_tokens, int32_t max_splits, float* part_o,
                                                    float* part_lse, int32_t* dev_err, void* stream);

/*
 * spec_verify_combine - log-sum-exp merge of the split-KV partials [P91, split-KV verify].
 *   LSE = ln sum_s exp(part_lse[s]);  out = sum_s exp(part_lse[s] - LSE) part_o[s]
 * over the ceil(seq_lens[r] / split_tokens) splits of each request; out bf16
 * [num_reqs*T][num_q_heads][head_dim].
 */
PKV_API pkv_status pkv_spec_verify_combine(const float* part_o, const float* part_lse,
                                   const int32_t* seq_lens, int32_t num_reqs, int32_t T,
                                   int32_t num_q_heads, int32_t head_dim, int32_t split_tokens,
                                   int32_t max_splits, void* out, void* stream);

/*
 * kv_cache_write - store a chunk's new K and V rows into the paged cache through the block table
 * [P109 item 1 and P91 kernel excerpt: block id widened to int64 before the stride product, the
 * int8 scales addressed by the same block id; P91 review: the int8-per-token-head and per-tensor
 * fp8 cache formats]. The pages do not print the writer; it is the step that fills the caches the
 * other calls read.
 *   k_new, v_new  bf16 [total_q][num_kv_heads][head_dim]; token t at k_new + t*new_stride_tok
 *                 (elements; >= num_kv_heads*head_dim, a multiple of 8), heads contiguous.
 *   Row t of request r (query_start_loc[r] <= t < query_start_loc[r+1]) goes to position
 *   seq_lens[r] - q_len + (t - query_start_loc[r]) with q_len = query_start_loc[r+1] -
 *   query_start_loc[r] (the attention calls' chunk convention), i.e. block
 *   block_table[r*bt_stride + pos/block_size], slot pos % block_size.
 *   kv_dtype PKV_KV_BF16: the row is copied. PKV_KV_INT8: codes = clamp(rint(x * (127/absmax)),
 *   -127, 127) and scale = absmax/127 (fp32 divides, ties to even; an all-zero row stores scale 0
 *   and zero codes, a row holding a NaN a NaN scale and zero codes) into the int8 caches and
 *   k_scale_cache / v_scale_cache [num_blocks][block_size][num_kv_heads] fp32 (element offset
 *   blk*scale_stride_blk + slot*scale_stride_tok + h). PKV_KV_FP8: code = e4m3(x / scale) with
 *   one fp32 divide, round to nearest even, magnitudes past 448 (infinity included) stored as
 *   +-448, NaN as a NaN code; k_scale / v_scale are device pointers to one fp32 each.
 *   Caches: element strides as for the other calls (elements of the cache dtype); bases 16-byte
 *   aligned, strides multiples of 8 elements. Scale pointers of the unused formats may be NULL.
 *   max_q_len >= every request's q_len (sizes the grid). Rows whose table entry is outside
 *   [0, num_blocks) or past max_blocks, and every row of a request whose q_len > seq_len, are not
 *   written and set PKV_ERR_DEVICE_BOUNDS in dev_err. Slots not addressed by a new row are untouched.
 */
PKV_API pkv_status pkv_kv_cache_write(const void* k_new, const void* v_new, int64_t new_stride_tok,
                                      const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                                      const int32_t* seq_lens, const int32_t* query_start_loc,
                                      int32_t num_reqs, int32_t max_q_len, int32_t kv_dtype, void* k_cache,
                                      void* v_cache, int64_t num_blocks, int64_t stride_blk,
                                      int64_t stride_tok, int64_t stride_head, float* k_scale_cache,
                                      float* v_scale_cache, int64_t scale_stride_blk,
                                      int64_t scale_stride_tok, const float* k_scale, const float* v_scale,
                                      int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t* dev_err, void* stream);

/*
 * paged_prefill_attn_fp8 - chunked causal prefill attention read straight from a per-tensor fp8
 * e4m3 paged cache, each K/V tile dequantized in shared memory [P3360 "What changed": the
 * alternative it measured against - dequantizing per read instead of once per layer into a dense
 * scratch; here both paths exist so that they can be measured against each other on GB300].
 *   k = bf16_rn(fp32(e4m3(k_fp8[...])) * (*k_scale)), the same for v - bit for bit the values
 *   pkv_kv_fp8_dequant_dense writes - then exactly the attention of pkv_paged_prefill_attn with
 *   qk_mode PKV_QK_BF16 (same chunk convention, causal mask and GQA map), out bf16
 *   [total_q][num_q_heads][head_dim].
 * k_fp8 / v_fp8: uint8 e4m3 pools [num_blocks][block_size][num_kv_heads][head_dim] with element
 * strides (16-byte aligned); k_scale / v_scale: device pointers to one fp32 each. Keys past
 * seq_len or in a block whose id is out of range read as zero (PKV_ERR_DEVICE_BOUNDS for the
 * latter). workspace / workspace_bytes: as pkv_paged_prefill_attn (NULL: one CTA per query tile;
 * given: the persistent grid). Requirements as pkv_paged_prefill_attn (head_dim == 256).
 */
PKV_API pkv_status pkv_paged_prefill_attn_fp8(const void* q, const uint8_t* k_fp8, const uint8_t* v_fp8,
                                              const float* k_scale, const float* v_scale, int64_t num_blocks,
                                              int64_t stride_blk, int64_t stride_tok, int64_t stride_head,
                                              const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                                              const int32_t* seq_lens, const int32_t* query_start_loc,
                                              int32_t num_reqs, int32_t total_q, int32_t max_q_len,
                                              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                              int32_t block_size, float softmax_scale, void* out,
                                              void* workspace, int64_t workspace_bytes, int32_t* dev_err,
                                              void* stream);

/*
 * spec_verify_attn_noalloc - pkv_spec_verify_attn_partial followed by pkv_spec_verify_combine, with
 * the split partials kept in a fixed scratch array inside the library instead of a caller
 * workspace. The paper has no counterpart; it exists for callers that cannot allocate device
 * memory (a plugin whose host owns the device allocator, a path that must not allocate between
 * steps, a caller that can only pass inputs and outputs). It allocates nothing.
 * Limit: the partials need num_reqs*T*num_q_heads*max_splits*(head_dim+1)*4 bytes (plus
 * alignment), at most pkv_spec_verify_noalloc_capacity_bytes() (32 MiB); larger calls return
 * PKV_ERR_INVALID_ARG with a message - use fewer splits (larger split_tokens) or the workspace call.
 * The array is reserved on every GPU that loads the library until the process exits. Its device
 * address is looked up on the first call made on each device (with that device current), so make
 * that first call before any stream capture; the address is then kept for the life of the process,
 * so do not cudaDeviceReset a device after calling this on it. All calls on a device share the array and overwrite
 * it; calls that overlap on the GPU race on it. Each call writes every partial it reads.
 * Arguments, layouts and requirements are those of pkv_spec_verify_attn_partial, with out bf16
 * [num_reqs*T][num_q_heads][head_dim] as in pkv_spec_verify_combine.
 */
PKV_API size_t pkv_spec_verify_noalloc_capacity_bytes(void);
PKV_API pkv_status pkv_spec_verify_attn_noalloc(const void* q, const int8_t* k_cache, const int8_t* v_cache,
                                                const float* k_scale, const float* v_scale,
                                                int64_t num_blocks, int64_t stride_blk, int64_t stride_tok,
                                                int64_t stride_head, int64_t scale_stride_blk,
                                                int64_t scale_stride_tok, const int32_t* block_table,
                                                int64_t bt_stride, int32_t max_blocks,
                                                const int32_t* seq_lens, int32_t num_reqs, int32_t T,
                                                int32_t num_q_heads, int32_t num_kv_heads,
                                                int32_t head_dim, int32_t block_size, float softmax_scale,
                                                int32_t split_tokens, int32_t max_splits, void* out,
                                                int32_t* dev_err, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H_ */

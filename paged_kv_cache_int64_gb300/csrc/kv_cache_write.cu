// kv_cache_write.cu - pkv_kv_cache_write: store a chunk's new K/V rows into the paged cache through
// the block table, as bf16, as int8 per (token, head) with fp32 scales, or as per-tensor e4m3.
//
// HyperQwen PR #109 (description item 1) and PR #91 (the kernel excerpt): the block id loaded from
// the int32 table is widened to int64 before it multiplies the cache stride, and the int8
// per-token-head scales are addressed by the same block id. PR #91's review names the two
// quantized cache formats this writes: int8 per token and head ("int8_per_token_head") and fp8
// with a per-tensor descale.
//
// Row t of request r (query_start_loc[r] <= t < query_start_loc[r+1]) is the token at position
// seq_len[r] - q_len[r] + (t - query_start_loc[r]), the same chunk convention as the attention calls.
//
// HBM-bound, one pass: per (token, head) and tensor, 512 B read and 512 B (bf16), 256 B + 4 B (int8)
// or 256 B (e4m3) written. One warp per (token, head, tensor) row: 16 contiguous bytes per lane, four
// rows in flight per warp; the int8 absmax is reduced with warp shuffles.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "host_common.h"
#include "sm103.cuh"

namespace pkv {

namespace {

constexpr int kD = 256;
constexpr int kWarps = 8;
constexpr int kRowsPerIter = 4;

struct WriteArgs {
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  int64_t new_stride_tok;
  const int32_t* block_table;
  int64_t bt_stride;
  int32_t max_blocks;
  const int32_t* seq_lens;
  const int32_t* qsl;
  uint8_t* k_cache;  // byte pointers: the element size depends on the cache dtype
  uint8_t* v_cache;
  int64_t num_blocks, stride_blk, stride_tok, stride_head;  // in elements
  float* k_scale_cache;
  float* v_scale_cache;
  int64_t scale_stride_blk, scale_stride_tok;
  const float* k_scale;  // e4m3: per-tensor scales (device)
  const float* v_scale;
  int32_t block_size, num_kv_heads;
  int* dev_err;
};

// 8 bf16 values of one lane -> 8 int8 codes of the row's symmetric quantizer (absmax over the warp's
// 256 values): scale = absmax / 127, code = clamp(rint(x * (127 / absmax)), -127, 127); an all-zero
// row gives scale 0, a row holding a NaN a NaN scale and zero codes.
__device__ __forceinline__ uint2 quantize_lane(const float (&x)[8], float& scale) {
  float amax = 0.0f;
  bool nan = false;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    nan |= (x[i] != x[i]);
    amax = fmaxf(amax, fabsf(x[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  nan = __any_sync(0xffffffffu, nan);
  if (nan) {
    scale = __int_as_float(0x7fc00000);
    return make_uint2(0, 0);
  }
  if (amax == 0.0f) {
    scale = 0.0f;
    return make_uint2(0, 0);
  }
  scale = __fdiv_rn(amax, 127.0f);
  const float inv = __fdiv_rn(127.0f, amax);
  uint32_t b[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = max(-127, min(127, __float2int_rn(__fmul_rn(x[i], inv))));
    b[i] = (uint32_t)(c & 0xff);
  }
  return make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24), b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
}

// 8 values -> 8 e4m3 codes of x / s (fp32 divide, then round to nearest even with saturation to
// +-448, the hardware conversion).
__device__ __forceinline__ uint2 e4m3_lane(const float (&x)[8], float s) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 y = make_float2(__fdiv_rn(x[2 * i], s), __fdiv_rn(x[2 * i + 1], s));
    w[i] = (uint32_t)__nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
  }
  return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

// kDt: 0 bf16, 1 int8 per (token, head), 2 e4m3 per tensor.
template <int kDt>
__global__ void __launch_bounds__(kWarps * 32) kv_cache_write_kernel(const WriteArgs a) {
  const int r = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int q0 = __ldg(a.qsl + r);
  const int q_len = __ldg(a.qsl + r + 1) - q0;
  const int seq_len = __ldg(a.seq_lens + r);
  if (q_len <= 0) return;
  if (q_len > seq_len) {  // the chunk would start before position 0: nothing is written
    if (blockIdx.x == 0 && threadIdx.x == 0) record_error(a.dev_err, kErrDeviceBounds);
    return;
  }
  const int hkv = a.num_kv_heads;
  // rows ordered (token, head, tensor): the K and V rows of one (token, head) share a table entry
  const int64_t nrows = (int64_t)q_len * hkv * 2;
  const int64_t stride = (int64_t)gridDim.x * kWarps * kRowsPerIter;
  float ts[2] = {1.0f, 1.0f};
  if (kDt == 2) {
    ts[0] = __ldg(a.k_scale);
    ts[1] = __ldg(a.v_scale);
  }
  for (int64_t base = ((int64_t)blockIdx.x * kWarps + warp) * kRowsPerIter; base < nrows; base += stride) {
    uint4 raw[kRowsPerIter];
    int64_t off[kRowsPerIter], soff[kRowsPerIter];
#pragma unroll
    for (int u = 0; u < kRowsPerIter; ++u) {
      const int64_t row = base + u;
      raw[u] = make_uint4(0, 0, 0, 0);
      off[u] = -1;
      soff[u] = -1;
      if (row >= nrows) continue;
      const int which = (int)(row & 1);
      const int h = (int)((row >> 1) % hkv);
      const int i = (int)((row >> 1) / hkv);
      const int64_t pos = (int64_t)seq_len - q_len + i;
      const int64_t col = pos / a.block_size;
      const int64_t blk = col < a.max_blocks ? (int64_t)__ldg(a.block_table + (int64_t)r * a.bt_stride + col) : -1;
      if (blk < 0 || blk >= a.num_blocks) {
        if (lane == 0) record_error(a.dev_err, kErrDeviceBounds);
        continue;  // not written
      }
      const int64_t slot = pos % a.block_size;
      off[u] = blk * a.stride_blk + slot * a.stride_tok + (int64_t)h * a.stride_head;  // 64-bit product
      soff[u] = blk * a.scale_stride_blk + slot * a.scale_stride_tok + h;
      const __nv_bfloat16* src = (which ? a.v_new : a.k_new) + (int64_t)(q0 + i) * a.new_stride_tok + (int64_t)h * kD;
      raw[u] = __ldg(reinterpret_cast<const uint4*>(src) + lane);
    }
#pragma unroll
    for (int u = 0; u < kRowsPerIter; ++u) {
      const int64_t row = base + u;
      if (row >= nrows) break;  // warp-uniform
      if (off[u] < 0) continue;  // warp-uniform (one table entry per row)
      const int which = (int)(row & 1);
      uint8_t* cache = which ? a.v_cache : a.k_cache;
      if (kDt == 0) {
        reinterpret_cast<uint4*>(cache + off[u] * 2)[lane] = raw[u];
        continue;
      }
      const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&raw[u]);
      float x[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(v2[e]);
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
      }
      if (kDt == 1) {
        float scale;
        const uint2 codes = quantize_lane(x, scale);
        reinterpret_cast<uint2*>(cache + off[u])[lane] = codes;
        if (lane == 0) (which ? a.v_scale_cache : a.k_scale_cache)[soff[u]] = scale;
      } else {
        reinterpret_cast<uint2*>(cache + off[u])[lane] = e4m3_lane(x, ts[which]);
      }
    }
  }
}

}  // namespace

}  // namespace pkv

extern "C" pkv_status pkv_kv_cache_write(const void* k_new, const void* v_new, int64_t new_stride_tok,
                                         const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                                         const int32_t* seq_lens, const int32_t* query_start_loc, int32_t num_reqs,
                                         int32_t max_q_len, int32_t kv_dtype, void* k_cache, void* v_cache,
                                         int64_t num_blocks, int64_t stride_blk, int64_t stride_tok,
                                         int64_t stride_head, float* k_scale_cache, float* v_scale_cache,
                                         int64_t scale_stride_blk, int64_t scale_stride_tok, const float* k_scale,
                                         const float* v_scale, int32_t block_size, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t* dev_err, void* stream) {
  using namespace pkv;
  clear_error();
  PKV_UNSUP(head_dim == kD, "kv_cache_write: head_dim must be 256 (got %d)", head_dim);
  PKV_ARG(kv_dtype == PKV_KV_BF16 || kv_dtype == PKV_KV_INT8 || kv_dtype == PKV_KV_FP8,
          "kv_cache_write: unknown kv_dtype %d", kv_dtype);
  PKV_ARG(num_reqs >= 0 && max_q_len >= 0, "kv_cache_write: bad size argument");
  if (num_reqs == 0 || max_q_len == 0) return PKV_OK;  // nothing to do, nothing read
  PKV_ARG(k_new && v_new && block_table && seq_lens && query_start_loc && k_cache && v_cache,
          "kv_cache_write: null pointer argument");
  PKV_ARG(kv_dtype != PKV_KV_INT8 || (k_scale_cache && v_scale_cache),
          "kv_cache_write: the int8 cache needs k_scale_cache and v_scale_cache");
  PKV_ARG(kv_dtype != PKV_KV_FP8 || (k_scale && v_scale), "kv_cache_write: the e4m3 cache needs k_scale and v_scale");
  PKV_ARG(num_blocks > 0 && block_size > 0 && num_kv_heads > 0 && max_blocks > 0 && bt_stride >= max_blocks &&
              new_stride_tok >= (int64_t)num_kv_heads * kD,
          "kv_cache_write: bad size argument");
  PKV_ARG(stride_blk > 0 && stride_tok > 0 && stride_head > 0, "kv_cache_write: strides must be positive");
  PKV_ARG(kv_dtype != PKV_KV_INT8 || (scale_stride_blk > 0 && scale_stride_tok >= num_kv_heads),
          "kv_cache_write: bad scale strides");
  // a lane moves 8 elements: 16 bytes of a bf16 row, 8 bytes of an int8 / e4m3 row
  PKV_ARG(aligned16(k_new) && aligned16(v_new) && new_stride_tok % 8 == 0 && aligned16(k_cache) &&
              aligned16(v_cache) && stride_blk % 8 == 0 && stride_tok % 8 == 0 && stride_head % 8 == 0,
          "kv_cache_write: bases must be 16-byte aligned and strides multiples of 8 elements");

  WriteArgs a{static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new), new_stride_tok,
              block_table, bt_stride, max_blocks, seq_lens, query_start_loc,
              static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), num_blocks, stride_blk, stride_tok,
              stride_head, k_scale_cache, v_scale_cache, scale_stride_blk, scale_stride_tok, k_scale, v_scale,
              block_size, num_kv_heads, dev_err};
  const int64_t rows = (int64_t)max_q_len * num_kv_heads * 2;
  const int64_t per_cta = (int64_t)kWarps * kRowsPerIter;
  int64_t want = (rows + per_cta - 1) / per_cta;
  int64_t cap = (int64_t)num_sms() * 8;  // 8 resident CTAs of 256 threads per SM
  cap = (cap + num_reqs - 1) / num_reqs;
  if (cap < 1) cap = 1;
  dim3 grid((unsigned)(want < cap ? want : cap), (unsigned)num_reqs);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (kv_dtype == PKV_KV_BF16) kv_cache_write_kernel<0><<<grid, kWarps * 32, 0, st>>>(a);
  else if (kv_dtype == PKV_KV_INT8) kv_cache_write_kernel<1><<<grid, kWarps * 32, 0, st>>>(a);
  else kv_cache_write_kernel<2><<<grid, kWarps * 32, 0, st>>>(a);
  return check_launch("kv_cache_write");
}

// kv_int8_quant.cu - pkv_kv_int8_stats_quant: per-token-head symmetric int8 quantization of the
// bf16 K cache into a dense, position-indexed scratch.
//
// HyperQwen PR #109 (int8 prefill attention, prefill_attn_hd256.py): _k_stats_kernel computes
// per-token-head statistics of K read through blk = block_table[...] and _k_quant_kernel writes
// int8 K into a dense scratch indexed by position with one scale per (token, head); the block id
// is widened to int64 before it multiplies the cache stride (description item 1).
//
// Optionally the same codes are also written as fp16 values (exact) to a second scratch: the
// tensor cores of sm_103a have no int8 MMA, so the int8-QK prefill multiplies the codes as fp16;
// widening each K row once here serves the 64 query tiles that read it.
//
// One pass, HBM-bound: 512 B read + 256 B + 4 B written per (token, head) row (+ 512 B with the fp16
// copy). One warp per row,
// 16 contiguous bytes per lane (coalesced 512-byte row), the absmax reduced with warp shuffles,
// four rows in flight per warp.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "host_common.h"
#include "sm103.cuh"

namespace pkv {

namespace {

constexpr int kD = 256;
constexpr int kWarps = 8;
constexpr int kRowsPerIter = 4;

struct QuantArgs {
  const __nv_bfloat16* k_cache;
  int64_t num_blocks, stride_blk, stride_tok, stride_head;
  const int32_t* block_table;
  int64_t bt_stride;
  int32_t max_blocks;
  const int32_t* pos_begin;
  const int32_t* pos_end;
  int32_t block_size, num_kv_heads;
  int8_t* k8;
  float* k8_scale;
  __half* k16;  // optional fp16 copy of the codes
  int64_t max_ctx;
  int* dev_err;
};

// Element offset of K row (request r, position pos, head h), or -1 with an error recorded when
// the table entry is outside the pool. 64-bit throughout: blk * stride_blk can exceed 2^31.
__device__ __forceinline__ int64_t row_offset(const QuantArgs& a, int r, int64_t pos, int h) {
  const int64_t col = pos / a.block_size;
  if (col >= a.max_blocks) {
    record_error(a.dev_err, kErrDeviceBounds);
    return -1;
  }
  const int64_t blk = (int64_t)__ldg(a.block_table + (int64_t)r * a.bt_stride + col);
  if (blk < 0 || blk >= a.num_blocks) {
    record_error(a.dev_err, kErrDeviceBounds);
    return -1;
  }
  return blk * a.stride_blk + (pos % a.block_size) * a.stride_tok + (int64_t)h * a.stride_head;
}

__global__ void __launch_bounds__(kWarps * 32) kv_int8_stats_quant_kernel(const QuantArgs a) {
  const int r = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t p0 = __ldg(a.pos_begin + r);
  const int64_t p1 = __ldg(a.pos_end + r);
  const int64_t nrows = (p1 - p0) * a.num_kv_heads;
  const int64_t stride = (int64_t)gridDim.x * kWarps * kRowsPerIter;
  for (int64_t base = ((int64_t)blockIdx.x * kWarps + warp) * kRowsPerIter; base < nrows; base += stride) {
    uint4 raw[kRowsPerIter];
#pragma unroll
    for (int u = 0; u < kRowsPerIter; ++u) {
      const int64_t row = base + u;
      raw[u] = make_uint4(0, 0, 0, 0);
      if (row < nrows) {
        const int64_t pos = p0 + row / a.num_kv_heads;
        const int h = (int)(row % a.num_kv_heads);
        const int64_t off = row_offset(a, r, pos, h);
        if (off >= 0) raw[u] = __ldg(reinterpret_cast<const uint4*>(a.k_cache + off) + lane);
      }
    }
#pragma unroll
    for (int u = 0; u < kRowsPerIter; ++u) {
      const int64_t row = base + u;
      if (row >= nrows) break;  // warp-uniform
      const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&raw[u]);
      float x[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(v2[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
      }
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
      float scale;
      uint32_t lo = 0, hi = 0;
      uint4 wide = make_uint4(0, 0, 0, 0);
      if (nan) {
        scale = __int_as_float(0x7fc00000);  // a NaN row: NaN scale, zero codes
      } else if (amax == 0.0f) {
        scale = 0.0f;
      } else {
        scale = __fdiv_rn(amax, 127.0f);
        const float inv = __fdiv_rn(127.0f, amax);
        uint32_t b[8];
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          int c = __float2int_rn(__fmul_rn(x[i], inv));
          c = max(-127, min(127, c));
          b[i] = (uint32_t)(c & 0xff);
          const uint32_t hbits = __half_as_ushort(__int2half_rn(c));  // exact: |c| <= 127
          if (i & 1) w[i >> 1] |= hbits << 16; else w[i >> 1] = hbits;
        }
        wide = make_uint4(w[0], w[1], w[2], w[3]);
        lo = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
        hi = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
      }
      const int64_t pos = p0 + row / a.num_kv_heads;
      const int h = (int)(row % a.num_kv_heads);
      const int64_t o = ((int64_t)r * a.max_ctx + pos) * a.num_kv_heads + h;
      reinterpret_cast<uint2*>(a.k8 + o * kD)[lane] = make_uint2(lo, hi);
      if (a.k16) reinterpret_cast<uint4*>(a.k16 + o * kD)[lane] = wide;
      if (lane == 0) a.k8_scale[o] = scale;
    }
  }
}

}  // namespace

}  // namespace pkv

extern "C" pkv_status pkv_kv_int8_stats_quant(const void* k_cache, int64_t num_blocks, int64_t stride_blk,
                                              int64_t stride_tok, int64_t stride_head,
                                              const int32_t* block_table, int64_t bt_stride,
                                              int32_t max_blocks, const int32_t* pos_begin,
                                              const int32_t* pos_end, int32_t num_reqs, int32_t max_tokens,
                                              int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                              int8_t* k8, float* k8_scale, void* k16, int64_t max_ctx,
                                              int32_t* dev_err, void* stream) {
  using namespace pkv;
  clear_error();
  PKV_UNSUP(head_dim == kD, "kv_int8_stats_quant: head_dim must be 256 (got %d)", head_dim);
  PKV_ARG(k_cache && block_table && pos_begin && pos_end && k8 && k8_scale,
          "kv_int8_stats_quant: null pointer argument");
  PKV_ARG(num_reqs >= 0 && max_tokens >= 0 && num_blocks > 0 && block_size > 0 && num_kv_heads > 0 &&
              max_blocks > 0 && max_ctx > 0 && bt_stride >= max_blocks,
          "kv_int8_stats_quant: bad size argument");
  PKV_ARG(stride_blk > 0 && stride_tok > 0 && stride_head > 0, "kv_int8_stats_quant: strides must be positive");
  PKV_ARG(aligned16(k_cache) && stride_blk % 8 == 0 && stride_tok % 8 == 0 && stride_head % 8 == 0,
          "kv_int8_stats_quant: k_cache rows must be 16-byte aligned");
  PKV_ARG(!k16 || aligned16(k16), "kv_int8_stats_quant: k16 must be 16-byte aligned");
  if (num_reqs == 0 || max_tokens == 0) return PKV_OK;
  QuantArgs a{static_cast<const __nv_bfloat16*>(k_cache), num_blocks, stride_blk, stride_tok, stride_head,
              block_table, bt_stride, max_blocks, pos_begin, pos_end, block_size, num_kv_heads,
              k8, k8_scale, static_cast<__half*>(k16), max_ctx, dev_err};
  const int64_t rows = (int64_t)max_tokens * num_kv_heads;
  const int64_t per_cta = (int64_t)kWarps * kRowsPerIter;
  int64_t want = (rows + per_cta - 1) / per_cta;
  int64_t cap = (int64_t)num_sms() * 8;  // 8 resident CTAs of 256 threads per SM
  cap = (cap + num_reqs - 1) / num_reqs;
  if (cap < 1) cap = 1;
  dim3 grid((unsigned)(want < cap ? want : cap), (unsigned)num_reqs);
  kv_int8_stats_quant_kernel<<<grid, kWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return check_launch("kv_int8_stats_quant");
}

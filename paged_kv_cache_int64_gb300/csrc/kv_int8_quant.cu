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
// copy). CTAs of four warps (so a 2,048-token chunk of four heads spreads over 256 CTAs, past the
// SM count); row, position and slot arithmetic in 32 bits, once per row. A warp takes four
// consecutive rows at a time, eight lanes per row: lane l holds elements
// 32 (l % 8) .. +31 of row l / 8 (four 16-byte loads), the row's absmax is three shuffles among its
// eight lanes, and the lane stores its 32 codes as two 16-byte words (and their fp16 copy as four);
// the four rows' scales leave in one store instruction (lanes 0, 8, 16, 24: consecutive floats).
// Two such quads are in flight per warp (eight 16-byte loads per lane before the first use).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "host_common.h"
#include "sm103.cuh"

namespace pkv {

namespace {

constexpr int kD = 256;
constexpr int kWarps = 4;
constexpr int kQuads = 2;                   // quads of rows in flight per warp
constexpr int kRowsPerWarpIter = 4 * kQuads;

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
// the table entry is outside the pool. Positions and rows fit 32 bits (checked on the host), so the
// divisions are 32-bit; the offset is 64-bit throughout: blk * stride_blk can exceed 2^31.
__device__ __forceinline__ int64_t row_offset(const QuantArgs& a, int r, int pos, int h) {
  const int col = pos / a.block_size;
  if (col >= a.max_blocks) {
    record_error(a.dev_err, kErrDeviceBounds);
    return -1;
  }
  const int64_t blk = (int64_t)__ldg(a.block_table + (int64_t)r * a.bt_stride + col);
  if (blk < 0 || blk >= a.num_blocks) {
    record_error(a.dev_err, kErrDeviceBounds);
    return -1;
  }
  return blk * a.stride_blk + (int64_t)(pos - col * a.block_size) * a.stride_tok + (int64_t)h * a.stride_head;
}

__global__ void __launch_bounds__(kWarps * 32, 8) kv_int8_stats_quant_kernel(const QuantArgs a) {
  const int r = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int sub = lane >> 3;       // the lane's row within a quad
  const int part = lane & 7;       // its 32-element part of the row
  const int H = a.num_kv_heads;
  const int p0 = __ldg(a.pos_begin + r);
  const int p1 = __ldg(a.pos_end + r);
  if ((int64_t)(p1 - p0) * H >= (1ll << 31)) {  // rows beyond 32-bit indexing (the host checks max_tokens)
    if (threadIdx.x == 0) record_error(a.dev_err, kErrDeviceBounds);
    return;
  }
  const int nrows = (p1 - p0) * H;
  const int stride = (int)gridDim.x * kWarps * kRowsPerWarpIter;
  for (int base = ((int)blockIdx.x * kWarps + warp) * kRowsPerWarpIter; base < nrows; base += stride) {
    uint4 raw[kQuads][4];
    int pos_q[kQuads], h_q[kQuads];  // the lane's row of each quad: position and head
#pragma unroll
    for (int qd = 0; qd < kQuads; ++qd) {
      const int row = base + 4 * qd + sub;
      const int t = row / H;
      pos_q[qd] = p0 + t;
      h_q[qd] = row - t * H;
#pragma unroll
      for (int c = 0; c < 4; ++c) raw[qd][c] = make_uint4(0, 0, 0, 0);
      if (row < nrows) {
        const int64_t off = row_offset(a, r, pos_q[qd], h_q[qd]);
        if (off >= 0) {
          const uint4* src = reinterpret_cast<const uint4*>(a.k_cache + off) + 4 * part;
#pragma unroll
          for (int c = 0; c < 4; ++c) raw[qd][c] = __ldg(src + c);
        }
      }
    }
#pragma unroll
    for (int qd = 0; qd < kQuads; ++qd) {
      if (base + 4 * qd >= nrows) break;  // warp-uniform
      const bool live_row = base + 4 * qd + sub < nrows;
      // absmax of the lane's 32 elements on their bit patterns: a bf16 magnitude orders as its low
      // 15 bits, so a packed 16-bit maximum of (bits & 0x7fff) gives it, and a maximum above 0x7f80
      // (infinity) means a NaN is present
      uint32_t mx2 = 0u;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t w[4] = {raw[qd][c].x, raw[qd][c].y, raw[qd][c].z, raw[qd][c].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) mx2 = __vmaxu2(mx2, w[e] & 0x7fff7fffu);
      }
      uint32_t mx = max(mx2 & 0xffffu, mx2 >> 16);
      // the row's eight lanes: lanes 8s .. 8s + 7
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const bool nan = mx > 0x7f80u;
      const float amax = __uint_as_float(mx << 16);
      const bool live = !nan && amax > 0.0f;
      const float scale = nan ? __int_as_float(0x7fc00000) : (amax > 0.0f ? __fdiv_rn(amax, 127.0f) : 0.0f);
      const float inv = live ? __fdiv_rn(127.0f, amax) : 0.0f;  // a NaN or all-zero row: zero codes
      const bool inv_inf = isinf(inv);
      if (!live_row) continue;
      const int64_t o = ((int64_t)r * a.max_ctx + pos_q[qd]) * H + h_q[qd];
      uint4* d8 = reinterpret_cast<uint4*>(a.k8 + o * kD) + 2 * part;
      uint4* d16 = a.k16 ? reinterpret_cast<uint4*>(a.k16 + o * kD) + 4 * part : nullptr;
      // 8 elements per chunk: their codes (two words) and the codes as fp16 (four words), stored as
      // soon as a 16-byte word is whole.
      // Rounding. With inv finite and nonzero, |x| <= amax and inv = 127 / amax correctly rounded give
      // |p| = |x * inv| <= 127 (1 + 2^-23) < 127.5: rint(p) is already in [-127, 127] (the definition's
      // clamp never acts), and adding 1.5 * 2^23 to p (one correctly rounded add; |p| < 2^22) leaves
      // rint(p), ties to even, in the sum's low mantissa bits in two's complement - its low byte is
      // the code. Rows whose 127 / amax overflows (amax below ~3.7e-37) or vanishes (an infinite
      // element) take the conversion instruction and the clamp instead.
      const bool fast = live && !inv_inf && inv > 0.0f;
      uint32_t b_prev[2] = {0u, 0u};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t w[4] = {raw[qd][c].x, raw[qd][c].y, raw[qd][c].z, raw[qd][c].w};
        uint32_t bw[2];
        if (fast) {
          constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
          uint32_t y[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            y[2 * e] = __float_as_uint(__fadd_rn(__fmul_rn(__uint_as_float(w[e] << 16), inv), kMagic));
            y[2 * e + 1] = __float_as_uint(__fadd_rn(__fmul_rn(__uint_as_float(w[e] & 0xffff0000u), inv), kMagic));
          }
#pragma unroll
          for (int k = 0; k < 2; ++k)
            bw[k] = __byte_perm(__byte_perm(y[4 * k], y[4 * k + 1], 0x0040), __byte_perm(y[4 * k + 2], y[4 * k + 3], 0x0040),
                                0x5410);
        } else {
          bw[0] = bw[1] = 0u;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            int c0 = 0, c1 = 0;
            if (live) {
              c0 = max(-127, min(127, __float2int_rn(__fmul_rn(__uint_as_float(w[e] << 16), inv))));
              c1 = max(-127, min(127, __float2int_rn(__fmul_rn(__uint_as_float(w[e] & 0xffff0000u), inv))));
            }
            bw[e >> 1] |= ((uint32_t)(c0 & 0xff) | ((uint32_t)(c1 & 0xff) << 8)) << (16 * (e & 1));
          }
        }
        if (d16) {
          // codes -> fp16 integers, exact: bytes (b ^ 0x80) under the fp16 exponent of 1024 give
          // 1024 + b + 128, and one fp16 subtraction of 1152 leaves b
          uint32_t hw[4];
          const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const uint32_t u = bw[k] ^ 0x80808080u;
            uint32_t lo = __byte_perm(u, 0x64646464u, 0x5140), hi = __byte_perm(u, 0x64646464u, 0x7362);
            const __half2 hl = __hsub2(*reinterpret_cast<__half2*>(&lo), bias);
            const __half2 hh = __hsub2(*reinterpret_cast<__half2*>(&hi), bias);
            hw[2 * k] = *reinterpret_cast<const uint32_t*>(&hl);
            hw[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&hh);
          }
          d16[c] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        }
        if (c & 1) d8[c >> 1] = make_uint4(b_prev[0], b_prev[1], bw[0], bw[1]);
        else {
          b_prev[0] = bw[0];
          b_prev[1] = bw[1];
        }
      }
      if (part == 0) a.k8_scale[o] = scale;
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
  PKV_UNSUP((int64_t)max_tokens * num_kv_heads < (1ll << 31) && max_ctx < (1ll << 31),
            "kv_int8_stats_quant: more than 2^31 rows in one call");
  if (num_reqs == 0 || max_tokens == 0) return PKV_OK;
  QuantArgs a{static_cast<const __nv_bfloat16*>(k_cache), num_blocks, stride_blk, stride_tok, stride_head,
              block_table, bt_stride, max_blocks, pos_begin, pos_end, block_size, num_kv_heads,
              k8, k8_scale, static_cast<__half*>(k16), max_ctx, dev_err};
  const int64_t rows = (int64_t)max_tokens * num_kv_heads;
  const int64_t per_cta = (int64_t)kWarps * kRowsPerWarpIter;
  int64_t want = (rows + per_cta - 1) / per_cta;
  // one 32-row slice of the range per CTA: the block scheduler balances the tail (the loop
  // strides only past 2^31 - 1 CTAs)
  const int64_t cap = (1ll << 31) - 1;
  dim3 grid((unsigned)(want < cap ? want : cap), (unsigned)num_reqs);
  kv_int8_stats_quant_kernel<<<grid, kWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return check_launch("kv_int8_stats_quant");
}

// kv_fp8_dequant.cu - pkv_kv_fp8_dequant_dense: per-tensor fp8 e4m3 K/V cache -> dense bf16
// scratch, once per layer.
//
// vllm.cpp PR #3360, "What changed": the fp8 cache is dequantized once per layer into a dense
// bf16 scratch holding one block per request (block_size = max_seq, identity block table), so the
// ordinary bf16 attention runs on it unchanged.
//
// One streaming pass, HBM-bound: 1 B read + 2 B written per element for K and for V. Each thread
// converts 16 e4m3 bytes per step with the hardware conversion (e4m3x2 -> f16x2, exact), widens
// to fp32, multiplies by the per-tensor scale (fp32, round to nearest) and rounds the product to
// bf16 (round to nearest even): bit-identical to the definition.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "host_common.h"
#include "sm103.cuh"

namespace pkv {

namespace {

constexpr int kThreads = 256;
constexpr int kChunksPerThread = 4;  // 16-byte chunks in flight per thread

struct DequantArgs {
  const uint8_t* src[2];
  __nv_bfloat16* dst[2];
  const float* scale[2];
  int64_t num_blocks, stride_blk, stride_tok, stride_head;
  const int32_t* block_table;
  int64_t bt_stride;
  int32_t max_blocks;
  const int32_t* seq_lens;
  int32_t max_seq, block_size, num_kv_heads, head_dim;
  int* dev_err;
};

__global__ void __launch_bounds__(kThreads) kv_fp8_dequant_dense_kernel(const DequantArgs a) {
  const int r = blockIdx.y;
  const int64_t L = __ldg(a.seq_lens + r);
  const int chunks_per_row = a.head_dim / 16;                       // 16 codes per chunk
  const int64_t per_tok = (int64_t)a.num_kv_heads * chunks_per_row;  // chunks per token
  const int64_t n = 2 * L * per_tok;                                 // K then V
  const float sk = __ldg(a.scale[0]), sv = __ldg(a.scale[1]);
  const int64_t stride = (int64_t)gridDim.x * kThreads * kChunksPerThread;
  for (int64_t base = (int64_t)blockIdx.x * kThreads * kChunksPerThread + threadIdx.x; base < n;
       base += stride) {
    uint4 raw[kChunksPerThread];
    int64_t dsto[kChunksPerThread];
#pragma unroll
    for (int u = 0; u < kChunksPerThread; ++u) {
      const int64_t i = base + (int64_t)u * kThreads;
      raw[u] = make_uint4(0, 0, 0, 0);
      dsto[u] = -1;
      if (i < n) {
        const int which = i >= L * per_tok;
        const int64_t j = which ? i - L * per_tok : i;
        const int64_t pos = j / per_tok;
        const int64_t rem = j % per_tok;
        const int h = (int)(rem / chunks_per_row);
        const int c = (int)(rem % chunks_per_row);
        dsto[u] = ((((int64_t)r * a.max_seq + pos) * a.num_kv_heads + h) * a.head_dim + c * 16) |
                  ((int64_t)which << 62);
        const int64_t col = pos / a.block_size;
        const int64_t blk = col < a.max_blocks ? (int64_t)__ldg(a.block_table + (int64_t)r * a.bt_stride + col) : -1;
        if (blk < 0 || blk >= a.num_blocks) {
          record_error(a.dev_err, kErrDeviceBounds);
        } else {
          const int64_t off = blk * a.stride_blk + (pos % a.block_size) * a.stride_tok +
                              (int64_t)h * a.stride_head + c * 16;
          raw[u] = __ldg(reinterpret_cast<const uint4*>(a.src[which] + off));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kChunksPerThread; ++u) {
      if (dsto[u] < 0) continue;
      const int which = (int)(dsto[u] >> 62);
      const int64_t o = dsto[u] & ((1ll << 62) - 1);
      uint4 hi;
      const uint4 lo = dequant16_e4m3_bf16(raw[u], which ? sv : sk, hi);
      uint4* dst = reinterpret_cast<uint4*>(a.dst[which] + o);
      dst[0] = lo;
      dst[1] = hi;
    }
  }
}

}  // namespace

}  // namespace pkv

extern "C" pkv_status pkv_kv_fp8_dequant_dense(const uint8_t* k_fp8, const uint8_t* v_fp8, int64_t num_blocks,
                                               int64_t stride_blk, int64_t stride_tok, int64_t stride_head,
                                               const int32_t* block_table, int64_t bt_stride,
                                               int32_t max_blocks, const int32_t* seq_lens, int32_t num_reqs,
                                               int32_t max_seq, int32_t block_size, int32_t num_kv_heads,
                                               int32_t head_dim, const float* k_scale, const float* v_scale,
                                               void* k_dense, void* v_dense, int32_t* dev_err, void* stream) {
  using namespace pkv;
  clear_error();
  PKV_UNSUP(head_dim == 256, "kv_fp8_dequant_dense: head_dim must be 256 (got %d)", head_dim);
  PKV_ARG(k_fp8 && v_fp8 && block_table && seq_lens && k_scale && v_scale && k_dense && v_dense,
          "kv_fp8_dequant_dense: null pointer argument");
  PKV_ARG(num_reqs >= 0 && max_seq > 0 && num_blocks > 0 && block_size > 0 && num_kv_heads > 0 &&
              max_blocks > 0 && bt_stride >= max_blocks,
          "kv_fp8_dequant_dense: bad size argument");
  PKV_ARG(stride_blk > 0 && stride_tok > 0 && stride_head > 0, "kv_fp8_dequant_dense: strides must be positive");
  PKV_ARG(aligned16(k_fp8) && aligned16(v_fp8) && aligned16(k_dense) && aligned16(v_dense) &&
              stride_blk % 16 == 0 && stride_tok % 16 == 0 && stride_head % 16 == 0,
          "kv_fp8_dequant_dense: caches and strides must be 16-byte aligned");
  if (num_reqs == 0) return PKV_OK;
  DequantArgs a{{k_fp8, v_fp8},
                {static_cast<__nv_bfloat16*>(k_dense), static_cast<__nv_bfloat16*>(v_dense)},
                {k_scale, v_scale},
                num_blocks, stride_blk, stride_tok, stride_head, block_table, bt_stride, max_blocks, seq_lens,
                max_seq, block_size, num_kv_heads, head_dim, dev_err};
  const int64_t chunks = 2ll * max_seq * num_kv_heads * (head_dim / 16);
  const int64_t per_cta = (int64_t)kThreads * kChunksPerThread;
  int64_t want = (chunks + per_cta - 1) / per_cta;
  int64_t cap = ((int64_t)num_sms() * 8 + num_reqs - 1) / num_reqs;
  if (cap < 1) cap = 1;
  dim3 grid((unsigned)(want < cap ? want : cap), (unsigned)num_reqs);
  kv_fp8_dequant_dense_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return check_launch("kv_fp8_dequant_dense");
}

// kv_fp8_dequant.cu - pkv_kv_fp8_dequant_dense: per-tensor fp8 e4m3 K/V cache -> dense bf16
// scratch, once per layer.
//
// vllm.cpp PR #3360, "What changed": the fp8 cache is dequantized once per layer into a dense
// bf16 scratch holding one block per request (block_size = max_seq, identity block table), so the
// ordinary bf16 attention runs on it unchanged.
//
// One streaming pass, HBM-bound: 1 B read + 2 B written per element for K and for V. One warp per
// (request, position) at a time: lanes 0-15 take K, lanes 16-31 V, lane q the 16 codes at bytes
// 16q .. 16q + 15 of every head's row, so each half-warp reads the token's Hkv x 256 codes as
// coalesced 256-byte rows and writes them as 512-byte bf16 rows. The block id and slot are found
// once per position; each warp keeps two positions (2 Hkv 16-byte loads a lane) in flight. A code
// converts with the hardware conversion (e4m3x2 -> f16x2, exact), widens to fp32, is multiplied by
// the per-tensor scale (fp32, round to nearest) and rounded to bf16 (round to nearest even):
// bit-identical to the definition.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "host_common.h"
#include "sm103.cuh"

namespace pkv {

namespace {

constexpr int kThreads = 256;
constexpr int kMaxHeads = 4;  // kv heads handled per lane step (more heads loop)
constexpr int kPosPerWarp = 2;

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
  const int L = __ldg(a.seq_lens + r);
  const int lane = threadIdx.x & 31;
  const int which = lane >> 4;  // 0: K, 1: V
  const int q = lane & 15;      // 16-byte column chunk of every head's row
  const uint8_t* src = a.src[which];
  __nv_bfloat16* dst = a.dst[which];
  const float sc = __ldg(a.scale[which]);
  const int H = a.num_kv_heads;
  const int nw = (int)((gridDim.x * (unsigned)kThreads) >> 5);
  for (int pos0 = (int)((blockIdx.x * (unsigned)kThreads + threadIdx.x) >> 5); pos0 < L; pos0 += kPosPerWarp * nw) {
    for (int h0 = 0; h0 < H; h0 += kMaxHeads) {
      const int nh = min(kMaxHeads, H - h0);
      uint4 raw[kPosPerWarp][kMaxHeads];
      bool live[kPosPerWarp];
#pragma unroll
      for (int u = 0; u < kPosPerWarp; ++u) {
        const int pos = pos0 + u * nw;
        live[u] = pos < L;
        int64_t base = -1;
        if (live[u]) {
          const int col = pos / a.block_size;
          const int slot = pos - col * a.block_size;
          const int64_t blk = col < a.max_blocks ? (int64_t)__ldg(a.block_table + (int64_t)r * a.bt_stride + col) : -1;
          if (blk < 0 || blk >= a.num_blocks) {
            if (lane == 0) record_error(a.dev_err, kErrDeviceBounds);
          } else {
            base = blk * a.stride_blk + (int64_t)slot * a.stride_tok + (int64_t)h0 * a.stride_head + q * 16;
          }
        }
#pragma unroll
        for (int t = 0; t < kMaxHeads; ++t) {
          raw[u][t] = make_uint4(0, 0, 0, 0);  // a bad block reads as zero codes, written as zeros
          if (base >= 0 && t < nh) raw[u][t] = __ldg(reinterpret_cast<const uint4*>(src + base + (int64_t)t * a.stride_head));
        }
      }
#pragma unroll
      for (int u = 0; u < kPosPerWarp; ++u) {
        if (!live[u]) continue;
        const int64_t row0 = ((int64_t)r * a.max_seq + pos0 + u * nw) * H + h0;
#pragma unroll
        for (int t = 0; t < kMaxHeads; ++t) {
          if (t >= nh) continue;
          uint4 hi;
          const uint4 lo = dequant16_e4m3_bf16(raw[u][t], sc, hi);
          uint4* d = reinterpret_cast<uint4*>(dst + (row0 + t) * a.head_dim + q * 16);
          d[0] = lo;
          d[1] = hi;
        }
      }
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
  // one warp per position: a CTA per 8 positions of max_seq (CTAs past a request's seq_len leave at
  // once; the block scheduler balances the tail). Each warp then takes positions w and w + nw.
  const int64_t warps_per_cta = kThreads / 32;
  const int64_t want = ((int64_t)max_seq + kPosPerWarp * warps_per_cta - 1) / (kPosPerWarp * warps_per_cta);
  dim3 grid((unsigned)want, (unsigned)num_reqs);
  kv_fp8_dequant_dense_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return check_launch("kv_fp8_dequant_dense");
}

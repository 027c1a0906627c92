// spec_verify_combine.cu - pkv_spec_verify_combine: log-sum-exp merge of split-KV partials.
//
// HyperQwen PR #91 / split-KV verify: each split of a request's key range yields a normalised
// partial output o_s and its log-sum-exp lse_s; the full result is
// sum_s exp(lse_s - LSE) o_s with LSE = ln sum_s exp(lse_s).
//
// One warp per (query row, head): the lanes reduce the split LSEs, then each lane merges 8 of the
// 256 output elements (two 16-byte loads per split) and writes 16 bytes of bf16. With at most 32
// splits, lane s holds split s's weight, so the partials' loads need no LSE load before them.
#include <cuda_bf16.h>

#include "host_common.h"
#include "sm103.cuh"

namespace pkv {

namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32)
    spec_verify_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                               const int32_t* __restrict__ seq_lens, int32_t T, int32_t num_q_heads,
                               int32_t head_dim, int32_t split_tokens, int32_t max_splits, int64_t rows,
                               __nv_bfloat16* __restrict__ out) {
  // launched as a programmatic dependent: wait until the previous kernel in the stream (the
  // partials' launch) has completed and its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);  // (token, head)
  if (row >= rows) return;
  const int64_t tok = row / num_q_heads;
  const int r = (int)(tok / T);
  const int64_t L = __ldg(seq_lens + r);
  int ns = (int)((L + split_tokens - 1) / split_tokens);
  ns = min(ns, max_splits);
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  auto add = [&](int s, float w) {  // w == 0: a split with no visible key (its partial is not read)
    const float4* src = reinterpret_cast<const float4*>(part_o + ((int64_t)s * rows + row) * head_dim) + lane * 2;
    const float4 a = __ldg(src), b = __ldg(src + 1);
    if (w != 0.0f) {
      acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
      acc[4] += w * b.x; acc[5] += w * b.y; acc[6] += w * b.z; acc[7] += w * b.w;
    }
  };
  if (ns <= 32) {
    // lane s holds split s's LSE and, after the two reductions, its weight; the partials' loads
    // then carry no dependence on an LSE load and run eight splits at a time (a row of the longest
    // request has ~20 splits: three memory round trips)
    const float l = lane < ns ? __ldg(part_lse + (int64_t)lane * rows + row) : -INFINITY;
    float m = l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float e = (m == -INFINITY || l == -INFINITY) ? 0.0f : expf(l - m);
    float sum = e;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float w_lane = sum > 0.0f ? e * (1.0f / sum) : 0.0f;
#pragma unroll 8
    for (int s = 0; s < ns; ++s) add(s, __shfl_sync(0xffffffffu, w_lane, s));
  } else {
    float m = -INFINITY;
    for (int s = lane; s < ns; s += 32) m = fmaxf(m, __ldg(part_lse + (int64_t)s * rows + row));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float sum = 0.0f;
    if (m != -INFINITY) {
      for (int s = lane; s < ns; s += 32) {
        const float l = __ldg(part_lse + (int64_t)s * rows + row);
        sum += (l == -INFINITY) ? 0.0f : expf(l - m);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (m != -INFINITY && sum > 0.0f) {
      const float inv = 1.0f / sum;
      for (int s = 0; s < ns; ++s) {
        const float l = __ldg(part_lse + (int64_t)s * rows + row);
        add(s, l == -INFINITY ? 0.0f : expf(l - m) * inv);
      }
    }
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  reinterpret_cast<uint4*>(out + row * head_dim)[lane] = o;
}

}  // namespace

}  // namespace pkv

extern "C" pkv_status pkv_spec_verify_combine(const float* part_o, const float* part_lse, const int32_t* seq_lens,
                                              int32_t num_reqs, int32_t T, int32_t num_q_heads, int32_t head_dim,
                                              int32_t split_tokens, int32_t max_splits, void* out, void* stream) {
  using namespace pkv;
  clear_error();
  PKV_UNSUP(head_dim == 256, "spec_verify_combine: head_dim must be 256 (got %d)", head_dim);
  PKV_ARG(part_o && part_lse && seq_lens && out, "spec_verify_combine: null pointer argument");
  PKV_ARG(num_reqs >= 0 && T > 0 && num_q_heads > 0 && split_tokens > 0 && max_splits > 0,
          "spec_verify_combine: bad size argument");
  PKV_ARG(aligned16(part_o) && aligned16(out), "spec_verify_combine: part_o and out must be 16-byte aligned");
  if (num_reqs == 0) return PKV_OK;
  const int64_t rows = (int64_t)num_reqs * T * num_q_heads;
  // programmatic dependent launch: the blocks may be scheduled while the partials' CTAs finish;
  // each waits (griddepcontrol.wait) for that grid's completion before its first read
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((rows + kWarps - 1) / kWarps));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, spec_verify_combine_kernel, part_o, part_lse, seq_lens, T, num_q_heads, head_dim,
                     split_tokens, max_splits, rows, static_cast<__nv_bfloat16*>(out));
  return check_launch("spec_verify_combine");
}

// spec_verify_noalloc.cu - pkv_spec_verify_attn_noalloc: the int8 split-KV verify (partials and
// log-sum-exp combine) with its partials held in a fixed scratch array owned by the library, for
// callers that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is not available or not allowed - a plugin
// loaded into a host process whose allocator owns all device memory, a real-time path that must
// not allocate between steps, a caller that only hands over input and output buffers. The regular
// pkv_spec_verify_attn_partial asks the caller for the partials workspace; this entry point uses
// the file-scope array below instead and allocates nothing at any time.
//
// The array is a `static __device__` object: every GPU that loads the library reserves it until
// the process exits. Host code cannot use its name as a device address (on the host it is only a
// stand-in), so the address is looked up once per device with cudaGetSymbolAddress, with that
// device current, on the first call made on it. That first call should therefore come before any
// stream capture. The address stays cached for the life of the process: after a cudaDeviceReset
// of a device that has made such a call the array may sit elsewhere, so such a device must not be
// reset while the library is in use. Every call on a device shares the one array and overwrites
// what the last call left there; calls that overlap on the GPU (different streams, no ordering
// between them) race on it. Each call writes every partial it reads (splits past a request's keys
// are neither written nor read), so nothing has to start at zero.
#include <mutex>

#include "host_common.h"

namespace pkv {
namespace {

// 32 MiB of fp32: partial outputs (head_dim floats per row and split) and their log-sum-exps.
constexpr size_t kScratchFloats = (32u << 20) / sizeof(float);
static __device__ __align__(256) float g_verify_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {nullptr};

pkv_status scratch_for_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    set_error("spec_verify_attn_noalloc: no current CUDA device (or device index >= %d)", kMaxDevices);
    return PKV_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_verify_scratch);
    if (e != cudaSuccess || !p) {
      set_error("spec_verify_attn_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
      return PKV_ERR_CUDA;
    }
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" size_t pkv_spec_verify_noalloc_capacity_bytes(void) { return pkv::kScratchFloats * sizeof(float); }

extern "C" pkv_status pkv_spec_verify_attn_noalloc(const void* q, const int8_t* k_cache, const int8_t* v_cache,
                                                   const float* k_scale, const float* v_scale, int64_t num_blocks,
                                                   int64_t stride_blk, int64_t stride_tok, int64_t stride_head,
                                                   int64_t scale_stride_blk, int64_t scale_stride_tok,
                                                   const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                                                   const int32_t* seq_lens, int32_t num_reqs, int32_t T,
                                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                                   int32_t block_size, float softmax_scale, int32_t split_tokens,
                                                   int32_t max_splits, void* out, int32_t* dev_err, void* stream) {
  using namespace pkv;
  clear_error();
  if (num_reqs == 0) return PKV_OK;
  PKV_ARG(num_reqs > 0 && T > 0 && num_q_heads > 0 && head_dim > 0 && max_splits > 0,
          "spec_verify_attn_noalloc: bad size argument");
  // partial outputs first, then the log-sum-exps, each 256-byte aligned inside the array. The row
  // count is built one factor at a time and checked against the capacity before each product, so
  // no product can wrap around and slip a huge request past the check.
  size_t rows = 1;
  bool fits = true;
  for (const int32_t f : {num_reqs, T, num_q_heads, max_splits}) {
    if (rows > kScratchFloats / (size_t)f) {
      fits = false;
      break;
    }
    rows *= (size_t)f;
  }
  fits = fits && rows <= kScratchFloats / ((size_t)head_dim + 1);
  const size_t o_floats = fits ? (rows * (size_t)head_dim + 63) & ~(size_t)63 : 0;
  PKV_ARG(fits && o_floats + rows <= kScratchFloats,
          "spec_verify_attn_noalloc: the partials (num_reqs*T*num_q_heads*max_splits*(head_dim+1)*4 bytes) do not "
          "fit the fixed %zu-byte scratch; use fewer splits (larger split_tokens) or the workspace call",
          kScratchFloats * sizeof(float));
  float* scratch = nullptr;
  pkv_status s = scratch_for_current_device(&scratch);
  if (s != PKV_OK) return s;
  float* part_o = scratch;
  float* part_lse = scratch + o_floats;
  s = pkv_spec_verify_attn_partial(q, k_cache, v_cache, k_scale, v_scale, num_blocks, stride_blk, stride_tok,
                                   stride_head, scale_stride_blk, scale_stride_tok, block_table, bt_stride,
                                   max_blocks, seq_lens, num_reqs, T, num_q_heads, num_kv_heads, head_dim,
                                   block_size, softmax_scale, split_tokens, max_splits, part_o, part_lse, dev_err,
                                   stream);
  if (s != PKV_OK) return s;
  return pkv_spec_verify_combine(part_o, part_lse, seq_lens, num_reqs, T, num_q_heads, head_dim, split_tokens,
                                 max_splits, out, stream);
}

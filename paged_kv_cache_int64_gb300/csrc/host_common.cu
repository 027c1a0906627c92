// host_common.cu - error message, launch checks, tensor-map encoding.
#include <cudaTypedefs.h>
#include <string.h>

#include <mutex>

#include "host_common.h"
#include "sm103.cuh"

namespace pkv {

static thread_local char g_last_error[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
}

void clear_error() { g_last_error[0] = '\0'; }

pkv_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("%s: launch failed: %s", what, cudaGetErrorString(e));
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

pkv_status encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                        const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                        const char* what, bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) {
    set_error("%s: cuTensorMapEncodeTiled is unavailable from the driver", what);
    return PKV_ERR_CUDA;
  }
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  cuuint64_t d[5], s[4];
  cuuint32_t b[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) s[i] = strides_bytes[i];
  CUresult r = fn(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, s, b, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("%s: cuTensorMapEncodeTiled failed (CUresult %d)", what, (int)r);
    return PKV_ERR_INVALID_ARG;
  }
  return PKV_OK;
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  static int cache[64] = {0};
  if (dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < 64) cache[dev] = n;
  return n;
}

static thread_local uint64_t g_next_wait_limit_ns = 0;  // 0: the default

uint64_t take_wait_limit_ns() {
  const uint64_t v = g_next_wait_limit_ns;
  g_next_wait_limit_ns = 0;
  return v ? v : kWaitLimitNs;
}

}  // namespace pkv

extern "C" const char* pkv_last_error(void) { return pkv::g_last_error; }
extern "C" void pkv_testing_set_wait_limit_ns(uint64_t ns) { pkv::g_next_wait_limit_ns = ns; }
extern "C" int32_t pkv_abi_version(void) { return PKV_ABI_VERSION; }

// host_common.h - host-side helpers shared by the launchers: the thread-local error message,
// argument checks, and TMA tensor-map encoding through the driver entry point.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>

#include <atomic>
#include <stdint.h>
#include <stdio.h>

#include "../../include/pkv.h"

namespace pkv {

void set_error(const char* fmt, ...);
void clear_error();

// Returns PKV_ERR_CUDA with a message when the last launch failed.
pkv_status check_launch(const char* what);

// Encode a tiled tensor map (128-byte swizzle unless swizzle128 is false; zero fill for
// out-of-range coordinates).
// dims / box are innermost-first; strides_bytes has rank-1 entries (dims 1..rank-1).
pkv_status encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                        const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                        const char* what, bool swizzle128 = true);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Runs fn once per (flag, current device): for kernel attributes the driver keeps per device, such
// as the dynamic shared-memory opt-in. Devices 64 and up run fn on every call.
template <typename F>
inline void once_per_device(std::atomic<uint64_t>& done, F&& fn) {
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
  if (bit && (done.load(std::memory_order_relaxed) & bit)) return;
  fn();
  if (bit) done.fetch_or(bit, std::memory_order_relaxed);
}

// SM count of the current device (cached per device).
int num_sms();

// The bound on each wait of the next attention kernel that the calling thread launches: the
// default (one second) unless pkv_testing_set_wait_limit_ns set another for that one launch.
uint64_t take_wait_limit_ns();

}  // namespace pkv

#define PKV_REQUIRE(cond, status, ...)   \
  do {                                   \
    if (!(cond)) {                       \
      ::pkv::set_error(__VA_ARGS__);     \
      return (status);                   \
    }                                    \
  } while (0)

#define PKV_ARG(cond, ...) PKV_REQUIRE(cond, PKV_ERR_INVALID_ARG, __VA_ARGS__)
#define PKV_UNSUP(cond, ...) PKV_REQUIRE(cond, PKV_ERR_UNSUPPORTED, __VA_ARGS__)

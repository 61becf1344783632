// Diagnostics of the library's failure paths that need no fault on the GPU:
//  * w4g128_selftest_wait launches one small kernel that waits, with the same
//    bounded flag wait the reduce kernel uses, on a workspace word; when
//    nothing sets the word the wait runs out after the given limit, the
//    kernel records W4G128_ERR_TIMEOUT in the status word and returns on its
//    own, so the context stays usable;
//  * fault_hook reads W4G128_FAULT once (host only): "launch" makes every
//    compute entry point return W4G128_ERR_CUDA and "workspace" makes it
//    return W4G128_ERR_WORKSPACE, after argument validation and before
//    anything touches the device.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "w4g128.h"
#include "w4g128_internal.h"
#include "w4g128_ptx.cuh"

namespace w4g128 {

int fault_hook() {
  static const int mode = [] {
    const char* v = std::getenv("W4G128_FAULT");
    if (v == nullptr) return static_cast<int>(W4G128_OK);
    if (std::strcmp(v, "launch") == 0) return static_cast<int>(W4G128_ERR_CUDA);
    if (std::strcmp(v, "workspace") == 0) return static_cast<int>(W4G128_ERR_WORKSPACE);
    return static_cast<int>(W4G128_OK);
  }();
  return mode;
}

namespace {

// ws[0]: status word; ws + 256: the 64-bit flag word.
__global__ void __launch_bounds__(32) selftest_wait_kernel(unsigned* status, unsigned long long* flag,
                                                          unsigned long long limit_ns, int set_flag) {
  if (threadIdx.x != 0) return;
  *status = 0u;
  st_relaxed_u64(flag, set_flag ? 1ull : 0ull);
  unsigned long long seen = 0ull;
  if (!wait_nonzero_bounded(flag, seen, limit_ns)) atomicCAS(status, 0u, static_cast<unsigned>(W4G128_ERR_TIMEOUT));
}

}  // namespace
}  // namespace w4g128

extern "C" int w4g128_selftest_wait(void* ws, size_t ws_bytes, unsigned long long limit_ns, int set_flag,
                                    void* stream) {
  if (ws == nullptr || (set_flag != 0 && set_flag != 1)) return W4G128_ERR_INVALID_ARG;
  if (limit_ns < 1ull || limit_ns > w4g128::kDefaultWaitNs) return W4G128_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ws) % 16 != 0) return W4G128_ERR_ALIGN;
  if (ws_bytes < W4G128_SELFTEST_WS_BYTES) return W4G128_ERR_WORKSPACE;
  const int fault = w4g128::fault_hook();
  if (fault != W4G128_OK) return fault;
  if (!w4g128::device_is_sm103()) return W4G128_ERR_DEVICE;
  auto* base = static_cast<unsigned char*>(ws);
  w4g128::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<unsigned*>(base), reinterpret_cast<unsigned long long*>(base + 256), limit_ns, set_flag);
  if (cudaGetLastError() != cudaSuccess) return W4G128_ERR_CUDA;
  return W4G128_OK;
}

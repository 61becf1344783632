// w4g128_gemv_noalloc: the M = 1 GEMV for callers that cannot hand the
// library a device workspace.
//
// Who needs it: code that is only given a stream and must not allocate device
// memory itself -- plugin hooks of another runtime that owns the device
// memory budget, fixed-pool serving processes, and latency-critical threads
// that must not call cudaMalloc/cudaFree (they can synchronise the device and
// stall every other stream).  Such callers pass only weights, input and
// output; the split-K partials, activation packages and status word
// live in one fixed scratch array that the library reserves on every GPU that
// loads it, for the life of the process.
//
// The scratch array is a plain __device__ variable.  In host code its name is
// a host-side stand-in, not a device address, so every call looks the address
// up with cudaGetSymbolAddress (with the call's device current) and passes it
// to the kernels like any caller-owned workspace.  The lookup is repeated on
// every call rather than cached: after cudaDeviceReset, or after the primary
// context is released and created again, the module is loaded afresh and the
// array may sit at another address.  The first call on a device loads the
// module there (the set-up); make it before any stream capture.
#include <cuda_runtime.h>

#include <cstdint>

#include "w4g128.h"
#include "w4g128_internal.h"

// Every call on a device shares this array; it keeps the previous call's
// contents.  The parts that must start at zero, the status word and the
// split-K arrival counters, are cleared by each call's first kernel;
// everything else is written before it is read within the call.
static __device__ __align__(256) unsigned char g_w4g128_scratch[W4G128_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of the scratch array in the current context.
int scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_w4g128_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return W4G128_ERR_CUDA;
  }
  *out = p;
  return W4G128_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int w4g128_gemv_noalloc(const void* packed, const w4g128_bf16* x, w4g128_bf16* y, int K, int N,
                                   void* stream) {
  if (packed == nullptr || x == nullptr || y == nullptr) return W4G128_ERR_INVALID_ARG;
  if (!(K >= 128 && K <= 65536 && K % 128 == 0 && N >= 16 && N <= (1 << 24) && N % 16 == 0))
    return W4G128_ERR_SHAPE;
  if (!aligned(packed, 16) || !aligned(x, 4) || !aligned(y, 4)) return W4G128_ERR_ALIGN;
  if (w4g128::fault_hook() != W4G128_OK) return w4g128::fault_hook();
  if (!w4g128::device_is_sm103()) return W4G128_ERR_DEVICE;
  const w4g128::HostMatrix m{packed, x, y, K, N};
  const size_t need = w4g128::stream_workspace_bytes(&m, 1, 1);
  if (need == 0) return W4G128_ERR_SHAPE;
  if (need > W4G128_NOALLOC_SCRATCH_BYTES) return W4G128_ERR_WORKSPACE;  // shape too large for the scratch
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != W4G128_OK) return rc;
  return w4g128::launch_stream(&m, 1, 1, nullptr, scratch, W4G128_NOALLOC_SCRATCH_BYTES,
                               static_cast<cudaStream_t>(stream));
}

extern "C" int w4g128_noalloc_status(int* status_out, void* stream) {
  if (status_out == nullptr) return W4G128_ERR_INVALID_ARG;
  if (!w4g128::device_is_sm103()) return W4G128_ERR_DEVICE;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != W4G128_OK) return rc;
  return w4g128::read_workspace_status(scratch, status_out, static_cast<cudaStream_t>(stream));
}

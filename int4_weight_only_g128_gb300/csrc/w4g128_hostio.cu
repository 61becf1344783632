// Host <-> device moves of a step's activations as kernels, for
// w4g128_decode_step_host: a copy-engine copy between two kernels ends the
// chain of programmatic dependent launches (the next kernel can no longer
// start early and prefetch its weights), so when the host buffers are
// device-mapped (pinned memory) the library moves them with two small kernels
// that take part in the chain instead:
//  * upload: reads x from host memory before its dependency wait (the host
//    wrote it before the call), then writes it to device memory once the
//    previous kernel has finished (that kernel may still read the old x);
//  * download: once the step's last kernel has finished, copies y to host
//    memory with 16-byte stores.
// One CTA of 256 threads per 4 KB (one 16-byte unit per thread), up to one
// per SM; beyond that each thread moves further units.  Spreading the bytes
// over more CTAs shortens both moves: every thread's host access is a full
// round trip over the chip-to-host link, so fewer accesses per thread means
// less latency on the step's critical path.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "w4g128.h"
#include "w4g128_internal.h"
#include "w4g128_ptx.cuh"

namespace w4g128 {
namespace {

constexpr int kIoThreads = 256;
constexpr int kIoPerThread = 16;  // uint4 loads in flight per thread, at most

__global__ void __launch_bounds__(kIoThreads) upload_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                            size_t n16) {
  grid_dependents_launch();
  const size_t stride = static_cast<size_t>(gridDim.x) * kIoThreads;
  size_t i0 = static_cast<size_t>(blockIdx.x) * kIoThreads + threadIdx.x;
  while (i0 < n16) {
    uint4 v[kIoPerThread];
#pragma unroll
    for (int k = 0; k < kIoPerThread; ++k) {
      const size_t i = i0 + k * stride;
      if (i < n16) v[k] = src[i];
    }
    grid_dependency_wait();  // the previous kernel has finished with the old x (a no-op after the first time)
#pragma unroll
    for (int k = 0; k < kIoPerThread; ++k) {
      const size_t i = i0 + k * stride;
      if (i < n16) dst[i] = v[k];
    }
    i0 += kIoPerThread * stride;
  }
  grid_dependency_wait();  // a thread with nothing to move still orders this grid after the previous one
}

__global__ void __launch_bounds__(kIoThreads) download_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                              size_t n16) {
  grid_dependents_launch();
  grid_dependency_wait();  // every y of the step is written and visible
  const size_t stride = static_cast<size_t>(gridDim.x) * kIoThreads;
  for (size_t i = static_cast<size_t>(blockIdx.x) * kIoThreads + threadIdx.x; i < n16; i += stride)
    dst[i] = __ldcg(src + i);
}

int launch_io(bool up, const void* src, void* dst, size_t bytes, cudaStream_t stream) {
  const size_t n16 = bytes / 16;
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess) {
    cudaGetLastError();
    return W4G128_ERR_CUDA;
  }
  const size_t per_cta = kIoThreads;  // 4 KB per CTA before a CTA takes more
  const unsigned grid = static_cast<unsigned>(std::max<size_t>(1, std::min<size_t>(sms, (n16 + per_cta - 1) / per_cta)));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kIoThreads);
  const cudaError_t e = up ? cudaLaunchKernelEx(&cfg, upload_kernel, static_cast<const uint4*>(src),
                                                static_cast<uint4*>(dst), n16)
                           : cudaLaunchKernelEx(&cfg, download_kernel, static_cast<const uint4*>(src),
                                                static_cast<uint4*>(dst), n16);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return W4G128_ERR_CUDA;
  }
  return W4G128_OK;
}

}  // namespace

// The device address of a host buffer the GPU can reach directly (pinned and
// mapped, 16-byte aligned, a whole number of 16-byte units), or nullptr.
const void* mapped_host(const void* host, size_t bytes) {
  if (host == nullptr || bytes == 0 || bytes % 16 != 0 || reinterpret_cast<uintptr_t>(host) % 16 != 0)
    return nullptr;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return nullptr;
  return a.devicePointer;
}

int launch_upload(const void* host_dev, void* dev, size_t bytes, cudaStream_t stream) {
  return launch_io(true, host_dev, dev, bytes, stream);
}

int launch_download(const void* dev, void* host_dev, size_t bytes, cudaStream_t stream) {
  return launch_io(false, dev, host_dev, bytes, stream);
}

}  // namespace w4g128

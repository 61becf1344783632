// HBM bandwidth probes: a read-only stream and a copy, each a grid-stride
// loop of 128-bit accesses with four independent loads in flight per thread,
// sized to a few resident blocks per SM.
#include <cuda_runtime.h>

#include <cstdint>

#include "w4g128_probe.h"

namespace {

constexpr int kThreads = 512;
constexpr int kBlocksPerSM = 4;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kThreads) read_kernel(const uint4* __restrict__ buf, long long n16,
                                                        uint32_t* __restrict__ sink) {
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
  uint32_t acc = 0;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = ld_stream(buf + i), b = ld_stream(buf + i + stride);
    const uint4 c = ld_stream(buf + i + 2 * stride), d = ld_stream(buf + i + 3 * stride);
    acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
  }
  for (; i < n16; i += stride) {
    const uint4 a = ld_stream(buf + i);
    acc ^= a.x ^ a.y ^ a.z ^ a.w;
  }
  // one digest per block
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  __shared__ uint32_t red[kThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t v = 0;
    for (int w = 0; w < kThreads / 32; ++w) v ^= red[w];
    sink[blockIdx.x] = v;
  }
}

__global__ void __launch_bounds__(kThreads) copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                        long long n16) {
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = ld_stream(src + i), b = ld_stream(src + i + stride);
    const uint4 c = ld_stream(src + i + 2 * stride), d = ld_stream(src + i + 3 * stride);
    __stcs(dst + i, a);
    __stcs(dst + i + stride, b);
    __stcs(dst + i + 2 * stride, c);
    __stcs(dst + i + 3 * stride, d);
  }
  for (; i < n16; i += stride) __stcs(dst + i, ld_stream(src + i));
}

int grid_blocks() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms * kBlocksPerSM;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

size_t w4g128_probe_sink_bytes(void) {
  const int b = grid_blocks();
  return b > 0 ? static_cast<size_t>(b) * sizeof(uint32_t) : 0;
}

int w4g128_probe_read(const void* buf, size_t bytes, void* sink, void* stream) {
  if (buf == nullptr || sink == nullptr || bytes == 0) return W4G128_ERR_INVALID_ARG;
  if (bytes % 16 != 0) return W4G128_ERR_SHAPE;
  if (!aligned16(buf) || !aligned16(sink)) return W4G128_ERR_ALIGN;
  const int blocks = grid_blocks();
  if (blocks == 0) return W4G128_ERR_DEVICE;
  read_kernel<<<blocks, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(buf), static_cast<long long>(bytes / 16), static_cast<uint32_t*>(sink));
  return cudaGetLastError() == cudaSuccess ? W4G128_OK : W4G128_ERR_CUDA;
}

int w4g128_probe_copy(const void* src, void* dst, size_t bytes, void* stream) {
  if (src == nullptr || dst == nullptr || bytes == 0) return W4G128_ERR_INVALID_ARG;
  if (bytes % 16 != 0) return W4G128_ERR_SHAPE;
  if (!aligned16(src) || !aligned16(dst)) return W4G128_ERR_ALIGN;
  const int blocks = grid_blocks();
  if (blocks == 0) return W4G128_ERR_DEVICE;
  copy_kernel<<<blocks, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(src), static_cast<uint4*>(dst), static_cast<long long>(bytes / 16));
  return cudaGetLastError() == cudaSuccess ? W4G128_OK : W4G128_ERR_CUDA;
}

}  // extern "C"

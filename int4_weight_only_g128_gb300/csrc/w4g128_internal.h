// Internal declarations shared by the translation units of libw4g128.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "w4g128.h"

namespace w4g128 {

constexpr int kGroup = 128;          // K-rows per scale/min group
constexpr int kTileN = 16;           // columns per packed tile
constexpr int kCodeBytes = 1024;     // codes of one (tile, group) block
constexpr int kBlockBytes = 1088;    // codes + 8 metadata entries of 8 bytes
constexpr int kQuadTiles = 4;        // tiles a warp streams together (64 columns)
constexpr int kSegGroups = 4;        // groups per fixed split-K segment (512 rows)
constexpr int kQuadBytes = kQuadTiles * kBlockBytes;  // one full quad, one group

// Byte offset of block (tile t, group g) in the packed layout: quads of 4
// tiles are contiguous runs over all groups, and one quad's tiles for one
// group are adjacent.  T = N/16 tiles, G = K/128 groups.
__host__ __device__ inline long long block_offset(int t, int g, int G, int T) {
  const int q = t / kQuadTiles, i = t % kQuadTiles;
  const int nt = (T - kQuadTiles * q) < kQuadTiles ? (T - kQuadTiles * q) : kQuadTiles;
  return static_cast<long long>(q) * G * kQuadBytes + static_cast<long long>(g) * nt * kBlockBytes +
         static_cast<long long>(i) * kBlockBytes;
}

int launch_pack(const uint32_t* codes, const uint16_t* scales, const uint16_t* mins, int K, int N,
                void* packed, cudaStream_t stream);
int launch_unpack(const void* packed, int K, int N, uint32_t* codes, uint16_t* scales, uint16_t* mins,
                  cudaStream_t stream);

int launch_quantize(const uint16_t* w, int K, int N, int search, uint32_t* codes, uint16_t* scales,
                    uint16_t* mins, cudaStream_t stream);

// One matrix of a streaming call, as the host hands it over.
struct HostMatrix {
  const void* packed;
  const uint16_t* x;
  uint16_t* y;
  int K, N;
};

// Workspace bytes for streaming these matrices at this M on the current
// device.  Returns 0 on invalid arguments.
size_t stream_workspace_bytes(const HostMatrix* mats, int count, int M);

// The residual add + RMS norm that a one-matrix call may end in: y becomes
// h = residual + x W and out = gamma h / rms(h) per row (device pointers).
struct NormArgs {
  const uint16_t* residual;
  const uint16_t* gamma;
  uint16_t* out;
  float eps;
};

// Launches the prep, streaming and (M >= 2) reduce kernels; the API layer
// validates arguments.  Every M uses the warp-MMA arithmetic, so row m of a
// result is bitwise the M = 1 result of row m.  norm: nullptr, or the
// residual add + RMS norm (count must be 1).
int launch_stream(const HostMatrix* mats, int count, int M, const NormArgs* norm, void* ws,
                  size_t ws_bytes, cudaStream_t stream);

int read_workspace_status(const void* ws, int* status_out, cudaStream_t stream);

// The schedule of a call (the fields of w4g128_schedule), launching nothing.
int describe_schedule(const HostMatrix* mats, int count, int M, long long* out, int n);

// Device address of a pinned, device-mapped host buffer (16-byte aligned,
// `bytes` a multiple of 16), or nullptr when the GPU cannot reach it.
const void* mapped_host(const void* host, size_t bytes);

// Moves `bytes` (a multiple of 16, 16-byte aligned ends) between a mapped
// host buffer and device memory with a small kernel launched as a
// programmatic dependent of whatever precedes it on the stream.
int launch_upload(const void* host_dev, void* dev, size_t bytes, cudaStream_t stream);
int launch_download(const void* dev, void* host_dev, size_t bytes, cudaStream_t stream);

// Current device is compute capability 10.3; caches per device.
bool device_is_sm103();

// Host-only fault injection for tests of the error paths: W4G128_OK, or the
// status that the environment variable W4G128_FAULT ("launch" ->
// W4G128_ERR_CUDA, "workspace" -> W4G128_ERR_WORKSPACE) makes every compute
// entry point return before it touches the device.  Read once per process.
int fault_hook();

}  // namespace w4g128

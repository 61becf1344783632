// Canonical int4-g128 weights <-> the packed (tiled) layout the streaming
// kernels read.  Both directions are pure bit permutations.
//
// Canonical: codes uint32 [K/8][N] (row k = 8j+i in bits 4i..4i+3 of word
// (j, n)), scales / mins bf16 [K/128][N].  Packed: see include/w4g128.h;
// block (t, g) of 1088 bytes = 1024 bytes of codes (two 512-byte halves of
// 32 lanes x 4 words) + 64 bytes of (scale, min) pairs, placed by
// block_offset() so that each 64-column quad is one contiguous run.
#include <cuda_runtime.h>

#include <cstdint>

#include "w4g128_internal.h"

namespace w4g128 {
namespace {

// One CTA of 64 threads per block (t, g): thread = 32*h + lane writes the
// 16 bytes of lane `lane` in half h; threads 0..7 also write metadata entry r.
__global__ void __launch_bounds__(64) pack_kernel(const uint32_t* __restrict__ codes,
                                                  const uint16_t* __restrict__ scales,
                                                  const uint16_t* __restrict__ mins, int K, int N,
                                                  uint8_t* __restrict__ packed) {
  const int G = K / 128;
  const int64_t blk = blockIdx.x;
  const int t = static_cast<int>(blk / G), g = static_cast<int>(blk % G);
  const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, c = lane & 3;
  const int n_lo = 16 * t + r, n_hi = n_lo + 8;
  uint32_t out[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int k0 = 128 * g + 64 * h + 16 * j;
    const int64_t row = k0 / 8;                 // canonical word row of k0 .. k0+7
    // canonical words: [a][e] = rows k0 + 8a .., column n_lo + 8e
    const uint32_t w00 = codes[row * N + n_lo], w01 = codes[row * N + n_hi];
    const uint32_t w10 = codes[(row + 1) * N + n_lo], w11 = codes[(row + 1) * N + n_hi];
    uint32_t word = 0;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const int b = (p >> 2) & 1, a = (p >> 1) & 1, e = p & 1;
      const uint32_t src = a ? (e ? w11 : w10) : (e ? w01 : w00);
      const uint32_t q = (src >> (4 * (2 * c + b))) & 0xFu;
      word |= q << (4 * p);
    }
    out[j] = word;
  }
  uint8_t* base = packed + block_offset(t, g, G, N / kTileN);
  *reinterpret_cast<uint4*>(base + 512 * h + 16 * lane) = make_uint4(out[0], out[1], out[2], out[3]);
  if (threadIdx.x < 8) {
    const int rr = threadIdx.x;
    const int64_t lo = static_cast<int64_t>(g) * N + 16 * t + rr, hi = lo + 8;
    const uint32_t e0 = static_cast<uint32_t>(scales[lo]) | (static_cast<uint32_t>(mins[lo]) << 16);
    const uint32_t e1 = static_cast<uint32_t>(scales[hi]) | (static_cast<uint32_t>(mins[hi]) << 16);
    *reinterpret_cast<uint2*>(base + kCodeBytes + 8 * rr) = make_uint2(e0, e1);
  }
}

// One thread per canonical word (jr, n): gathers its 8 nibbles from the 4
// packed words (lanes 4r + c, c = 0..3) that hold them.
__global__ void unpack_codes_kernel(const uint8_t* __restrict__ packed, int K, int N,
                                    uint32_t* __restrict__ codes) {
  const int64_t total = static_cast<int64_t>(K / 8) * N;
  const int G = K / 128;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int jr = static_cast<int>(idx / N), n = static_cast<int>(idx % N);
    const int k_first = 8 * jr;
    const int g = k_first / 128, h = (k_first % 128) / 64, j = (k_first % 64) / 16, a = jr & 1;
    const int t = n / 16, e = (n % 16) / 8, r = (n % 16) % 8;
    const uint8_t* base = packed + block_offset(t, g, G, N / kTileN) + 512 * h;
    uint32_t word = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t pw = *reinterpret_cast<const uint32_t*>(base + 16 * (4 * r + c) + 4 * j);
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int p = 4 * b + 2 * a + e;
        const uint32_t q = (pw >> (4 * p)) & 0xFu;
        word |= q << (4 * (2 * c + b));
      }
    }
    codes[idx] = word;
  }
}

__global__ void unpack_meta_kernel(const uint8_t* __restrict__ packed, int K, int N,
                                   uint16_t* __restrict__ scales, uint16_t* __restrict__ mins) {
  const int G = K / 128;
  const int64_t total = static_cast<int64_t>(G) * N;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int g = static_cast<int>(idx / N), n = static_cast<int>(idx % N);
    const int t = n / 16, e = (n % 16) / 8, r = (n % 16) % 8;
    const uint8_t* ent = packed + block_offset(t, g, G, N / kTileN) + kCodeBytes + 8 * r + 4 * e;
    const uint32_t v = *reinterpret_cast<const uint32_t*>(ent);
    scales[idx] = static_cast<uint16_t>(v & 0xFFFFu);
    mins[idx] = static_cast<uint16_t>(v >> 16);
  }
}

int grid_stride_blocks(int64_t n, int threads) {
  const int64_t b = (n + threads - 1) / threads;
  return static_cast<int>(b < 65536 ? (b > 0 ? b : 1) : 65536);
}

}  // namespace

int launch_pack(const uint32_t* codes, const uint16_t* scales, const uint16_t* mins, int K, int N,
                void* packed, cudaStream_t stream) {
  const int64_t blocks = static_cast<int64_t>(N / 16) * (K / 128);
  if (blocks > 0x7FFFFFFFLL) return W4G128_ERR_SHAPE;
  pack_kernel<<<static_cast<unsigned>(blocks), 64, 0, stream>>>(codes, scales, mins, K, N,
                                                                 static_cast<uint8_t*>(packed));
  return cudaGetLastError() == cudaSuccess ? W4G128_OK : W4G128_ERR_CUDA;
}

int launch_unpack(const void* packed, int K, int N, uint32_t* codes, uint16_t* scales, uint16_t* mins,
                  cudaStream_t stream) {
  const auto* p = static_cast<const uint8_t*>(packed);
  const int64_t nc = static_cast<int64_t>(K / 8) * N, nm = static_cast<int64_t>(K / 128) * N;
  unpack_codes_kernel<<<grid_stride_blocks(nc, 256), 256, 0, stream>>>(p, K, N, codes);
  if (cudaGetLastError() != cudaSuccess) return W4G128_ERR_CUDA;
  unpack_meta_kernel<<<grid_stride_blocks(nm, 256), 256, 0, stream>>>(p, K, N, scales, mins);
  return cudaGetLastError() == cudaSuccess ? W4G128_OK : W4G128_ERR_CUDA;
}

}  // namespace w4g128

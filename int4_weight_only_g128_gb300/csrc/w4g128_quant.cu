// w4g128_quantize: bf16 weights -> canonical int4-g128 codes, scales, minimums.
//
// The format (Token Rush README, "Quantization"): 128 weights of one column
// share a bf16 scale and minimum, w = min + q * scale, q in 0..15.  Codes are
// chosen by round-to-nearest on the group's 16-level grid, optionally with a
// range search that clips outliers ("an MSE range search per group that clips
// a few outliers"):
//
//   lo, hi = min and max of the group; for a candidate p the grid spans
//   [a, b] = [p lo, p hi] in 15 steps: s = (b - a) / 15, scale = bf16(s),
//   min = bf16(a), q = clamp(round_half_even((w - min) / scale), 0, 15)
//   (q = 0 when scale = 0), error = sum over the group in row order of
//   (w - (min + q scale))^2.  Round-to-nearest is p = 1; the search tries
//   p = (100 - i) / 100, i = 0..20, and keeps the smallest error (the widest
//   range on ties).
//
// Every step is a single IEEE fp32 operation rounded to nearest, written with
// the _rn intrinsics so that no multiply-add is contracted: the codes and the
// chosen candidate are integer decisions, reproduced bit for bit by any
// implementation that performs the same operations.
//
// One thread per (group, column); a block stages a 128 x 128 tile of bf16
// weights (32 KB) in shared memory with coalesced loads.  This is a one-time
// preprocessing step, not part of the weight stream.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "w4g128.h"
#include "w4g128_internal.h"

namespace w4g128 {
namespace {

constexpr int kCols = 128;       // columns per block (one thread each)
constexpr int kCandidates = 21;  // p = 1.00, 0.99, ..., 0.80

__device__ __forceinline__ float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

__device__ __forceinline__ int code_of(float w, float mb, float sb) {
  if (sb == 0.0f) return 0;
  const float r = rintf(__fdiv_rn(__fsub_rn(w, mb), sb));  // ties to even
  if (!(r > 0.0f)) return 0;
  if (r > 15.0f) return 15;
  return static_cast<int>(r);
}

__global__ void __launch_bounds__(kCols) quantize_kernel(const uint16_t* __restrict__ w, int K, int N, int search,
                                                         uint32_t* __restrict__ codes, uint16_t* __restrict__ scales,
                                                         uint16_t* __restrict__ mins) {
  __shared__ uint16_t tile[kGroup][kCols];
  const int g = blockIdx.y;
  const int t = threadIdx.x;
  const int n = blockIdx.x * kCols + t;
  const bool live = n < N;
  // stage: for each row, the block's threads read consecutive columns
  for (int k = 0; k < kGroup; ++k)
    tile[k][t] = live ? w[static_cast<long long>(kGroup * g + k) * N + n] : 0;
  __syncthreads();
  if (!live) return;

  float lo = 0.f, hi = 0.f;
  for (int k = 0; k < kGroup; ++k) {
    const float v = __uint_as_float(static_cast<uint32_t>(tile[k][t]) << 16);
    if (k == 0 || v < lo) lo = v;
    if (k == 0 || v > hi) hi = v;
  }

  const int ncand = search ? kCandidates : 1;
  float best_e = 0.f, best_s = 0.f, best_m = 0.f;
  for (int i = 0; i < ncand; ++i) {
    const float p = __fdiv_rn(static_cast<float>(100 - i), 100.0f);
    const float a = __fmul_rn(p, lo), b = __fmul_rn(p, hi);
    const float sb = bf16_round(__fdiv_rn(__fsub_rn(b, a), 15.0f));
    const float mb = bf16_round(a);
    float e = 0.f;
    for (int k = 0; k < kGroup; ++k) {
      const float v = __uint_as_float(static_cast<uint32_t>(tile[k][t]) << 16);
      const int q = code_of(v, mb, sb);
      const float dq = __fadd_rn(mb, __fmul_rn(static_cast<float>(q), sb));
      const float r = __fsub_rn(v, dq);
      e = __fadd_rn(e, __fmul_rn(r, r));
    }
    if (i == 0 || e < best_e) {
      best_e = e;
      best_s = sb;
      best_m = mb;
    }
  }

  // codes of the chosen grid, 8 per word along K
#pragma unroll 1
  for (int j = 0; j < kGroup / 8; ++j) {
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float v = __uint_as_float(static_cast<uint32_t>(tile[8 * j + i][t]) << 16);
      word |= static_cast<uint32_t>(code_of(v, best_m, best_s)) << (4 * i);
    }
    codes[static_cast<long long>(16 * g + j) * N + n] = word;
  }
  scales[static_cast<long long>(g) * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(best_s));
  mins[static_cast<long long>(g) * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(best_m));
}

}  // namespace

int launch_quantize(const uint16_t* w, int K, int N, int search, uint32_t* codes, uint16_t* scales,
                    uint16_t* mins, cudaStream_t stream) {
  const dim3 grid((N + kCols - 1) / kCols, K / kGroup);
  quantize_kernel<<<grid, kCols, 0, stream>>>(w, K, N, search ? 1 : 0, codes, scales, mins);
  return cudaGetLastError() == cudaSuccess ? W4G128_OK : W4G128_ERR_CUDA;
}

}  // namespace w4g128

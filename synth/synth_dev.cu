// Seeded synthetic inputs, device side: fills the large weight arrays (codes,
// scales, mins) straight into device memory with the same counter-based
// SplitMix64 streams as synth.c, so that multi-gigabyte workloads need no
// host generation or host-to-device copy.  Every value is bit-identical to the
// host generator: integer hashing, IEEE double add/mul with explicit
// round-to-nearest intrinsics (no contraction into FMA) and an integer-only
// round-to-nearest-even conversion to bf16.  No arithmetic of the method
// itself lives here.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ULL;

__host__ __device__ inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

__host__ __device__ inline uint64_t key_of(uint64_t seed, uint64_t matrix_id, uint32_t array_id) {
  return mix64(seed ^ mix64(matrix_id * kGamma + (uint64_t)array_id + 1ULL));
}

__device__ inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1ULL) * kGamma); }

__device__ inline double u53(uint64_t v) {
  return __dmul_rn((double)(v >> 11), 1.0 / 9007199254740992.0);
}

__device__ inline uint16_t bf16_rn(double d) {
  uint64_t b = (uint64_t)__double_as_longlong(d);
  uint16_t sign = (uint16_t)((b >> 63) << 15);
  int e = (int)((b >> 52) & 0x7FF);
  uint64_t mant = b & ((1ULL << 52) - 1);
  if (e == 0x7FF) return (uint16_t)(sign | 0x7F80 | (mant ? 0x40 : 0));
  if (e == 0) return sign;
  int E = e - 1023;
  uint64_t m = (1ULL << 52) | mant;
  if (E >= -126) {
    uint64_t q = m >> 45, rem = m & ((1ULL << 45) - 1), half = 1ULL << 44;
    if (rem > half || (rem == half && (q & 1))) q++;
    if (q == 256) { q = 128; E++; }
    if (E > 127) return (uint16_t)(sign | 0x7F80);
    return (uint16_t)(sign | ((uint16_t)(E + 127) << 7) | (uint16_t)(q & 0x7F));
  }
  int s = -(E + 81);
  if (s >= 54) return sign;
  uint64_t q = m >> s, rem = m & ((1ULL << s) - 1), half = 1ULL << (s - 1);
  if (rem > half || (rem == half && (q & 1))) q++;
  return (uint16_t)(sign | (uint16_t)q);
}

__device__ inline double bf16_to_double(uint16_t h) {
  return (double)__uint_as_float((uint32_t)h << 16);
}

__device__ inline uint16_t scale_at(uint64_t ks, uint64_t idx) {
  double u = u53(draw(ks, idx));
  return bf16_rn(__dadd_rn(0.002, __dmul_rn(0.018, u)));
}

__device__ inline uint16_t min_at(uint64_t ks, uint64_t km, uint64_t idx) {
  double sb = bf16_to_double(scale_at(ks, idx));
  double v = u53(draw(km, idx));
  double b = __dadd_rn(__dmul_rn(2.0, v), -1.0);
  double f = __dadd_rn(1.0, __dmul_rn(0.1, b));
  double p = __dmul_rn(-8.0, sb);
  return bf16_rn(__dmul_rn(p, f));
}

__global__ void fill_codes_kernel(uint64_t key, int64_t n, uint32_t* out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = (uint32_t)draw(key, (uint64_t)i);
}

__global__ void fill_meta_kernel(uint64_t ks, uint64_t km, int64_t n, uint16_t* scales, uint16_t* mins) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    scales[i] = scale_at(ks, (uint64_t)i);
    mins[i] = min_at(ks, km, (uint64_t)i);
  }
}

int grid_for(int64_t n) {
  int64_t b = (n + 255) / 256;
  return (int)(b < 4096 ? (b > 0 ? b : 1) : 4096);
}

}  // namespace

extern "C" {

// codes[n_words] in device memory; returns a cudaError_t value.
int synth_dev_codes(uint64_t seed, uint64_t matrix_id, int64_t n_words, uint32_t* out, cudaStream_t s) {
  if (n_words <= 0) return 0;
  fill_codes_kernel<<<grid_for(n_words), 256, 0, s>>>(key_of(seed, matrix_id, 0), n_words, out);
  return (int)cudaGetLastError();
}

// scales[n], mins[n] in device memory.
int synth_dev_meta(uint64_t seed, uint64_t matrix_id, int64_t n, uint16_t* scales, uint16_t* mins,
                   cudaStream_t s) {
  if (n <= 0) return 0;
  fill_meta_kernel<<<grid_for(n), 256, 0, s>>>(key_of(seed, matrix_id, 1), key_of(seed, matrix_id, 2), n,
                                                scales, mins);
  return (int)cudaGetLastError();
}

}  // extern "C"

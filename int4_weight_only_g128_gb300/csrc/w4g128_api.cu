// The extern "C" entry points of libw4g128: argument validation (returned
// synchronously, before anything is launched), then the launchers.
#include <cuda_runtime.h>

#include <cstdint>

#include "w4g128.h"
#include "w4g128_internal.h"

namespace {

using w4g128::HostMatrix;

bool shape_ok(int K, int N) {
  return K >= 128 && K <= 65536 && K % 128 == 0 && N >= 16 && N <= (1 << 24) && N % 16 == 0;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

int check_matrix(const w4g128_matrix& m) {
  if (m.packed == nullptr || m.x == nullptr || m.y == nullptr) return W4G128_ERR_INVALID_ARG;
  if (!shape_ok(m.K, m.N)) return W4G128_ERR_SHAPE;
  if (!aligned(m.packed, 16) || !aligned(m.x, 4) || !aligned(m.y, 4)) return W4G128_ERR_ALIGN;
  return W4G128_OK;
}

int check_stream_call(const w4g128_matrix* mats, int count, int M, void* ws) {
  if (mats == nullptr || count < 1 || count > W4G128_MAX_MATRICES) return W4G128_ERR_INVALID_ARG;
  if (M < 1 || M > W4G128_MAX_M) return W4G128_ERR_INVALID_ARG;
  if (ws == nullptr) return W4G128_ERR_INVALID_ARG;
  if (!aligned(ws, 16)) return W4G128_ERR_ALIGN;
  for (int i = 0; i < count; ++i) {
    const int rc = check_matrix(mats[i]);
    if (rc != W4G128_OK) return rc;
  }
  return W4G128_OK;
}

int run_stream(const w4g128_matrix* mats, int count, int M, void* ws, size_t ws_bytes, void* stream,
               const w4g128::NormArgs* norm = nullptr) {
  int rc = check_stream_call(mats, count, M, ws);
  if (rc != W4G128_OK) return rc;
  rc = w4g128::fault_hook();
  if (rc != W4G128_OK) return rc;
  if (!w4g128::device_is_sm103()) return W4G128_ERR_DEVICE;
  static_assert(sizeof(HostMatrix) == sizeof(w4g128_matrix), "descriptor layout");
  HostMatrix hm[W4G128_MAX_MATRICES];
  for (int i = 0; i < count; ++i) hm[i] = HostMatrix{mats[i].packed, mats[i].x, mats[i].y, mats[i].K, mats[i].N};
  return w4g128::launch_stream(hm, count, M, norm, ws, ws_bytes, as_stream(stream));
}

size_t stream_bytes(const w4g128_matrix* mats, int count, int M) {
  if (mats == nullptr || count < 1 || count > W4G128_MAX_MATRICES || M < 1 || M > W4G128_MAX_M) return 0;
  HostMatrix hm[W4G128_MAX_MATRICES];
  for (int i = 0; i < count; ++i) {
    if (!shape_ok(mats[i].K, mats[i].N)) return 0;
    hm[i] = HostMatrix{mats[i].packed, mats[i].x, mats[i].y, mats[i].K, mats[i].N};
  }
  return w4g128::stream_workspace_bytes(hm, count, M);
}

}  // namespace

extern "C" {

const char* w4g128_status_string(int status) {
  switch (status) {
    case W4G128_OK: return "ok";
    case W4G128_ERR_INVALID_ARG: return "invalid argument";
    case W4G128_ERR_SHAPE: return "unsupported shape (K % 128, N % 16 or size limits)";
    case W4G128_ERR_ALIGN: return "misaligned pointer";
    case W4G128_ERR_WORKSPACE: return "workspace too small";
    case W4G128_ERR_CUDA: return "CUDA runtime or launch error";
    case W4G128_ERR_DEVICE: return "current device is not compute capability 10.3 (sm_103)";
    case W4G128_ERR_TIMEOUT: return "a bounded device-side wait timed out";
    case W4G128_ERR_INTERNAL: return "a kernel found its launch inconsistent and skipped its work";
    default: return "unknown status";
  }
}

size_t w4g128_packed_bytes(int K, int N) {
  if (!shape_ok(K, N)) return 0;
  return static_cast<size_t>(N / 16) * static_cast<size_t>(K / 128) * 1088u;
}

int w4g128_pack(const uint32_t* codes, const w4g128_bf16* scales, const w4g128_bf16* mins, int K, int N,
                void* packed, void* stream) {
  if (codes == nullptr || scales == nullptr || mins == nullptr || packed == nullptr) return W4G128_ERR_INVALID_ARG;
  if (!shape_ok(K, N)) return W4G128_ERR_SHAPE;
  if (!aligned(codes, 4) || !aligned(scales, 4) || !aligned(mins, 4) || !aligned(packed, 16))
    return W4G128_ERR_ALIGN;
  if (w4g128::fault_hook() != W4G128_OK) return w4g128::fault_hook();
  if (!w4g128::device_is_sm103()) return W4G128_ERR_DEVICE;
  return w4g128::launch_pack(codes, scales, mins, K, N, packed, as_stream(stream));
}

int w4g128_unpack(const void* packed, int K, int N, uint32_t* codes, w4g128_bf16* scales, w4g128_bf16* mins,
                  void* stream) {
  if (codes == nullptr || scales == nullptr || mins == nullptr || packed == nullptr) return W4G128_ERR_INVALID_ARG;
  if (!shape_ok(K, N)) return W4G128_ERR_SHAPE;
  if (!aligned(codes, 4) || !aligned(scales, 4) || !aligned(mins, 4) || !aligned(packed, 16))
    return W4G128_ERR_ALIGN;
  if (w4g128::fault_hook() != W4G128_OK) return w4g128::fault_hook();
  if (!w4g128::device_is_sm103()) return W4G128_ERR_DEVICE;
  return w4g128::launch_unpack(packed, K, N, codes, scales, mins, as_stream(stream));
}

int w4g128_quantize(const w4g128_bf16* w, int K, int N, int search, uint32_t* codes, w4g128_bf16* scales,
                    w4g128_bf16* mins, void* stream) {
  if (w == nullptr || codes == nullptr || scales == nullptr || mins == nullptr) return W4G128_ERR_INVALID_ARG;
  if (search != 0 && search != 1) return W4G128_ERR_INVALID_ARG;
  if (!shape_ok(K, N)) return W4G128_ERR_SHAPE;
  if (!aligned(w, 4) || !aligned(codes, 4) || !aligned(scales, 4) || !aligned(mins, 4)) return W4G128_ERR_ALIGN;
  if (w4g128::fault_hook() != W4G128_OK) return w4g128::fault_hook();
  if (!w4g128::device_is_sm103()) return W4G128_ERR_DEVICE;
  return w4g128::launch_quantize(w, K, N, search, codes, scales, mins, as_stream(stream));
}

size_t w4g128_workspace_bytes(int M, int K, int N) {
  const w4g128_matrix m{nullptr, nullptr, nullptr, K, N};
  return stream_bytes(&m, 1, M);
}

int w4g128_gemv(const void* packed, const w4g128_bf16* x, w4g128_bf16* y, int K, int N, void* ws,
                size_t ws_bytes, void* stream) {
  const w4g128_matrix m{packed, x, y, K, N};
  return run_stream(&m, 1, 1, ws, ws_bytes, stream);
}

int w4g128_gemm_verify(const void* packed, const w4g128_bf16* x, w4g128_bf16* y, int M, int K, int N,
                       void* ws, size_t ws_bytes, void* stream) {
  const w4g128_matrix m{packed, x, y, K, N};
  return run_stream(&m, 1, M, ws, ws_bytes, stream);
}

size_t w4g128_decode_step_workspace_bytes(const w4g128_matrix* mats, int count, int M) {
  return stream_bytes(mats, count, M);
}

int w4g128_schedule(const w4g128_matrix* mats, int count, int M, long long* out, int n) {
  if (mats == nullptr || out == nullptr || n < 1 || count < 1 || count > W4G128_MAX_MATRICES || M < 1 ||
      M > W4G128_MAX_M)
    return W4G128_ERR_INVALID_ARG;
  HostMatrix hm[W4G128_MAX_MATRICES];
  for (int i = 0; i < count; ++i) {
    if (!shape_ok(mats[i].K, mats[i].N)) return W4G128_ERR_SHAPE;
    hm[i] = HostMatrix{mats[i].packed, mats[i].x, mats[i].y, mats[i].K, mats[i].N};
  }
  if (!w4g128::device_is_sm103()) return W4G128_ERR_DEVICE;
  return w4g128::describe_schedule(hm, count, M, out, n);
}

int w4g128_decode_step(const w4g128_matrix* mats, int count, int M, void* ws, size_t ws_bytes, void* stream) {
  return run_stream(mats, count, M, ws, ws_bytes, stream);
}

int w4g128_decode_step_host(const w4g128_matrix* mats, int count, int M, const void* x_host, void* x_dev,
                            size_t x_bytes, void* y_host, const void* y_dev, size_t y_bytes, void* ws,
                            size_t ws_bytes, void* stream) {
  if ((x_bytes > 0 && (x_host == nullptr || x_dev == nullptr)) ||
      (y_bytes > 0 && (y_host == nullptr || y_dev == nullptr)))
    return W4G128_ERR_INVALID_ARG;
  int rc = check_stream_call(mats, count, M, ws);
  if (rc != W4G128_OK) return rc;
  rc = w4g128::fault_hook();
  if (rc != W4G128_OK) return rc;
  if (!w4g128::device_is_sm103()) return W4G128_ERR_DEVICE;
  const cudaStream_t s = as_stream(stream);
  // Pinned (device-mapped) host buffers move through small kernels that keep
  // the chain of programmatic dependent launches; other memory through the
  // copy engines.
  if (x_bytes > 0) {
    const void* xh = aligned(x_dev, 16) ? w4g128::mapped_host(x_host, x_bytes) : nullptr;
    if (xh != nullptr) {
      rc = w4g128::launch_upload(xh, x_dev, x_bytes, s);
      if (rc != W4G128_OK) return rc;
    } else if (cudaMemcpyAsync(x_dev, x_host, x_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
      cudaGetLastError();
      return W4G128_ERR_CUDA;
    }
  }
  rc = run_stream(mats, count, M, ws, ws_bytes, stream);
  if (rc != W4G128_OK) return rc;
  if (y_bytes > 0) {
    const void* yh = aligned(y_dev, 16) ? w4g128::mapped_host(y_host, y_bytes) : nullptr;
    if (yh != nullptr) {
      rc = w4g128::launch_download(y_dev, const_cast<void*>(yh), y_bytes, s);
      if (rc != W4G128_OK) return rc;
    } else if (cudaMemcpyAsync(y_host, y_dev, y_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) {
      cudaGetLastError();
      return W4G128_ERR_CUDA;
    }
  }
  return W4G128_OK;
}

int w4g128_verify_step(const w4g128_matrix* mats, int count, int M, void* ws, size_t ws_bytes, void* stream) {
  return run_stream(mats, count, M, ws, ws_bytes, stream);  // one arithmetic at every M
}

int w4g128_gemm_add_rmsnorm(const void* packed, const w4g128_bf16* x, const w4g128_bf16* residual,
                            const w4g128_bf16* gamma, float eps, w4g128_bf16* h, w4g128_bf16* out, int M, int K,
                            int N, int verify, void* ws, size_t ws_bytes, void* stream) {
  if (residual == nullptr || gamma == nullptr || out == nullptr) return W4G128_ERR_INVALID_ARG;
  if (!(eps >= 0.0f && eps <= 3.0e38f)) return W4G128_ERR_INVALID_ARG;  // finite, not negative, not NaN
  if (verify != 0 && verify != 1) return W4G128_ERR_INVALID_ARG;
  if (out == h || out == residual || out == x || static_cast<const void*>(h) == static_cast<const void*>(x))
    return W4G128_ERR_INVALID_ARG;
  if (!aligned(residual, 4) || !aligned(gamma, 4) || !aligned(out, 4)) return W4G128_ERR_ALIGN;
  const w4g128_matrix m{packed, x, h, K, N};
  const w4g128::NormArgs norm{residual, gamma, out, eps};
  return run_stream(&m, 1, M, ws, ws_bytes, stream, &norm);
}

int w4g128_workspace_status(const void* ws, int* status_out, void* stream) {
  if (ws == nullptr || status_out == nullptr) return W4G128_ERR_INVALID_ARG;
  return w4g128::read_workspace_status(ws, status_out, as_stream(stream));
}

}  // extern "C"

/*
 * Bandwidth probes shipped with libw4g128, used to state GEMV throughput as a
 * fraction of what this GPU's HBM actually delivers.  The Token Rush README
 * ("bandwidth ceiling" paragraph) quotes decode speed against the measured
 * read bandwidth of the card; these two kernels measure it here: a pure read
 * stream and a plain copy.  They are not part of the GEMV path.
 */
#ifndef W4G128_PROBE_H
#define W4G128_PROBE_H

#include <stddef.h>
#include <stdint.h>

#include "w4g128.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Reads `bytes` (a multiple of 16) from the device buffer `buf` (16-byte
 * aligned) once with 128-bit streaming loads spread over every SM, and
 * writes one 32-bit XOR digest per thread block into `sink` (device, at least
 * w4g128_probe_sink_bytes() bytes) so the reads cannot be elided.
 * Asynchronous on `stream`; time it with CUDA events. */
W4G128_API int w4g128_probe_read(const void* buf, size_t bytes, void* sink, void* stream);

/* Copies `bytes` (a multiple of 16) from src to dst (both device, 16-byte
 * aligned, not overlapping).  Asynchronous on `stream`. */
W4G128_API int w4g128_probe_copy(const void* src, void* dst, size_t bytes, void* stream);

/* Size of the sink buffer w4g128_probe_read needs on the current device. */
W4G128_API size_t w4g128_probe_sink_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* W4G128_PROBE_H */

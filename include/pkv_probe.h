/*
 * pkv_probe.h -- read-bandwidth probes of the device's HBM.
 *
 * A measurement aid, not part of the decode path (the pages have no counterpart):
 * the decode kernels only read the KV pool, so their roofline is the rate at which
 * the GPU can stream bytes out of HBM, which a copy benchmark (reading and writing)
 * does not give.  Each probe reads every byte of a caller buffer once and writes one
 * 32-bit word per CTA to `sink` (so that the reads cannot be optimised away).  Time a
 * call with CUDA events on its stream; use a buffer much larger than the L2 cache.
 *
 *   pkv_probe_read_ldg  16-byte vector loads (non-coherent, L1 no-allocate) by
 *                       `ctas_per_sm` CTAs of 512 threads per SM, four loads in
 *                       flight per thread.
 *   pkv_probe_read_bulk one-dimensional TMA bulk copies (cp.async.bulk) of 32 KiB
 *                       into a three-stage shared-memory ring per CTA, `ctas_per_sm`
 *                       CTAs per SM (1 or 2), the copy engine the decode kernels use.
 *                       Every wait is bounded; a wait that gives up counts in
 *                       sink[gridDim] (must then be 0).
 *
 * buf: device pointer, 16-byte aligned; bytes: a multiple of 32768 (bulk) or 16
 * (ldg), at least one chunk.  sink: device array of at least (number of SMs x
 * ctas_per_sm + 1) uint32.  Returns PKV_OK, PKV_ERR_INVALID_ARG or PKV_ERR_CUDA;
 * launches are asynchronous on the stream.
 */
#ifndef PKV_PROBE_H
#define PKV_PROBE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int pkv_probe_read_ldg(const void *buf, size_t bytes, uint32_t *sink, int ctas_per_sm, void *cuda_stream);
int pkv_probe_read_bulk(const void *buf, size_t bytes, uint32_t *sink, int ctas_per_sm, void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif

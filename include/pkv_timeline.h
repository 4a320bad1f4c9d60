/*
 * pkv_timeline.h -- per-CTA timeline of the fused decode step's grid schedule.
 *
 * A measurement aid, not part of the decode path: only a library compiled with
 * -DPKV_TIMELINE (paged_kv_decode_12_gb300._build.build(timeline=True), which
 * writes libpkv_timeline.so beside libpkv.so) records it and exports the function
 * below; the default libpkv.so has neither the records nor the symbol.
 *
 * Each launch of the BF16 grid kernel (pkv_decode_step, and pkv_decode_attention
 * without PKV_DECODE_SPLIT_MERGE) stores, for every CTA linear index
 * i = x + 8 (y + B z) below 16384:
 *   stamps[i][0..4]  %globaltimer (ns) at CTA entry, once its work unit is known,
 *                    after the wait for the previous launch, after its page loop,
 *                    and at its end (after the combine / merge);
 *   meta[i][0..3]    SM id, sequence, chunk, pages of the unit; SM = -1 for a CTA
 *                    without a unit (an empty chunk slot, or an invalid length).
 * Later launches overwrite the same indices, so read it after the launch of interest.
 */
#ifndef PKV_TIMELINE_H
#define PKV_TIMELINE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Copy the first n records (n <= 16384) to host arrays stamps[n][5] and meta[n][4].
 * Synchronous (cudaMemcpyFromSymbol on the legacy stream, after all prior work on the
 * device).  Returns the number of records copied, PKV_ERR_INVALID_ARG (-1) for null
 * pointers or n < 1, PKV_ERR_CUDA (-4) on a copy error. */
int pkv_timeline_read(uint64_t *stamps, int32_t *meta, int n);

#ifdef __cplusplus
}
#endif

#endif

/*
 * mla_calibration.h -- a measurement aid shipped in libmla_combine_uv: a
 * read-only streaming kernel that gives the fastest time one launch of this
 * library's launch shape can take to read a given number of bytes.
 *
 * It has no counterpart on the pages that define the stage; the bench uses it
 * to measure, in the same harness as the decode-size combine calls (a CUDA
 * graph of back-to-back launches with programmatic dependent launch, inputs
 * rotated so that every launch reads HBM), the ceiling that any single kernel
 * of that byte count meets: launch, ramp-up and the HBM round trips.
 */
#ifndef MLA_CALIBRATION_H
#define MLA_CALIBRATION_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * mla_calib_stream_read -- enqueue on `stream` one kernel that reads `bytes`
 * bytes starting at device pointer `src` with 16-byte streaming loads, every
 * thread's loads in flight before any is used, and writes nothing unless the
 * xor of everything read equals a fixed 32-bit pattern (then one word at
 * `sink`, a device uint32).  `dependent_round_trips` (0..4) first reads that
 * many words one after another, each address depending on the word before
 * (as a kernel that must read its LSE values before its rows), before the
 * stream starts.  Launched with programmatic stream serialization: it waits
 * for the previous kernel on the stream before its first read and lets the
 * next one begin its prologue at once.
 * Returns 0 once enqueued; 2 (MLA_ERR_SHAPE) for bytes < 16, a byte count
 * not a multiple of 16 or dependent_round_trips outside 0..4; 4
 * (MLA_ERR_ALIGN) for a `src` not 16-byte aligned; 1 (MLA_ERR_NULL) for a
 * NULL pointer; 7 (MLA_ERR_CUDA) if the launch fails.
 */
int32_t mla_calib_stream_read(const void *src, int64_t bytes, int32_t dependent_round_trips, uint32_t *sink,
                              void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_CALIBRATION_H */

/*
 * The index-checked debug build of the verifier library (libspecverify_debug.so: the same
 * sources compiled with -DSPEC_DEBUG). It exports everything include/spec_verify.h declares, with
 * the same behaviour, plus the call below. Its kernels check each index of their main global
 * accesses (logit rows and vectors, the workspace's per-chunk and per-row arrays, the per-row and
 * per-request outputs, the compaction's packed outputs, the truncation cuts) against the array's
 * length. A failed check does not trap: it records the first failure and skips the access.
 *
 * The pages define no such build: it is a test aid of this library, for runs where a memory
 * checker is not available.
 */
#ifndef SPEC_DEBUG_H
#define SPEC_DEBUG_H

#include <stdint.h>

#include "spec_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Waits for the device (cudaDeviceSynchronize), then reads and clears the library's debug words:
 * out[0] the first failure's code (0: none; 1 logit rows, 2 per-chunk workspace, 3 per-row
 * workspace, 4 per-row outputs, 5 per-request outputs, 6 packed outputs, 7 truncation cuts),
 * out[1] its source line, out[2] its index (low 32 bits), out[3] the number of failures.
 * out: host array of 4 words, owned by the caller. Returns SPEC_ERR_INVALID_ARG for a NULL out,
 * SPEC_ERR_CUDA when the device or the copy fails, else SPEC_OK. */
spec_status spec_debug_fetch(unsigned int *out);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_DEBUG_H */

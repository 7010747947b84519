/*
 * spl_calib.h: data-movement reference kernels, for calibrating the codec kernels' roofline.
 * They have no counterpart on the pages and do none of the codec's arithmetic: each moves the
 * bytes of one codec kernel the way that kernel moves them (the same chunking, the same bulk
 * copies into a shared-memory stage completing on an mbarrier, the same stores, the same CTA
 * size, CTAs per SM and order of chunks) and does one trivial operation per value, so that its
 * time is the floor the codec kernel's own access pattern sets on this GPU.
 *
 *   SPL_CALIB_SENDER_MOVES   out0[i] = in0[i] + in1[i]   (fp32, rounded to nearest)
 *       the sender's movement: per 4,096-value chunk, in0 (the error buffer's place) and in1
 *       (delta's) arrive by two 16 KB bulk copies in one stage, the next chunk's copies start
 *       once every thread has read the stage, and out0 is written with plain 16-byte stores;
 *       12 bytes per value.  in1 and out0 may not be NULL; out1 is unused.
 *   SPL_CALIB_RECEIVER_MOVES out0[i] = -in0[i], out1[i] = in0[i]
 *       the receiver's dense movement with the outer step fused: per chunk, in0 (theta's place)
 *       arrives by one 16 KB bulk copy into one stage, and out0 (the mean's place) and out1
 *       (theta's) are written with plain 16-byte stores; 12 bytes per value.  in1 is unused.
 *
 * persistent: 0: chunks in the codec kernel's order (waves of resident CTAs, 16 chunks each
 *           for the sender, 32 for the receiver);
 *           nonzero: one persistent wave, each resident CTA taking every resident-th chunk
 *           (the order the codec kernels used before; for comparison)
 * n:        a multiple of 4,096 (SPL_ERR_INVALID_ARG otherwise); 0 does nothing
 * in0, in1, out0, out1: device memory, 16-byte aligned (SPL_ERR_ALIGNMENT), n fp32 each,
 *           no output overlapping another array (SPL_ERR_INVALID_ARG)
 * d_flags:  device uint32 or NULL; SPL_FLAG_TIMEOUT (and SPL_FLAG_COPY_PENDING) as for the
 *           codec calls if a bulk copy does not land within the bounded wait
 * The call enqueues one kernel on the stream, allocates nothing and does not synchronise.
 */
#ifndef SPL_CALIB_H_
#define SPL_CALIB_H_

#include <stddef.h>
#include <stdint.h>

#include "spl.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SPL_CALIB_SENDER_MOVES = 0, SPL_CALIB_RECEIVER_MOVES = 1 } spl_calib_pattern;

spl_status spl_calib_moves(spl_calib_pattern pattern, int persistent, const float* in0,
                           const float* in1, float* out0, float* out1, size_t n,
                           uint32_t* d_flags, spl_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPL_CALIB_H_ */

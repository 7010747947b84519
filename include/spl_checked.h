/*
 * spl_checked.h: the one extra entry point of the library's checked build (libspl_checked.so),
 * a diagnostic build of the same kernels compiled with -DSPL_CHECKED=1.  It has no counterpart
 * on the pages: it exists to test the kernels' memory accesses without a memory checker.
 *
 * In the checked build every shared- and global-memory index of the kernels is tested before
 * the access.  An index out of range does not trap: the kernel records it in a device-side
 * debug array and skips the access (so its outputs may then be wrong).  The same arrays count
 * which select path each sender chunk took.  The normal library (libspl.so) has neither the
 * checks nor this call; every call of spl.h behaves the same in both builds.
 */
#ifndef SPL_CHECKED_H_
#define SPL_CHECKED_H_

#include <stdint.h>

#include "spl.h"

#ifdef __cplusplus
extern "C" {
#endif

enum {
    SPL_DEBUG_WORDS = 16,
    SPL_DEBUG_SITES = 0,       /* OR of (1 << site) over the failed checks (0: none failed) */
    SPL_DEBUG_FIRST_SITE = 1,  /* site + 1 of the first failed check (0: none) */
    SPL_DEBUG_FIRST_INDEX = 2, /* the index that failed it (low 32 bits) */
    SPL_DEBUG_FAILURES = 3,    /* failed checks */
    SPL_DEBUG_CHUNKS = 8,      /* sender chunks on the fast flow (device-resident error buffer) */
    SPL_DEBUG_WHOLE = 9,       /* ... whose boundary bin was taken whole */
    SPL_DEBUG_RANK32 = 10,     /* ... whose boundary bin of <= 32 keys was ranked */
    SPL_DEBUG_RANK64 = 11,     /* ... whose boundary bin of 33..64 keys was ranked */
    SPL_DEBUG_FULL_SCAN = 12,  /* ... whose bin search went past the top 512 bins */
    SPL_DEBUG_GENERIC = 13     /* ... that took the generic radix select */
};

/*
 * Copies the debug words accumulated since the last reset (all kernels, all calls on the
 * current device) into out[SPL_DEBUG_WORDS] and, when reset is nonzero, clears them.  Waits for
 * the device (it copies device symbols).  SPL_ERR_INVALID_ARG for a NULL out, SPL_ERR_CUDA if a
 * copy fails.  Exported by libspl_checked.so only.
 */
spl_status spl_debug_read(uint32_t* out, int reset);

#ifdef __cplusplus
}
#endif

#endif /* SPL_CHECKED_H_ */

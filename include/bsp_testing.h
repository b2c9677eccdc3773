/*
 * bsp_testing.h - switches of the test build of the library only.
 *
 * These entry points exist in libbsp_test.so (the same sources built with
 * BSP_TESTING defined) and not in libbsp.so: a production library cannot be
 * told to skip its copies or to give up its waits early.  They have no
 * counterpart on the pages; the tests use them to make a bounded
 * device-side wait run out, and check that the kernel then reports
 * BSP_ERR_TIMEOUT and the next call is correct.
 */
#ifndef BSP_TESTING_H
#define BSP_TESTING_H

#include <stdint.h>

#include "bsp.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * on = 1: the producers of every product kernel launched afterwards skip
 * the copies of their first tile, so the wait for it can only run out.
 * on = 0 restores normal operation.  BSP_ERR_INVALID_ARG for other values.
 */
bsp_status_t bsp_testing_set_stall(int on);

/*
 * Polls of a device-side wait before it gives up, for kernels launched
 * afterwards; 0 restores the library's default.  A short cap (a few
 * thousand polls) makes a stalled wait end in microseconds.
 */
bsp_status_t bsp_testing_set_spin_cap(uint32_t polls);

#ifdef __cplusplus
}
#endif

#endif /* BSP_TESTING_H */

/*
 * mla_decode_debug.h -- test hook of the debug build of the MLA decode library
 * (libmla_decode_debug.so, the same sources compiled with MLA_DEBUG).  The
 * product library does not export it.
 *
 * Every wait inside the split-KV kernel is bounded; when one runs out the
 * kernel records MLA_ERR_TIMEOUT in the workspace's error word, every role of
 * the cluster gives up, lets copies already in flight land, writes the
 * affected rows as NaN and exits, leaving the context usable.  A healthy call
 * never comes near the built-in limit (1 s), so the path can only be exercised
 * by shortening it: this hook makes a surfaced error visible without breaking
 * anything on the device (the TokenSpeed MLA summary, risks and impact item 6,
 * warns that failures hidden behind a fallback go unnoticed).
 */
#ifndef MLA_DECODE_DEBUG_H_
#define MLA_DECODE_DEBUG_H_

#include <stdint.h>

#include "mla_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * mla_debug_set_wait_limit_ns -- limit of every bounded device wait of the
 * launches that follow, in nanoseconds (0 restores the built-in 1 s).  Process
 * wide, not thread safe; host only.
 */
mla_status_t mla_debug_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_DEBUG_H_ */

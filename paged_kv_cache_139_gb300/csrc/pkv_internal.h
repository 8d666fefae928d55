// Host-side helpers shared by the library's translation units.
#pragma once

#include <cstdint>

#include "pkv.h"

namespace pkv {

// Record a printf-style message as this thread's last error; returns `st`.
pkv_status fail(pkv_status st, const char *fmt, ...)
#if defined(__GNUC__)
    __attribute__((format(printf, 2, 3)))
#endif
    ;

// Count `n` kernel launches made by the library.
void count_launches(int n);

// How many times pkv_check has reported (and cleared) a device-wait timeout
// on the current device.  A kernel that gave up may leave the work-ticket
// counters of its workspace mid-count, so scratch the library prepares itself
// is prepared again whenever this number changes.
unsigned int timeout_epoch();

}  // namespace pkv

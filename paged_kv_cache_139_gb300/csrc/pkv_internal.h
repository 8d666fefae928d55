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

}  // namespace pkv

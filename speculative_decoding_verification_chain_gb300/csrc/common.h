// Host helpers shared by the translation units of libspecverify.
#pragma once

#include "spec_verify.h"

namespace sv {

// Clears the message spec_last_error() returns (at the start of a call).
void clear_error();

// Records the message (fmt with one %s for detail) for spec_last_error() and
// returns s.
spec_status_t fail(spec_status_t s, const char *fmt, const char *detail = "");

// SPEC_OK when the current device is compute capability 10.3; fills *sms with
// its SM count.
spec_status_t require_sm103(int *sms);

// Limit in nanoseconds of the kernels' waits on other blocks and warps
// (spec_set_wait_limit_ns); copies still in flight at a kernel's exit are
// always waited for with the default limit.
unsigned long long wait_limit_ns();

}  // namespace sv

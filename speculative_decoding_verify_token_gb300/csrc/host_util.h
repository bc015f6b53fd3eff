// Host-side helpers of the specverify library: per-thread error text.
#pragma once

#include "specverify.h"

namespace sv {
// Record `code` with a printf-style description for spec_last_error(); returns `code`.
int set_error(int code, const char* fmt, ...);
void clear_error();
}  // namespace sv

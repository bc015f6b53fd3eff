// Per-thread last-error text of the C ABI.
#include <cstdarg>
#include <cstdio>

#include "host_util.h"

namespace sv {

static thread_local char g_err[512] = "";

int set_error(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

void clear_error() { g_err[0] = '\0'; }

}  // namespace sv

extern "C" const char* spec_last_error(void) { return sv::g_err; }

extern "C" const char* spec_version(void) { return "specverify 0.1 (sm_103a)"; }

// Thread-local error message and version for the libpa C ABI.
#include <cstdarg>
#include <cstdio>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {
thread_local char g_msg[512] = "";
}

namespace pa {

int set_error(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return code;
}

}  // namespace pa

extern "C" const char *pa_last_error(void) { return g_msg; }

extern "C" int pa_version(void) { return 10000; }  // 1.0.0

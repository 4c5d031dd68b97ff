// Internal declarations shared by libpa's translation units.
#pragma once

#include <cstdarg>

namespace pa {

// Record a message for pa_last_error() on the calling thread; returns `code`.
int set_error(int code, const char *fmt, ...);

}  // namespace pa

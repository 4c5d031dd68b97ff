// Internal declarations shared by libpa's translation units.
#pragma once

#include <cstdarg>

namespace pa {

// Record a message for pa_last_error() on the calling thread; returns `code`.
int set_error(int code, const char *fmt, ...);

// Read and clear the prefill kernels' device error word (PA_DEVERR_* bits)
// on the current device. Returns a cudaError_t value (0 on success).
int prefill_take_device_error(int *bits);

}  // namespace pa

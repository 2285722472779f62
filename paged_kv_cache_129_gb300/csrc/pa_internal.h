// Host-side helpers shared by the C-ABI translation units (no device code).
#pragma once

#include <cstdarg>
#include <cstddef>

namespace pa {

// Record a thread-local error message and return `code` (for `return fail(...)`).
int fail(int code, const char* fmt, ...);

// Clear the thread-local message (called on success paths that want it empty).
void clear_error();

}  // namespace pa

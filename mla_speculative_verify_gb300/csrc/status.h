// status.h -- thread-local error message behind mla_last_error().
#pragma once

namespace mla {

// Record a printf-style message for mla_last_error() and return `code`.
int set_error(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
void clear_error();

}  // namespace mla

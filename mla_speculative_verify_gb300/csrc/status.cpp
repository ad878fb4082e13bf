// status.cpp -- thread-local error message behind mla_last_error().
#include "status.h"

#include <cstdarg>
#include <cstdio>

#include "mla_decode.h"

namespace mla {

static thread_local char g_error[512] = "";

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_error, sizeof g_error, fmt, ap);
  va_end(ap);
  return code;
}

void clear_error() { g_error[0] = '\0'; }

}  // namespace mla

extern "C" const char* mla_last_error(void) { return mla::g_error; }

extern "C" int mla_version(void) { return 100; }

// Thread-local error messages and the library version.
#include <cstdarg>
#include <cstdio>

#include "pagedattn.h"
#include "status.h"

namespace {
thread_local char g_message[512] = "no error";
}

namespace pa {

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_message, sizeof(g_message), fmt, ap);
  va_end(ap);
  return code;
}

}  // namespace pa

extern "C" {

PA_API const char* pa_last_error(void) { return g_message; }

PA_API int pa_version(void) { return 100; }

}  // extern "C"

#include "status.h"

#include <cstdarg>
#include <cstdio>

namespace {
thread_local char g_msg[512] = "";
}

namespace gtp {
gtp_status fail(gtp_status s, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return s;
}
void clear_error() { g_msg[0] = '\0'; }
}  // namespace gtp

extern "C" const char *gtp_last_error(void) { return g_msg; }

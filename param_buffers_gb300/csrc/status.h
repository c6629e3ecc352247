// Error reporting shared by the C-ABI entry points: a status code plus a thread-local
// message readable through gtp_last_error().
#pragma once
#include "gtp.h"

namespace gtp {
// Records a printf-style message for gtp_last_error() and returns `s`.
gtp_status fail(gtp_status s, const char *fmt, ...)
#if defined(__GNUC__)
    __attribute__((format(printf, 2, 3)))
#endif
    ;
// Clears the message; entry points call it on entry.
void clear_error();
}  // namespace gtp

// libvc_core: status strings and the per-thread last-error text shared by the
// four compute libraries (see include/vc.h, "Conventions").
#include <cstdarg>
#include <cstdio>

#include "vc.h"
#include "vc_internal.h"

namespace {
thread_local char g_last_error[512] = "";
}

extern "C" const char* vc_status_str(vc_status_t s) {
  switch (s) {
    case VC_OK: return "ok";
    case VC_ERR_INVALID_ARG: return "invalid argument";
    case VC_ERR_UNSUPPORTED: return "unsupported configuration";
    case VC_ERR_CUDA: return "CUDA error";
    case VC_ERR_TIMEOUT: return "timed out";
    case VC_ERR_WORKSPACE: return "workspace missing or too small";
    case VC_ERR_CAPACITY: return "capacity exceeded";
  }
  return "unknown status";
}

extern "C" const char* vc_last_error(void) { return g_last_error; }

extern "C" vc_status_t vc_internal_fail(vc_status_t s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

extern "C" void vc_internal_clear(void) { g_last_error[0] = '\0'; }

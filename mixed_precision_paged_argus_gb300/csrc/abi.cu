// Host-side status reporting shared by every entry point of the C ABI.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "common.cuh"

namespace argus {

static thread_local char g_last_error[512] = "";

argus_status fail(argus_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

argus_status launch_status(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    return fail(ARGUS_E_LAUNCH, "%s: launch failed: %s", what, cudaGetErrorString(e));
  }
  return ARGUS_OK;
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

}  // namespace argus

extern "C" const char* argus_status_string(argus_status s) {
  switch (s) {
    case ARGUS_OK: return "ok";
    case ARGUS_E_INVALID: return "invalid argument";
    case ARGUS_E_UNSUPPORTED: return "unsupported shape or codec";
    case ARGUS_E_WORKSPACE: return "workspace too small";
    case ARGUS_E_LAUNCH: return "kernel launch failed";
  }
  return "unknown status";
}

extern "C" const char* argus_last_error(void) { return argus::g_last_error; }

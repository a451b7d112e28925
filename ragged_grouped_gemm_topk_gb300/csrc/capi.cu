// Host-side pieces of the C ABI shared by every entry point: error text, launch
// checks, device capability checks and the library version.
#include <stdarg.h>
#include <stdio.h>

#include "common.cuh"

namespace moe {

namespace {
thread_local char g_err[512] = "";

struct DevInfo {
  int checked = 0;  // 0 unknown, 1 ok, -1 not sm_103
  int sms = 0;
};
DevInfo g_dev[64];
}  // namespace

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

moe_status_t check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("%s: launch failed: %s", what, cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool device_is_sm103(int* sm_count) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    set_error("no current CUDA device");
    return false;
  }
  DevInfo& di = g_dev[dev];
  if (di.checked == 0) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    di.sms = sms;
    di.checked = (major == 10 && minor == 3) ? 1 : -1;
    if (di.checked < 0)
      set_error("device %d is sm_%d%d; libmoe is built for sm_103a only", dev, major, minor);
  }
  if (sm_count) *sm_count = di.sms;
  if (di.checked < 0) {
    set_error("device %d is not sm_103; libmoe is built for sm_103a only", dev);
    return false;
  }
  return true;
}

}  // namespace moe

extern "C" int moe_version(void) { return (0 << 16) | (1 << 8) | 0; }

extern "C" const char* moe_last_error_string(void) { return moe::g_err; }

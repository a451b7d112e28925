// Host-side pieces of the C ABI shared by every entry point: error text, launch
// checks, device capability checks and the library version.
#include <stdarg.h>
#include <stdio.h>

#include <atomic>

#include "common.cuh"

namespace moe {

namespace {
thread_local char g_err[512] = "";

// Per-device capability cache, safe to fill from several host threads: the SM
// count is stored before the capability flag, which is published with release order.
struct DevInfo {
  std::atomic<int> checked{0};  // 0 unknown, 1 ok, -1 not sm_103
  std::atomic<int> sms{0};
};
constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
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

moe_status_t device_check(int* sm_count) {
  int dev = 0;
  const cudaError_t ge = cudaGetDevice(&dev);
  if (ge != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    set_error("no usable current CUDA device: %s", ge != cudaSuccess ? cudaGetErrorString(ge) : "ordinal out of range");
    return ge != cudaSuccess ? MOE_ERR_CUDA : MOE_ERR_UNSUPPORTED;
  }
  DevInfo& di = g_dev[dev];
  int capable = di.checked.load(std::memory_order_acquire);
  if (capable == 0) {
    // a failed query (for example a sticky error of an earlier call) is reported
    // as a CUDA error and not cached: the next call asks again
    int major = 0, minor = 0, sms = 0;
    cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
      set_error("device %d: attribute query failed: %s", dev, cudaGetErrorString(e));
      return MOE_ERR_CUDA;
    }
    capable = (major == 10 && minor == 3 && sms > 0) ? 1 : -1;
    di.sms.store(sms, std::memory_order_relaxed);
    di.checked.store(capable, std::memory_order_release);
  }
  if (sm_count) *sm_count = di.sms.load(std::memory_order_relaxed);
  if (capable < 0) {
    set_error("device %d is not sm_103; libmoe is built for sm_103a only", dev);
    return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

}  // namespace moe

extern "C" int moe_version(void) { return (0 << 16) | (1 << 8) | 0; }

extern "C" const char* moe_last_error_string(void) { return moe::g_err; }

namespace moe {
namespace {

// One CTA waits on an mbarrier that nothing ever arrives at, through the same
// bounded wait every pipeline stage of the GEMM uses, with a caller-chosen limit.
__global__ void wait_timeout_kernel(int32_t* status, uint64_t limit_ns) {
  pdl_begin();
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, status, &abort_flag, limit_ns);
}

// One thread runs a device-side check that always fails.
__global__ void debug_selftest_kernel(int32_t* status) {
  pdl_begin();
  if (threadIdx.x == 0) (void)dbg_check(status == nullptr, status);
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_debug_selftest(int32_t* dev_status, int* is_debug, cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_debug_selftest");
  using namespace moe;
#ifdef MOE_DEBUG
  const int dbg = 1;
#else
  const int dbg = 0;
#endif
  if (is_debug) *is_debug = dbg;
  if (!dev_status) {
    set_error("moe_debug_selftest: need a status word");
    return MOE_ERR_INVALID_ARG;
  }
  int sms = 0;
  if (const moe_status_t dst = device_check(&sms); dst != MOE_OK) return dst;
  launch_pdl(debug_selftest_kernel, 1, 32, 0, stream, dev_status);
  return check_launch("moe_debug_selftest");
}

extern "C" moe_status_t moe_check_wait_timeout(int32_t* dev_status, int limit_us, cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_check_wait_timeout");
  using namespace moe;
  if (!dev_status || limit_us < 1 || limit_us > 2000000) {
    set_error("moe_check_wait_timeout: need a status word and 1 <= limit_us <= 2000000");
    return MOE_ERR_INVALID_ARG;
  }
  int sms = 0;
  if (const moe_status_t dst = device_check(&sms); dst != MOE_OK) return dst;
  launch_pdl(wait_timeout_kernel, 1, 32, 0, stream, dev_status, static_cast<uint64_t>(limit_us) * 1000ull);
  return check_launch("moe_check_wait_timeout");
}

// moe_permute_noalloc: the dispatch of moe_permute for callers that cannot
// allocate device memory.
//
// Some callers are handed device pointers and nothing else: a plugin running
// inside another runtime that owns the allocator, a serving process whose whole
// device memory was reserved up front by its own pool, or code that must not
// allocate while a stream is being captured.  They cannot cudaMalloc the scratch
// buffer moe_permute asks for.  This entry point uses a fixed scratch array that
// lives in the library's own device memory instead.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchInts int32
// (1 MiB).  Every GPU that loads the library holds it until the process exits.
// It stores the per-block, per-expert histogram of the rank kernel, which needs
// ceil(T / 256) * E entries; larger problems are rejected with
// MOE_ERR_WORKSPACE.  Every entry the kernels read is written earlier in the
// same call, so nothing has to start at zero, but every call shares the one
// array: two calls whose kernels overlap on the GPU (different streams, or
// different host threads) race on it and give wrong results.
//
// In host code the array's name is only a host-side stand-in, so its device
// address is looked up with cudaGetSymbolAddress, with the device current, on the
// first call made in each CUDA context (normally once per device; again after the
// device's primary context was reset).  Make that first call before any stream
// capture.
#include <mutex>
#include <vector>

#include "common.cuh"

namespace moe {

moe_status_t permute_validate(const void* x, moe_dtype_t x_dtype, int T, int d,
                              const int32_t* topk_idx, int k, int E, const int32_t* counts,
                              int32_t* offsets, int32_t* dest_row, int32_t* src_pair, void* xp,
                              moe_dtype_t xp_dtype, uint8_t* xp_scales);
moe_status_t permute_launch(const void* x, moe_dtype_t x_dtype, int T, int d,
                            const int32_t* topk_idx, int k, int E, const int32_t* counts,
                            int32_t* offsets, int32_t* dest_row, int32_t* src_pair, void* xp,
                            moe_dtype_t xp_dtype, uint8_t* xp_scales, int32_t* hist,
                            int32_t* dev_status, cudaStream_t stream, int sms,
                            uint32_t* amax_bits, float* tensor_scale);
size_t permute_hist_bytes(int T, int E);

namespace {

constexpr size_t kNoAllocScratchInts = 262144;   // 1 MiB

__device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchInts];

// Looked-up addresses, keyed by the CUDA context they belong to.  The key is the
// driver's context id, which no later context reuses: after cudaDeviceReset (or
// any other teardown of the primary context) the new context gets a new id, so
// an address that belonged to the old one is never handed out again.
struct ScratchEntry {
  unsigned long long ctx_id;
  int32_t* ptr;
};
std::mutex g_mu;
std::vector<ScratchEntry> g_scratch;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name, int version) {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &ptr, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(ptr);
}

// Device address of the scratch array in the current context (looked up once per
// context).
int32_t* scratch_in_current_context() {
  // make the runtime bind the current device's primary context if nothing has yet
  // (cudaSetDevice initialises it; it allocates nothing)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) {
    set_error("moe_permute_noalloc: no usable CUDA device");
    return nullptr;
  }
  static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent", 4000);
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId", 12000);
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) {
    set_error("moe_permute_noalloc: cannot identify the current CUDA context");
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  for (const ScratchEntry& e : g_scratch)
    if (e.ctx_id == id) return e.ptr;
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_permute_scratch);
  if (e != cudaSuccess || !ptr) {
    set_error("moe_permute_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
    return nullptr;
  }
  g_scratch.push_back({id, static_cast<int32_t*>(ptr)});
  return static_cast<int32_t*>(ptr);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_permute_noalloc(const void* x, moe_dtype_t x_dtype, int T, int d,
                                            const int32_t* topk_idx, int k, int E,
                                            const int32_t* counts, int32_t* offsets,
                                            int32_t* dest_row, int32_t* src_pair, void* xp,
                                            moe_dtype_t xp_dtype, uint8_t* xp_scales,
                                            int32_t* dev_status, cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_permute_noalloc");
  moe_status_t st = permute_validate(x, x_dtype, T, d, topk_idx, k, E, counts, offsets, dest_row,
                                     src_pair, xp, xp_dtype, xp_scales);
  if (st != MOE_OK) return st;
  if (permute_hist_bytes(T, E) > kNoAllocScratchInts * sizeof(int32_t)) {
    set_error("moe_permute_noalloc: ceil(T/256)*E = %zu int32 exceeds the fixed scratch of %zu "
              "(use moe_permute with a caller workspace)",
              permute_hist_bytes(T, E) / sizeof(int32_t), kNoAllocScratchInts);
    return MOE_ERR_WORKSPACE;
  }
  int sms = 0;
  if (const moe_status_t dst = device_check(&sms); dst != MOE_OK) return dst;
  int32_t* scratch = scratch_in_current_context();
  if (!scratch) return MOE_ERR_CUDA;
  return permute_launch(x, x_dtype, T, d, topk_idx, k, E, counts, offsets, dest_row, src_pair, xp,
                        xp_dtype, xp_scales, scratch, dev_status, stream, sms, nullptr, nullptr);
}

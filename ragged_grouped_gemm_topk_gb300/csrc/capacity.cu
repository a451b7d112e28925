// Capacity-based dispatch: the contrast case of "Accelerating Dropless MoE Training
// in JAX with NVIDIA Transformer Engine" (first section: a fixed per-expert capacity
// pads experts that receive fewer tokens and drops the tokens that overflow the
// busy ones; dropless routing avoids both, which is the point of the method).
//
// Every expert owns exactly C rows of the output, [e*C, (e+1)*C).  Expert e's pairs,
// in the dropless order (token ascending), fill its first min(count_e, C) rows;
// the rest of its rows are zero padding; its pairs past the first C are dropped
// (dest_row = -1, and the combine leaves them out).  The per-expert order comes from
// the dropless maps (the rank kernel of moe_permute), so the kept tokens of an
// expert are exactly its first C tokens.
#include "common.cuh"

namespace moe {

moe_status_t permute_launch(const void* x, moe_dtype_t x_dtype, int T, int d,
                            const int32_t* topk_idx, int k, int E, const int32_t* counts,
                            int32_t* offsets, int32_t* dest_row, int32_t* src_pair, void* xp,
                            moe_dtype_t xp_dtype, uint8_t* xp_scales, int32_t* hist,
                            int32_t* dev_status, cudaStream_t stream, int sms,
                            uint32_t* amax_bits, float* tensor_scale);
size_t permute_hist_bytes(int T, int E);

namespace {

constexpr int kCapThreads = 256;

// Pair p: its dropless row (in dest_row) -> its capacity row, or -1 past capacity.
__global__ void __launch_bounds__(kCapThreads) capacity_remap_kernel(
    const int32_t* __restrict__ topk_idx, int pairs, int E, int C, const int32_t* __restrict__ off_drop,
    int32_t* __restrict__ dest_row, int32_t* status) {
  pdl_begin();
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < pairs; p += gridDim.x * blockDim.x) {
    const int e = topk_idx[p];
    if (e < 0 || e >= E) {            // flagged by the rank kernel already
      dest_row[p] = -1;
      continue;
    }
    const int r = dest_row[p] - off_drop[e];
    if (r < 0) flag_error(status, MOE_DEV_BAD_INDEX);
    dest_row[p] = (r >= 0 && r < C) ? e * C + r : -1;
  }
}

// One warp per capacity row: the row of the token its pair came from, or zeros.
// Also writes the uniform offsets e*C.
__global__ void __launch_bounds__(kCapThreads) capacity_fill_kernel(
    const uint8_t* __restrict__ x, int row_bytes, int k, int E, int C, const int32_t* __restrict__ off_drop,
    const int32_t* __restrict__ src_drop, int32_t* __restrict__ src_pair, int32_t* __restrict__ offsets,
    uint8_t* __restrict__ xp) {
  pdl_begin();
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = e * C;
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const long long rows = static_cast<long long>(E) * C;
  const int n16 = row_bytes / 16;
  for (long long row = static_cast<long long>(blockIdx.x) * wpb + (threadIdx.x >> 5); row < rows;
       row += static_cast<long long>(gridDim.x) * wpb) {
    const int e = static_cast<int>(row / C), r = static_cast<int>(row % C);
    const int beg = off_drop[e], n = off_drop[e + 1] - beg;
    const int pair = r < n ? src_drop[beg + r] : -1;
    if (lane == 0) src_pair[row] = pair;
    uint4* dst = reinterpret_cast<uint4*>(xp + row * row_bytes);
    if (pair >= 0) {
      const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(pair / k) * row_bytes);
      for (int c = lane; c < n16; c += 32) dst[c] = src[c];
    } else {
      for (int c = lane; c < n16; c += 32) dst[c] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

}  // namespace

size_t permute_capacity_workspace_bytes(int T, int k, int E) {
  const size_t pairs = static_cast<size_t>(T > 0 ? T : 0) * static_cast<size_t>(k > 0 ? k : 0);
  return permute_hist_bytes(T, E) + (static_cast<size_t>(E > 0 ? E : 0) + 1) * sizeof(int32_t) +
         pairs * sizeof(int32_t);
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_permute_capacity_workspace_size(int T, int k, int E) {
  return permute_capacity_workspace_bytes(T, k, E);
}

extern "C" moe_status_t moe_permute_capacity(const void* x, moe_dtype_t x_dtype, int T, int d,
                                             const int32_t* topk_idx, int k, int E, int capacity,
                                             const int32_t* counts, int32_t* offsets, int32_t* dest_row,
                                             int32_t* src_pair, void* xp, void* workspace,
                                             size_t workspace_bytes, int32_t* dev_status,
                                             cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_permute_capacity");
  const char* fn = "moe_permute_capacity";
  const int eb = x_dtype == MOE_F32 ? 4 : 2;
  if (T < 0 || d < 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E || capacity < 0 ||
      (x_dtype != MOE_BF16 && x_dtype != MOE_F32) || (d * eb) % 16) {
    set_error("%s: need T, d, capacity >= 0, 1 <= E <= 1024, 1 <= k <= min(E, 32), BF16/F32 rows of a "
              "multiple of 16 bytes", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (static_cast<long long>(T) * k >= (1LL << 31) || static_cast<long long>(E) * capacity >= (1LL << 31)) {
    set_error("%s: T*k and E*capacity must fit in int32", fn);
    return MOE_ERR_INVALID_ARG;
  }
  const bool any_rows = static_cast<long long>(E) * capacity > 0 && d > 0;
  if (!counts || !offsets || (T > 0 && (!topk_idx || !dest_row || !x)) ||
      (any_rows && (!src_pair || !xp)) || !aligned16(x) || !aligned16(xp)) {
    set_error("%s: null or misaligned pointer", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (!workspace || workspace_bytes < permute_capacity_workspace_bytes(T, k, E)) {
    set_error("%s: workspace of %zu bytes needed", fn, permute_capacity_workspace_bytes(T, k, E));
    return MOE_ERR_WORKSPACE;
  }
  int sms = 0;
  if (const moe_status_t dst = device_check(&sms); dst != MOE_OK) return dst;
  // workspace: rank histogram | dropless offsets [E+1] | dropless src_pair [T*k]
  int32_t* hist = static_cast<int32_t*>(workspace);
  int32_t* off_drop = hist + permute_hist_bytes(T, E) / sizeof(int32_t);
  int32_t* src_drop = off_drop + (E + 1);
  const int pairs = T * k;
  // dropless maps only (no rows): dest_row receives the dropless rows
  moe_status_t st = permute_launch(nullptr, x_dtype, T, d, topk_idx, k, E, counts, off_drop, dest_row, src_drop,
                                   nullptr, x_dtype, nullptr, hist, dev_status, stream, sms, nullptr, nullptr);
  if (st != MOE_OK) return st;
  if (pairs > 0) {
    const int g = (pairs + kCapThreads - 1) / kCapThreads;
    launch_pdl(capacity_remap_kernel, g < sms * 8 ? g : sms * 8, kCapThreads, 0, stream, topk_idx, pairs, E,
               capacity, static_cast<const int32_t*>(off_drop), dest_row, dev_status);
  }
  const long long rows = static_cast<long long>(E) * capacity;
  const long long wgrid = (rows + kCapThreads / 32 - 1) / (kCapThreads / 32);
  const int grid = static_cast<int>(wgrid < 1 ? 1 : (wgrid < sms * 8 ? wgrid : sms * 8));
  launch_pdl(capacity_fill_kernel, grid, kCapThreads, 0, stream, static_cast<const uint8_t*>(x), d * eb, k, E,
             capacity, static_cast<const int32_t*>(off_drop), static_cast<const int32_t*>(src_drop), src_pair,
             offsets, static_cast<uint8_t*>(xp));
  return check_launch(fn);
}

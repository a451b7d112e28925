// Top-k routing (forward and backward).
//
// The router of "Accelerating Dropless MoE Training in JAX with NVIDIA Transformer
// Engine" (opening section; "Optimisation 2": a fused router kernel assigns each
// token its experts before dispatch).  One warp owns one token: the E logits of
// the row are spread over the lanes (E <= 32 * V), k rounds of a warp arg-max
// pick the experts (value descending, expert id ascending on ties), the softmax
// weights come from the selected logits, and the per-expert counts are gathered
// in a shared-memory histogram before one global atomic per (block, expert).
#include <math.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kRouteThreads = 256;
constexpr uint32_t kFull = 0xFFFFFFFFu;

__global__ void zero_i32_kernel(int32_t* p, int n) {
  pdl_begin();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = 0;
}

// (v, e) beats (ov, oe) when v is larger, or equal with a smaller expert id.
// e == INT32_MAX marks "no candidate".
__device__ __forceinline__ bool beats(float v, int e, float ov, int oe) {
  if (e == INT32_MAX) return false;
  if (oe == INT32_MAX) return true;
  return v > ov || (v == ov && e < oe);
}

template <int V>
__global__ void __launch_bounds__(kRouteThreads) route_topk_kernel(
    const float* __restrict__ logits, int T, int E, int k, int renormalize,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int32_t* __restrict__ counts,
    int32_t* status) {
  pdl_begin();
  extern __shared__ int hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += gridDim.x * wpb) {
    const float* row = logits + static_cast<size_t>(t) * E;
    float v[V];
    uint32_t taken = 0;
    bool nan = false;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        v[i] = __ldg(row + e);
        if (isnan(v[i])) {
          nan = true;
          v[i] = -INFINITY;
        }
      } else {
        v[i] = -INFINITY;
        taken |= 1u << i;
      }
    }
    if (__any_sync(kFull, nan) && lane == 0) flag_error(status, MOE_DEV_NAN_LOGIT);

    float sel_v = -INFINITY, top0 = -INFINITY;
    int sel_e = 0;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int be = INT32_MAX;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        if (!((taken >> i) & 1u) && beats(v[i], lane + 32 * i, bv, be)) {
          bv = v[i];
          be = lane + 32 * i;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(kFull, bv, off);
        const int oe = __shfl_xor_sync(kFull, be, off);
        if (beats(ov, oe, bv, be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      if (lane == j) {
        sel_v = bv;
        sel_e = be;
      }
      if (j == 0) top0 = bv;
    }

    // a token whose experts are all masked (-inf) has no softmax mass: weight 0
    float w;
    if (top0 == -INFINITY) {
      w = 0.f;
    } else if (renormalize) {
      const float ex = lane < k ? expf(sel_v - top0) : 0.f;
      float s = ex;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
      w = ex / s;
    } else {
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < V; ++i)
        if (lane + 32 * i < E) s += expf(v[i] - top0);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
      w = expf(sel_v - top0) / s;
    }
    if (lane < k) {
      topk_idx[static_cast<size_t>(t) * k + lane] = sel_e;
      topk_w[static_cast<size_t>(t) * k + lane] = w;
      atomicAdd(&hist[sel_e], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (hist[e]) atomicAdd(&counts[e], hist[e]);
}

// One warp per token.  dlogits row: renormalised -> zero except the selected
// experts; otherwise -p_e * inner everywhere, the selected experts overwritten.
__global__ void __launch_bounds__(kRouteThreads) route_topk_bwd_kernel(
    const float* __restrict__ dw, const float* __restrict__ topk_w,
    const int32_t* __restrict__ topk_idx, const float* __restrict__ logits, int T, int E, int k,
    int renormalize, float* __restrict__ dlogits, int32_t* status) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += gridDim.x * wpb) {
    const size_t base = static_cast<size_t>(t) * k;
    float wj = 0.f, dwj = 0.f;
    int ej = 0;
    if (lane < k) {
      wj = topk_w[base + lane];
      dwj = dw[base + lane];
      ej = topk_idx[base + lane];
      if (ej < 0 || ej >= E) {
        flag_error(status, MOE_DEV_BAD_INDEX);
        ej = -1;
      }
    }
    float inner = wj * dwj;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) inner += __shfl_xor_sync(kFull, inner, off);
    float* out = dlogits + static_cast<size_t>(t) * E;
    if (renormalize) {
      for (int e = lane; e < E; e += 32) out[e] = 0.f;
    } else {
      const float* row = logits + static_cast<size_t>(t) * E;
      float m = -INFINITY;
      for (int e = lane; e < E; e += 32) m = fmaxf(m, row[e]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
      if (m == -INFINITY) {
        // every expert masked: no probability mass, no gradient
        for (int e = lane; e < E; e += 32) out[e] = 0.f;
      } else {
        float s = 0.f;
        for (int e = lane; e < E; e += 32) s += expf(row[e] - m);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
        const float scale = -inner / s;
        for (int e = lane; e < E; e += 32) out[e] = expf(row[e] - m) * scale;
      }
    }
    __syncwarp();
    if (lane < k && ej >= 0) out[ej] = wj * (dwj - inner);
  }
}

template <int V>
void launch_route(const float* logits, int T, int E, int k, int renorm, int32_t* idx, float* w,
                  int32_t* counts, int32_t* status, cudaStream_t stream, int sms) {
  const int wpb = kRouteThreads / 32;
  int grid = (T + wpb - 1) / wpb;
  grid = grid < sms * 4 ? grid : sms * 4;
  if (grid < 1) grid = 1;
  launch_pdl(route_topk_kernel<V>, grid, kRouteThreads, E * sizeof(int), stream, logits, T, E, k, renorm,
                                                                          idx, w, counts, status);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_route_topk(const float* logits, int T, int E, int k, int renormalize,
                                       int32_t* topk_idx, float* topk_w, int32_t* counts,
                                       int32_t* dev_status, cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_route_topk");
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E || k > 32) {
    set_error("moe_route_topk: need T >= 0, 1 <= E <= 1024, 1 <= k <= min(E, 32) (T=%d E=%d k=%d)",
              T, E, k);
    return MOE_ERR_INVALID_ARG;
  }
  if (!counts || (T > 0 && (!logits || !topk_idx || !topk_w))) {
    set_error("moe_route_topk: null pointer");
    return MOE_ERR_INVALID_ARG;
  }
  int sms = 0;
  if (const moe_status_t dst = device_check(&sms); dst != MOE_OK) return dst;
  launch_pdl(zero_i32_kernel, (E + 255) / 256, 256, 0, stream, counts, E);
  if (T > 0) {
    const int V = (E + 31) / 32;
    if (V <= 1) launch_route<1>(logits, T, E, k, renormalize, topk_idx, topk_w, counts, dev_status, stream, sms);
    else if (V <= 2) launch_route<2>(logits, T, E, k, renormalize, topk_idx, topk_w, counts, dev_status, stream, sms);
    else if (V <= 4) launch_route<4>(logits, T, E, k, renormalize, topk_idx, topk_w, counts, dev_status, stream, sms);
    else if (V <= 8) launch_route<8>(logits, T, E, k, renormalize, topk_idx, topk_w, counts, dev_status, stream, sms);
    else if (V <= 16) launch_route<16>(logits, T, E, k, renormalize, topk_idx, topk_w, counts, dev_status, stream, sms);
    else launch_route<32>(logits, T, E, k, renormalize, topk_idx, topk_w, counts, dev_status, stream, sms);
  }
  return check_launch("moe_route_topk");
}

extern "C" moe_status_t moe_route_topk_bwd(const float* dw, const float* topk_w,
                                           const int32_t* topk_idx, const float* logits, int T,
                                           int E, int k, int renormalize, float* dlogits,
                                           int32_t* dev_status, cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_route_topk_bwd");
  if (T < 0 || E < 1 || k < 1 || k > E || k > 32) {
    set_error("moe_route_topk_bwd: need T >= 0, 1 <= k <= min(E, 32)");
    return MOE_ERR_INVALID_ARG;
  }
  if (T > 0 && (!dw || !topk_w || !topk_idx || !dlogits || (!renormalize && !logits))) {
    set_error("moe_route_topk_bwd: null pointer");
    return MOE_ERR_INVALID_ARG;
  }
  int sms = 0;
  if (const moe_status_t dst = device_check(&sms); dst != MOE_OK) return dst;
  if (T == 0) return MOE_OK;
  const int wpb = kRouteThreads / 32;
  int grid = (T + wpb - 1) / wpb;
  grid = grid < sms * 8 ? grid : sms * 8;
  launch_pdl(route_topk_bwd_kernel, grid, kRouteThreads, 0, stream, dw, topk_w, topk_idx, logits, T, E, k,
                                                           renormalize, dlogits, dev_status);
  return check_launch("moe_route_topk_bwd");
}

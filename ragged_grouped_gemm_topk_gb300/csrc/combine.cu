// Weighted unpermute (combine) and its backward.
//
// Combine per "Accelerating Dropless MoE Training in JAX with NVIDIA Transformer
// Engine", "Optimisation 2" (processed tokens are routed back and the expert
// results accumulated per token) and Figure 3 (back to the original order).
// A warp owns one column slice of one token: the token's k source rows are
// gathered with 16-byte loads, up to 8 rows in flight per lane, and summed in slot
// order in fp32.
#include "common.cuh"

namespace moe {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr int kThreads = 256;

struct alignas(16) Vec16 {
  uint32_t w[4];
};

template <typename T>
struct Elt;
template <>
struct Elt<uint16_t> {
  static constexpr int kN = 8;
  __device__ static void unpack(const Vec16& v, float (&f)[8]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = bf16_to_f32(static_cast<uint16_t>(v.w[i] & 0xFFFFu));
      f[2 * i + 1] = bf16_to_f32(static_cast<uint16_t>(v.w[i] >> 16));
    }
  }
  __device__ static void store(uint8_t* dst, const float (&f)[8]) {
    Vec16 o;
#pragma unroll
    for (int i = 0; i < 4; ++i) o.w[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
    *reinterpret_cast<Vec16*>(dst) = o;
  }
};
template <>
struct Elt<float> {
  static constexpr int kN = 4;
  __device__ static void unpack(const Vec16& v, float (&f)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = __uint_as_float(v.w[i]);
  }
  __device__ static void store(uint8_t* dst, const float (&f)[4]) {
    *reinterpret_cast<float4*>(dst) = make_float4(f[0], f[1], f[2], f[3]);
  }
};

// Store N floats (N = elements of one 16-byte input chunk) in the output dtype.
template <typename Tout, int N>
__device__ __forceinline__ void store_out(uint8_t* dst, const float (&f)[N]) {
  if constexpr (sizeof(Tout) == 2) {
    uint32_t w[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) w[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
    if constexpr (N == 8) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < N; i += 4)
      *reinterpret_cast<float4*>(dst + 4 * i) = make_float4(f[i], f[i + 1], f[i + 2], f[i + 3]);
  }
}

// Work item = (token, column slice of kSliceChunks 16-byte chunks), so that a
// few thousand tokens still spread over every SM; each lane keeps up to 8 source
// rows' loads in flight per chunk.
constexpr int kSliceChunks = 128;

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kThreads) combine_kernel(
    const uint8_t* __restrict__ yp, int M, int T, int d, int k, const int32_t* __restrict__ dest_row,
    const float* __restrict__ topk_w, uint8_t* __restrict__ y, int allow_drop, int32_t* status) {
  pdl_begin();
  constexpr int N = Elt<Tin>::kN;
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const size_t in_row = static_cast<size_t>(d) * sizeof(Tin);
  const size_t out_row = static_cast<size_t>(d) * sizeof(Tout);
  const int n16 = static_cast<int>(in_row / 16);
  const int nslice = (n16 + kSliceChunks - 1) / kSliceChunks;
  const long long tasks = static_cast<long long>(T) * nslice;
  for (long long task = static_cast<long long>(blockIdx.x) * wpb + (threadIdx.x >> 5); task < tasks;
       task += static_cast<long long>(gridDim.x) * wpb) {
    const int t = static_cast<int>(task / nslice);
    const int slice = static_cast<int>(task % nslice);
    int src = -1;
    float w = 0.f;
    if (lane < k) {
      const size_t p = static_cast<size_t>(t) * k + lane;
      src = dest_row[p];
      w = topk_w ? topk_w[p] : 1.f;
      if ((src < 0 || src >= M) && !(src == -1 && allow_drop)) {   // -1: a dropped slot (capacity mode)
        if (slice == 0) flag_error(status, MOE_DEV_BAD_INDEX);
        src = -1;
      }
    }
    const int c_end = min(n16, (slice + 1) * kSliceChunks);
    for (int base = slice * kSliceChunks; base < c_end; base += 32) {
      const int c = base + lane;
      const bool active = c < c_end;
      float acc[N];
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = 0.f;
      for (int j0 = 0; j0 < k; j0 += 8) {
        Vec16 v[8];
        float wj[8];
        int sj[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          sj[u] = __shfl_sync(kFull, src, (j0 + u) & 31);
          wj[u] = __shfl_sync(kFull, w, (j0 + u) & 31);
          if (active && j0 + u < k && sj[u] >= 0)
            v[u] = reinterpret_cast<const Vec16*>(yp + static_cast<size_t>(sj[u]) * in_row)[c];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (active && j0 + u < k && sj[u] >= 0) {
            float f[N];
            Elt<Tin>::unpack(v[u], f);
#pragma unroll
            for (int i = 0; i < N; ++i) acc[i] = fmaf(wj[u], f[i], acc[i]);
          }
        }
      }
      if (active)
        store_out<Tout, N>(y + static_cast<size_t>(t) * out_row + static_cast<size_t>(c) * N * sizeof(Tout), acc);
    }
  }
}

// Same sum for a compile-time k in {1, 2, 4, 8}: a lane gathers U chunks of each
// of the k source rows before it sums any of them, so that U*k = 8 or 16 16-byte
// loads are in flight per lane (the runtime-k loop above has only k of them, too
// few to cover HBM latency at k = 2).  Slot order and fp32 fmaf as above.
constexpr int kFixedSlice = 256;   // 16-byte chunks per work item

template <typename Tin, typename Tout, int K>
__global__ void __launch_bounds__(kThreads) combine_fixed_kernel(
    const uint8_t* __restrict__ yp, int M, int T, int d, const int32_t* __restrict__ dest_row,
    const float* __restrict__ topk_w, uint8_t* __restrict__ y, int allow_drop, int32_t* status) {
  pdl_begin();
  constexpr int N = Elt<Tin>::kN;
  constexpr int U = (16 / K) < 8 ? (16 / K) : 8;
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const size_t in_row = static_cast<size_t>(d) * sizeof(Tin);
  const size_t out_row = static_cast<size_t>(d) * sizeof(Tout);
  const int n16 = static_cast<int>(in_row / 16);
  const int nslice = (n16 + kFixedSlice - 1) / kFixedSlice;
  const long long tasks = static_cast<long long>(T) * nslice;
  for (long long task = static_cast<long long>(blockIdx.x) * wpb + (threadIdx.x >> 5); task < tasks;
       task += static_cast<long long>(gridDim.x) * wpb) {
    const int t = static_cast<int>(task / nslice);
    const int slice = static_cast<int>(task % nslice);
    int src = -1;
    float w = 0.f;
    if (lane < K) {
      const size_t p = static_cast<size_t>(t) * K + lane;
      src = dest_row[p];
      w = topk_w ? topk_w[p] : 1.f;
      if ((src < 0 || src >= M) && !(src == -1 && allow_drop)) {   // -1: a dropped slot (capacity mode)
        if (slice == 0) flag_error(status, MOE_DEV_BAD_INDEX);
        src = -1;
      }
    }
    const Vec16* rows[K];
    float wj[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      const int sj = __shfl_sync(kFull, src, j);
      wj[j] = __shfl_sync(kFull, w, j);
      rows[j] = sj >= 0 ? reinterpret_cast<const Vec16*>(yp + static_cast<size_t>(sj) * in_row) : nullptr;
    }
    const int c_end = min(n16, (slice + 1) * kFixedSlice);
    for (int base = slice * kFixedSlice; base < c_end; base += 32 * U) {
      Vec16 v[U][K];
#pragma unroll
      for (int i = 0; i < U; ++i) {
        const int c = base + 32 * i + lane;
#pragma unroll
        for (int j = 0; j < K; ++j)
          if (c < c_end && rows[j] != nullptr) v[i][j] = rows[j][c];
      }
#pragma unroll
      for (int i = 0; i < U; ++i) {
        const int c = base + 32 * i + lane;
        if (c < c_end) {
          float acc[N];
#pragma unroll
          for (int e = 0; e < N; ++e) acc[e] = 0.f;
#pragma unroll
          for (int j = 0; j < K; ++j) {
            if (rows[j] != nullptr) {
              float f[N];
              Elt<Tin>::unpack(v[i][j], f);
#pragma unroll
              for (int e = 0; e < N; ++e) acc[e] = fmaf(wj[j], f[e], acc[e]);
            }
          }
          store_out<Tout, N>(y + static_cast<size_t>(t) * out_row + static_cast<size_t>(c) * N * sizeof(Tout), acc);
        }
      }
    }
  }
}

// One warp per (token, slot): dyp[dest_row[t,j]] = w[t,j] dy[t] and
// dw[t,j] = <dy[t], yp[dest_row[t,j]]> (warp reduction).  dy[t] is re-read by the
// token's k warps, from L2.
template <typename Tin>
__global__ void __launch_bounds__(kThreads) combine_bwd_kernel(
    const uint8_t* __restrict__ dy, const uint8_t* __restrict__ yp, int T, int d, int k,
    const int32_t* __restrict__ dest_row, const float* __restrict__ topk_w,
    uint8_t* __restrict__ dyp, float* __restrict__ dw, int32_t* status) {
  pdl_begin();
  constexpr int N = Elt<Tin>::kN;
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int M = T * k;
  const size_t row = static_cast<size_t>(d) * sizeof(Tin);
  const int n16 = static_cast<int>(row / 16);
  const long long pairs = static_cast<long long>(T) * k;
  for (long long p = static_cast<long long>(blockIdx.x) * wpb + (threadIdx.x >> 5); p < pairs;
       p += static_cast<long long>(gridDim.x) * wpb) {
    const int t = static_cast<int>(p / k);
    const int sj = dest_row[p];
    const float wj = topk_w[p];
    float part = 0.f;
    if (sj >= 0 && sj < M) {
      const Vec16* dyr = reinterpret_cast<const Vec16*>(dy + static_cast<size_t>(t) * row);
      const Vec16* ypr = reinterpret_cast<const Vec16*>(yp + static_cast<size_t>(sj) * row);
      uint8_t* out = dyp + static_cast<size_t>(sj) * row;
      for (int c = lane; c < n16; c += 32) {
        float a[N], b[N], o[N];
        Elt<Tin>::unpack(dyr[c], a);
        Elt<Tin>::unpack(ypr[c], b);
#pragma unroll
        for (int i = 0; i < N; ++i) {
          part = fmaf(a[i], b[i], part);
          o[i] = wj * a[i];
        }
        Elt<Tin>::store(out + static_cast<size_t>(c) * 16, o);
      }
    } else if (lane == 0) {
      flag_error(status, MOE_DEV_BAD_INDEX);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(kFull, part, off);
    if (lane == 0) dw[p] = part;
  }
}

// As combine_bwd_kernel (bf16), with dYp leaving as its row-wise MXFP8 (codes
// [T*k, d], E8M0 scales [T*k, d/32]) instead of in bf16: each row value is first
// rounded to bf16, exactly as the bf16 kernel stores it, then quantised, so the
// codes and scales equal the row-wise quantiser's on the bf16 dYp.  A lane's
// 16-byte chunk holds 8 elements, four adjacent lanes one 32-element block (d % 32
// == 0); the warp walks the row in 32-chunk steps so every lane joins the block
// shuffles.
__global__ void __launch_bounds__(kThreads) combine_bwd_mx_kernel(
    const uint8_t* __restrict__ dy, const uint8_t* __restrict__ yp, int T, int d, int k,
    const int32_t* __restrict__ dest_row, const float* __restrict__ topk_w, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales, float* __restrict__ dw, int32_t* status) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int M = T * k;
  const size_t row = static_cast<size_t>(d) * 2;
  const int n16 = d / 8;
  const long long pairs = static_cast<long long>(T) * k;
  for (long long p = static_cast<long long>(blockIdx.x) * wpb + (threadIdx.x >> 5); p < pairs;
       p += static_cast<long long>(gridDim.x) * wpb) {
    const int t = static_cast<int>(p / k);
    const int sj = dest_row[p];
    const float wj = topk_w[p];
    float part = 0.f;
    if (sj >= 0 && sj < M) {                    // warp-uniform
      const Vec16* dyr = reinterpret_cast<const Vec16*>(dy + static_cast<size_t>(t) * row);
      const Vec16* ypr = reinterpret_cast<const Vec16*>(yp + static_cast<size_t>(sj) * row);
      const Vec16 zero = {{0u, 0u, 0u, 0u}};
      // one chunk: accumulate dw, round w*dy to bf16, quantise its 32-element block
      auto chunk = [&](const Vec16& va, const Vec16& vb, int c, bool on) {
        float a[8], b[8], o[8];
        Elt<uint16_t>::unpack(va, a);
        Elt<uint16_t>::unpack(vb, b);
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          part = fmaf(a[i], b[i], part);
          o[i] = bf16_to_f32(f32_to_bf16(wj * a[i]));
          amax = fmaxf(amax, fabsf(o[i]));
        }
        amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
        uint32_t sbyte;
        float inv;
        mx_scale(amax, &sbyte, &inv);
        uint32_t q[2];
#pragma unroll
        for (int h = 0; h < 2; ++h)
          q[h] = static_cast<uint32_t>(f32x2_to_e4m3x2(o[4 * h] * inv, o[4 * h + 1] * inv)) |
                 (static_cast<uint32_t>(f32x2_to_e4m3x2(o[4 * h + 2] * inv, o[4 * h + 3] * inv)) << 16);
        if (on) {
          *reinterpret_cast<uint2*>(codes + static_cast<size_t>(sj) * d + static_cast<size_t>(c) * 8) =
              make_uint2(q[0], q[1]);
          if ((lane & 3) == 0) scales[static_cast<size_t>(sj) * (d / 32) + c / 4] = static_cast<uint8_t>(sbyte);
        }
      };
      // two 32-chunk steps per pass, all four loads issued first; chunks are taken in
      // the order lane, lane + 32, lane + 64, ... (the bf16 kernel's dw order)
      for (int base = 0; base < n16; base += 64) {
        const int c0 = base + lane, c1 = base + 32 + lane;
        const bool on0 = c0 < n16, on1 = c1 < n16;   // a block's four lanes agree (n16 % 4 == 0)
        const Vec16 a0 = on0 ? dyr[c0] : zero, b0 = on0 ? ypr[c0] : zero;
        const Vec16 a1 = on1 ? dyr[c1] : zero, b1 = on1 ? ypr[c1] : zero;
        chunk(a0, b0, c0, on0);
        if (base + 32 < n16) chunk(a1, b1, c1, on1);  // warp-uniform
      }
    } else if (lane == 0) {
      flag_error(status, MOE_DEV_BAD_INDEX);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(kFull, part, off);
    if (lane == 0) dw[p] = part;
  }
}

int grid_for(long long tasks, int sms) {
  const int wpb = kThreads / 32;
  const long long g = (tasks + wpb - 1) / wpb;
  const long long cap = static_cast<long long>(sms) * 8;
  return static_cast<int>(g < 1 ? 1 : (g < cap ? g : cap));
}

template <typename Tin, typename Tout>
void launch_fixed(int k, int grid, cudaStream_t stream, const uint8_t* a, int M, int T, int d,
                  const int32_t* dest_row, const float* topk_w, uint8_t* o, int drop, int32_t* dev_status) {
  switch (k) {
    case 1: launch_pdl(combine_fixed_kernel<Tin, Tout, 1>, grid, kThreads, 0, stream, a, M, T, d, dest_row, topk_w, o, drop, dev_status); break;
    case 2: launch_pdl(combine_fixed_kernel<Tin, Tout, 2>, grid, kThreads, 0, stream, a, M, T, d, dest_row, topk_w, o, drop, dev_status); break;
    case 4: launch_pdl(combine_fixed_kernel<Tin, Tout, 4>, grid, kThreads, 0, stream, a, M, T, d, dest_row, topk_w, o, drop, dev_status); break;
    default: launch_pdl(combine_fixed_kernel<Tin, Tout, 8>, grid, kThreads, 0, stream, a, M, T, d, dest_row, topk_w, o, drop, dev_status); break;
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

namespace moe {
namespace {
moe_status_t combine_impl(const char* fn, const void* yp, moe_dtype_t dtype, int M, int T, int d, int k,
                          const int32_t* dest_row, const float* topk_w, void* y, moe_dtype_t y_dtype,
                          int drop, int32_t* dev_status, cudaStream_t stream) {
  if (T < 0 || d < 0 || M < 0 || k < 1 || k > 32 || d % 8 ||
      (dtype != MOE_BF16 && dtype != MOE_F32) || (y_dtype != MOE_BF16 && y_dtype != MOE_F32)) {
    set_error("%s: need T, d, rows >= 0, d %% 8 == 0, 1 <= k <= 32, BF16/F32", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (static_cast<long long>(T) * k >= (1LL << 31)) {
    set_error("%s: T*k must fit in int32", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (T > 0 && d > 0 && (!y || !dest_row || !aligned16(yp) || !aligned16(y) || (M > 0 && !yp))) {
    set_error("%s: null or misaligned pointer", fn);
    return MOE_ERR_INVALID_ARG;
  }
  int sms = 0;
  if (const moe_status_t dst = device_check(&sms); dst != MOE_OK) return dst;
  if (T == 0 || d == 0) return MOE_OK;
  const long long n16 = static_cast<long long>(d) * (dtype == MOE_BF16 ? 2 : 4) / 16;
  const uint8_t* a = static_cast<const uint8_t*>(yp);
  uint8_t* o = static_cast<uint8_t*>(y);
  if (k == 1 || k == 2 || k == 4 || k == 8) {
    const int grid = grid_for(static_cast<long long>(T) * ((n16 + kFixedSlice - 1) / kFixedSlice), sms);
    if (dtype == MOE_BF16 && y_dtype == MOE_BF16) launch_fixed<uint16_t, uint16_t>(k, grid, stream, a, M, T, d, dest_row, topk_w, o, drop, dev_status);
    else if (dtype == MOE_BF16) launch_fixed<uint16_t, float>(k, grid, stream, a, M, T, d, dest_row, topk_w, o, drop, dev_status);
    else if (y_dtype == MOE_BF16) launch_fixed<float, uint16_t>(k, grid, stream, a, M, T, d, dest_row, topk_w, o, drop, dev_status);
    else launch_fixed<float, float>(k, grid, stream, a, M, T, d, dest_row, topk_w, o, drop, dev_status);
    return check_launch(fn);
  }
  const int grid = grid_for(static_cast<long long>(T) * ((n16 + kSliceChunks - 1) / kSliceChunks), sms);
  if (dtype == MOE_BF16 && y_dtype == MOE_BF16)
    launch_pdl(combine_kernel<uint16_t, uint16_t>, grid, kThreads, 0, stream, a, M, T, d, k, dest_row, topk_w, o, drop, dev_status);
  else if (dtype == MOE_BF16)
    launch_pdl(combine_kernel<uint16_t, float>, grid, kThreads, 0, stream, a, M, T, d, k, dest_row, topk_w, o, drop, dev_status);
  else if (y_dtype == MOE_BF16)
    launch_pdl(combine_kernel<float, uint16_t>, grid, kThreads, 0, stream, a, M, T, d, k, dest_row, topk_w, o, drop, dev_status);
  else
    launch_pdl(combine_kernel<float, float>, grid, kThreads, 0, stream, a, M, T, d, k, dest_row, topk_w, o, drop, dev_status);
  return check_launch(fn);
}
}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_unpermute_combine(const void* yp, moe_dtype_t dtype, int T, int d,
                                              int k, const int32_t* dest_row,
                                              const float* topk_w, void* y, moe_dtype_t y_dtype,
                                              int32_t* dev_status, cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_unpermute_combine");
  if (static_cast<long long>(T) * k >= (1LL << 31)) {
    set_error("moe_unpermute_combine: T*k must fit in int32");
    return MOE_ERR_INVALID_ARG;
  }
  return combine_impl("moe_unpermute_combine", yp, dtype, T > 0 && k > 0 ? T * k : 0, T, d, k, dest_row, topk_w,
                      y, y_dtype, 0, dev_status, stream);
}

extern "C" moe_status_t moe_unpermute_combine_capacity(const void* yp, moe_dtype_t dtype, int rows, int T,
                                                       int d, int k, const int32_t* dest_row,
                                                       const float* topk_w, void* y, moe_dtype_t y_dtype,
                                                       int32_t* dev_status, cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_unpermute_combine_capacity");
  return combine_impl("moe_unpermute_combine_capacity", yp, dtype, rows, T, d, k, dest_row, topk_w, y, y_dtype,
                      1, dev_status, stream);
}

extern "C" moe_status_t moe_unpermute_combine_bwd(const void* dy, const void* yp,
                                                  moe_dtype_t dtype, int T, int d, int k,
                                                  const int32_t* dest_row, const float* topk_w,
                                                  void* dyp, float* dw, int32_t* dev_status,
                                                  cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_unpermute_combine_bwd");
  if (T < 0 || d < 0 || k < 1 || k > 32 || d % 8 || (dtype != MOE_BF16 && dtype != MOE_F32)) {
    set_error("moe_unpermute_combine_bwd: need T, d >= 0, d %% 8 == 0, 1 <= k <= 32, BF16/F32");
    return MOE_ERR_INVALID_ARG;
  }
  if (static_cast<long long>(T) * k >= (1LL << 31)) {
    set_error("moe_unpermute_combine_bwd: T*k must fit in int32");
    return MOE_ERR_INVALID_ARG;
  }
  if (T > 0 && (!dy || !yp || !dest_row || !topk_w || !dyp || !dw || !aligned16(dy) ||
                !aligned16(yp) || !aligned16(dyp))) {
    set_error("moe_unpermute_combine_bwd: null or misaligned pointer");
    return MOE_ERR_INVALID_ARG;
  }
  int sms = 0;
  if (const moe_status_t dst = device_check(&sms); dst != MOE_OK) return dst;
  if (T == 0) return MOE_OK;
  const int grid = grid_for(static_cast<long long>(T) * k, sms);
  const uint8_t* a = static_cast<const uint8_t*>(dy);
  const uint8_t* b = static_cast<const uint8_t*>(yp);
  uint8_t* o = static_cast<uint8_t*>(dyp);
  if (dtype == MOE_BF16)
    launch_pdl(combine_bwd_kernel<uint16_t>, grid, kThreads, 0, stream, a, b, T, d, k, dest_row, topk_w, o, dw, dev_status);
  else
    launch_pdl(combine_bwd_kernel<float>, grid, kThreads, 0, stream, a, b, T, d, k, dest_row, topk_w, o, dw, dev_status);
  return check_launch("moe_unpermute_combine_bwd");
}

extern "C" moe_status_t moe_unpermute_combine_bwd_mxfp8(const void* dy, const void* yp, moe_dtype_t dtype, int T,
                                                        int d, int k, const int32_t* dest_row,
                                                        const float* topk_w, uint8_t* dyp_codes,
                                                        uint8_t* dyp_scales, float* dw, int32_t* dev_status,
                                                        cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_unpermute_combine_bwd_mxfp8");
  const char* fn = "moe_unpermute_combine_bwd_mxfp8";
  if (T < 0 || d < 0 || k < 1 || k > 32 || d % 32 || dtype != MOE_BF16) {
    set_error("%s: need T, d >= 0, d %% 32 == 0, 1 <= k <= 32, BF16 dy and yp", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (static_cast<long long>(T) * k >= (1LL << 31)) {
    set_error("%s: T*k must fit in int32", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (T > 0 && (!dy || !yp || !dest_row || !topk_w || !dyp_codes || !dyp_scales || !dw || !aligned16(dy) ||
                !aligned16(yp) || !aligned16(dyp_codes))) {
    set_error("%s: null or misaligned pointer", fn);
    return MOE_ERR_INVALID_ARG;
  }
  int sms = 0;
  if (const moe_status_t dst = device_check(&sms); dst != MOE_OK) return dst;
  if (T == 0) return MOE_OK;
  const int grid = grid_for(static_cast<long long>(T) * k, sms);
  launch_pdl(combine_bwd_mx_kernel, grid, kThreads, 0, stream, static_cast<const uint8_t*>(dy),
             static_cast<const uint8_t*>(yp), T, d, k, dest_row, topk_w, dyp_codes, dyp_scales, dw, dev_status);
  return check_launch(fn);
}

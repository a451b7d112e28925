// NVFP4 quantisation (E2M1 elements, an E4M3 scale per 16 elements, an fp32 scale
// for the whole tensor): the Blackwell FP4 recipe that "Deep reading of arXiv
// 2603.07685" (contribution 3) names beside MXFP8.
//
// Two kernels: the tensor's amax (a grid-stride max, one atomicMax of the float's
// bits per CTA: non-negative floats order like their bit patterns), then one
// thread per 16-element block.  Every rounding that decides a code is an fp32
// operation in this order: g = 2688 / amax (1 for an all-zero tensor); block
// scale s = E4M3_rn_sat((amax_block / 6) * g); y = v * (g / s) (0 when s is 0);
// code = E2M1_rn_sat(y).  Codes are packed two per byte, element 2i in the low
// nibble; scales are [rows, K/16] bytes; g is written for the GEMM epilogue.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kQThreads = 256;

template <typename Tin>
__global__ void __launch_bounds__(kQThreads) nvfp4_amax_kernel(const uint8_t* __restrict__ in, long long n16,
                                                               uint32_t* amax_bits) {
  pdl_begin();
  nvfp4_amax_body<Tin>(in, n16, amax_bits, blockIdx.x, gridDim.x);
}

template <typename Tin>
__global__ void __launch_bounds__(kQThreads) nvfp4_quantize_kernel(
    const uint8_t* __restrict__ in, long long nblk, const uint32_t* amax_bits, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales, float* g_out) {
  pdl_begin();
  const float g = nvfp4_tensor_scale(__uint_as_float(*amax_bits));
  if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;
  for (long long b = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; b < nblk;
       b += static_cast<long long>(gridDim.x) * blockDim.x) {
    float v[16];
    const uint4* src = reinterpret_cast<const uint4*>(in + b * 16 * sizeof(Tin));
    if constexpr (sizeof(Tin) == 2) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 u = src[h];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[8 * h + 2 * j] = bf16_to_f32(static_cast<uint16_t>(w[j] & 0xFFFFu));
          v[8 * h + 2 * j + 1] = bf16_to_f32(static_cast<uint16_t>(w[j] >> 16));
        }
      }
    } else {
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint4 u = src[h];
        v[4 * h] = __uint_as_float(u.x);
        v[4 * h + 1] = __uint_as_float(u.y);
        v[4 * h + 2] = __uint_as_float(u.z);
        v[4 * h + 3] = __uint_as_float(u.w);
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    uint32_t scode;
    float inv;
    nvfp4_block_scale(amax, g, &scode, &inv);
    float y[2][8];
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i / 8][i % 8] = __fmul_rn(v[i], inv);
    *reinterpret_cast<uint2*>(codes + b * 8) = make_uint2(f32x8_to_e2m1x8(y[0]), f32x8_to_e2m1x8(y[1]));
    scales[b] = static_cast<uint8_t>(scode);
  }
}

}  // namespace

// The tensor amax into *amax_bits (as float bits; the caller zeroes it first).
void nvfp4_amax_launch(const void* in, moe_dtype_t dtype, long long elems, uint32_t* amax_bits,
                       cudaStream_t stream, int sms) {
  const long long n16 = elems * (dtype == MOE_BF16 ? 2 : 4) / 16;
  const long long g1 = (n16 + kQThreads - 1) / kQThreads;
  const int grid = static_cast<int>(g1 < 1 ? 1 : (g1 < sms * 8 ? g1 : sms * 8));
  if (dtype == MOE_BF16)
    launch_pdl(nvfp4_amax_kernel<uint16_t>, grid, kQThreads, 0, stream, static_cast<const uint8_t*>(in), n16,
               amax_bits);
  else
    launch_pdl(nvfp4_amax_kernel<float>, grid, kQThreads, 0, stream, static_cast<const uint8_t*>(in), n16,
               amax_bits);
}

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_quantize_nvfp4(const void* in, moe_dtype_t in_dtype, int rows, int K, uint8_t* codes,
                                           uint8_t* scales, float* tensor_scale, cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_quantize_nvfp4");
  const char* fn = "moe_quantize_nvfp4";
  if (rows < 0 || K < 0 || K % 16 || (in_dtype != MOE_BF16 && in_dtype != MOE_F32)) {
    set_error("%s: need rows >= 0, K %% 16 == 0, BF16/F32 input", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (!tensor_scale || (rows > 0 && K > 0 && (!in || !codes || !scales)) || !aligned16(in) ||
      (reinterpret_cast<uintptr_t>(codes) & 7) || (reinterpret_cast<uintptr_t>(tensor_scale) & 3)) {
    set_error("%s: null or misaligned pointer (in 16-byte, codes 8-byte aligned)", fn);
    return MOE_ERR_INVALID_ARG;
  }
  int sms = 0;
  if (const moe_status_t dst = device_check(&sms); dst != MOE_OK) return dst;
  uint32_t* amax_bits = reinterpret_cast<uint32_t*>(tensor_scale + 1);
  cudaError_t e = cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) {
    set_error("%s: cudaMemsetAsync: %s", fn, cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  const long long elems = static_cast<long long>(rows) * K;
  const int eb = in_dtype == MOE_BF16 ? 2 : 4;
  const long long n16 = elems * eb / 16;
  const long long nblk = elems / 16;
  const uint8_t* src = static_cast<const uint8_t*>(in);
  (void)n16;
  const long long g2 = (nblk + kQThreads - 1) / kQThreads;
  const int grid2 = static_cast<int>(g2 < 1 ? 1 : (g2 < sms * 8 ? g2 : sms * 8));
  nvfp4_amax_launch(in, in_dtype, elems, amax_bits, stream, sms);
  if (in_dtype == MOE_BF16)
    launch_pdl(nvfp4_quantize_kernel<uint16_t>, grid2, kQThreads, 0, stream, src, nblk,
               static_cast<const uint32_t*>(amax_bits), codes, scales, tensor_scale);
  else
    launch_pdl(nvfp4_quantize_kernel<float>, grid2, kQThreads, 0, stream, src, nblk,
               static_cast<const uint32_t*>(amax_bits), codes, scales, tensor_scale);
  return check_launch(fn);
}

// Ragged grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// "Accelerating Dropless MoE Training in JAX with NVIDIA Transformer Engine",
// "Optimisation 1: grouped GEMM": one launch covers every expert's matmul, each
// computed at its own (data-dependent) token count, with no device-to-host copy
// of the counts and no padding to a worst-case capacity.
//
// Design (one persistent CTA per SM, 6 warps):
//   warp 0     TMA producer: streams K-blocks of the A rows and B rows of the
//              current tile into a 4-stage shared-memory ring (128-byte swizzle).
//   warp 1     allocates TMEM; one lane issues tcgen05.mma (M=128, N=256) into a
//              double-buffered fp32 accumulator in TMEM and commits each stage
//              back to the producer and each finished tile to the epilogue.
//   warps 2-5  epilogue: tcgen05.ld the accumulator (one TMEM lane = one row per
//              thread), apply the fused epilogue and store rows with 16-byte
//              stores, masked at the expert's last row.
// Tiles are enumerated on the device from `offsets`: expert e has
// ceil(count_e / 128) row tiles times the column tiles; row tiles vary fastest
// so neighbouring CTAs share the same weight slice in L2.  Rows past an expert's
// end inside its last tile belong to the next expert (or lie past M and are
// zero-filled by TMA): they are computed but never stored.
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"

namespace moe {
namespace gemm {

constexpr int kBM = 128;
constexpr int kBN = 256;              // MMA N (SwiGLU: 128 gate + 128 up rows)
constexpr int kBKBytes = 128;         // one 128-byte swizzle atom of K per stage
constexpr int kStages = 4;
constexpr int kAStage = kBM * kBKBytes;           // 16 KB
constexpr int kBStage = kBN * kBKBytes;           // 32 KB
constexpr int kStageBytes = kAStage + kBStage;    // 48 KB
constexpr int kThreads = 192;
constexpr int kTmemCols = 2 * kBN;                // double-buffered accumulator
constexpr int kMaxE = 1024;

// Instruction descriptor (kind::f16 / kind::tf32): D=f32, A/B format, K-major
// operands, N >> 3 at bit 17, M >> 4 at bit 24.
template <int kKind>
__host__ __device__ constexpr uint32_t make_idesc(int m, int n) {
  return (1u << 4) | (static_cast<uint32_t>(kKind == 0 ? 2 : 1) << 7) |
         (static_cast<uint32_t>(kKind == 0 ? 2 : 1) << 10) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

struct Smem {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int pad;
  int prefix[kMaxE + 1];
  int offs[kMaxE + 1];
};

constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(kStages) * kStageBytes + sizeof(Smem);

struct TileInfo {
  int e;      // expert
  int row0;   // first row of the tile (global row index)
  int rows;   // valid rows in the tile (<= 128)
  int n0;     // first output column (or first B row)
};

__device__ __forceinline__ TileInfo tile_info(const Smem& s, int tile, int E, int nt) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s.prefix[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int local = tile - s.prefix[e];
  const int cnt = s.offs[e + 1] - s.offs[e];
  const int mt = (cnt + kBM - 1) / kBM;
  const int m_tile = local % mt;
  const int n_tile = local / mt;
  TileInfo t;
  t.e = e;
  t.row0 = s.offs[e] + m_tile * kBM;
  const int left = s.offs[e + 1] - t.row0;
  t.rows = left < kBM ? left : kBM;
  t.n0 = n_tile;  // scaled by the caller
  return t;
}

// Build the per-expert tile prefix in shared memory (all threads participate).
__device__ void build_tiles(Smem& s, const int32_t* offsets, int E, int M, int nt, int32_t* status) {
  for (int e = threadIdx.x; e <= E; e += blockDim.x) s.offs[e] = offsets[e];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int cnt = s.offs[e + 1] - s.offs[e];
    if (cnt < 0 || s.offs[e + 1] > M || s.offs[e] < 0) {
      flag_error(status, MOE_DEV_BAD_INDEX);
      cnt = 0;
    }
    s.prefix[e + 1] = ((cnt + kBM - 1) / kBM) * nt;
  }
  if (threadIdx.x == 0) s.prefix[0] = 0;
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    for (int base = 1; base <= E; base += 32) {
      const int i = base + lane;
      int v = i <= E ? s.prefix[i] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xFFFFFFFFu, v, off);
        if (lane >= off) v += u;
      }
      if (i <= E) s.prefix[i] = v + carry;
      carry += __shfl_sync(0xFFFFFFFFu, v, 31);
    }
    if (lane == 0) s.total_tiles = carry;
  }
  __syncthreads();
}

__device__ __forceinline__ float silu_f(float g) { return g * __frcp_rn(1.f + __expf(-g)); }

// Store 32 consecutive fp32 values as OutT (16-byte stores).
template <typename OutT>
__device__ __forceinline__ void store32(OutT* dst, const float (&v)[32]) {
  if constexpr (sizeof(OutT) == 2) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      d4[q] = make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                         pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
  } else {
    float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int q = 0; q < 8; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  }
}

// kKind: 0 = tf32 (fp32 storage), 1 = bf16.  kSwiglu: fused SwiGLU epilogue.
template <int kKind, bool kSwiglu, typename OutT>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_fwd_kernel(
    const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
    const int32_t* __restrict__ offsets, int M, int N, int K, int E, OutT* __restrict__ C,
    OutT* __restrict__ preact, int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Smem& s = *reinterpret_cast<Smem*>(tiles + kStages * kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int n_out = kSwiglu ? N / 2 : N;                 // output columns
  const int bn_out = kSwiglu ? kBN / 2 : kBN;            // output columns per tile
  const int nt = (n_out + bn_out - 1) / bn_out;
  const int kb_count = (K * (kKind == 0 ? 4 : 2) + kBKBytes - 1) / kBKBytes;
  const int bk_elems = kBKBytes / (kKind == 0 ? 4 : 2);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], 128);
    }
    s.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  build_tiles(s, offsets, E, M, nt, status);   // contains __syncthreads
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const int total = s.total_tiles;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = blockIdx.x; tile < total && !s.abort; tile += gridDim.x) {
        const TileInfo ti = tile_info(s, tile, E, nt);
        const int n0 = ti.n0 * bn_out;
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!mbar_wait(&s.empty[stage], phase ^ 1u, status, &s.abort)) break;
          uint8_t* sa = tiles + stage * kStageBytes;
          uint8_t* sb = sa + kAStage;
          mbar_arrive_expect_tx(&s.full[stage], kStageBytes);
          const int kx = kb * bk_elems;
          tma_load_2d(sa, &tmA, &s.full[stage], kx, ti.row0);
          if (kSwiglu) {
            tma_load_3d(sb, &tmB, &s.full[stage], kx, n0, ti.e);
            tma_load_3d(sb + kBStage / 2, &tmB, &s.full[stage], kx, n_out + n0, ti.e);
          } else {
            tma_load_3d(sb, &tmB, &s.full[stage], kx, n0, ti.e);
          }
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc<kKind>(kBM, kBN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int tile = blockIdx.x; tile < total && !s.abort; tile += gridDim.x) {
        if (!mbar_wait(&s.tempty[acc], acc_phase ^ 1u, status, &s.abort)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * kBN);
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!mbar_wait(&s.full[stage], phase, status, &s.abort)) break;
          tc_fence_after();
          const uint32_t sa = smem_u32(tiles + stage * kStageBytes);
          const uint32_t sb = sa + kAStage;
#pragma unroll
          for (int kk = 0; kk < kBKBytes / 32; ++kk) {
            const uint64_t ad = make_sdesc(sa + kk * 32, 16, 1024, 2);
            const uint64_t bd = make_sdesc(sb + kk * 32, 16, 1024, 2);
            tc_mma<kKind>(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(&s.empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        tc_commit(&s.tfull[acc]);
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
    }
  } else {
    // Epilogue warps 2..5 -> TMEM lane quarter (warp % 4).
    const int q = warp & 3;
    const int r = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total && !s.abort; tile += gridDim.x) {
      const TileInfo ti = tile_info(s, tile, E, nt);
      const int n0 = ti.n0 * bn_out;
      if (!mbar_wait(&s.tfull[acc], acc_phase, status, &s.abort)) break;
      tc_fence_after();
      const uint32_t tb = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kBN);
      const bool valid = r < ti.rows;
      const size_t grow = static_cast<size_t>(ti.row0 + r);
      if constexpr (kSwiglu) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(tb + c * 32, g);
          tmem_ld32(tb + 128 + c * 32, u);
          tmem_ld_wait();
          const int col = n0 + c * 32;
          if (valid && col < n_out) {
            float h[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float gv = __uint_as_float(g[i]);
              h[i] = silu_f(gv) * __uint_as_float(u[i]);
            }
            store32<OutT>(C + grow * n_out + col, h);
            if (preact != nullptr) {
              float gf[32], uf[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                gf[i] = __uint_as_float(g[i]);
                uf[i] = __uint_as_float(u[i]);
              }
              store32<OutT>(preact + grow * N + col, gf);
              store32<OutT>(preact + grow * N + n_out + col, uf);
            }
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tb + c * 32, v);
          tmem_ld_wait();
          const int col = n0 + c * 32;
          if (valid && col < n_out) {
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
            store32<OutT>(C + grow * n_out + col, f);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&s.tempty[acc]);
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ----------------------------------------------------------------------------- host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Tiled tensor map over a row-major tensor with dims (innermost first) and the
// given box; 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* ptr, int rank,
              const uint64_t* dims, const uint32_t* box, CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return false;
  }
  cuuint64_t gdim[3];
  cuuint64_t gstride[2];
  cuuint32_t bdim[3], estr[3] = {1, 1, 1};
  uint64_t stride = static_cast<uint64_t>(elem_bytes);
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    if (i > 0) gstride[i - 1] = stride;
    stride *= dims[i];
  }
  CUresult r = fn(map, dt, rank, const_cast<void*>(ptr), gdim, gstride, bdim, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return false;
  }
  return true;
}

template <typename Kern>
bool ensure_smem(Kern k, size_t bytes) {
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) {
    set_error("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    return false;
  }
  return true;
}

template <int kKind, bool kSwiglu, typename OutT>
moe_status_t launch_fwd(const CUtensorMap& ta, const CUtensorMap& tb, const int32_t* offsets, int M,
                        int N, int K, int E, void* C, void* preact, int32_t* status,
                        cudaStream_t stream, int sms) {
  auto kern = grouped_gemm_fwd_kernel<kKind, kSwiglu, OutT>;
  if (!ensure_smem(kern, kSmemBytes)) return MOE_ERR_CUDA;
  kern<<<sms, kThreads, kSmemBytes, stream>>>(ta, tb, offsets, M, N, K, E, static_cast<OutT*>(C),
                                              static_cast<OutT*>(preact), status);
  return check_launch("moe_grouped_gemm_fwd");
}

}  // namespace gemm
}  // namespace moe

using namespace moe;
using namespace moe::gemm;

static int elem_bytes(moe_dtype_t t) { return t == MOE_F32 ? 4 : (t == MOE_BF16 ? 2 : 1); }

extern "C" moe_status_t moe_grouped_gemm_fwd(const moe_operand_t* A, const moe_operand_t* B,
                                             const int32_t* offsets, int M, int N, int K, int E,
                                             moe_epilogue_t epi, void* C, moe_dtype_t c_dtype,
                                             void* preact, int32_t* dev_status,
                                             cudaStream_t stream) {
  if (!A || !B) {
    set_error("moe_grouped_gemm_fwd: null operand");
    return MOE_ERR_INVALID_ARG;
  }
  if (M < 0 || N <= 0 || K <= 0 || E < 1 || E > kMaxE || K % 32 || N % 32 ||
      (epi == MOE_EPI_SWIGLU && N % 64) || (epi != MOE_EPI_NONE && epi != MOE_EPI_SWIGLU)) {
    set_error("moe_grouped_gemm_fwd: need M >= 0, K %% 32 == 0, N %% 32 == 0 (SwiGLU: N %% 64), 1 <= E <= %d, epi NONE|SWIGLU (M=%d N=%d K=%d E=%d)",
              kMaxE, M, N, K, E);
    return MOE_ERR_INVALID_ARG;
  }
  if (A->dtype != B->dtype || (c_dtype != MOE_BF16 && c_dtype != MOE_F32)) {
    set_error("moe_grouped_gemm_fwd: A and B must share a dtype; C must be BF16 or F32");
    return MOE_ERR_INVALID_ARG;
  }
  if (!offsets || (M > 0 && (!A->ptr || !B->ptr || !C)) || !aligned16(A->ptr) || !aligned16(B->ptr) ||
      !aligned16(C) || !aligned16(preact)) {
    set_error("moe_grouped_gemm_fwd: null or misaligned pointer");
    return MOE_ERR_INVALID_ARG;
  }
  int sms = 0;
  if (!device_is_sm103(&sms)) return MOE_ERR_UNSUPPORTED;
  if (M == 0) return MOE_OK;
  if (A->dtype == MOE_E4M3) {
    set_error("moe_grouped_gemm_fwd: MXFP8 operands are not built in this library");
    return MOE_ERR_UNSUPPORTED;
  }
  const int eb = elem_bytes(A->dtype);
  const CUtensorMapDataType dt =
      A->dtype == MOE_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint32_t bk = kBKBytes / eb;
  CUtensorMap ta, tb;
  const uint64_t adims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
  const uint32_t abox[2] = {bk, kBM};
  const uint64_t bdims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(E)};
  const uint32_t bbox[3] = {bk, static_cast<uint32_t>(epi == MOE_EPI_SWIGLU ? kBN / 2 : kBN), 1};
  if (!make_map(&ta, dt, eb, A->ptr, 2, adims, abox, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&tb, dt, eb, B->ptr, 3, bdims, bbox, CU_TENSOR_MAP_SWIZZLE_128B))
    return MOE_ERR_INVALID_ARG;
  const bool sw = epi == MOE_EPI_SWIGLU;
  if (A->dtype == MOE_F32) {
    if (c_dtype == MOE_F32)
      return sw ? launch_fwd<0, true, float>(ta, tb, offsets, M, N, K, E, C, preact, dev_status, stream, sms)
                : launch_fwd<0, false, float>(ta, tb, offsets, M, N, K, E, C, preact, dev_status, stream, sms);
    return sw ? launch_fwd<0, true, uint16_t>(ta, tb, offsets, M, N, K, E, C, preact, dev_status, stream, sms)
              : launch_fwd<0, false, uint16_t>(ta, tb, offsets, M, N, K, E, C, preact, dev_status, stream, sms);
  }
  if (c_dtype == MOE_F32)
    return sw ? launch_fwd<1, true, float>(ta, tb, offsets, M, N, K, E, C, preact, dev_status, stream, sms)
              : launch_fwd<1, false, float>(ta, tb, offsets, M, N, K, E, C, preact, dev_status, stream, sms);
  return sw ? launch_fwd<1, true, uint16_t>(ta, tb, offsets, M, N, K, E, C, preact, dev_status, stream, sms)
            : launch_fwd<1, false, uint16_t>(ta, tb, offsets, M, N, K, E, C, preact, dev_status, stream, sms);
}

extern "C" moe_status_t moe_grouped_gemm_dgrad(const moe_operand_t* dC, const moe_operand_t* B,
                                               const int32_t* offsets, int M, int N, int K, int E,
                                               moe_epilogue_t epi, const void* preact, void* dA,
                                               moe_dtype_t dA_dtype, int32_t* dev_status,
                                               cudaStream_t stream) {
  (void)dC; (void)B; (void)offsets; (void)M; (void)N; (void)K; (void)E; (void)epi; (void)preact;
  (void)dA; (void)dA_dtype; (void)dev_status; (void)stream;
  set_error("moe_grouped_gemm_dgrad: not built yet");
  return MOE_ERR_UNSUPPORTED;
}

extern "C" moe_status_t moe_grouped_gemm_wgrad(const moe_operand_t* A, const moe_operand_t* dC,
                                               const int32_t* offsets, int M, int N, int K, int E,
                                               void* dB, moe_dtype_t dB_dtype, int32_t* dev_status,
                                               cudaStream_t stream) {
  (void)A; (void)dC; (void)offsets; (void)M; (void)N; (void)K; (void)E; (void)dB; (void)dB_dtype;
  (void)dev_status; (void)stream;
  set_error("moe_grouped_gemm_wgrad: not built yet");
  return MOE_ERR_UNSUPPORTED;
}

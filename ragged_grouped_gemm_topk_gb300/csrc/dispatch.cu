// Local dispatch (token permutation) and row-wise group-aware MXFP8 quantisation.
//
// Dispatch per "Accelerating Dropless MoE Training in JAX with NVIDIA Transformer
// Engine", "Optimisation 2" (dispatch = local rearrangement of tokens by expert)
// and Figure 3.  Rows are ordered by (expert, token), so the permutation is
// unique and the kernels reproduce it exactly without sorting:
//
//   rank     one block per 256 tokens; each warp builds, for its 32 tokens, a
//            32-bit mask per expert (atomicOr in shared memory, order-free), so
//            a pair's rank among earlier tokens of the same expert is a popcount;
//            per-warp counts are scanned inside the block and the block's
//            per-expert totals go to the workspace.
//   scatter  every CTA scans the routed counts into offsets (CTA 0 publishes
//            them and checks them against the rank pass); one warp per token
//            adds the counts of its expert in the earlier rank blocks (a warp
//            reduction) to get dest_row / src_pair, then copies the token's row
//            with 16-byte loads (8 per lane in flight) and stores to its k rows,
//            optionally quantised to MXFP8 on the way.
//
// MXFP8 follows the OCP Microscaling Formats v1.0 conversion (shared exponent
// floor(log2 amax) - 8, clamped to [-127, 127]; E4M3 round-to-nearest-even with
// saturation); an all-zero block gets scale byte 127.  Blocks run along a row,
// and a row belongs to one expert, so no block mixes two experts ("group-aware").
#include "common.cuh"

namespace moe {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr int kRankThreads = 256;                    // 8 warps x 32 tokens per block
constexpr int kTokensPerRankBlock = kRankThreads;
constexpr int kScatterThreads = 256;

__device__ __forceinline__ void permute_rank_body(const int32_t* __restrict__ idx, int T, int k, int E,
                                                  int32_t* __restrict__ local_rank, int32_t* __restrict__ block_hist,
                                                  int32_t* status) {
  extern __shared__ uint32_t sm[];
  uint32_t* mask = sm;                                      // [8][E]
  int32_t* wbase = reinterpret_cast<int32_t*>(sm + 8 * E);  // [8][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 8 * E; i += blockDim.x) mask[i] = 0;
  __syncthreads();
  const int t = blockIdx.x * kTokensPerRankBlock + warp * 32 + lane;
  if (t < T) {
    for (int j = 0; j < k; ++j) {
      const int e = idx[static_cast<size_t>(t) * k + j];
      if (e < 0 || e >= E) {
        flag_error(status, MOE_DEV_BAD_INDEX);
        continue;
      }
      atomicOr(&mask[warp * E + e], 1u << lane);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      wbase[w * E + e] = run;
      run += __popc(mask[w * E + e]);
    }
    block_hist[static_cast<size_t>(blockIdx.x) * E + e] = run;
  }
  __syncthreads();
  if (t < T) {
    const uint32_t below = (1u << lane) - 1u;
    for (int j = 0; j < k; ++j) {
      const int e = idx[static_cast<size_t>(t) * k + j];
      int r = -1;
      if (e >= 0 && e < E) r = wbase[warp * E + e] + __popc(mask[warp * E + e] & below);
      local_rank[static_cast<size_t>(t) * k + j] = r;
    }
  }
}

__global__ void __launch_bounds__(kRankThreads) permute_rank_kernel(
    const int32_t* __restrict__ idx, int T, int k, int E, int32_t* __restrict__ local_rank,
    int32_t* __restrict__ block_hist, int32_t* status) {
  pdl_begin();
  permute_rank_body(idx, T, k, E, local_rank, block_hist, status);
}

// NVFP4 dispatch, first pass: the rank blocks (the first nblk) and the tensor amax of
// x (the other blocks) in one launch, as the two are independent.
template <typename Tin>
__global__ void __launch_bounds__(kRankThreads) permute_rank_amax_kernel(
    const int32_t* __restrict__ idx, int T, int k, int E, int32_t* __restrict__ local_rank,
    int32_t* __restrict__ block_hist, int32_t* status, int nblk, const uint8_t* __restrict__ x, long long n16,
    uint32_t* amax_bits) {
  pdl_begin();
  if (static_cast<int>(blockIdx.x) < nblk)
    permute_rank_body(idx, T, k, E, local_rank, block_hist, status);
  else
    nvfp4_amax_body<Tin>(x, n16, amax_bits, blockIdx.x - nblk, gridDim.x - nblk);
}

struct alignas(16) Vec16 {
  uint32_t w[4];
};

// MXFP8 of one 16-byte chunk held by a lane: returns the E4M3 bytes of its
// elements; the 32-element block is shared by LPB consecutive lanes.
template <typename Tin>
struct Mx;

template <>
struct Mx<uint16_t> {  // bf16: 8 elements per lane, 4 lanes per block
  static constexpr int kEpl = 8;
  static constexpr int kLpb = 4;
  __device__ static void values(const Vec16& v, float (&f)[8]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = bf16_to_f32(static_cast<uint16_t>(v.w[i] & 0xFFFFu));
      f[2 * i + 1] = bf16_to_f32(static_cast<uint16_t>(v.w[i] >> 16));
    }
  }
};

template <>
struct Mx<float> {  // f32: 4 elements per lane, 8 lanes per block
  static constexpr int kEpl = 4;
  static constexpr int kLpb = 8;
  __device__ static void values(const Vec16& v, float (&f)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = __uint_as_float(v.w[i]);
  }
};

// Quantise one lane's chunk; all 32 lanes must call (inactive lanes pass zeros).
template <typename Tin>
__device__ __forceinline__ void mx_chunk(const Vec16& v, uint32_t (&codes)[2], uint32_t* sbyte) {
  constexpr int EPL = Mx<Tin>::kEpl;
  float f[EPL];
  Mx<Tin>::values(v, f);
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
  for (int off = 1; off < Mx<Tin>::kLpb; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
  float inv;
  mx_scale(amax, sbyte, &inv);
  codes[0] = codes[1] = 0;
#pragma unroll
  for (int i = 0; i < EPL; i += 2) {
    const uint32_t pr = f32x2_to_e4m3x2(f[i] * inv, f[i + 1] * inv);
    codes[i / 4] |= pr << (16 * ((i / 2) & 1));
  }
}

// One warp per token.  Each lane keeps kScatterU 16-byte chunks of the row in
// flight (8 KB per warp), and the first batch is requested before the token's
// destinations are resolved so that the two latencies overlap.
constexpr int kScatterU = 8;
// Quantising scatter: each warp quantises a segment of 32 * kScatterU chunks of its
// token once, into a shared-memory buffer (codes, then scales), and copies the segment
// out to the token's k rows with wide stores.
constexpr int kSegCodes = 32 * kScatterU * 8;       // MXFP8 from bf16: 8 code bytes a chunk
constexpr int kSegBytes = kSegCodes + 32 * kScatterU * 8 / 16;   // + NVFP4 scales from bf16 (the most)

// Warp-cooperative copy of n bytes from shared memory (16-byte aligned) to global
// memory: 16-byte stores where the destination and the length allow, else 4- or 1-byte.
__device__ __forceinline__ void warp_copy_out(uint8_t* dst, const uint8_t* src, int n, int lane) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(dst) | static_cast<uintptr_t>(n);
  if ((a & 15) == 0) {
    for (int o = lane * 16; o < n; o += 512)
      *reinterpret_cast<uint4*>(dst + o) = *reinterpret_cast<const uint4*>(src + o);
  } else if ((a & 3) == 0) {
    for (int o = lane * 4; o < n; o += 128)
      *reinterpret_cast<uint32_t*>(dst + o) = *reinterpret_cast<const uint32_t*>(src + o);
  } else {
    for (int o = lane; o < n; o += 32) dst[o] = src[o];
  }
}

// kQuant: 0 = copy rows, 1 = MXFP8 rows, 2 = NVFP4 rows (packed E2M1 codes [.., d/2],
// E4M3 scales per 16 [.., d/16], tensor scale from the amax of x in *amax_bits, which
// is the amax of the permuted rows: every token is routed).
// Chunk of a segment held in a lane's slot i: chunks i*32 + lane (coalesced), or, for
// bf16 rows quantised to NVFP4, each lane two adjacent chunks (one whole 16-element
// block) per pair of slots.
template <bool kBlockLane>
__device__ __forceinline__ int chunk_of(int i, int lane) {
  return kBlockLane ? 64 * (i / 2) + 2 * lane + (i & 1) : 32 * i + lane;
}

// (four CTAs per SM: 64 registers, no spill, for every row type)
template <typename Tin, int kQuant>
__global__ void __launch_bounds__(kScatterThreads, 4) permute_scatter_kernel(
    const uint8_t* __restrict__ x, int T, int d, const int32_t* __restrict__ idx, int k, int E,
    const int32_t* __restrict__ counts, const int32_t* local_rank, const int32_t* __restrict__ block_hist,
    int nblk, int32_t* __restrict__ offsets, int32_t* dest_row, int32_t* __restrict__ src_pair,
    uint8_t* __restrict__ xp, uint8_t* __restrict__ xp_scales, const uint32_t* amax_bits, float* tensor_scale,
    int32_t* status) {
  pdl_begin();
  float g4 = 1.f;
  // NVFP4: the multiplier of every scale byte (g / its value), computed once per CTA
  __shared__ float s_inv[kQuant == 2 ? 256 : 1];
  // quantising scatter: one staging segment per warp
  __shared__ __align__(16) uint8_t s_seg[kQuant ? kScatterThreads / 32 : 1][kQuant ? kSegBytes : 16];
  if constexpr (kQuant == 2) {
    g4 = nvfp4_tensor_scale(__uint_as_float(*amax_bits));
    if (blockIdx.x == 0 && threadIdx.x == 0) *tensor_scale = g4;
    for (int c = threadIdx.x; c < 256; c += blockDim.x) s_inv[c] = nvfp4_block_inv(static_cast<uint32_t>(c), g4);
  }
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  // offsets = exclusive scan of the routed counts, in every CTA (E <= 1024)
  __shared__ int s_off[1025];
  __shared__ int s_part[kScatterThreads / 32];
  {
    constexpr int G = 1024 / kScatterThreads;
    int c[G], sum = 0;
#pragma unroll
    for (int u = 0; u < G; ++u) {
      const int e = threadIdx.x * G + u;
      c[u] = e < E ? counts[e] : 0;
      sum += c[u];
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int w = __shfl_up_sync(kFull, incl, off);
      if (lane >= off) incl += w;
    }
    if (lane == 31) s_part[threadIdx.x >> 5] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < static_cast<int>(threadIdx.x >> 5); ++w) before += s_part[w];
    int run = before + incl - sum;
#pragma unroll
    for (int u = 0; u < G; ++u) {
      const int e = threadIdx.x * G + u;
      if (e <= E) s_off[e] = run;
      run += c[u];
    }
    // the loop reaches index G * kScatterThreads - 1 at most: at E = 1024 the end
    // of the scan (every routed pair) is written by the last thread
    if (E == G * kScatterThreads && threadIdx.x == kScatterThreads - 1) s_off[E] = run;
    __syncthreads();
  }
  if (blockIdx.x == 0) {
    // publish offsets; the routed counts must cover every pair and agree with the
    // per-block histograms of the rank pass
    for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = s_off[e];
    if (threadIdx.x == 0 && s_off[E] != T * k) flag_error(status, MOE_DEV_BAD_INDEX);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int col = 0;
      for (int b = 0; b < nblk; ++b) col += block_hist[static_cast<size_t>(b) * E + e];
      if (col != s_off[e + 1] - s_off[e]) flag_error(status, MOE_DEV_BAD_INDEX);
    }
  }
  const size_t in_row = static_cast<size_t>(d) * sizeof(Tin);
  const size_t out_row = kQuant == 2 ? static_cast<size_t>(d) / 2 : (kQuant ? static_cast<size_t>(d) : in_row);
  const int n16 = static_cast<int>(in_row / 16);
  constexpr bool kBlockLane = kQuant == 2 && Mx<Tin>::kEpl == 8;
  for (int tw = blockIdx.x * wpb + (threadIdx.x >> 5); tw < T; tw += gridDim.x * wpb) {
    // NVFP4: the tensor-amax pass has just streamed x, last rows last, so the scatter
    // takes the tokens from the end and finds the most recent of them still in L2
    const int t = kQuant == 2 ? T - 1 - tw : tw;
    const Vec16* src = reinterpret_cast<const Vec16*>(x + static_cast<size_t>(t) * in_row);
    Vec16 v[kScatterU];
    auto load = [&](int base) {
#pragma unroll
      for (int i = 0; i < kScatterU; ++i) {
        const int c = base + chunk_of<kBlockLane>(i, lane);
        if (c < n16) {
          v[i] = src[c];
        } else {
          v[i].w[0] = v[i].w[1] = v[i].w[2] = v[i].w[3] = 0;
        }
      }
    };
    if (xp != nullptr) load(0);
    // destination of slot j (lane j): offsets[e] + the pairs of expert e in the rank
    // blocks before this token's (summed by the warp) + the rank inside its block
    const int blk = t / kTokensPerRankBlock;
    int e_l = -1, r_l = -1;
    if (lane < k) {
      const size_t p = static_cast<size_t>(t) * k + lane;
      e_l = idx[p];
      r_l = local_rank[p];
    }
    int before = 0;
    for (int j = 0; j < k; ++j) {
      const int e = __shfl_sync(kFull, e_l, j);
      int part = 0;
      if (e >= 0 && e < E)
        for (int b = lane; b < blk; b += 32) part += block_hist[static_cast<size_t>(b) * E + e];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(kFull, part, off);
      if (lane == j) before = part;
    }
    int dest = -1;
    if (lane < k) {
      const size_t p = static_cast<size_t>(t) * k + lane;
      if (e_l >= 0 && e_l < E && r_l >= 0) dest = s_off[e_l] + before + r_l;
      if (dest >= T * k) {
        flag_error(status, MOE_DEV_BAD_INDEX);
        dest = -1;
      }
      dest_row[p] = dest;
      if (dest >= 0) src_pair[dest] = static_cast<int32_t>(p);
    }
    if (xp == nullptr) continue;
    for (int base = 0; base < n16; base += 32 * kScatterU) {
      if (kQuant == 0 && base > 0) load(base);
      if constexpr (kQuant != 0) {
        // quantise the segment once into this warp's staging buffer: codes at
        // [0, kSegCodes), the scale bytes after them
        constexpr int EPL = Mx<Tin>::kEpl;
        constexpr int CB = kQuant == 2 ? EPL / 2 : EPL;      // code bytes per chunk
        constexpr int BLK = kQuant == 2 ? 16 : 32;           // elements per scale byte
        uint8_t* seg = s_seg[threadIdx.x >> 5];
        if constexpr (kBlockLane) {
          // bf16 to NVFP4: each lane one whole 16-element block per pair of slots (no
          // shuffle for the block amax, one scale per lane); n16 is even (d % 16 == 0)
#pragma unroll
          for (int m = 0; m < kScatterU / 2; ++m) {
            if (base + 64 * m >= n16) break;   // warp-uniform
            const int cl = 64 * m + 2 * lane;  // the block's first chunk within the segment
            float f0[8], f1[8];
            Mx<Tin>::values(v[2 * m], f0);
            Mx<Tin>::values(v[2 * m + 1], f1);
            float amax = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fmaxf(fabsf(f0[e]), fabsf(f1[e])));
            const uint32_t scode = nvfp4_block_code(amax, g4);
            const float inv = s_inv[scode];
            float y0[8], y1[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              y0[e] = __fmul_rn(f0[e], inv);
              y1[e] = __fmul_rn(f1[e], inv);
            }
            if (base + cl < n16) {
              *reinterpret_cast<uint2*>(seg + cl * 4) = make_uint2(f32x8_to_e2m1x8(y0), f32x8_to_e2m1x8(y1));
              seg[kSegCodes + cl / 2] = static_cast<uint8_t>(scode);
            }
          }
        } else {
#pragma unroll
        for (int i = 0; i < kScatterU; ++i) {
          if (base + 32 * i >= n16) break;     // warp-uniform: no lane of this chunk row is active
          const int cl = 32 * i + lane;        // chunk within the segment
          const bool active = base + cl < n16;
          if constexpr (kQuant == 2) {
            // a 16-element block spans 16 / EPL lanes
            constexpr int LPB = 16 / EPL;
            float f[EPL];
            Mx<Tin>::values(v[i], f);
            float amax = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(f[e]));
#pragma unroll
            for (int off = 1; off < LPB; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
            const uint32_t scode = nvfp4_block_code(amax, g4);
            const float inv = s_inv[scode];
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = e < EPL ? __fmul_rn(f[e < EPL ? e : 0], inv) : 0.f;
            const uint32_t packed = f32x8_to_e2m1x8(y);   // EPL codes in the low EPL nibbles
            if (active) {
              if (EPL == 8)
                *reinterpret_cast<uint32_t*>(seg + cl * CB) = packed;
              else
                *reinterpret_cast<uint16_t*>(seg + cl * CB) = static_cast<uint16_t>(packed);
              if ((lane % LPB) == 0) seg[kSegCodes + (cl * EPL) / BLK] = static_cast<uint8_t>(scode);
            }
          } else {
            uint32_t codes[2], sbyte;
            mx_chunk<Tin>(v[i], codes, &sbyte);
            if (active) {
              if (EPL == 8)
                *reinterpret_cast<uint2*>(seg + cl * CB) = make_uint2(codes[0], codes[1]);
              else
                *reinterpret_cast<uint32_t*>(seg + cl * CB) = codes[0];
              if ((lane % Mx<Tin>::kLpb) == 0) seg[kSegCodes + (cl * EPL) / BLK] = static_cast<uint8_t>(sbyte);
            }
          }
        }
        }
        __syncwarp();
        // the next segment's loads (the registers are free now) overlap this one's stores
        if (base + 32 * kScatterU < n16) load(base + 32 * kScatterU);
        // then copy it out to each of the token's rows
        const int nvalid = n16 - base < 32 * kScatterU ? n16 - base : 32 * kScatterU;
        const size_t srow = static_cast<size_t>(d) / BLK;
        // MOE_DEBUG: the segment's codes and scales lie inside the warp's buffer
        const bool seg_ok = dbg_check(nvalid * CB <= kSegCodes && nvalid * EPL / BLK <= kSegBytes - kSegCodes, status);
        for (int j = 0; j < k && seg_ok; ++j) {
          const int dj = __shfl_sync(kFull, dest, j);
          if (dj < 0) continue;                // warp-uniform
          warp_copy_out(xp + static_cast<size_t>(dj) * out_row + static_cast<size_t>(base) * CB, seg, nvalid * CB,
                        lane);
          warp_copy_out(xp_scales + static_cast<size_t>(dj) * srow + static_cast<size_t>(base) * EPL / BLK,
                        seg + kSegCodes, nvalid * EPL / BLK, lane);
        }
        __syncwarp();                          // the segment is read before the next one is written
      } else {
#pragma unroll
        for (int i = 0; i < kScatterU; ++i) {
          const int c = base + 32 * i + lane;
          const bool active = c < n16;
          for (int j = 0; j < k; ++j) {
            const int dj = __shfl_sync(kFull, dest, j);
            if (active && dj >= 0)
              reinterpret_cast<Vec16*>(xp + static_cast<size_t>(dj) * out_row)[c] = v[i];
          }
        }
      }
    }
  }
}

template <typename Tin>
__global__ void __launch_bounds__(kScatterThreads) quantize_rowwise_kernel(
    const uint8_t* __restrict__ in, int rows, int K, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  constexpr int EPL = Mx<Tin>::kEpl;
  const size_t in_row = static_cast<size_t>(K) * sizeof(Tin);
  const int n16 = static_cast<int>(in_row / 16);
  for (int r = blockIdx.x * wpb + (threadIdx.x >> 5); r < rows; r += gridDim.x * wpb) {
    const Vec16* src = reinterpret_cast<const Vec16*>(in + static_cast<size_t>(r) * in_row);
    constexpr int U = kScatterU / 2;     // chunks per lane in flight
    for (int base = 0; base < n16; base += 32 * U) {
      Vec16 v[U];
#pragma unroll
      for (int i = 0; i < U; ++i) {
        const int c = base + 32 * i + lane;
        if (c < n16) {
          v[i] = src[c];
        } else {
          v[i].w[0] = v[i].w[1] = v[i].w[2] = v[i].w[3] = 0;
        }
      }
#pragma unroll
      for (int i = 0; i < U; ++i) {
        if (base + 32 * i >= n16) break;      // warp-uniform
        const int c = base + 32 * i + lane;
        uint32_t q[2], sbyte;
        mx_chunk<Tin>(v[i], q, &sbyte);
        if (c < n16) {
          uint8_t* orow = codes + static_cast<size_t>(r) * K + static_cast<size_t>(c) * EPL;
          if (EPL == 8)
            *reinterpret_cast<uint2*>(orow) = make_uint2(q[0], q[1]);
          else
            *reinterpret_cast<uint32_t*>(orow) = q[0];
          if ((lane % Mx<Tin>::kLpb) == 0)
            scales[static_cast<size_t>(r) * (K / 32) + (c * EPL) / 32] = static_cast<uint8_t>(sbyte);
        }
      }
    }
  }
}

// Column-wise, group-aware MXFP8: a block is 32 consecutive rows of one column,
// blocks restart at every group start, and the rows of a group's last block past
// its end count as zeros (they never change the amax and get no codes).  Block
// rows are numbered group by group: group e's first is sum over e' < e of
// ceil(count_e' / 32).  One work item = (block row, strip of columns); each thread
// owns 4 adjacent columns (an 8- or 16-byte chunk) and keeps the block's 32 rows of
// them in registers (32 loads in flight), so reads and writes stay row-contiguous
// across the warp.
//
// kTiled: the scales leave in the layout the block-scaled weight-gradient GEMM reads
// straight into its tensor-memory scale slots.  Group e's 32-row blocks are taken
// four at a time (a quad: 128 rows); quad q of group e has index
// Q = floor(offsets[e] / 128) + e + q (distinct for every group and quad, and below
// ceil(rows / 128) + E).  The scales of quad Q and columns [128c, 128c + 128) form
// one 512-byte tile at ((Q * K / 128) + c) * 512, where column m of the 128 and block
// j of the quad sit at byte (m % 32) * 16 + (m / 32) * 4 + j.  Bytes of blocks past a
// group's last one are not written.
//
// gather (optional): the rows to quantise are the dispatched rows Xp[r] =
// in[gather[r] / gk] (gather = the dispatch's src_pair, gk = top-k), read straight
// from the token rows instead of from a materialised Xp.  Each warp loads its
// block's 32 pair indices with one coalesced load into shared memory; a pair index
// outside [0, gpairs) flags MOE_DEV_BAD_INDEX and its row reads as zeros.  With
// gweight (per-pair weights, the routing weights) the rows are gweight[p] *
// in[p / gk], the product taken in fp32 and rounded to Tin: the rows the combine
// backward writes as dYp, quantised without being stored.
//
// slots (gathered form): every token row is read by k blocks, one per expert it routes
// to.  Taken in group order, those reads are far apart and each comes from DRAM.  With
// slots > 0 the blocks are taken slot by slot instead: block b of a group with nb blocks
// goes to slot floor(b * slots / nb), i.e. by its position in its group, and so, since a
// group's rows are in token order, roughly by the tokens it reads; inside a slot, group
// by group.  The blocks of one slot read one token range, which stays in L2 for its k
// readers.  The slot tables sit in dynamic shared memory: qtab[s][e] = sum over e' < e of
// ceil(s * nb_e' / slots), for s = 0..slots and e = 0..E.  The output does not depend on
// the order.
constexpr int kColThreads = 128;

template <typename Tin, bool kTiled>
__global__ void __launch_bounds__(kColThreads) quantize_colwise_kernel(
    const uint8_t* __restrict__ in, int rows, int K, const int32_t* __restrict__ offsets, int E,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, const int32_t* __restrict__ gather,
    const float* __restrict__ gweight, int gk, int gpairs, int32_t* status, int slots) {
  pdl_begin();
  extern __shared__ int qtab[];                // slots > 0: [slots + 1][E + 1]
  constexpr int EB = sizeof(Tin);
  constexpr int CPT = 4;                       // columns per thread
  constexpr int NW = CPT * EB / 4;             // 32-bit words per chunk
  constexpr int kStrip = kColThreads * CPT;
  __shared__ int bpre[1025];                   // block-row prefix per group
  __shared__ int part[kColThreads];
  __shared__ int grow[kColThreads / 32][32];   // gathered source rows of the task's block, per warp
  __shared__ float gwt[kColThreads / 32][32];  // and their weights
  // blocks per group (invalid groups count as empty), then an exclusive scan
  constexpr int G = 1024 / kColThreads;        // groups per thread (E <= 1024)
  int cnt[G], sum = 0;
#pragma unroll
  for (int u = 0; u < G; ++u) {
    const int e = threadIdx.x * G + u;
    int c = 0;
    if (e < E) {
      const int lo = offsets[e], hi = offsets[e + 1];
      if (lo >= 0 && hi >= lo && hi <= rows) c = (hi - lo + 31) / 32;
    }
    cnt[u] = c;
    sum += c;
  }
  part[threadIdx.x] = sum;
  __syncthreads();
  if (threadIdx.x < 32) {
    int carry = 0;
    for (int base = 0; base < kColThreads; base += 32) {
      int v = part[base + threadIdx.x];
      const int own = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int w = __shfl_up_sync(kFull, v, off);
        if (static_cast<int>(threadIdx.x) >= off) v += w;
      }
      part[base + threadIdx.x] = carry + v - own;   // exclusive
      carry += __shfl_sync(kFull, v, 31);
    }
  }
  __syncthreads();
  {
    int run = part[threadIdx.x];
#pragma unroll
    for (int u = 0; u < G; ++u) {
      const int e = threadIdx.x * G + u;
      if (e < E) bpre[e] = run;
      run += cnt[u];
    }
    if (threadIdx.x == kColThreads - 1) bpre[E] = run;   // every block row
  }
  __syncthreads();
  if (slots > 0) {
    // qtab[s][e]: exclusive scan over the groups of ceil(s * nb_e / slots)
    for (int sl = 0; sl <= slots; ++sl) {
      int* q = qtab + sl * (E + 1);
      int own = 0;
#pragma unroll
      for (int u = 0; u < G; ++u) {
        const int e = threadIdx.x * G + u;
        const int nb = e < E ? bpre[e + 1] - bpre[e] : 0;
        cnt[u] = (sl * nb + slots - 1) / slots;
        own += cnt[u];
      }
      part[threadIdx.x] = own;
      __syncthreads();
      if (threadIdx.x < 32) {
        int carry = 0;
        for (int base = 0; base < kColThreads; base += 32) {
          int v = part[base + threadIdx.x];
          const int mine = v;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const int w = __shfl_up_sync(kFull, v, off);
            if (static_cast<int>(threadIdx.x) >= off) v += w;
          }
          part[base + threadIdx.x] = carry + v - mine;   // exclusive
          carry += __shfl_sync(kFull, v, 31);
        }
      }
      __syncthreads();
      int run = part[threadIdx.x];
#pragma unroll
      for (int u = 0; u < G; ++u) {
        const int e = threadIdx.x * G + u;
        if (e < E) q[e] = run;
        run += cnt[u];
      }
      if (threadIdx.x == kColThreads - 1) q[E] = run;
      __syncthreads();
    }
  }
  const int total = bpre[E];
  const int nstrip = (K + kStrip - 1) / kStrip;
  const size_t in_row = static_cast<size_t>(K) * EB;
  for (long long task = blockIdx.x; task < static_cast<long long>(total) * nstrip; task += gridDim.x) {
    const int strip = static_cast<int>(task % nstrip);
    int br, lo_e = 0;
    if (slots > 0) {
      // block ordinal i -> slot sl (blocks of slots < sl: qtab[sl][E]) -> group (blocks of
      // slot sl in groups < e: qtab[sl + 1][e] - qtab[sl][e]) -> block in the group
      const int i = static_cast<int>(task / nstrip);
      int sl = 0, hs = slots - 1;
      while (sl < hs) {
        const int mid = (sl + hs + 1) >> 1;
        if (qtab[mid * (E + 1) + E] <= i) sl = mid; else hs = mid - 1;
      }
      const int* q0 = qtab + sl * (E + 1);
      const int* q1 = q0 + (E + 1);
      const int j = i - q0[E];
      int hi_e = E - 1;
      while (lo_e < hi_e) {
        const int mid = (lo_e + hi_e + 1) >> 1;
        if (q1[mid] - q0[mid] <= j) lo_e = mid; else hi_e = mid - 1;
      }
      const int b = (q0[lo_e + 1] - q0[lo_e]) + (j - (q1[lo_e] - q0[lo_e]));
      br = bpre[lo_e] + b;
    } else {
      br = static_cast<int>(task / nstrip);
      int hi_e = E - 1;                         // last group whose first block row <= br
      while (lo_e < hi_e) {
        const int mid = (lo_e + hi_e + 1) >> 1;
        if (bpre[mid] <= br) lo_e = mid; else hi_e = mid - 1;
      }
    }
    const int r0 = offsets[lo_e] + (br - bpre[lo_e]) * 32;
    const int n = min(32, offsets[lo_e + 1] - r0);
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (gather) {                                // every lane, before any lane leaves the task
      __syncwarp();                              // the previous task's reads of grow are done
      int srow = -1;
      float wr = 1.f;
      if (lane < n) {
        const int p = gather[r0 + lane];
        if (p >= 0 && p < gpairs) {
          srow = p / gk;
          if (gweight) wr = gweight[p];
        } else {
          flag_error(status, MOE_DEV_BAD_INDEX);
        }
      }
      grow[wid][lane] = srow;
      gwt[wid][lane] = wr;
      __syncwarp();
    }
    const int col = strip * kStrip + CPT * threadIdx.x;   // K % 32 == 0: a chunk is all in or all out
    if (col >= K) continue;
    uint32_t raw[32][NW];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int srow = gather ? grow[wid][i] : r0 + i;
      const bool ok = i < n && srow >= 0;
      const uint8_t* src = in + static_cast<size_t>(ok ? srow : 0) * in_row + static_cast<size_t>(col) * EB;
      if constexpr (NW == 2) {
        const uint2 u = ok ? *reinterpret_cast<const uint2*>(src) : make_uint2(0u, 0u);
        raw[i][0] = u.x;
        raw[i][1] = u.y;
      } else {
        const uint4 u = ok ? *reinterpret_cast<const uint4*>(src) : make_uint4(0u, 0u, 0u, 0u);
        raw[i][0] = u.x;
        raw[i][1] = u.y;
        raw[i][2] = u.z;
        raw[i][3] = u.w;
      }
    }
    if (gweight) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float wr = gwt[wid][i];
#pragma unroll
        for (int j = 0; j < NW; ++j) {
          if constexpr (NW == 2)
            raw[i][j] = pack_bf16x2(wr * bf16_to_f32(static_cast<uint16_t>(raw[i][j] & 0xFFFFu)),
                                    wr * bf16_to_f32(static_cast<uint16_t>(raw[i][j] >> 16)));
          else
            raw[i][j] = __float_as_uint(wr * __uint_as_float(raw[i][j]));
        }
      }
    }
    auto decode = [](const uint32_t (&w)[NW], float (&f)[CPT]) {
      if constexpr (NW == 2) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          f[2 * j] = bf16_to_f32(static_cast<uint16_t>(w[j] & 0xFFFFu));
          f[2 * j + 1] = bf16_to_f32(static_cast<uint16_t>(w[j] >> 16));
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) f[j] = __uint_as_float(w[j]);
      }
    };
    float amax[CPT];
#pragma unroll
    for (int j = 0; j < CPT; ++j) amax[j] = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      float f[CPT];
      decode(raw[i], f);
#pragma unroll
      for (int j = 0; j < CPT; ++j) amax[j] = fmaxf(amax[j], fabsf(f[j]));
    }
    uint32_t sb[CPT];
    float inv[CPT];
#pragma unroll
    for (int j = 0; j < CPT; ++j) mx_scale(amax[j], &sb[j], &inv[j]);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (i < n) {
        float f[CPT];
        decode(raw[i], f);
        *reinterpret_cast<uint32_t*>(codes + static_cast<size_t>(r0 + i) * K + col) =
            static_cast<uint32_t>(f32x2_to_e4m3x2(f[0] * inv[0], f[1] * inv[1])) |
            (static_cast<uint32_t>(f32x2_to_e4m3x2(f[2] * inv[2], f[3] * inv[3])) << 16);
      }
    }
    if constexpr (kTiled) {
      const int b = br - bpre[lo_e];                         // block within the group
      const size_t quad = static_cast<size_t>(offsets[lo_e] / 128 + lo_e + b / 4);
      uint8_t* tile = scales + (quad * (K / 128) + col / 128) * 512 + (b % 4);
#pragma unroll
      for (int j = 0; j < CPT; ++j) {
        const int m = col % 128 + j;
        tile[(m % 32) * 16 + (m / 32) * 4] = static_cast<uint8_t>(sb[j]);
      }
    } else {
      *reinterpret_cast<uint32_t*>(scales + static_cast<size_t>(br) * K + col) =
          sb[0] | (sb[1] << 8) | (sb[2] << 16) | (sb[3] << 24);
    }
  }
}

// Transposed row-wise MXFP8 of a batch of matrices: in [G, R, C] -> codes [G, C, R]
// and scales [G, C, R / 32], blocks of 32 along R (so the transposed matrix is
// quantised row-wise along its rows).  For weights read along their output dim: the
// data gradient contracts B [E, N, K] over N, so it needs B^T [E, K, N] with scales
// along N.  A CTA task is one matrix, kTrCols(Tin) columns (512 bytes of a row) and
// kTrRb 32-row blocks.  Thread j owns column j: per block it quantises the 32
// values of its column (read back from shared memory) and writes them as one
// 32-byte run of the transposed row; its kTrRb scale bytes leave as one 16-byte
// store at the end, so scale writes fill whole sectors.  Row blocks stream through
// two shared-memory buffers with cp.async, the next block loading while this one
// is encoded.
constexpr int kTrRb = 16;
template <typename Tin>
constexpr int tr_cols() { return 512 / static_cast<int>(sizeof(Tin)); }

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sa), "l"(gmem), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <typename Tin>
__global__ void __launch_bounds__(tr_cols<Tin>(), 4) quantize_transposed_kernel(
    const uint8_t* __restrict__ in, int G, int R, int C, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales) {
  pdl_begin();
  constexpr int EB = sizeof(Tin);
  constexpr int COLS = tr_cols<Tin>();
  constexpr int kChunks = COLS * EB / 16;                    // 16-byte chunks per tile row (32)
  __shared__ __align__(16) Tin tile[2][32][COLS];
  const int nrb = R / 32, ncb = (C + COLS - 1) / COLS, nrg = (nrb + kTrRb - 1) / kTrRb;
  const long long tasks = static_cast<long long>(G) * ncb * nrg;
  const bool vec_scales = nrb % kTrRb == 0;                   // 16-byte aligned scale runs
  for (long long task = blockIdx.x; task < tasks; task += gridDim.x) {
    const int g = static_cast<int>(task / (static_cast<long long>(ncb) * nrg));
    const int rem = static_cast<int>(task % (static_cast<long long>(ncb) * nrg));
    const int rg = rem / ncb, c0 = (rem % ncb) * COLS;
    const int rb0 = rg * kTrRb, nb = min(kTrRb, nrb - rb0);
    const uint8_t* src = in + static_cast<size_t>(g) * R * C * EB;
    auto load = [&](int rb, int buf) {
#pragma unroll
      for (int i = threadIdx.x; i < 32 * kChunks; i += COLS) {
        const int r = i / kChunks, ch = i % kChunks;
        const int c = c0 + ch * (16 / EB);
        const bool ok = c < C;
        const uint8_t* gp = src + (static_cast<size_t>(rb * 32 + r) * C + (ok ? c : 0)) * EB;
        cp_async16(&tile[buf][r][ch * (16 / EB)], gp, ok);
      }
      cp_async_commit();
    };
    load(rb0, 0);
    const int c = c0 + threadIdx.x;
    uint32_t sc[kTrRb / 4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < kTrRb; ++i) {
      if (i < nb) {
        if (i + 1 < nb) {
          load(rb0 + i + 1, (i + 1) & 1);
          cp_async_wait<1>();
        } else {
          cp_async_wait<0>();
        }
        __syncthreads();
        if (c < C) {
          const Tin* col = &tile[i & 1][0][threadIdx.x];
          float amax = 0.f;
#pragma unroll
          for (int r = 0; r < 32; ++r) {
            float v;
            if constexpr (EB == 2) v = bf16_to_f32(static_cast<uint16_t>(col[r * COLS]));
            else v = static_cast<float>(col[r * COLS]);
            amax = fmaxf(amax, fabsf(v));
          }
          uint32_t sb;
          float inv;
          mx_scale(amax, &sb, &inv);
          uint32_t w[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if constexpr (EB == 2) v[u] = bf16_to_f32(static_cast<uint16_t>(col[(4 * q + u) * COLS]));
              else v[u] = static_cast<float>(col[(4 * q + u) * COLS]);
            }
            w[q] = static_cast<uint32_t>(f32x2_to_e4m3x2(v[0] * inv, v[1] * inv)) |
                   (static_cast<uint32_t>(f32x2_to_e4m3x2(v[2] * inv, v[3] * inv)) << 16);
          }
          uint8_t* dst = codes + (static_cast<size_t>(g) * C + c) * R + static_cast<size_t>(rb0 + i) * 32;
          reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
          reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
          sc[i / 4] |= sb << (8 * (i % 4));
        }
        __syncthreads();                  // the buffer is reloaded two blocks on
      }
    }
    if (c < C) {
      uint8_t* sdst = scales + (static_cast<size_t>(g) * C + c) * nrb + rb0;
      if (vec_scales) {
        *reinterpret_cast<uint4*>(sdst) = make_uint4(sc[0], sc[1], sc[2], sc[3]);
      } else {
#pragma unroll
        for (int i = 0; i < kTrRb; ++i)
          if (i < nb) sdst[i] = static_cast<uint8_t>(sc[i / 4] >> (8 * (i % 4)));
      }
    }
  }
}

int scatter_grid(int T, int sms) {
  const int wpb = kScatterThreads / 32;
  int g = (T + wpb - 1) / wpb;
  const int cap = sms * 8;
  return g < 1 ? 1 : (g < cap ? g : cap);
}

}  // namespace

// Launches the permute kernels (the rank pass, then the scatter); shared by the
// workspace and the fixed-scratch entry points.
// xp_dtype MOE_E2M1 (x not null): NVFP4 rows; the first launch also takes the tensor
// amax of x into *amax_bits (zeroed by the caller), and the scatter writes the tensor
// scale to *tensor_scale.
moe_status_t permute_launch(const void* x, moe_dtype_t x_dtype, int T, int d,
                            const int32_t* topk_idx, int k, int E, const int32_t* counts,
                            int32_t* offsets, int32_t* dest_row, int32_t* src_pair, void* xp,
                            moe_dtype_t xp_dtype, uint8_t* xp_scales, int32_t* hist,
                            int32_t* dev_status, cudaStream_t stream, int sms,
                            uint32_t* amax_bits, float* tensor_scale) {
  const int nblk = (T + kTokensPerRankBlock - 1) / kTokensPerRankBlock;
  const size_t rank_smem = static_cast<size_t>(2) * 8 * E * sizeof(uint32_t);  // mask + base, [8][E] each
  // NVFP4 rows: the rank pass and the tensor amax of x (zeroed by the caller) share a launch
  const bool with_amax = xp_dtype == MOE_E2M1;
  const void* first = with_amax ? (x_dtype == MOE_BF16 ? reinterpret_cast<const void*>(permute_rank_amax_kernel<uint16_t>)
                                                        : reinterpret_cast<const void*>(permute_rank_amax_kernel<float>))
                                : reinterpret_cast<const void*>(permute_rank_kernel);
  if (rank_smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(first, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(rank_smem));
    if (e != cudaSuccess) {
      set_error("moe_permute: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
      return MOE_ERR_CUDA;
    }
  }
  if (with_amax) {
    const long long n16 = static_cast<long long>(T) * d * (x_dtype == MOE_BF16 ? 2 : 4) / 16;
    const long long g1 = (n16 + kRankThreads - 1) / kRankThreads;
    const int agrid = static_cast<int>(g1 < 1 ? 1 : (g1 < sms * 8 ? g1 : sms * 8));
    const uint8_t* xb = static_cast<const uint8_t*>(x);
    if (x_dtype == MOE_BF16)
      launch_pdl(permute_rank_amax_kernel<uint16_t>, nblk + agrid, kRankThreads, rank_smem, stream, topk_idx, T, k,
                 E, dest_row, hist, dev_status, nblk, xb, n16, amax_bits);
    else
      launch_pdl(permute_rank_amax_kernel<float>, nblk + agrid, kRankThreads, rank_smem, stream, topk_idx, T, k, E,
                 dest_row, hist, dev_status, nblk, xb, n16, amax_bits);
  } else if (nblk > 0) {
    launch_pdl(permute_rank_kernel, nblk, kRankThreads, rank_smem, stream, topk_idx, T, k, E, dest_row,
                                                                   hist, dev_status);
  }
  // the scatter also publishes offsets (so it runs even for T == 0)
  const int grid = scatter_grid(T, sms);
  const uint8_t* xb = static_cast<const uint8_t*>(x);
  uint8_t* xpb = static_cast<uint8_t*>(xp);
  // dest_row holds each pair's within-block rank until the scatter overwrites that
  // same element with the pair's final row (read and write by the same thread).
  if (xp_dtype == MOE_E2M1) {
    if (x_dtype == MOE_BF16)
      launch_pdl(permute_scatter_kernel<uint16_t, 2>, grid, kScatterThreads, 0, stream, xb, T, d, topk_idx, k, E,
                 counts, dest_row, hist, nblk, offsets, dest_row, src_pair, xpb, xp_scales, amax_bits, tensor_scale,
                 dev_status);
    else
      launch_pdl(permute_scatter_kernel<float, 2>, grid, kScatterThreads, 0, stream, xb, T, d, topk_idx, k, E,
                 counts, dest_row, hist, nblk, offsets, dest_row, src_pair, xpb, xp_scales, amax_bits, tensor_scale,
                 dev_status);
  } else if (xp_dtype == MOE_E4M3) {
    if (x_dtype == MOE_BF16)
      launch_pdl(permute_scatter_kernel<uint16_t, 1>, grid, kScatterThreads, 0, stream, 
          xb, T, d, topk_idx, k, E, counts, dest_row, hist, nblk, offsets, dest_row, src_pair, xpb, xp_scales,
          nullptr, nullptr, dev_status);
    else
      launch_pdl(permute_scatter_kernel<float, 1>, grid, kScatterThreads, 0, stream, 
          xb, T, d, topk_idx, k, E, counts, dest_row, hist, nblk, offsets, dest_row, src_pair, xpb, xp_scales,
          nullptr, nullptr, dev_status);
  } else if (x_dtype == MOE_BF16) {
    launch_pdl(permute_scatter_kernel<uint16_t, 0>, grid, kScatterThreads, 0, stream, 
        xb, T, d, topk_idx, k, E, counts, dest_row, hist, nblk, offsets, dest_row, src_pair, xpb, nullptr,
        nullptr, nullptr, dev_status);
  } else {
    launch_pdl(permute_scatter_kernel<float, 0>, grid, kScatterThreads, 0, stream, 
        xb, T, d, topk_idx, k, E, counts, dest_row, hist, nblk, offsets, dest_row, src_pair, xpb, nullptr,
        nullptr, nullptr, dev_status);
  }
  return check_launch("moe_permute");
}

moe_status_t permute_validate(const void* x, moe_dtype_t x_dtype, int T, int d,
                              const int32_t* topk_idx, int k, int E, const int32_t* counts,
                              int32_t* offsets, int32_t* dest_row, int32_t* src_pair, void* xp,
                              moe_dtype_t xp_dtype, uint8_t* xp_scales) {
  if (T < 0 || d < 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E) {
    set_error("moe_permute: need T, d >= 0, 1 <= E <= 1024, 1 <= k <= min(E, 32)");
    return MOE_ERR_INVALID_ARG;
  }
  if (static_cast<long long>(T) * k >= (1LL << 31)) {
    set_error("moe_permute: T*k must fit in int32");
    return MOE_ERR_INVALID_ARG;
  }
  if (!counts || !offsets || (T > 0 && (!topk_idx || !dest_row || !src_pair))) {
    set_error("moe_permute: null pointer");
    return MOE_ERR_INVALID_ARG;
  }
  if (xp) {
    if (!x || (x_dtype != MOE_BF16 && x_dtype != MOE_F32)) {
      set_error("moe_permute: x must be a BF16 or F32 device buffer");
      return MOE_ERR_INVALID_ARG;
    }
    if (xp_dtype != x_dtype && xp_dtype != MOE_E4M3) {
      set_error("moe_permute: xp_dtype must equal x_dtype or be MOE_E4M3");
      return MOE_ERR_INVALID_ARG;
    }
    if (d % 8 || !aligned16(x) || !aligned16(xp)) {
      set_error("moe_permute: d %% 8 == 0 and 16-byte aligned x / xp required");
      return MOE_ERR_INVALID_ARG;
    }
    if (xp_dtype == MOE_E4M3 && (d % 32 || !xp_scales)) {
      set_error("moe_permute: MXFP8 output needs d %% 32 == 0 and xp_scales");
      return MOE_ERR_INVALID_ARG;
    }
  }
  return MOE_OK;
}

size_t permute_hist_bytes(int T, int E) {
  const size_t nblk = (static_cast<size_t>(T > 0 ? T : 0) + kTokensPerRankBlock - 1) / kTokensPerRankBlock;
  return nblk * static_cast<size_t>(E > 0 ? E : 0) * sizeof(int32_t);
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_permute_workspace_size(int T, int k, int E) {
  (void)k;
  const size_t b = permute_hist_bytes(T, E);
  return b < 256 ? 256 : b;
}

extern "C" moe_status_t moe_permute(const void* x, moe_dtype_t x_dtype, int T, int d,
                                    const int32_t* topk_idx, int k, int E, const int32_t* counts,
                                    int32_t* offsets, int32_t* dest_row, int32_t* src_pair,
                                    void* xp, moe_dtype_t xp_dtype, uint8_t* xp_scales,
                                    void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                    cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_permute");
  moe_status_t st = permute_validate(x, x_dtype, T, d, topk_idx, k, E, counts, offsets, dest_row,
                                     src_pair, xp, xp_dtype, xp_scales);
  if (st != MOE_OK) return st;
  if (!workspace || workspace_bytes < permute_hist_bytes(T, E)) {
    set_error("moe_permute: workspace of %zu bytes needed", permute_hist_bytes(T, E));
    return MOE_ERR_WORKSPACE;
  }
  int sms = 0;
  if (const moe_status_t dst = device_check(&sms); dst != MOE_OK) return dst;
  return permute_launch(x, x_dtype, T, d, topk_idx, k, E, counts, offsets, dest_row, src_pair, xp,
                        xp_dtype, xp_scales, static_cast<int32_t*>(workspace), dev_status, stream,
                        sms, nullptr, nullptr);
}

namespace {
void colwise_launch(const void* in, moe_dtype_t in_dtype, int rows, int K, const int32_t* offsets, int E, int axis,
                    uint8_t* codes, uint8_t* scales, const int32_t* gather, const float* gweight, int gk,
                    int gpairs, int32_t* status, cudaStream_t stream, int sms) {
  const int strip = kColThreads * 4;
  const long long items = (static_cast<long long>(rows) / 32 + E) * ((K + strip - 1) / strip);
  // the gathered form takes its blocks slot by slot (see the kernel); its slot tables
  // take (slots + 1) * (E + 1) ints of dynamic shared memory
  const int slots = gather ? (E <= 512 ? 16 : 8) : 0;
  const size_t dyn = slots > 0 ? static_cast<size_t>(slots + 1) * (E + 1) * sizeof(int) : 0;
  const uint8_t* src = static_cast<const uint8_t*>(in);
  auto go = [&](auto kern) {
    // as many CTAs as stay resident (they walk the work in a grid-stride loop)
    int per_sm = 8;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kColThreads, dyn) != cudaSuccess || per_sm < 1)
      per_sm = 1;
    per_sm = per_sm < 8 ? per_sm : 8;
    const long long cap = static_cast<long long>(sms) * per_sm;
    const int grid = static_cast<int>(items < cap ? (items > 0 ? items : 1) : cap);
    launch_pdl(kern, grid, kColThreads, dyn, stream, src, rows, K, offsets, E, codes, scales, gather, gweight, gk,
               gpairs, status, slots);
  };
  if (in_dtype == MOE_BF16) {
    if (axis == 2) go(quantize_colwise_kernel<uint16_t, true>);
    else go(quantize_colwise_kernel<uint16_t, false>);
  } else {
    if (axis == 2) go(quantize_colwise_kernel<float, true>);
    else go(quantize_colwise_kernel<float, false>);
  }
}
}  // namespace

extern "C" moe_status_t moe_quantize_mxfp8_gathered(const void* x, moe_dtype_t x_dtype, int T, int K, int k,
                                                    const int32_t* src_pair, const float* row_w,
                                                    const int32_t* offsets, int E,
                                                    int axis, uint8_t* codes, uint8_t* scales,
                                                    int32_t* dev_status, cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_quantize_mxfp8_gathered");
  const char* fn = "moe_quantize_mxfp8_gathered";
  if (axis != 1 && axis != 2) {
    set_error("%s: axis 1 (column-wise) or 2 (column-wise, tiled scales)", fn);
    return MOE_ERR_UNSUPPORTED;
  }
  if (T < 0 || K < 0 || K % 32 || k < 1 || k > 32 || !offsets || E < 1 || E > 1024 ||
      (axis == 2 && K % 128) || (x_dtype != MOE_BF16 && x_dtype != MOE_F32)) {
    set_error("%s: need T, K >= 0, K %% 32 == 0 (axis 2: %% 128), 1 <= k <= 32, offsets, 1 <= E <= 1024, "
              "BF16/F32 rows", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (static_cast<long long>(T) * k >= (1LL << 31)) {
    set_error("%s: T*k must fit in int32", fn);
    return MOE_ERR_INVALID_ARG;
  }
  const int rows = T * k;
  if (rows > 0 && K > 0 && (!x || !src_pair || !codes || !scales || !aligned16(x) || !aligned16(codes))) {
    set_error("%s: null or misaligned pointer", fn);
    return MOE_ERR_INVALID_ARG;
  }
  int sms = 0;
  if (const moe_status_t dst = device_check(&sms); dst != MOE_OK) return dst;
  if (rows == 0 || K == 0) return MOE_OK;
  colwise_launch(x, x_dtype, rows, K, offsets, E, axis, codes, scales, src_pair, row_w, k, rows, dev_status, stream,
                 sms);
  return check_launch(fn);
}

extern "C" moe_status_t moe_quantize_mxfp8_grouped(const void* in, moe_dtype_t in_dtype, int rows,
                                                   int K, const int32_t* offsets, int E, int axis,
                                                   uint8_t* codes, uint8_t* scales,
                                                   cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_quantize_mxfp8_grouped");
  if (axis != 0 && axis != 1 && axis != 2) {
    set_error("moe_quantize_mxfp8_grouped: axis 0 (row-wise), 1 (column-wise) or 2 (column-wise, tiled scales)");
    return MOE_ERR_UNSUPPORTED;
  }
  if (axis >= 1 && (!offsets || E < 1 || E > 1024)) {
    set_error("moe_quantize_mxfp8_grouped: column-wise needs offsets and 1 <= E <= 1024");
    return MOE_ERR_INVALID_ARG;
  }
  if (axis == 2 && K % 128) {
    set_error("moe_quantize_mxfp8_grouped: tiled column-wise scales need K %% 128 == 0");
    return MOE_ERR_INVALID_ARG;
  }
  if (rows < 0 || K < 0 || K % 32 || (in_dtype != MOE_BF16 && in_dtype != MOE_F32)) {
    set_error("moe_quantize_mxfp8_grouped: need rows >= 0, K %% 32 == 0, BF16/F32 input");
    return MOE_ERR_INVALID_ARG;
  }
  if (rows > 0 && K > 0 && (!in || !codes || !scales || !aligned16(in) || !aligned16(codes))) {
    set_error("moe_quantize_mxfp8_grouped: null or misaligned pointer");
    return MOE_ERR_INVALID_ARG;
  }
  int sms = 0;
  if (const moe_status_t dst = device_check(&sms); dst != MOE_OK) return dst;
  if (rows == 0 || K == 0) return MOE_OK;
  if (axis >= 1) {
    colwise_launch(in, in_dtype, rows, K, offsets, E, axis, codes, scales, nullptr, nullptr, 1, 0, nullptr, stream,
                   sms);
    return check_launch("moe_quantize_mxfp8_grouped");
  }
  const int grid = scatter_grid(rows, sms);
  if (in_dtype == MOE_BF16)
    launch_pdl(quantize_rowwise_kernel<uint16_t>, grid, kScatterThreads, 0, stream, 
        static_cast<const uint8_t*>(in), rows, K, codes, scales);
  else
    launch_pdl(quantize_rowwise_kernel<float>, grid, kScatterThreads, 0, stream, 
        static_cast<const uint8_t*>(in), rows, K, codes, scales);
  return check_launch("moe_quantize_mxfp8_grouped");
}

extern "C" moe_status_t moe_quantize_mxfp8_transposed(const void* in, moe_dtype_t in_dtype, int G, int R,
                                                      int C, uint8_t* codes, uint8_t* scales,
                                                      cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_quantize_mxfp8_transposed");
  if (G < 0 || R < 0 || C < 0 || R % 32 || C % 8 || (in_dtype != MOE_BF16 && in_dtype != MOE_F32)) {
    set_error("moe_quantize_mxfp8_transposed: need G, R, C >= 0, R %% 32 == 0, C %% 8 == 0, BF16/F32 input");
    return MOE_ERR_INVALID_ARG;
  }
  if (G > 0 && R > 0 && C > 0 && (!in || !codes || !scales || !aligned16(in) || !aligned16(codes))) {
    set_error("moe_quantize_mxfp8_transposed: null or misaligned pointer");
    return MOE_ERR_INVALID_ARG;
  }
  int sms = 0;
  if (const moe_status_t dst = device_check(&sms); dst != MOE_OK) return dst;
  if (G == 0 || R == 0 || C == 0) return MOE_OK;
  if (in_dtype == MOE_BF16) {
    const long long items = static_cast<long long>(G) * ((R / 32 + kTrRb - 1) / kTrRb) *
                            ((C + tr_cols<uint16_t>() - 1) / tr_cols<uint16_t>());
    const int grid = static_cast<int>(items < static_cast<long long>(sms) * 4 ? items : sms * 4);
    launch_pdl(quantize_transposed_kernel<uint16_t>, grid, tr_cols<uint16_t>(), 0, stream,
               static_cast<const uint8_t*>(in), G, R, C, codes, scales);
  } else {
    const long long items = static_cast<long long>(G) * ((R / 32 + kTrRb - 1) / kTrRb) *
                            ((C + tr_cols<float>() - 1) / tr_cols<float>());
    const int grid = static_cast<int>(items < static_cast<long long>(sms) * 6 ? items : sms * 6);
    launch_pdl(quantize_transposed_kernel<float>, grid, tr_cols<float>(), 0, stream,
               static_cast<const uint8_t*>(in), G, R, C, codes, scales);
  }
  return check_launch("moe_quantize_mxfp8_transposed");
}

extern "C" moe_status_t moe_permute_nvfp4(const void* x, moe_dtype_t x_dtype, int T, int d,
                                          const int32_t* topk_idx, int k, int E, const int32_t* counts,
                                          int32_t* offsets, int32_t* dest_row, int32_t* src_pair,
                                          uint8_t* xp_codes, uint8_t* xp_scales, float* tensor_scale,
                                          void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                          cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_permute_nvfp4");
  const char* fn = "moe_permute_nvfp4";
  if (T < 0 || d < 0 || d % 16 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E ||
      (x_dtype != MOE_BF16 && x_dtype != MOE_F32) || static_cast<long long>(T) * k >= (1LL << 31)) {
    set_error("%s: need T, d >= 0, d %% 16 == 0, 1 <= E <= 1024, 1 <= k <= min(E, 32), BF16/F32 x", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (!counts || !offsets || !tensor_scale || (T > 0 && (!x || !topk_idx || !dest_row || !src_pair ||
                                                        (d > 0 && (!xp_codes || !xp_scales)))) ||
      !aligned16(x) || (reinterpret_cast<uintptr_t>(xp_codes) & 3) || (reinterpret_cast<uintptr_t>(tensor_scale) & 3)) {
    set_error("%s: null or misaligned pointer", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (!workspace || workspace_bytes < permute_hist_bytes(T, E)) {
    set_error("%s: workspace of %zu bytes needed", fn, permute_hist_bytes(T, E));
    return MOE_ERR_WORKSPACE;
  }
  int sms = 0;
  if (const moe_status_t dst = device_check(&sms); dst != MOE_OK) return dst;
  uint32_t* amax_bits = reinterpret_cast<uint32_t*>(tensor_scale + 1);
  cudaError_t e = cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) {
    set_error("%s: cudaMemsetAsync: %s", fn, cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  // the amax of x is the amax of the permuted rows (every token is routed); the
  // first of the dispatch's two launches takes it beside the rank pass
  return permute_launch(x, x_dtype, T, d, topk_idx, k, E, counts, offsets, dest_row, src_pair, xp_codes,
                        MOE_E2M1, xp_scales, static_cast<int32_t*>(workspace), dev_status, stream, sms,
                        amax_bits, tensor_scale);
}

// Shared device helpers for libmoe (sm_103a): error bits, bounded waits and thin
// inline-PTX wrappers for mbarrier, TMA and tcgen05 (written from the public PTX
// ISA description of each instruction).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// ----------------------------------------------------------------------------- host helpers

void set_error(const char* fmt, ...);
moe_status_t check_launch(const char* what);

// An NVTX range named after the C entry point, for the span of the call (the
// host-side work and the launches it enqueues show up under that name in a
// timeline tool; with no tool attached the push and pop do nothing).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// MOE_OK on an sm_103 device (and its SM count), MOE_ERR_UNSUPPORTED on another
// architecture, MOE_ERR_CUDA when the runtime cannot be queried.
moe_status_t device_check(int* sm_count);
bool aligned16(const void* p);

// ----------------------------------------------------------------------------- device basics

__device__ __forceinline__ void flag_error(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

// Device-side invariant check of a MOE_DEBUG build: a failed condition ORs
// MOE_DEV_ASSERT into the status word (never a trap) and the result lets the caller
// skip the access it guards.  In a release build it is `true` and costs nothing.
#ifdef MOE_DEBUG
__device__ __forceinline__ bool dbg_check(bool cond, int32_t* status) {
  if (!cond) flag_error(status, MOE_DEV_ASSERT);
  return cond;
}
#else
__device__ __forceinline__ constexpr bool dbg_check(bool, int32_t*) { return true; }
#endif

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Any single pipeline wait longer than this is a broken invariant, not a slow GPU.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// Round-to-nearest-even float -> bf16 bits (hardware conversion).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Two floats -> two bf16 (lo in bits 0..15), round-to-nearest-even, in one packed
// conversion instruction: the same bits as two single conversions, at several times
// their throughput (the GEMM epilogues that drain an accumulator are bound by it).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two floats -> two E4M3 bytes (lo in bits 0..7), round-to-nearest-even with
// saturation to the largest finite value.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight floats -> eight E2M1 codes packed in 32 bits (element i in bits 4i..4i+3),
// round-to-nearest-even with saturation to +-6.  The cvt puts its first source in
// the high nibble.
__device__ __forceinline__ uint32_t f32x8_to_e2m1x8(const float (&v)[8]) {
  uint32_t r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// Value of a non-negative E4M3 byte (sign bit clear, not NaN) from its bit fields:
// exponent field 0 -> man * 2^-9, else (8 + man) * 2^(exp - 10).  Exact.
__device__ __forceinline__ float ue4m3_value(uint32_t code) {
  const uint32_t exp = (code >> 3) & 0xFu, man = code & 0x7u;
  if (exp == 0) return static_cast<float>(man) * 0.001953125f;
  return __uint_as_float(((exp + 120u) << 23) | (man << 20));
}

// NVFP4 scaling of one 16-element block with block amax `amax` in a tensor whose
// encode scale is g: the E4M3 scale byte s = E4M3_rn_sat((amax / 6) * g) and the
// multiplier g / s (0 when s decodes to 0), every step one fp32 rounding.
__device__ __forceinline__ float nvfp4_tensor_scale(float amax_t) { return amax_t == 0.f ? 1.f : 2688.f / amax_t; }
__device__ __forceinline__ uint32_t nvfp4_block_code(float amax, float g) {
  return f32x2_to_e4m3x2(__fmul_rn(__fdiv_rn(amax, 6.f), g), 0.f) & 0xFFu;
}
// The multiplier of a block whose scale byte is `code`: g / value(code), 0 for a zero scale.
__device__ __forceinline__ float nvfp4_block_inv(uint32_t code, float g) {
  const float sval = ue4m3_value(code);
  return sval == 0.f ? 0.f : __fdiv_rn(g, sval);
}
__device__ __forceinline__ void nvfp4_block_scale(float amax, float g, uint32_t* scode, float* inv) {
  *scode = nvfp4_block_code(amax, g);
  *inv = nvfp4_block_inv(*scode, g);
}

// Tensor amax of a bf16 (Tin = uint16_t) or fp32 array of n16 16-byte chunks, the part
// of block blk of nblocks (blockDim.x threads each), merged into *amax_bits (the fp32
// bits of a non-negative value, so an integer max orders them): four chunks in flight
// per thread.  Every thread of the block calls it.
template <typename Tin>
__device__ __forceinline__ void nvfp4_amax_body(const uint8_t* __restrict__ in, long long n16, uint32_t* amax_bits,
                                                long long blk, long long nblocks) {
  float m = 0.f;
  const uint4* v4 = reinterpret_cast<const uint4*>(in);
  const long long stride = nblocks * blockDim.x;
  for (long long i = blk * blockDim.x + threadIdx.x; i < n16; i += 4 * stride) {
    uint4 u[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) u[q] = i + q * stride < n16 ? v4[i + q * stride] : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t w[4] = {u[q].x, u[q].y, u[q].z, u[q].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if constexpr (sizeof(Tin) == 2) {
          m = fmaxf(m, fabsf(bf16_to_f32(static_cast<uint16_t>(w[j] & 0xFFFFu))));
          m = fmaxf(m, fabsf(bf16_to_f32(static_cast<uint16_t>(w[j] >> 16))));
        } else {
          m = fmaxf(m, fabsf(__uint_as_float(w[j])));
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  __shared__ float part[32];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < static_cast<int>(blockDim.x >> 5); ++i) m = fmaxf(m, part[i]);
    atomicMax(amax_bits, __float_as_uint(m));
  }
}

// MXFP8 shared-exponent rule (OCP Microscaling Formats v1.0): X = floor(log2 amax)
// - 8 (8 = E4M3's largest exponent), clamped at -127, stored as the E8M0 byte
// X + 127; an all-zero block gets byte 127.  Returns the byte and the exact power
// of two 2^-X to multiply the block by before the E4M3 conversion.
__device__ __forceinline__ void mx_scale(float amax, uint32_t* sbyte, float* inv) {
  if (amax == 0.f) {
    *sbyte = 127u;
    *inv = 1.f;
    return;
  }
  const int eb = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);  // biased exponent
  const int s = eb - 8 > 0 ? eb - 8 : 0;                                     // X + 127
  *sbyte = static_cast<uint32_t>(s);
  *inv = __uint_as_float(static_cast<uint32_t>(254 - s) << 23);              // 2^(127 - s)
}

// ----------------------------------------------------------------------------- dependent launch

// Every kernel of the library starts with pdl_begin(): wait until the preceding
// kernel in the stream has completed and its writes are visible (a no-op when the
// launch carried no programmatic dependency), then allow the next kernel to be
// scheduled, so its launch and prologue overlap this kernel instead of following
// it.  The next kernel still waits for this one to complete before reading
// anything it wrote.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with a programmatic stream dependency on the preceding kernel, in thread-
// block clusters of `cluster` CTAs along x when cluster > 1 (grid.x a multiple of it).
template <typename... KArgs, typename... Args>
inline void launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                               int cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  (void)cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Launch with a programmatic stream dependency on the preceding kernel.
template <typename... KArgs, typename... Args>
inline void launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  launch_pdl_cluster(kern, grid, block, smem, stream, 1, static_cast<Args&&>(args)...);
}

// ----------------------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete.  Gives up after
// kWaitLimitNs, flags MOE_DEV_TIMEOUT and sets *abort so the other roles of the
// block stop too; returns false in that case.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* status,
                                          volatile int* abort, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++n & 255u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        flag_error(status, MOE_DEV_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
  return true;
}

// ----------------------------------------------------------------------------- clusters
// Distributed shared memory between the CTAs of a thread-block cluster: an address
// of this CTA's shared memory mapped into a peer's window, plain loads and stores
// through it, and mbarrier arrivals on a peer's barrier (release at cluster scope,
// paired with the acquire-at-cluster-scope wait below).

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %cluster_ctarank;" : "=r"(r));
  return r;
}

// The address of `saddr` (this CTA's shared window) in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t caddr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(caddr)
               : "memory");
  return v;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t caddr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(caddr), "r"(v) : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t caddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}

__device__ __forceinline__ void fence_acq_rel_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }

// Every thread of every CTA of the cluster: the barrier initialisations of each CTA
// are visible to the others before any of them arrives remotely.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// A wait for arrivals from the peers of the cluster: gives up after limit_ns and
// flags MOE_DEV_TIMEOUT, but is not cut short by this CTA's own abort flag (a CTA
// whose pipeline gave up still completes its exchanges with its peers, so none of
// them accesses its shared memory after it has exited).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, int32_t* status,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (!mbar_try_wait_cluster(bar, parity)) {
    if ((++n & 255u) == 0 && globaltimer_ns() - t0 > limit_ns) {
      flag_error(status, MOE_DEV_TIMEOUT);
      return false;
    }
  }
  return true;
}

// ----------------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Untiled global -> shared bulk copy completing on an mbarrier (16-byte aligned
// addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Shared -> global tiled store through the tensor map (bulk async group of this
// thread); out-of-range parts of the box are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Shared -> global tiled reduction: each element of the box is added to the one in
// global memory (in the tensor map's element type), out-of-range parts untouched.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, const void* src, int x, int y,
                                                  int z) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// L2 policy for data written once and not read again by this kernel: its lines are
// the first to be evicted, so streaming output does not push operands out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void st_global_hint(void* dst, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(dst), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Allow at most N of this thread's committed bulk store groups to be still
// reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until this thread's committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until this thread's committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ----------------------------------------------------------------------------- tcgen05

// Shared-memory matrix descriptor (tcgen05 "matrix descriptor"): start address,
// leading / stride byte offsets (all >> 4), the fixed version bits 46..48 = 0b001
// and the swizzle mode in bits 61..63 (2 = 128-byte swizzle, 0 = none).
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                               uint32_t swizzle) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(swizzle & 7u) << 61;
  return d;
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

template <int kKind>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate);

// kind 0: tf32 x tf32 -> f32
template <>
__device__ __forceinline__ void tc_mma<0>(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// kind 1: bf16 x bf16 -> f32
template <>
__device__ __forceinline__ void tc_mma<1>(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Block-scaled E4M3 x E4M3 -> f32 with E8M0 scale vectors read from tensor memory.
__device__ __forceinline__ void tc_mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// NVFP4 block-scaled MMA: E2M1 operands (K = 64 per instruction), four E4M3 scale
// bytes per row per instruction (one per 16 elements).
__device__ __forceinline__ void tc_mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Copy 128 rows x 16 bytes from shared memory (no-swizzle descriptor) into 128
// TMEM lanes x 4 columns.
__device__ __forceinline__ void tc_cp_128x128b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x128b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Copy 32 rows x 16 bytes from shared memory (no-swizzle descriptor) into TMEM
// lanes 0-31 x 4 columns, replicated into all four 32-lane quarters.  With the
// 512-byte scale-factor atom (byte (m % 32) * 16 + (m / 32) * 4 + kb for row m of
// 128 and scale block kb of 4) this is the layout block-scaled MMAs read.
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Each thread of the warp reads 32 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace moe

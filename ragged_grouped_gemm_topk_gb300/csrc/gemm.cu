// Ragged grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA):
// forward, data gradient and weight gradient.
//
// "Accelerating Dropless MoE Training in JAX with NVIDIA Transformer Engine",
// "Optimisation 1: grouped GEMM": one launch covers every expert's matmul, each
// computed at its own (data-dependent) token count, with no device-to-host copy
// of the counts and no padding to a worst-case capacity.
//
// One persistent CTA per SM, 6 warps:
//   warp 0     TMA producer: streams the A and B slices of the current tile into a
//              4-stage shared-memory ring (48 KB per stage, 128-byte swizzle).
//   warp 1     allocates TMEM; one lane issues tcgen05.mma (M=128, N=256, K=16 per
//              instruction) into a double-buffered fp32 accumulator in TMEM and
//              commits each stage back to the producer and each tile to the epilogue.
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (TMEM lane = tile row, one
//              row per thread), the fused epilogue, release of the accumulator,
//              then the stores: forward bf16 output and the plain data gradient by
//              TMA store from a per-warp shared staging box (a warp whose rows cross
//              the group's end stores its valid rows directly), wgrad likewise per
//              dW box, other outputs by 16-byte stores masked at the group's end and
//              the edge.
// Tiles are enumerated on the device from `offsets`, so the host never learns the
// per-expert sizes:
//   forward / dgrad  expert e owns ceil(count_e / 128) row tiles x the column
//                    tiles, taken in blocks of row tiles that fit L2 (all column
//                    tiles of a block, row tiles fastest), so neighbouring CTAs
//                    share a weight slice and each activation row is read from
//                    DRAM about once.  Rows of the last row tile past the
//                    group's end are computed but never stored.
//   wgrad            every expert owns ceil(N/128) x ceil(K/256) tiles of dB[e]
//                    (experts largest first, so the equal tiles of a big expert
//                    run in step on every SM and share its rows in L2);
//                    the contraction runs over the group's own rows in 64-row
//                    blocks; rows of the last block past the group's end are
//                    zeroed in shared memory (and whole 16-row MMA steps beyond it
//                    skipped), and an empty group writes exact zeros.
// Operand majors: forward A and B, and dgrad A, are K-major; dgrad B (the weight
// read along its output dim) and both wgrad operands are MN-major.  MN-major
// tiles arrive as 64-column x 64-row TMA boxes (128 B rows, 128-byte swizzle);
// their descriptors step 8 KB between 64-column chunks (leading byte offset) and
// 1 KB between 8-row groups (stride byte offset).
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "common.cuh"

namespace moe {
namespace gemm {

constexpr int kBM = 128;
constexpr int kBN = 256;                          // MMA N
constexpr int kBKBytes = 128;                     // K-major: one swizzle atom of K per stage
constexpr int kMnRows = 64;                       // MN-major: contraction rows per stage
constexpr int kStages = 4;
constexpr int kAStage = kBM * kBKBytes;           // 16 KB
constexpr int kBStage = kBN * kBKBytes;           // 32 KB
constexpr int kStageBytes = kAStage + kBStage;    // 48 KB
constexpr int kBox = 8192;                        // one 64 x 64 bf16 MN-major box
constexpr int kSfAStage = 2048;                   // MXFP8: raw A scale rows, 128 x 16 bytes
constexpr int kSfBStage = 4096;                   // MXFP8: raw B scale rows, 256 x 16 bytes
constexpr int kSfSlot = kSfAStage + kSfBStage;    // one raw scale slot (4 K-blocks' worth)
constexpr int kAtomBytes = 1536;                  // MXFP8 per-stage atoms: A 512 B, B 2 x 512 B
// Forward kernels' extra shared memory (after the operand stages): epilogue staging
// boxes (two per epilogue warp, one for MXFP8; 32 rows x 64 bytes: 32 bf16 or 64
// E4M3 columns; 1 KB aligned for the 64-byte swizzle), then for MXFP8 the scale
// atoms of every stage and the two raw scale-row slots.  64-byte boxes measured
// faster than 128-byte ones for bf16 too (and MXFP8 has room for no more).
constexpr int kEpiRowBytes = 64;
constexpr int kEpiBox = 32 * kEpiRowBytes;
constexpr int kEpiOff = 0;
// staging boxes per epilogue warp (rotating: a box is staged while the previous
// ones are still being read by their TMA stores) and raw scale-row slots (MXFP8)
template <int kKind>
constexpr int epi_bufs() { return kKind == 2 ? 1 : (kKind == 3 ? 0 : 2); }
// NVFP4 (kind 3): each stage's raw E4M3 scale rows (A 128 x 16 B, B 256 x 16 B) land
// next to the stage and are re-laid in place into its twelve 512-byte atoms (A: one
// per 64-element MMA; B: two per MMA, rows 0-127 and 128-255).  No staging boxes:
// the epilogue stores directly, so the four 48 KB stages still fit.
constexpr int kNvAtomBytes = 6144;
template <int kKind>
constexpr int raw_slots() { return 2; }
template <int kKind>
constexpr int atom_off() { return kEpiOff + 4 * epi_bufs<kKind>() * kEpiBox; }
template <int kKind>
constexpr int raw_off() { return atom_off<kKind>() + kStages * kAtomBytes; }
constexpr int kTmemCols = 512;
constexpr int kMaxE = 1024;

enum { kFwd = 0, kDgrad = 1, kWgrad = 2 };
enum { kEpiNone = 0, kEpiSwiglu = 1, kEpiDswiglu = 2, kEpiTopk = 3 };
constexpr int kTopkMax = 8;                       // router epilogue: experts per token
constexpr int kMaxSplit = 4;                      // router: CTAs of a cluster sharing one tile
constexpr int kMinSliceBlocks = 8;                // router: K blocks of a contraction slice, at least

// Instruction descriptor (kind::f16 / kind::tf32): D = f32 (bit 4), A/B format
// (bits 7-9 / 10-12: 1 = bf16, 2 = tf32), A/B major (bits 15 / 16: 1 = MN-major),
// N >> 3 at bit 17, M >> 4 at bit 24.
template <int kKind>
__host__ __device__ constexpr uint32_t make_idesc(int m, int n, int a_mn, int b_mn) {
  return (1u << 4) | (static_cast<uint32_t>(kKind == 0 ? 2 : 1) << 7) |
         (static_cast<uint32_t>(kKind == 0 ? 2 : 1) << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

struct Smem {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t sfready[kStages];
  uint64_t sfull[2];       // MXFP8 raw scale slots loaded
  uint64_t sempty[2];      // MXFP8 raw scale slots read into registers
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t xready;         // router split over a cluster: every peer's partial logits are staged
  uint64_t xdone;          //   every peer has finished reading this CTA's partial logits
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int nnz;                 // wgrad: experts with rows
  int epi_ok;              // router: the accumulator is ready (else the pipeline gave up)
  int x_ok;                // router split: every CTA of the cluster staged its partial
  int peer_ok[kMaxSplit];  // router split: written by each peer before it arrives on xready
  int prefix[kMaxE + 1];   // fwd/dgrad: tile prefix; wgrad: expert ids, non-empty then empty
};

// Per-kind configuration.  kind 0 = tf32, 1 = bf16: 6 warps.  kind 2 = MXFP8: a
// 7th warp lays the E8M0 scales of each stage out as 512-byte scale atoms, which
// are copied to TMEM scale slots (see Tl for the TMEM layout).
template <int kKind>
struct Cfg {
  static constexpr bool kMx = kKind >= 2;     // block-scaled (2 = MXFP8, 3 = NVFP4)
  static constexpr int kStage = kStageBytes;
  static constexpr int kEb = kKind == 0 ? 4 : (kKind == 1 ? 2 : 1);
};

// Wide tiles (bf16 operands, bf16 output, plain epilogue: GEMM2, the GEMM1 data
// gradient, the weight gradients): 256 rows x 256 columns, computed as two M=128 MMAs that share each
// stage's B slice, their accumulators in TMEM columns 0-255 and 256-511.  Per
// FLOP each SM then takes in a third fewer operand bytes, and each 64 KB stage
// carries twice the MMA work, so three stages cover more load latency than four
// 48 KB stages of 128-row tiles.  Eight epilogue warps (two per TMEM lane
// quarter, one set per 128-row half) drain the two accumulators side by side.
// A group's last tile computes its second half only if it has rows there, so no
// more rows are padded than with 128-row tiles.  GEMM1 (SwiGLU, with the pre-
// activation store that holds the accumulator while it writes) keeps 128-row tiles
// and its double-buffered accumulator: measured no faster wide on the DeepSeek-V3
// training layer and 6% slower on a smaller one.
template <int kKind, int kMode, int kEpi, int kOutBytes>
constexpr bool wide_tile() {
  return kKind == 1 && kOutBytes == 2 && kEpi == kEpiNone;
}
constexpr int kWideM = 256;
constexpr int kWideStages = 3;
constexpr int kWideStage = kWideM * kBKBytes + kBStage;      // 64 KB
constexpr int kWideEpiWarps = 8;
// first epilogue warp: after the producer and the MMA warp, and for the weight
// gradient the zero-fill warp (warp 2)
template <int kMode>
constexpr int wide_epi_warp0() { return kMode == kWgrad ? 3 : 2; }

// wgrad: each epilogue warp stages its 32 dW rows in wg_bufs rotating 2 KB boxes of
// 32 columns for the TMA store (so the 4-stage operand ring still fits), and a 7th
// warp writes the dW of experts without rows.  MXFP8 wgrad keeps two boxes per warp
// to make room for each stage's 1.5 KB of scale atoms, which arrive ready-made (the
// tiled column-wise scale layout) by bulk copy with the stage's operands.  Forward:
// each epilogue warp stages one 32-row x 32-column bf16 box (2 KB) of its output
// for the TMA store.
template <int kKind>
constexpr int wg_bufs() { return kKind == 2 ? 2 : 3; }   // 2 KB staging boxes per epilogue warp
template <int kKind>
constexpr int wg_stage() { return 2048 * wg_bufs<kKind>(); }
template <int kKind>
constexpr int wg_atom_off() { return 4 * wg_stage<kKind>(); }
constexpr int kMxWgRows = 128;                    // MXFP8 wgrad: contraction rows per stage (4 blocks)
template <int kKind, int kMode, bool kW = false>
constexpr int stages_for() { return kW ? kWideStages : kStages; }
template <int kKind, int kMode, bool kW = false>
constexpr int threads_for() {
  return kW ? 32 * (wide_epi_warp0<kMode>() + kWideEpiWarps) : ((kKind >= 2 || kMode == kWgrad) ? 224 : 192);
}
// Router (top-k epilogue): 16 warps, so that 14 epilogue warps share the selection
// (the 4 of a 128-row tile's lane quarters stage the logits from TMEM).
constexpr int kRouterWarps = 16;
template <int kKind, int kMode, int kEpi, int kOutBytes>
constexpr int block_threads() {
  return kEpi == kEpiTopk ? 32 * kRouterWarps
                          : threads_for<kKind, kMode, wide_tile<kKind, kMode, kEpi, kOutBytes>()>();
}
template <bool kW>
constexpr int stage_bytes() { return kW ? kWideStage : kStageBytes; }
// wide tiles: one 2 KB staging box per epilogue warp (forward and weight gradient)
template <int kKind, int kMode, bool kW = false>
constexpr size_t extra_smem() {
  return kW ? kWideEpiWarps * kEpiBox
            : kMode == kWgrad ? wg_atom_off<kKind>() + (kKind == 2 ? kStages * kAtomBytes : 0)
                              : (kMode == kFwd ? (kKind == 3 ? kStages * kNvAtomBytes
                                                             : kKind == 2 ? raw_off<kKind>() + raw_slots<kKind>() * kSfSlot
                                                             : atom_off<kKind>())
                                               : 0);
}
template <int kKind, int kMode, bool kW = false>
constexpr size_t smem_for() {
  return 1024 + static_cast<size_t>(stages_for<kKind, kMode, kW>()) * stage_bytes<kW>() +
         extra_smem<kKind, kMode, kW>() + sizeof(Smem);
}

// Tile shape and TMEM layout per instantiation: 128 x 256 tiles everywhere.
// tf32 / bf16 double-buffer the accumulator (2 x 256 TMEM columns).  MXFP8 keeps
// one accumulator (columns 0-255) so that columns 256-383 can hold one 32-column
// scale slot per pipeline stage (A scales at +0, B scales at +16).
template <int kKind, int kMode, int kEpi>
struct Tl {
  static constexpr int BN = kBN;
  static constexpr int kAcc = kKind >= 2 ? 1 : 2;   // block-scaled: columns 256-511 hold the scales
  static constexpr uint32_t kSfBase = 256u;
  static constexpr uint32_t kSfStride = 32u;
  static constexpr uint32_t kSfB = 16u;
};

// Block-scaled instruction descriptor (kind::mxf8f6f4): E4M3 A and B (format 0),
// K-major, N >> 3 at bit 17, E8M0 scales (bit 23), M >> 4 at bit 24; the scale
// byte of each k-step is selected by the A / B scale ids (bits 29-30 / 4-5).
__host__ __device__ constexpr uint32_t make_idesc_mx(int m, int n) {
  return (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(m >> 4) << 24);
}

// Block-scaled instruction descriptor (kind::mxf4nvf4): E2M1 A and B (format 1),
// K-major, N >> 3 at bit 17, E4M3 scales (bit 23 clear), M >> 4 at bit 24; with
// 16-element blocks each MMA (K = 64) reads four scale bytes per row, so no scale ids.
__host__ __device__ constexpr uint32_t make_idesc_nvf4(int m, int n) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

struct Params {
  const int32_t* offsets;
  int M, N, K, E;
  void* out;               // C / dA / dB
  void* preact_out;        // forward SwiGLU: G|U store (may be null)
  const void* preact_in;   // dgrad dSwiGLU: G|U input
  uint8_t* out_scales;     // forward with MXFP8 output: E8M0 [M, n_out / 32]
  int32_t* status;
  const uint8_t* sfa;      // MXFP8 wgrad: tiled column-wise scales of dC (the MMA's A) ...
  const uint8_t* sfb;      // ... and of A (the MMA's B)
  const float* ts_a;       // NVFP4: tensor encode scales of A and B (the product is
  const float* ts_b;       //   multiplied by 1 / (g_A * g_B))
  int32_t* topk_idx;       // router epilogue: [M, k] selected experts,
  float* topk_w;           //   [M, k] their weights,
  int32_t* counts;         //   [N] tokens per expert (zeroed by the host entry)
  int k_sel;               //   experts per token (<= kTopkMax)
  int renorm;              //   softmax over the selected logits (1) or over all (0)
  int n_mma;               //   MMA width: E rounded up to 16 (the B tile holds that many rows)
  int split;               //   CTAs (one cluster) sharing a tile's contraction: 1, 2 or 4
  int accumulate;          // wgrad, fp32 dB: add to dB (TMA reductions) instead of writing it
};

// Rows of group e.  Without an offsets array the problem is one dense group of M rows.
__device__ __forceinline__ void group_range(const Params& p, int e, int& beg, int& end) {
  if (p.offsets == nullptr) {
    beg = 0;
    end = p.M;
  } else {
    beg = __ldg(p.offsets + e);
    end = __ldg(p.offsets + e + 1);
  }
}

struct Tile {
  int e;
  int row0;    // fwd/dgrad: first row; wgrad: first row of the group
  int rows;    // fwd/dgrad: valid rows (<= the tile rows); wgrad: rows of the group
  int col0;    // first output column (fwd/dgrad) / first dB column (wgrad)
  int n0;      // wgrad: first dB row
  int kblocks; // contraction blocks
  int kb0;     // first contraction block (the router's slice of a split contraction)
};

__device__ __forceinline__ bool group_ok(int beg, int end, int M) { return beg >= 0 && end >= beg && end <= M; }

// Forward / dgrad raster: an expert's tiles are taken in blocks of `rb` row tiles,
// all column tiles of a block before the next block, row tiles fastest inside it.
// rb is chosen so that a block's A rows (rb x 128 rows of the contraction) take about
// this many bytes: they stay in L2 while every column tile of the block reads them,
// so each A row comes from DRAM about once instead of once per column tile (the hot
// experts of a skewed layer hold far more rows than L2), and the block's column
// slices of B, read by its rb row tiles, stay in L2 as well.
constexpr long long kRasterABytes = 32ll << 20;

template <int kMode, int kEpi>
struct Geo {
  int nt;       // column tiles per row tile (fwd/dgrad); dB row tiles (wgrad)
  int nt2;      // wgrad: dB column tiles
  int n_out;    // output columns (fwd/dgrad)
  int bn_out;   // output columns per tile
  int kb_fixed; // contraction blocks (fwd/dgrad)
  int mn_rows;  // wgrad: contraction rows per stage
  int rb;       // fwd/dgrad: row tiles per raster block
  int tm;       // tile rows (fwd/dgrad: rows of the group; wgrad: dB rows): 128, or 256 for wide tiles
  int split;    // CTAs sharing a tile (router: a cluster, each a slice of the contraction); else 1
  int crank;    // this CTA's rank in that cluster
  __device__ Geo(const Params& p, int elem_bytes, int bn, int tile_m = kBM) {
    mn_rows = elem_bytes == 1 ? kMxWgRows : kMnRows;
    rb = 1;
    tm = tile_m;
    split = kEpi == kEpiTopk && p.split > 1 ? p.split : 1;
    crank = kEpi == kEpiTopk && split > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    if (kMode == kWgrad) {
      nt = (p.N + tm - 1) / tm;
      nt2 = (p.K + kBN - 1) / kBN;
      n_out = p.K;
      bn_out = kBN;
      kb_fixed = 0;
    } else {
      n_out = kMode == kFwd ? (kEpi == kEpiSwiglu ? p.N / 2 : p.N) : p.K;
      bn_out = kEpi == kEpiSwiglu ? bn / 2 : bn;
      nt = (n_out + bn_out - 1) / bn_out;
      nt2 = 1;
      kb_fixed = kMode == kFwd ? (p.K * elem_bytes + kBKBytes - 1) / kBKBytes
                               : (p.N + kMnRows - 1) / kMnRows;
      const long long a_row = kMode == kFwd ? static_cast<long long>(p.K) * elem_bytes
                                            : static_cast<long long>(p.N) * 2;   // dgrad: dC is bf16
      const long long r = kRasterABytes / (static_cast<long long>(tm) * (a_row > 0 ? a_row : 1));
      rb = r < 1 ? 1 : (r > 1024 ? 1024 : static_cast<int>(r));
    }
  }
  __device__ int tiles_of(int cnt) const {
    if (kMode == kWgrad) return nt * nt2;
    return ((cnt + tm - 1) / tm) * nt;
  }
  // this CTA's first tile and its stride through the tile list (a router cluster
  // shares one tile)
  __device__ int first_tile() const {
    return kEpi == kEpiTopk ? static_cast<int>(blockIdx.x) / split : static_cast<int>(blockIdx.x);
  }
  __device__ int tile_stride() const {
    return kEpi == kEpiTopk ? static_cast<int>(gridDim.x) / split : static_cast<int>(gridDim.x);
  }
};

template <int kMode, int kEpi>
__device__ __forceinline__ Tile tile_info(const Smem& s, const Geo<kMode, kEpi>& g, int tile, const Params& p) {
  const int E = p.E, M = p.M;
  int lo = 0, local = 0;
  if (kMode == kWgrad) {
    // only experts with rows own tiles (in id order); empty ones are zero-filled
    const int tpe = g.nt * g.nt2;
    lo = s.prefix[tile / tpe];
    local = tile % tpe;
  } else {
    int hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s.prefix[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    local = tile - s.prefix[lo];
  }
  Tile t;
  t.e = lo;
  int beg, end;
  group_range(p, lo, beg, end);
  const int cnt = group_ok(beg, end, M) ? end - beg : 0;
  if (kMode == kWgrad) {
    t.n0 = (local % g.nt) * g.tm;
    t.col0 = (local / g.nt) * kBN;
    t.row0 = cnt > 0 ? beg : 0;
    t.rows = cnt;
    t.kblocks = (cnt + g.mn_rows - 1) / g.mn_rows;
    t.kb0 = 0;
  } else {
    const int mt = (cnt + g.tm - 1) / g.tm;   // >= 1: only non-empty groups own tiles
    const int blk = local / (g.rb * g.nt);   // raster block (see kRasterABytes)
    const int rem = local - blk * g.rb * g.nt;
    const int in_blk = mt - blk * g.rb < g.rb ? mt - blk * g.rb : g.rb;   // row tiles in this block
    t.row0 = beg + (blk * g.rb + rem % in_blk) * g.tm;
    const int left = beg + cnt - t.row0;
    t.rows = left < g.tm ? left : g.tm;
    t.col0 = (rem / in_blk) * g.bn_out;
    t.n0 = 0;
    if constexpr (kEpi == kEpiTopk) {
      // a split contraction: slice crank of split near-equal runs of K blocks
      t.kb0 = g.crank * g.kb_fixed / g.split;
      t.kblocks = (g.crank + 1) * g.kb_fixed / g.split - t.kb0;
    } else {
      t.kb0 = 0;
      t.kblocks = g.kb_fixed;
    }
  }
  return t;
}

// Per-expert tile prefix in shared memory (all threads participate).  A group
// whose offsets are out of range is flagged and treated as empty.  `scratch` is
// shared memory for E ints that nothing else uses yet (the first operand stage).
template <int kMode, int kEpi>
__device__ void build_tiles(Smem& s, const Geo<kMode, kEpi>& g, const Params& p, int* scratch) {
  const int32_t* offs = p.offsets;
  if (kMode == kWgrad) {
    // Expert list: the experts with rows by row count, largest first (ties: lower
    // id), then the empty (or invalid) ones in id order.  Tiles are dealt to the
    // CTAs round-robin, so the equal-cost tiles of one expert run side by side on
    // every SM, in step through its rows, and share them in L2; the many short
    // tiles of the small experts come last.
    int* cnt = scratch;
    if (threadIdx.x == 0) s.nnz = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
      const int beg = offs[e], end = offs[e + 1];
      const bool ok = group_ok(beg, end, p.M);
      if (!ok && blockIdx.x == 0) flag_error(p.status, MOE_DEV_BAD_INDEX);
      cnt[e] = ok ? end - beg : 0;
      if (ok && end > beg) atomicAdd(&s.nnz, 1);
    }
    __syncthreads();
    const int nh = s.nnz;
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
      const int c = cnt[e];
      int rank = 0;
      if (c > 0) {
        for (int j = 0; j < p.E; ++j) {
          const int cj = cnt[j];
          rank += (cj > c || (cj == c && j < e)) ? 1 : 0;
        }
      } else {
        rank = nh;
        for (int j = 0; j < e; ++j) rank += cnt[j] == 0 ? 1 : 0;
      }
      s.prefix[rank] = e;
    }
    if (threadIdx.x == 0) s.total_tiles = nh * g.nt * g.nt2;
    fence_proxy_async_smem();   // the scratch is the first stage, which TMA writes next
    __syncthreads();
    return;
  }
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
    int beg, end;
    group_range(p, e, beg, end);
    int cnt = end - beg;
    if (!group_ok(beg, end, p.M)) {
      if (blockIdx.x == 0) flag_error(p.status, MOE_DEV_BAD_INDEX);
      cnt = 0;
    }
    s.prefix[e + 1] = g.tiles_of(cnt);
  }
  if (threadIdx.x == 0) s.prefix[0] = 0;
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    for (int base = 1; base <= p.E; base += 32) {
      const int i = base + lane;
      int v = i <= p.E ? s.prefix[i] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xFFFFFFFFu, v, off);
        if (lane >= off) v += u;
      }
      if (i <= p.E) s.prefix[i] = v + carry;
      carry += __shfl_sync(0xFFFFFFFFu, v, 31);
    }
    if (lane == 0) s.total_tiles = carry;
  }
  __syncthreads();
}

// silu(g) = g * sigmoid(g) with the fast exponential and division (the MXFP8 GEMM's
// accumulator waits for this epilogue, so it must be short); for g < -88 the
// exponential overflows and both give the exact limit 0.
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.f + __expf(-g)); }
__device__ __forceinline__ float sigmoid_f(float g) { return __fdividef(1.f, 1.f + __expf(-g)); }

// NVFP4: scale 32 accumulator words by alpha (a no-op for the other kinds).
template <int kKind>
__device__ __forceinline__ void nv_scale(uint32_t (&v)[32], float alpha) {
  if constexpr (kKind == 3) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
  }
}

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

// Load 32 consecutive values (bf16 or fp32) as fp32.
template <typename T>
__device__ __forceinline__ void load32(const T* src, float (&v)[32]) {
  if constexpr (sizeof(T) == 2) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = s4[q];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[8 * q + 2 * i] = bf16_to_f32(static_cast<uint16_t>(w[i] & 0xFFFFu));
        v[8 * q + 2 * i + 1] = bf16_to_f32(static_cast<uint16_t>(w[i] >> 16));
      }
    }
  } else {
    const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 u = s4[q];
      v[4 * q] = u.x; v[4 * q + 1] = u.y; v[4 * q + 2] = u.z; v[4 * q + 3] = u.w;
    }
  }
}

// MOE_DEBUG: a TMA copy's x coordinate starts on a 16-byte boundary and no coordinate
// is negative (a copy that breaks either faults); a release build takes it as true.
__device__ __forceinline__ bool tma_x_ok(long long x, int elem_bytes, long long y, int32_t* status) {
  return dbg_check(x >= 0 && y >= 0 && (x * elem_bytes) % 16 == 0, status);
}

// Write one warp's 32 tile rows of output, held one row per lane as 32-bit words
// (two bf16 or four E4M3 values each).  A warp whose 32 rows all belong to the
// group sends boxes of kRowB-byte rows (kBoxElems elements) through its kBufs
// rotating staging buffers of 32 x kRowB bytes by TMA store; 16-byte chunk h of row
// r sits at chunk h ^ ((r >> 1) & 3) for 64-byte rows (64-byte swizzle) and h ^
// ((r >> 2) & 1) for 32-byte rows (32-byte swizzle).  Two 1 KB boxes in place of one
// 2 KB box let a box be staged while the previous one is still read by its store.
// A warp whose rows cross the group's end (the next group's rows follow) stores its
// valid rows directly.  `box` counts the warp's staged boxes across its tiles: the
// buffers rotate over that count, so the buffer a box takes was last used kBufs boxes
// before whatever the number of boxes of a tile.
template <int kBoxElems, int kBufs, int kRowB, int kWords>
__device__ __forceinline__ void epi_store_rows(const CUtensorMap* tmD, uint8_t* stg, const uint32_t (&pk)[kWords],
                                               int lane, uint8_t* out, int row0, int rows_valid, int col0,
                                               int n_out, int& box, int32_t* status) {
  static_assert(kRowB == 64 || kRowB == 32, "box rows of 64 or 32 bytes");
  constexpr int kElemBytes = kRowB / kBoxElems;
  constexpr int kRowWords = kRowB / 4;       // 32-bit words per box row
  constexpr int kChunks = kRowB / 16;        // 16-byte chunks per box row
  const size_t row_bytes = static_cast<size_t>(n_out) * kElemBytes;
  if constexpr (kBufs == 0) {
    // no staging boxes (NVFP4): every row is stored directly below
  } else if (rows_valid >= 32) {
#pragma unroll
    for (int c = 0; c < kWords / kRowWords; ++c) {
      if (col0 + c * kBoxElems >= n_out) break;
      uint8_t* buf = stg + (box++ % (kBufs > 0 ? kBufs : 1)) * (32 * kRowB);
      if (lane == 0) bulk_wait_read<(kBufs > 0 ? kBufs - 1 : 0)>();   // the box that last used buf has been read
      __syncwarp();
      const int sw = kRowB == 64 ? (lane >> 1) & 3 : (lane >> 2) & 1;
#pragma unroll
      for (int h = 0; h < kChunks; ++h) {
        const int w0 = c * kRowWords + 4 * h;
        *reinterpret_cast<uint4*>(buf + lane * kRowB + ((h ^ sw) * 16)) =
            make_uint4(pk[w0], pk[w0 + 1], pk[w0 + 2], pk[w0 + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && tma_x_ok(col0 + c * kBoxElems, kElemBytes, row0, status)) {
        tma_store_2d(tmD, buf, col0 + c * kBoxElems, row0);
        bulk_commit();
      }
    }
  }
  if ((kBufs == 0 || rows_valid < 32) && lane < rows_valid) {
#pragma unroll
    for (int c = 0; c < kWords / kRowWords; ++c) {
      const int col = col0 + c * kBoxElems;
      uint4* d4 = reinterpret_cast<uint4*>(out + static_cast<size_t>(row0 + lane) * row_bytes +
                                           static_cast<size_t>(col) * kElemBytes);
#pragma unroll
      for (int h = 0; h < kChunks; ++h)   // n_out is a multiple of 16 bytes' worth: check per chunk
        if (col + h * (16 / kElemBytes) < n_out)
          d4[h] = make_uint4(pk[c * kRowWords + 4 * h], pk[c * kRowWords + 4 * h + 1], pk[c * kRowWords + 4 * h + 2],
                             pk[c * kRowWords + 4 * h + 3]);
    }
  }
}

// Named barrier 1 over the epilogue warps (kThreads threads from warp 2 on).
template <int kThreads>
__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }

template <int kKind, int kMode, int kEpi, typename OutT>
__global__ void __launch_bounds__((block_threads<kKind, kMode, kEpi, static_cast<int>(sizeof(OutT))>()), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                        const __grid_constant__ CUtensorMap tmD, const Params p) {
  using C = Cfg<kKind>;
  constexpr bool kW = wide_tile<kKind, kMode, kEpi, static_cast<int>(sizeof(OutT))>();
  constexpr int TM = kW ? kWideM : kBM;                 // tile rows
  constexpr int NS = stages_for<kKind, kMode, kW>();
  constexpr int kStageSz = stage_bytes<kW>();
  constexpr int kASize = TM * kBKBytes;                 // A part of a stage
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Smem& s = *reinterpret_cast<Smem*>(tiles + NS * kStageSz + extra_smem<kKind, kMode, kW>());
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int eb = C::kEb;
  using TL = Tl<kKind, kMode, kEpi>;
  constexpr int BN = TL::BN;
  constexpr int kAccN = kW ? 1 : TL::kAcc;              // accumulator buffers (wide: one, in two halves)
  const Geo<kMode, kEpi> g(p, eb, BN, TM);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
      mbar_init(&s.sfready[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.sfull[i], 1);
      mbar_init(&s.sempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], kW ? 32 * kWideEpiWarps : 128);
    }
    // router split: one arrival from each peer of the cluster
    mbar_init(&s.xready, g.split > 1 ? g.split - 1 : 1);
    mbar_init(&s.xdone, g.split > 1 ? g.split - 1 : 1);
    s.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (C::kMx) {
      tma_prefetch_desc(&tmSA);
      tma_prefetch_desc(&tmSB);
    }
    if (kMode == kWgrad || (kMode == kFwd && sizeof(OutT) <= 2) || kW) tma_prefetch_desc(&tmD);
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  pdl_begin();             // the prologue above overlaps the preceding kernel
  build_tiles(s, g, p, reinterpret_cast<int*>(tiles));   // contains __syncthreads
  // a cluster's CTAs see each other's barriers initialised before any remote arrival
  // (reached by every thread, before any other wait)
  if (kEpi == kEpiTopk && g.split > 1) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const int total = s.total_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0, ss = 0;
      uint32_t phase = 0, ss_phase = 0;
      for (int tile = g.first_tile(); tile < total && !s.abort; tile += g.tile_stride()) {
        const Tile t = tile_info(s, g, tile, p);
        for (int kb = 0; kb < t.kblocks; ++kb) {
          if (kKind == 2 && kMode == kFwd && kb % 4 == 0) {
            // raw E8M0 rows, 16 bytes per row = the scales of 4 K-blocks, into slot ss
            if (!mbar_wait(&s.sempty[ss], ss_phase ^ 1u, p.status, &s.abort)) break;
            uint8_t* rsa = tiles + NS * kStageSz + raw_off<kKind>() + ss * kSfSlot;
            uint8_t* rsb = rsa + kSfAStage;
            const int sx = 16 * (kb / 4);
            const int brow = t.e * p.N;
            mbar_arrive_expect_tx(&s.sfull[ss], kSfSlot);
            tma_load_2d(rsa, &tmSA, &s.sfull[ss], sx, t.row0);
            if (kEpi == kEpiSwiglu) {
              tma_load_2d(rsb, &tmSB, &s.sfull[ss], sx, brow + t.col0);
              tma_load_2d(rsb + kSfBStage / 2, &tmSB, &s.sfull[ss], sx, brow + g.n_out + t.col0);
            } else {
              tma_load_2d(rsb, &tmSB, &s.sfull[ss], sx, brow + t.col0);
              tma_load_2d(rsb + kSfBStage / 2, &tmSB, &s.sfull[ss], sx, brow + t.col0 + kBM);
            }
            if (++ss == raw_slots<kKind>()) { ss = 0; ss_phase ^= 1u; }
          }
          if (!mbar_wait(&s.empty[stage], phase ^ 1u, p.status, &s.abort)) break;
          uint8_t* sa = tiles + stage * kStageSz;
          uint8_t* sb = sa + kASize;
          uint64_t* bar = &s.full[stage];
          {
            // MOE_DEBUG: the stage's TMA x coordinates (a misaligned copy faults); a
            // failed check completes the stage without copies (garbage, flagged)
            bool xok;
            if constexpr (kMode == kFwd) xok = tma_x_ok((t.kb0 + kb) * (kBKBytes / eb), eb, t.row0, p.status);
            else if constexpr (kMode == kDgrad) xok = tma_x_ok(kb * kMnRows, 2, t.row0, p.status) &&
                                                      tma_x_ok(t.col0, 2, 0, p.status);
            else if constexpr (C::kMx) xok = tma_x_ok(t.n0, 1, t.row0, p.status) && tma_x_ok(t.col0, 1, 0, p.status);
            else xok = tma_x_ok(t.n0, 2, t.row0, p.status) && tma_x_ok(t.col0, 2, 0, p.status);
            if (!xok) {
              mbar_arrive(bar);
              if (++stage == NS) { stage = 0; phase ^= 1u; }
              continue;
            }
          }
          mbar_arrive_expect_tx(bar, (kEpi == kEpiTopk ? kAStage + p.n_mma * kBKBytes : kStageSz) +
                                         (C::kMx && kMode == kWgrad ? kAtomBytes : 0) +
                                         (kKind == 3 ? kNvAtomBytes : 0));
          if (kMode == kFwd) {
            const int kx = (t.kb0 + kb) * (kBKBytes / eb);
            tma_load_2d(sa, &tmA, bar, kx, t.row0);
            if (kEpi == kEpiSwiglu) {
              tma_load_3d(sb, &tmB, bar, kx, t.col0, t.e);
              tma_load_3d(sb + kBStage / 2, &tmB, bar, kx, g.n_out + t.col0, t.e);
            } else {
              tma_load_3d(sb, &tmB, bar, kx, t.col0, t.e);
            }
            if constexpr (kKind == 3) {
              // raw scale rows of this stage: 16 bytes (= 256 elements) per row
              uint8_t* at = tiles + NS * kStageSz + stage * kNvAtomBytes;
              const int brow = t.e * p.N;
              tma_load_2d(at, &tmSA, bar, 16 * kb, t.row0);
              tma_load_2d(at + 2048, &tmSB, bar, 16 * kb, brow + t.col0);
              tma_load_2d(at + 4096, &tmSB, bar, 16 * kb, brow + (kEpi == kEpiSwiglu ? g.n_out : kBM) + t.col0);
            }
          } else if (kMode == kDgrad) {
            const int nx = kb * kMnRows;                  // contraction index (N of B)
            tma_load_2d(sa, &tmA, bar, nx, t.row0);
#pragma unroll
            for (int j = 0; j < kBN / 64; ++j) tma_load_3d(sb + j * kBox, &tmB, bar, t.col0 + 64 * j, nx, t.e);
          } else if constexpr (C::kMx) {
            // 128 rows of the group: one 128-column box of dC^T, two of A, and the
            // quad's scale tiles (dC: 512 B for rows n0.., A: 1 KB for columns col0..)
            const int r = t.row0 + kb * kMxWgRows;
            tma_load_2d(sa, &tmA, bar, t.n0, r);
            tma_load_2d(sb, &tmB, bar, t.col0, r);
            tma_load_2d(sb + kBStage / 2, &tmB, bar, t.col0 + 128, r);
            const size_t quad = static_cast<size_t>(t.row0 / 128 + t.e + kb);
            uint8_t* at = tiles + NS * kStageSz + wg_atom_off<kKind>() + stage * kAtomBytes;
            bulk_load(at, p.sfa + (quad * (p.N / 128) + t.n0 / 128) * 512, 512, bar);
            bulk_load(at + 512, p.sfb + (quad * (p.K / 128) + t.col0 / 128) * 512, 1024, bar);
          } else {
            const int r = t.row0 + kb * kMnRows;          // contraction index (rows of the group)
#pragma unroll
            for (int j = 0; j < TM / 64; ++j) tma_load_2d(sa + j * kBox, &tmA, bar, t.n0 + 64 * j, r);
#pragma unroll
            for (int j = 0; j < kBN / 64; ++j) tma_load_2d(sb + j * kBox, &tmB, bar, t.col0 + 64 * j, r);
          }
          if (++stage == NS) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // the router's MMA is only as wide as its (16-rounded) expert count
    const uint32_t idesc = kKind == 3 ? make_idesc_nvf4(kBM, BN)
                           : C::kMx ? make_idesc_mx(kBM, BN) | (kMode == kWgrad ? (3u << 15) : 0u)
                                    : make_idesc<kKind>(kBM, kEpi == kEpiTopk ? p.n_mma : kBN, kMode == kWgrad,
                                                        kMode != kFwd);
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    for (int tile = g.first_tile(); tile < total && !s.abort; tile += g.tile_stride()) {
      const Tile t = tile_info(s, g, tile, p);
      if (!mbar_wait(&s.tempty[acc], acc_phase ^ 1u, p.status, &s.abort)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BN);
      for (int kb = 0; kb < t.kblocks; ++kb) {
        if (C::kMx && kMode == kWgrad) {
          // Both operands MN-major (A = dC^T, B = A), 128 contraction rows per stage.
          // Last block of the group: zero rows [valid, 32*steps) of dC^T and skip
          // 32-row steps wholly past the group (their scales are never read).
          if (!mbar_wait(&s.full[stage], phase, p.status, &s.abort)) break;
          tc_fence_after();
          uint8_t* sa_ptr = tiles + stage * kStageSz;
          const int valid = t.rows - kb * kMxWgRows;
          int steps = 4;
          if (valid < kMxWgRows) {
            steps = (valid + 31) / 32;
            const int zrows = steps * 32 - valid;
            for (int i = lane; i < zrows * 8; i += 32)
              *reinterpret_cast<uint4*>(sa_ptr + (valid + i / 8) * 128 + (i % 8) * 16) = make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0) {
            const uint32_t sa = smem_u32(sa_ptr);
            const uint32_t sb = sa + kAStage;
            const uint32_t ssa = smem_u32(tiles + NS * kStageSz + wg_atom_off<kKind>() + stage * kAtomBytes);
            const uint32_t slot = tmem + TL::kSfBase + TL::kSfStride * static_cast<uint32_t>(stage);
            tc_cp_32x128b_warpx4(slot, make_sdesc(ssa, 0, 128, 0));
            tc_cp_32x128b_warpx4(slot + TL::kSfB, make_sdesc(ssa + 512, 0, 128, 0));
            tc_cp_32x128b_warpx4(slot + TL::kSfB + 4, make_sdesc(ssa + 1024, 0, 128, 0));
            for (int kk = 0; kk < steps; ++kk) {
              // 32 rows x 128 bytes per step; 128-column atoms 16 KB apart, 8-row groups 1 KB apart
              const uint64_t ad = make_sdesc(sa + kk * 4096, kBStage / 2, 1024, 2);
              const uint64_t bd = make_sdesc(sb + kk * 4096, kBStage / 2, 1024, 2);
              const uint32_t id = idesc | (static_cast<uint32_t>(kk) << 29) | (static_cast<uint32_t>(kk) << 4);
              tc_mma_mxf8(d_tmem, ad, bd, id, slot, slot + TL::kSfB, (kb | kk) != 0 ? 1u : 0u);
            }
            tc_commit(&s.empty[stage]);
          }
          __syncwarp();
          if (++stage == NS) { stage = 0; phase ^= 1u; }
          continue;
        }
        if (kKind == 3) {
          // NVFP4: wait for the atoms (the scale warp saw the stage land), then per
          // MMA kk copy its atoms into a 32-column region (A at +0, B rows 0-127 at
          // +16, rows 128-255 at +20: the alignments of the MXFP8 slots) and issue the
          // K=64 MMA.  Two region sets alternate by stage: a copy is issued after the
          // MMAs that read the set before, by the same thread, and runs after them.
          if (!mbar_wait(&s.sfready[stage], phase, p.status, &s.abort)) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t sa = smem_u32(tiles + stage * kStageSz);
            const uint32_t sb = sa + kAStage;
            const uint32_t at = smem_u32(tiles + NS * kStageSz + stage * kNvAtomBytes);
            const uint32_t set = tmem + TL::kSfBase + 128u * static_cast<uint32_t>(stage & 1);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t slot = set + 32u * static_cast<uint32_t>(kk);
              tc_cp_32x128b_warpx4(slot, make_sdesc(at + kk * 512, 0, 128, 0));
              tc_cp_32x128b_warpx4(slot + 16, make_sdesc(at + 2048 + kk * 1024, 0, 128, 0));
              tc_cp_32x128b_warpx4(slot + 20, make_sdesc(at + 2048 + kk * 1024 + 512, 0, 128, 0));
              const uint64_t ad = make_sdesc(sa + kk * 32, 16, 1024, 2);
              const uint64_t bd = make_sdesc(sb + kk * 32, 16, 1024, 2);
              tc_mma_nvf4(d_tmem, ad, bd, idesc, slot, slot + 16, (kb | kk) != 0 ? 1u : 0u);
            }
            tc_commit(&s.empty[stage]);
          }
          __syncwarp();
          if (++stage == NS) { stage = 0; phase ^= 1u; }
          continue;
        }
        if (C::kMx) {
          if (!mbar_wait(&s.sfready[stage], phase, p.status, &s.abort)) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t sa = smem_u32(tiles + stage * kStageSz);
            const uint32_t sb = sa + kAStage;
            const uint32_t ssa = smem_u32(tiles + NS * kStageSz + atom_off<kKind>() + stage * kAtomBytes);  // atoms
            const uint32_t ssb = ssa + 512;
            // scale slot of this stage: A atom at +0 (4 columns), B atoms at +kSfB, +kSfB+4
            const uint32_t slot = tmem + TL::kSfBase + TL::kSfStride * static_cast<uint32_t>(stage);
            tc_cp_32x128b_warpx4(slot, make_sdesc(ssa, 0, 128, 0));
            tc_cp_32x128b_warpx4(slot + TL::kSfB, make_sdesc(ssb, 0, 128, 0));
            tc_cp_32x128b_warpx4(slot + TL::kSfB + 4, make_sdesc(ssb + 512, 0, 128, 0));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = make_sdesc(sa + kk * 32, 16, 1024, 2);
              const uint64_t bd = make_sdesc(sb + kk * 32, 16, 1024, 2);
              const uint32_t id = idesc | (static_cast<uint32_t>(kk) << 29) | (static_cast<uint32_t>(kk) << 4);
              tc_mma_mxf8(d_tmem, ad, bd, id, slot, slot + TL::kSfB, (kb | kk) != 0 ? 1u : 0u);
            }
            tc_commit(&s.empty[stage]);
          }
          __syncwarp();
          if (++stage == NS) { stage = 0; phase ^= 1u; }
          continue;
        }
        if (!mbar_wait(&s.full[stage], phase, p.status, &s.abort)) break;
        tc_fence_after();
        uint8_t* sa_ptr = tiles + stage * kStageSz;
        const uint32_t sa = smem_u32(sa_ptr);
        const uint32_t sb = sa + kASize;
        int steps = 4;
        if (kMode == kWgrad) {
          // Last block of the group: zero rows [valid, 16*steps) of the A operand
          // (dC^T) so the next group's rows contribute nothing, and skip 16-row
          // MMA steps that lie wholly past the group.
          const int valid = t.rows - kb * kMnRows;
          if (valid < kMnRows) {
            steps = (valid + 15) / 16;
            const int zrows = steps * 16 - valid;
            for (int i = lane; i < zrows * 8 * (TM / 64); i += 32) {
              const int box = i / (zrows * 8), rem = i % (zrows * 8);
              const int row = valid + rem / 8, chunk = rem % 8;
              *reinterpret_cast<uint4*>(sa_ptr + box * kBox + row * 128 + chunk * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
        }
        if (lane == 0) {
          // wide tiles: the second 128-row half (A rows / dB rows 128-255, accumulator
          // columns 256-511) only where the tile has rows there
          const int halves = kW ? ((kMode == kWgrad ? t.n0 + kBM < p.N : t.rows > kBM) ? 2 : 1) : 1;
          for (int kk = 0; kk < steps; ++kk) {
            uint64_t bd;
            if (kMode == kFwd) bd = make_sdesc(sb + kk * 32, 16, 1024, 2);
            else bd = make_sdesc(sb + kk * 2048, kBox, 1024, 2);
            for (int h = 0; h < halves; ++h) {
              // half h of A: 128 K-major rows further (16 KB), or two 64-column MN-major boxes
              const uint64_t ad = kMode == kWgrad ? make_sdesc(sa + h * 2 * kBox + kk * 2048, kBox, 1024, 2)
                                                  : make_sdesc(sa + h * kAStage + kk * 32, 16, 1024, 2);
              tc_mma<kKind>(d_tmem + static_cast<uint32_t>(h) * 256u, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            }
          }
          tc_commit(&s.empty[stage]);
        }
        __syncwarp();
        if (++stage == NS) { stage = 0; phase ^= 1u; }
      }
      if (lane == 0) tc_commit(&s.tfull[acc]);
      __syncwarp();
      if (++acc == kAccN) { acc = 0; acc_phase ^= 1u; }
    }
  } else if (kKind == 3 && warp == 6) {
    // ------------------------------------------------------------------ NVFP4 scale layout
    // Each stage's raw rows (A 128 x 16 B at +0, B 256 x 16 B at +2048) become, in
    // place, the atoms of its four MMAs: byte (m % 32) * 16 + (m / 32) * 4 + j of atom
    // kk is the scale of row m, 16-element block 4 kk + j (word kk of the row).
    int stage = 0;
    uint32_t phase = 0;
    for (int tile = blockIdx.x; tile < total && !s.abort; tile += gridDim.x) {
      const Tile t = tile_info(s, g, tile, p);
      for (int kb = 0; kb < t.kblocks; ++kb) {
        if (!mbar_wait(&s.full[stage], phase, p.status, &s.abort)) break;
        uint8_t* at = tiles + NS * kStageSz + stage * kNvAtomBytes;
        uint4 ra[4], rb[2][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) ra[i] = *reinterpret_cast<const uint4*>(at + (lane + 32 * i) * 16);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < 4; ++i) rb[h][i] = *reinterpret_cast<const uint4*>(at + 2048 + h * 2048 + (lane + 32 * i) * 16);
        __syncwarp();
        auto word = [](const uint4& v, int w) { return w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w)); };
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          *reinterpret_cast<uint4*>(at + kk * 512 + lane * 16) =
              make_uint4(word(ra[0], kk), word(ra[1], kk), word(ra[2], kk), word(ra[3], kk));
#pragma unroll
          for (int h = 0; h < 2; ++h)
            *reinterpret_cast<uint4*>(at + 2048 + kk * 1024 + h * 512 + lane * 16) =
                make_uint4(word(rb[h][0], kk), word(rb[h][1], kk), word(rb[h][2], kk), word(rb[h][3], kk));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.sfready[stage]);
        if (++stage == NS) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (kKind == 2 && kMode == kFwd && warp == 6) {
    // ------------------------------------------------------------------ MXFP8 scale layout
    // Every 4 K-blocks: take the raw scale rows of the slot (row r: 16 bytes, the
    // scales of 4 K-blocks) into registers and free the slot.  Every K-block: write
    // its 512-byte atoms (byte (m % 32) * 16 + (m / 32) * 4 + j for row m of 128 and
    // 32-element block j of the K-block) into the stage's atom area, once the stage's
    // previous atoms have been consumed (the stage is full again).
    int stage = 0, ss = 0;
    uint32_t phase = 0, ss_phase = 0;
    uint4 ra[4], rb[8];
    for (int tile = blockIdx.x; tile < total && !s.abort; tile += gridDim.x) {
      const Tile t = tile_info(s, g, tile, p);
      for (int kb = 0; kb < t.kblocks; ++kb) {
        if (kb % 4 == 0) {
          if (!mbar_wait(&s.sfull[ss], ss_phase, p.status, &s.abort)) break;
          const uint8_t* rsa = tiles + NS * kStageSz + raw_off<kKind>() + ss * kSfSlot;
          const uint8_t* rsb = rsa + kSfAStage;
#pragma unroll
          for (int j = 0; j < 4; ++j) ra[j] = *reinterpret_cast<const uint4*>(rsa + (lane + 32 * j) * 16);
#pragma unroll
          for (int j = 0; j < 8; ++j) rb[j] = *reinterpret_cast<const uint4*>(rsb + (lane + 32 * j) * 16);
          __syncwarp();
          if (lane == 0) mbar_arrive(&s.sempty[ss]);
          if (++ss == raw_slots<kKind>()) { ss = 0; ss_phase ^= 1u; }
        }
        if (!mbar_wait(&s.full[stage], phase, p.status, &s.abort)) break;
        uint8_t* at = tiles + NS * kStageSz + atom_off<kKind>() + stage * kAtomBytes;
        const int w = kb % 4;
        auto word = [w](const uint4& v) { return w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w)); };
        *reinterpret_cast<uint4*>(at + lane * 16) = make_uint4(word(ra[0]), word(ra[1]), word(ra[2]), word(ra[3]));
        *reinterpret_cast<uint4*>(at + 512 + lane * 16) = make_uint4(word(rb[0]), word(rb[1]), word(rb[2]), word(rb[3]));
        *reinterpret_cast<uint4*>(at + 1024 + lane * 16) = make_uint4(word(rb[4]), word(rb[5]), word(rb[6]), word(rb[7]));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.sfready[stage]);
        if (++stage == NS) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (kMode == kWgrad && warp == (kW ? 2 : 6)) {
    // ------------------------------------------------------------------ wgrad zero fill
    // Experts without rows own no tiles; their dW (exact zeros) is written here,
    // alongside the MMA work, with plain 16-byte stores (not through the TMA unit,
    // which the operand loads need) marked evict-first in L2 (so the zeros do not
    // push the operands out).  An expert's dW is N*K*2 bytes, a multiple of 2048
    // since N and K are multiples of 32.  The CTA's chunks are c = blockIdx.x +
    // i * gridDim.x; a warp writes four of them (8 KB) per pass, which measured a few
    // percent faster than one (the fill ends earlier, ahead of the store-bound tiles
    // of the small experts at the end).
    // Accumulating into dW, the experts without rows keep theirs: nothing to write.
    constexpr int kZfU = 4;
    const uint64_t pol = l2_evict_first_policy();
    const size_t per = static_cast<size_t>(p.N) * p.K * sizeof(OutT);
    const size_t cpe = per / 2048;
    const size_t chunks = p.accumulate ? 0 : static_cast<size_t>(p.E - s.nnz) * cpe;
    uint8_t* outb = static_cast<uint8_t*>(p.out);
    for (size_t c0 = blockIdx.x; c0 < chunks && !s.abort; c0 += kZfU * static_cast<size_t>(gridDim.x)) {
#pragma unroll
      for (int u = 0; u < kZfU; ++u) {
        const size_t c = c0 + static_cast<size_t>(u) * gridDim.x;
        if (c < chunks) {
          const size_t ci = c / cpe;
          const int e = s.prefix[s.nnz + static_cast<int>(ci)];
          uint4* dst = reinterpret_cast<uint4*>(outb + static_cast<size_t>(e) * per + (c - ci * cpe) * 2048);
#pragma unroll
          for (int i = lane; i < 128; i += 32) st_global_hint(dst + i, make_uint4(0, 0, 0, 0), pol);
        }
      }
    }
  } else if (warp >= 2 &&
             warp <= (kW ? wide_epi_warp0<kMode>() + kWideEpiWarps - 1 : (kEpi == kEpiTopk ? kRouterWarps - 1 : 5))) {
    // ------------------------------------------------------------------ epilogue
    // The accumulator is released (tempty) as soon as its last TMEM read is done;
    // the global stores of the tile follow from registers (or, for wgrad, from a
    // shared-memory staging buffer by TMA), overlapping the next tile's MMAs.
    // Wide tiles: the first four epilogue warps take the first 128-row half, the
    // next four the second.
    constexpr int kW0 = kW ? wide_epi_warp0<kMode>() : 2;
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int hh = kW ? (warp - kW0) >> 2 : 0;        // half of a wide tile
    const int si = kW ? warp - kW0 : q;               // staging box set of this warp
    constexpr int kEB = kW ? 1 : epi_bufs<kKind>();   // forward staging: 2 KB units per warp
    // MXFP8 has one 2 KB unit per warp: it holds two 1 KB boxes of 32-byte rows,
    // double-buffered; the others use 2 KB boxes of 64-byte rows (on wide tiles 1 KB
    // boxes measured slower: more, smaller stores)
    constexpr bool kHalfBox = kKind == 2;
    constexpr int kRB = kHalfBox ? 32 : kEpiRowBytes;    // box row bytes
    constexpr int kNB = kHalfBox ? 2 * kEB : kEB;        // staging boxes per warp
    float alpha = 1.f;                      // NVFP4: undo the two tensor encode scales
    if constexpr (kKind == 3) alpha = __fdiv_rn(1.f, __fmul_rn(__ldg(p.ts_a), __ldg(p.ts_b)));
    const int r = q * 32 + lane;            // tile row owned by this thread
    OutT* out = static_cast<OutT*>(p.out);
    int acc = 0;
    uint32_t acc_phase = 0;
    // wgrad: boxes this warp has staged so far; the staging buffers rotate over all of
    // them, across tiles, so the buffer a box takes was last used kWgBufs boxes before
    int wbox = 0;
    bool xchg = false;                      // router split: this CTA exchanged partials with its peers
    // (the router's epilogue warps meet at named barriers, so they all enter the
    // loop and all take the same decision to leave it: see below)
    for (int tile = g.first_tile(); tile < total && (kEpi == kEpiTopk || !s.abort); tile += g.tile_stride()) {
      Tile t = tile_info(s, g, tile, p);
      if (kW) {                              // this warp's half of the wide tile
        if (kMode == kWgrad) {
          t.n0 += hh * kBM;
        } else {
          t.row0 += hh * kBM;
          t.rows -= hh * kBM;
        }
      }
      [[maybe_unused]] bool acc_ok = true;
      if constexpr (kEpi == kEpiTopk) {
        // one bounded wait for all the router's epilogue warps; its outcome reaches
        // them through a barrier that every one of them always reaches
        if (warp == 2) {
          const bool ok = mbar_wait(&s.tfull[acc], acc_phase, p.status, &s.abort);
          if (lane == 0) s.epi_ok = ok ? 1 : 0;
        }
        epi_bar_sync<32 * (kRouterWarps - 2)>();
        acc_ok = *reinterpret_cast<volatile int*>(&s.epi_ok) != 0;
        // a CTA of a split cluster goes on to its exchanges with its peers either way
        if (!acc_ok && g.split == 1) break;
      } else {
        if (!mbar_wait(&s.tfull[acc], acc_phase, p.status, &s.abort)) break;
      }
      tc_fence_after();
      if (kW && (kMode == kWgrad ? t.n0 >= p.N : t.rows <= 0)) {
        // no rows in this half: nothing was computed for it
        tc_fence_before();
        mbar_arrive(&s.tempty[acc]);
        if (++acc == kAccN) { acc = 0; acc_phase ^= 1u; }
        continue;
      }
      const uint32_t tb = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN) +
                          static_cast<uint32_t>(hh) * 256u;
      bool released = false;
      if constexpr (kMode == kWgrad && sizeof(OutT) == 4) {
        // fp32 dW rows n0 + 32q .. +31 (this warp): each 32-column chunk read from TMEM
        // leaves as two 16-column boxes (64-byte rows, 64-byte swizzle) through the
        // warp's rotating 2 KB staging buffers, written by TMA (clipped at N and K) or,
        // accumulating, added to dW by a TMA reduction (one fp32 rounding an element).
        // The accumulator is released once its last chunk is read.
        constexpr int kWgBufs = wg_bufs<kKind>();
        uint8_t* stg = tiles + NS * kStageSz + si * wg_stage<kKind>();
        const int sw = (lane >> 1) & 3;
        const int nch = (p.K - t.col0) / 32 < kBN / 32 ? (p.K - t.col0) / 32 : kBN / 32;   // K % 32 == 0
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
          uint32_t v[32];
          tmem_ld32(tb + c * 32, v);
          tmem_ld_wait();
          if (c == nch - 1) {
            tc_fence_before();
            mbar_arrive(&s.tempty[acc]);
            released = true;
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint8_t* buf = stg + (wbox++ % kWgBufs) * 2048;
            if (lane == 0) bulk_wait_read<kWgBufs - 1>();   // the box that last used buf is read
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<uint4*>(buf + lane * 64 + ((j ^ sw) * 16)) =
                  make_uint4(v[16 * h + 4 * j], v[16 * h + 4 * j + 1], v[16 * h + 4 * j + 2], v[16 * h + 4 * j + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && tma_x_ok(t.col0 + 32 * c + 16 * h, 4, t.n0 + 32 * q, p.status)) {
              if (p.accumulate)
                tma_reduce_add_3d(&tmD, buf, t.col0 + 32 * c + 16 * h, t.n0 + 32 * q, t.e);
              else
                tma_store_3d(&tmD, buf, t.col0 + 32 * c + 16 * h, t.n0 + 32 * q, t.e);
              bulk_commit();
            }
          }
        }
      } else if constexpr (kMode == kWgrad) {
        // bf16 dW rows n0 + 32q .. +31 (this warp) x 256 columns: the accumulator is read
        // whole into registers and released, then written by TMA (clipped at N and K) in
        // 32-column boxes (64-byte swizzle) through the warp's wg_bufs rotating 2 KB
        // staging buffers, so boxes are staged while earlier ones are still read.
        uint32_t pk[kBN / 2];
#pragma unroll
        for (int c = 0; c < kBN / 32; c += 2) {   // two loads per wait
          uint32_t v[2][32];
          tmem_ld32(tb + c * 32, v[0]);
          tmem_ld32(tb + (c + 1) * 32, v[1]);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[(c + h) * 16 + i] = pack_bf16x2(__uint_as_float(v[h][2 * i]), __uint_as_float(v[h][2 * i + 1]));
        }
        tc_fence_before();
        mbar_arrive(&s.tempty[acc]);
        released = true;
        constexpr int kWgBufs = kW ? 1 : wg_bufs<kKind>();
        uint8_t* stg = tiles + NS * kStageSz + si * (kW ? 2048 : wg_stage<kKind>());
        const int sw = (lane >> 1) & 3;
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) {
          if (t.col0 + 32 * c >= p.K) break;      // warp-uniform: past the last dW column
          uint8_t* buf = stg + (wbox++ % kWgBufs) * 2048;
          if (lane == 0) bulk_wait_read<kWgBufs - 1>();   // the box that last used buf is read
          __syncwarp();
#pragma unroll
          for (int h = 0; h < 4; ++h)
            *reinterpret_cast<uint4*>(buf + lane * 64 + ((h ^ sw) * 16)) =
                make_uint4(pk[c * 16 + 4 * h], pk[c * 16 + 4 * h + 1], pk[c * 16 + 4 * h + 2], pk[c * 16 + 4 * h + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && tma_x_ok(t.col0 + 32 * c, 2, t.n0 + 32 * q, p.status)) {
            tma_store_3d(&tmD, buf, t.col0 + 32 * c, t.n0 + 32 * q, t.e);
            bulk_commit();
          }
        }
      } else if constexpr (sizeof(OutT) == 1) {
        // MXFP8 output: the 32 consecutive columns a thread holds of its row are one
        // 32-element block.  The values are rounded to bf16 while the accumulator is
        // read (so the result equals a bf16 store followed by row-wise quantisation);
        // after its release, each block's shared exponent comes from its amax and the
        // codes are E4M3 with round-to-nearest-even and saturation.
        constexpr int NB = (kEpi == kEpiSwiglu ? BN / 2 : BN) / 32;   // blocks per tile row
        uint32_t pk[NB * 16];
#pragma unroll
        for (int c = 0; c < NB; ++c) {
          if constexpr (kEpi == kEpiSwiglu) {
            uint32_t gv[32], uv[32];
            tmem_ld32(tb + c * 32, gv);
            tmem_ld32(tb + BN / 2 + c * 32, uv);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[c * 16 + i] = pack_bf16x2(silu_f(__uint_as_float(gv[2 * i])) * __uint_as_float(uv[2 * i]),
                                           silu_f(__uint_as_float(gv[2 * i + 1])) * __uint_as_float(uv[2 * i + 1]));
          } else {
            uint32_t v[32];
            tmem_ld32(tb + c * 32, v);
            tmem_ld_wait();
            nv_scale<kKind>(v, alpha);
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[c * 16 + i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          }
        }
        tc_fence_before();
        mbar_arrive(&s.tempty[acc]);
        released = true;
        uint32_t cw[NB * 8];
        uint32_t sb[NB];
#pragma unroll
        for (int c = 0; c < NB; ++c) {
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            amax = fmaxf(amax, fmaxf(fabsf(bf16_to_f32(static_cast<uint16_t>(pk[c * 16 + i] & 0xFFFFu))),
                                     fabsf(bf16_to_f32(static_cast<uint16_t>(pk[c * 16 + i] >> 16)))));
          float inv;
          mx_scale(amax, &sb[c], &inv);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t w0 = pk[c * 16 + 2 * i], w1 = pk[c * 16 + 2 * i + 1];
            cw[c * 8 + i] =
                static_cast<uint32_t>(f32x2_to_e4m3x2(bf16_to_f32(static_cast<uint16_t>(w0 & 0xFFFFu)) * inv,
                                                      bf16_to_f32(static_cast<uint16_t>(w0 >> 16)) * inv)) |
                (static_cast<uint32_t>(f32x2_to_e4m3x2(bf16_to_f32(static_cast<uint16_t>(w1 & 0xFFFFu)) * inv,
                                                       bf16_to_f32(static_cast<uint16_t>(w1 >> 16)) * inv)) << 16);
          }
        }
        epi_store_rows<kRB, kNB, kRB>(&tmD, tiles + NS * kStageSz + kEpiOff + si * kEB * kEpiBox, cw, lane,
                           reinterpret_cast<uint8_t*>(out), t.row0 + q * 32, t.rows - q * 32, t.col0, g.n_out, wbox, p.status);
        if (r < t.rows) {
          uint8_t* srow = p.out_scales + static_cast<size_t>(t.row0 + r) * (g.n_out / 32);
          if (g.n_out % 128 == 0 && t.col0 + 32 * NB <= g.n_out) {
            // the NB scale bytes of this row are consecutive and 4-byte aligned
#pragma unroll
            for (int c = 0; c < NB; c += 4)
              *reinterpret_cast<uint32_t*>(srow + t.col0 / 32 + c) =
                  sb[c] | (sb[c + 1] << 8) | (sb[c + 2] << 16) | (sb[c + 3] << 24);
          } else {
#pragma unroll
            for (int c = 0; c < NB; ++c)
              if (t.col0 + 32 * c < g.n_out) srow[t.col0 / 32 + c] = static_cast<uint8_t>(sb[c]);
          }
        }
      } else if constexpr (kEpi == kEpiSwiglu) {
        const bool valid = r < t.rows;
        const size_t grow = static_cast<size_t>(t.row0 + r);
        OutT* pre = static_cast<OutT*>(p.preact_out);
        if (sizeof(OutT) == 2 && pre == nullptr) {
          uint32_t pk[64];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t gv[32], uv[32];
            tmem_ld32(tb + c * 32, gv);
            tmem_ld32(tb + 128 + c * 32, uv);
            tmem_ld_wait();
            nv_scale<kKind>(gv, alpha);
            nv_scale<kKind>(uv, alpha);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[c * 16 + i] = pack_bf16x2(silu_f(__uint_as_float(gv[2 * i])) * __uint_as_float(uv[2 * i]),
                                           silu_f(__uint_as_float(gv[2 * i + 1])) * __uint_as_float(uv[2 * i + 1]));
          }
          tc_fence_before();
          mbar_arrive(&s.tempty[acc]);
          released = true;
          epi_store_rows<kRB / 2, kNB, kRB>(&tmD, tiles + NS * kStageSz + kEpiOff + si * kEB * kEpiBox, pk, lane,
                             reinterpret_cast<uint8_t*>(out), t.row0 + q * 32, t.rows - q * 32, t.col0, g.n_out, wbox, p.status);
        } else {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t gv[32], uv[32];
            tmem_ld32(tb + c * 32, gv);
            tmem_ld32(tb + 128 + c * 32, uv);
            tmem_ld_wait();
            nv_scale<kKind>(gv, alpha);
            nv_scale<kKind>(uv, alpha);
            const int col = t.col0 + c * 32;
            if (valid && col < g.n_out) {
              float h[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) h[i] = silu_f(__uint_as_float(gv[i])) * __uint_as_float(uv[i]);
              store32<OutT>(out + grow * g.n_out + col, h);
              if (pre != nullptr) {
                float gf[32], uf[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                  gf[i] = __uint_as_float(gv[i]);
                  uf[i] = __uint_as_float(uv[i]);
                }
                store32<OutT>(pre + grow * p.N + col, gf);
                store32<OutT>(pre + grow * p.N + g.n_out + col, uf);
              }
            }
          }
        }
      } else if constexpr (kEpi == kEpiDswiglu) {
        // the product is dH [M, f]; preact (G | U) is [M, 2f]; output [dG | dU]
        const bool valid = r < t.rows;
        const size_t grow = static_cast<size_t>(t.row0 + r);
        const OutT* pre = static_cast<const OutT*>(p.preact_in);
        const int f = g.n_out;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tb + c * 32, v);
          tmem_ld_wait();
          const int col = t.col0 + c * 32;
          if (valid && col < f) {
            float gf[32], uf[32], dg[32], du[32];
            load32<OutT>(pre + grow * 2 * f + col, gf);
            load32<OutT>(pre + grow * 2 * f + f + col, uf);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float dh = __uint_as_float(v[i]);
              const float sg = sigmoid_f(gf[i]);
              du[i] = dh * gf[i] * sg;
              dg[i] = dh * uf[i] * sg * (1.f + gf[i] * (1.f - sg));
            }
            store32<OutT>(out + grow * 2 * f + col, dg);
            store32<OutT>(out + grow * 2 * f + f + col, du);
          }
        }
      } else if constexpr (kEpi == kEpiTopk) {
        // Router: the tile's logits (128 tokens x E experts, fp32).  The selection runs
        // one token at a time per warp with the experts spread over the lanes (lane l
        // holds experts l, l + 32, ...): k rounds of a warp-wide max, the lowest expert
        // id winning ties, so equal logits go to the lower id, -inf (masked) experts are
        // taken last in id order, and NaN logits are flagged and treated as -inf.  (A
        // thread-per-token insertion pass cost several times the whole contraction.)
        // The launch gives every CTA exactly one tile, so the operand stages are free
        // once the accumulator is ready: the logits are staged there (128 rows x 256
        // floats; 16-byte chunk u of row j at chunk (u & ~7) | ((u ^ j) & 7)), and the
        // tile's per-expert counts are summed in shared memory first.
        const int E = p.N;
        const int ew = ((E + 31) / 32) * 32;
        float* lout = static_cast<float*>(p.out);
        fence_proxy_async_smem();            // the stages' TMA writes precede these stores
        float* stg = reinterpret_cast<float*>(tiles);                       // [128][256]
        int* tcnt = reinterpret_cast<int*>(tiles + kBM * kBN * sizeof(float));   // [256]
        constexpr int kEpiThreads = 32 * (kRouterWarps - 2);
        for (int i = threadIdx.x - 64; i < kBN; i += kEpiThreads) tcnt[i] = 0;
        if (acc_ok && warp <= 5) {           // one warp per TMEM lane quarter
#pragma unroll 1
          for (int c = 0; c < ew / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tb + c * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int uu = c * 8 + u;
              const int ph = (uu & ~7) | ((uu ^ r) & 7);
              *reinterpret_cast<float4*>(stg + r * kBN + ph * 4) =
                  make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                              __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3]));
            }
          }
          tc_fence_before();
          mbar_arrive(&s.tempty[acc]);
        }
        released = true;
        epi_bar_sync<kEpiThreads>();         // every row staged, the counts zeroed
        // Rows this CTA selects: the whole tile, or with a split contraction (a
        // cluster of g.split CTAs, each holding the partial logits of one run of K
        // blocks) its 128 / g.split rows, the partials summed in slice order (so the
        // logits do not depend on which CTA sums them) from the peers' staging
        // through distributed shared memory.
        const int rbeg = g.crank * (kBM / g.split);
        const int rend = t.rows < rbeg + kBM / g.split ? t.rows : rbeg + kBM / g.split;
        bool go = acc_ok;
        if (g.split > 1) {
          // (1) tell every peer whether this CTA's partial is staged, then wait for theirs
          if (warp == 2 && lane == 0) {
            fence_acq_rel_cluster();
            for (int j = 1; j < g.split; ++j) {
              const uint32_t pr = static_cast<uint32_t>((g.crank + j) % g.split);
              st_cluster_u32(cluster_map(smem_u32(&s.peer_ok[g.crank]), pr), acc_ok ? 1u : 0u);
              mbar_arrive_cluster(cluster_map(smem_u32(&s.xready), pr));
            }
          }
          if (warp == 2) {
            const bool ok = mbar_wait_cluster(&s.xready, 0, p.status);
            fence_acq_rel_cluster();
            if (lane == 0) {
              bool all = ok && acc_ok;
              for (int j = 0; j < g.split; ++j)
                if (j != g.crank) all = all && *reinterpret_cast<volatile int*>(&s.peer_ok[j]) != 0;
              s.x_ok = all ? 1 : 0;
            }
          }
          epi_bar_sync<kEpiThreads>();
          go = *reinterpret_cast<volatile int*>(&s.x_ok) != 0;
          // (2) the sums of this CTA's rows, in place (the peers read only their own rows
          // of this CTA's staging); the chunk swizzle stays within a row, so chunk c of a
          // row is the same 4 experts in every CTA
          if (go && rend > rbeg) {
            const int nch = ew / 4;
            const uint32_t lb = smem_u32(stg);
            uint32_t pb[kMaxSplit];
#pragma unroll
            for (int j = 0; j < kMaxSplit; ++j) pb[j] = j < g.split ? cluster_map(lb, static_cast<uint32_t>(j)) : 0u;
#pragma unroll 2
            for (int i = threadIdx.x - 64; i < (rend - rbeg) * nch; i += kEpiThreads) {
              const int row = rbeg + i / nch, ch = i % nch;
              const uint32_t off = static_cast<uint32_t>(row * kBN + ch * 4) * 4u;
              if (!dbg_check(row < kBM && off + 16u <= static_cast<uint32_t>(kBM * kBN * 4), p.status)) break;
              float4 a = ld_cluster_f4(pb[0] + off);
#pragma unroll
              for (int j = 1; j < kMaxSplit; ++j) {
                if (j < g.split) {
                  const float4 v = ld_cluster_f4(pb[j] + off);
                  a.x += v.x;
                  a.y += v.y;
                  a.z += v.z;
                  a.w += v.w;
                }
              }
              *reinterpret_cast<float4*>(stg + row * kBN + ch * 4) = a;
            }
          }
          epi_bar_sync<kEpiThreads>();
          // (3) done with the peers' staging (each waits for this before it exits)
          if (warp == 2 && lane == 0) {
            fence_acq_rel_cluster();
            for (int j = 1; j < g.split; ++j)
              mbar_arrive_cluster(cluster_map(smem_u32(&s.xdone), static_cast<uint32_t>((g.crank + j) % g.split)));
          }
          xchg = true;
        }
        if (!go) break;
        {
          const int ksel = p.k_sel;
          const bool full_softmax = p.renorm == 0;
          bool nan = false;
          // kRb tokens at a time per warp (their rounds are independent), the warps
          // taking the tile's rows in turn
          constexpr int kRb = 2;
#pragma unroll 1
          for (int jb = rbeg + (warp - 2) * kRb; jb < rend; jb += (kRouterWarps - 2) * kRb) {
            float val[kRb][8];
            uint32_t taken[kRb];                       // bit m: expert lane + 32 m is out
            float run_m[kRb], run_s[kRb], top0[kRb], my_v[kRb];
            int my_i[kRb];
#pragma unroll
            for (int b = 0; b < kRb; ++b) {
              const int row = jb + b;
              const bool rok = row < rend;
              taken[b] = rok ? 0u : 0xFFu;
#pragma unroll
              for (int m = 0; m < 8; ++m) {
                const int col = lane + 32 * m;
                float x = -INFINITY;
                if (rok && col < E) {
                  const int uu = col >> 2;
                  x = stg[row * kBN + (((uu & ~7) | ((uu ^ row) & 7)) << 2) + (col & 3)];
                  if (lout != nullptr) lout[static_cast<size_t>(t.row0 + row) * E + col] = x;
                  nan = nan || isnan(x);
                  x = isnan(x) ? -INFINITY : x;
                } else {
                  taken[b] |= 1u << m;
                }
                val[b][m] = x;
              }
              run_m[b] = -INFINITY;
              run_s[b] = 0.f;
              top0[b] = -INFINITY;
              my_v[b] = -INFINITY;
              my_i[b] = -1;
            }
            // full softmax: max and sum of exp over the experts that are not masked
            if (full_softmax) {
#pragma unroll
              for (int b = 0; b < kRb; ++b) {
#pragma unroll
                for (int m = 0; m < 8; ++m) run_m[b] = fmaxf(run_m[b], val[b][m]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) run_m[b] = fmaxf(run_m[b], __shfl_xor_sync(0xFFFFFFFFu, run_m[b], o));
              }
#pragma unroll
              for (int b = 0; b < kRb; ++b) {
                if (run_m[b] != -INFINITY) {
#pragma unroll
                  for (int m = 0; m < 8; ++m) run_s[b] += val[b][m] == -INFINITY ? 0.f : expf(val[b][m] - run_m[b]);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) run_s[b] += __shfl_xor_sync(0xFFFFFFFFu, run_s[b], o);
              }
            }
            // k rounds: the largest value not yet taken, the lowest expert id among equals
            for (int j = 0; j < ksel; ++j) {
              uint32_t key[kRb];
              int bm[kRb];
#pragma unroll
              for (int b = 0; b < kRb; ++b) {
                bm[b] = -1;
                float bv = -INFINITY;
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                  const bool ok = !((taken[b] >> m) & 1u) && (bm[b] < 0 || val[b][m] > bv);
                  bv = ok ? val[b][m] : bv;
                  bm[b] = ok ? m : bm[b];
                }
                // order-preserving key of the value (0: this lane has nothing left)
                const uint32_t bu = __float_as_uint(bv);
                key[b] = bm[b] < 0 ? 0u : ((bu & 0x80000000u) ? ~bu : (bu | 0x80000000u));
              }
              uint32_t wkey[kRb], mycol[kRb];
#pragma unroll
              for (int b = 0; b < kRb; ++b) wkey[b] = __reduce_max_sync(0xFFFFFFFFu, key[b]);
#pragma unroll
              for (int b = 0; b < kRb; ++b)
                mycol[b] = bm[b] >= 0 && key[b] == wkey[b] ? static_cast<uint32_t>(lane + 32 * bm[b]) : 0xFFFFFFFFu;
#pragma unroll
              for (int b = 0; b < kRb; ++b) {
                const uint32_t wkey_b = wkey[b];
                const uint32_t wcol = __reduce_min_sync(0xFFFFFFFFu, mycol[b]);
                if (mycol[b] == wcol) taken[b] |= 1u << bm[b];
                const float wv = __uint_as_float((wkey_b & 0x80000000u) ? (wkey_b & 0x7FFFFFFFu) : ~wkey_b);
                if (j == 0) top0[b] = wv;
                if (lane == j) {
                  my_v[b] = wv;
                  my_i[b] = wkey_b == 0u ? -1 : static_cast<int>(wcol);
                }
              }
            }
            // weights: softmax over the k selected (renormalize) or the full softmax;
            // every expert masked (-inf): no softmax mass, weight 0
#pragma unroll
            for (int b = 0; b < kRb; ++b) {
              float w;
              if (!full_softmax) {
                const float e = lane < ksel && top0[b] != -INFINITY ? expf(my_v[b] - top0[b]) : 0.f;
                float den = e;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xFFFFFFFFu, den, o);
                w = top0[b] == -INFINITY ? 0.f : e / den;
              } else {
                w = top0[b] == -INFINITY || lane >= ksel ? 0.f : expf(my_v[b] - run_m[b]) / run_s[b];
              }
              const int row = jb + b;
              if (lane < ksel && row < rend) {
                const size_t grow = static_cast<size_t>(t.row0 + row);
                p.topk_idx[grow * ksel + lane] = my_i[b];
                p.topk_w[grow * ksel + lane] = w;
                if (my_i[b] >= 0) atomicAdd(&tcnt[my_i[b]], 1);   // k <= E: always an expert
              }
            }
          }
          if (__any_sync(0xFFFFFFFFu, nan) && lane == 0) flag_error(p.status, MOE_DEV_NAN_LOGIT);
          epi_bar_sync<kEpiThreads>();       // the tile's counts are complete
          for (int i = threadIdx.x - 64; i < E; i += kEpiThreads) {
            const int cnt = tcnt[i];
            if (cnt > 0) atomicAdd(&p.counts[i], cnt);
          }
        }
      } else {
        const bool valid = r < t.rows;
        const size_t grow = static_cast<size_t>(t.row0 + r);
        if constexpr (sizeof(OutT) == 2) {
          uint32_t pk[BN / 2];
#pragma unroll
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tb + c * 32, v);
            tmem_ld_wait();
            nv_scale<kKind>(v, alpha);
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[c * 16 + i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          }
          tc_fence_before();
          mbar_arrive(&s.tempty[acc]);
          released = true;
          if constexpr (kMode == kFwd || kW) {
            epi_store_rows<kRB / 2, kNB, kRB>(&tmD, tiles + NS * kStageSz + kEpiOff + si * kEB * kEpiBox, pk, lane,
                               reinterpret_cast<uint8_t*>(out), t.row0 + q * 32, t.rows - q * 32, t.col0, g.n_out, wbox, p.status);
          } else if (valid) {
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
              const int col = t.col0 + c * 32;
              if (col < g.n_out) {
                uint4* d4 = reinterpret_cast<uint4*>(out + grow * g.n_out + col);
#pragma unroll
                for (int h = 0; h < 4; ++h)
                  d4[h] = make_uint4(pk[c * 16 + 4 * h], pk[c * 16 + 4 * h + 1], pk[c * 16 + 4 * h + 2],
                                     pk[c * 16 + 4 * h + 3]);
              }
            }
          }
        } else {
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tb + c * 32, v);
            tmem_ld_wait();
            nv_scale<kKind>(v, alpha);
            const int col = t.col0 + c * 32;
            if (valid && col < g.n_out) {
              float f[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
              store32<OutT>(out + grow * g.n_out + col, f);
            }
          }
        }
      }
      if (!released) {
        tc_fence_before();
        mbar_arrive(&s.tempty[acc]);
      }
      if (++acc == kAccN) { acc = 0; acc_phase ^= 1u; }
    }
    // a CTA of a split cluster exits only after its peers have read its staging
    if (kEpi == kEpiTopk && xchg && warp == 2) (void)mbar_wait_cluster(&s.xdone, 0, p.status);
    if constexpr (kMode == kWgrad || kMode == kFwd || kW) {
      if (lane == 0) bulk_wait_all0();      // every TMA store has landed
      __syncwarp();
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
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// Tiled tensor map over a dense row-major tensor: dims innermost first, box
// sizes, 128-byte swizzle (or none), zero fill out of bounds.
bool make_map(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* ptr, int rank,
              const uint64_t* dims, const uint32_t* box,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
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
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return false;
  }
  return true;
}

}  // namespace gemm
namespace {
// Kernels whose shared-memory attribute is set, per device.  Internal linkage on
// purpose: a function-local static in a template would be merged across every
// copy of this library loaded into one process.
struct SmemSet {
  const void* fn;
  uint64_t devs;
};
SmemSet g_smem_set[64];
std::mutex g_smem_mu;
}  // namespace
namespace gemm {

template <typename Kern>
bool ensure_smem(Kern k, size_t bytes) {
  // once per kernel and device: the attribute sticks, and setting it costs a driver call
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 63;
  const uint64_t bit = 1ull << dev;
  const void* fn = reinterpret_cast<const void*>(k);
  std::lock_guard<std::mutex> lock(g_smem_mu);
  int slot = -1;
  for (int i = 0; i < 64 && slot < 0; ++i)
    if (g_smem_set[i].fn == fn || g_smem_set[i].fn == nullptr) slot = i;
  if (slot >= 0 && g_smem_set[slot].fn == fn && (g_smem_set[slot].devs & bit)) return true;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) {
    set_error("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    return false;
  }
  if (slot >= 0) {
    g_smem_set[slot].fn = fn;
    g_smem_set[slot].devs |= bit;
  }
  return true;
}

template <int kKind, int kMode, int kEpi, typename OutT>
moe_status_t launch(const CUtensorMap& ta, const CUtensorMap& tb, const Params& p, cudaStream_t stream,
                    int sms, const char* what, const CUtensorMap* tsa = nullptr,
                    const CUtensorMap* tsb = nullptr, const CUtensorMap* td = nullptr, int cluster = 1) {
  constexpr bool kW = wide_tile<kKind, kMode, kEpi, static_cast<int>(sizeof(OutT))>();
  constexpr size_t smem = smem_for<kKind, kMode, kW>();
  static_assert(smem <= 232448, "shared memory budget");
  auto kern = grouped_gemm_kernel<kKind, kMode, kEpi, OutT>;
  if (!ensure_smem(kern, smem)) return MOE_ERR_CUDA;
  launch_pdl_cluster(kern, sms, block_threads<kKind, kMode, kEpi, static_cast<int>(sizeof(OutT))>(), smem, stream,
                     cluster, ta, tb, tsa ? *tsa : ta, tsb ? *tsb : tb, td ? *td : ta, p);
  return check_launch(what);
}

int elem_bytes(moe_dtype_t t) { return t == MOE_F32 ? 4 : (t == MOE_BF16 ? 2 : 1); }

CUtensorMapDataType map_type(moe_dtype_t t) {
  return t == MOE_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                      : (t == MOE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

moe_status_t common_checks(const char* fn, const moe_operand_t* A, const moe_operand_t* B,
                           const int32_t* offsets, int M, int N, int K, int E, const void* out, int* sms) {
  if (!A || !B) {
    set_error("%s: null operand", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (M < 0 || N <= 0 || K <= 0 || E < 1 || E > kMaxE || K % 32 || N % 32) {
    set_error("%s: need M >= 0, N %% 32 == 0, K %% 32 == 0, 1 <= E <= %d (M=%d N=%d K=%d E=%d)", fn,
              kMaxE, M, N, K, E);
    return MOE_ERR_INVALID_ARG;
  }
  if (A->dtype != B->dtype) {
    set_error("%s: both operands must have the same dtype", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (!offsets || (M > 0 && (!A->ptr || !B->ptr || !out)) || !aligned16(A->ptr) || !aligned16(B->ptr) ||
      !aligned16(out)) {
    set_error("%s: null or misaligned pointer", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (const moe_status_t dst = device_check(sms); dst != MOE_OK) return dst;
  return MOE_OK;
}

}  // namespace gemm
}  // namespace moe

using namespace moe;
using namespace moe::gemm;

extern "C" moe_status_t moe_grouped_gemm_fwd(const moe_operand_t* A, const moe_operand_t* B,
                                             const int32_t* offsets, int M, int N, int K, int E,
                                             moe_epilogue_t epi, void* C, moe_dtype_t c_dtype,
                                             void* preact, int32_t* dev_status,
                                             cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_grouped_gemm_fwd");
  const char* fn = "moe_grouped_gemm_fwd";
  int sms = 0;
  moe_status_t st = common_checks(fn, A, B, offsets, M, N, K, E, C, &sms);
  if (st != MOE_OK) return st;
  if ((epi != MOE_EPI_NONE && epi != MOE_EPI_SWIGLU) || (epi == MOE_EPI_SWIGLU && N % 64) ||
      (c_dtype != MOE_BF16 && c_dtype != MOE_F32) || !aligned16(preact)) {
    set_error("%s: epi NONE|SWIGLU (SWIGLU: N %% 64 == 0), C BF16|F32, aligned preact", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (A->dtype == MOE_E4M3 && (!A->scales || !B->scales || K % 512 || !aligned16(A->scales) ||
                               !aligned16(B->scales))) {
    set_error("%s: MXFP8 needs 16-byte aligned A and B scales and K %% 512 == 0", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (A->dtype == MOE_E2M1 && (!A->scales || !B->scales || !A->tensor_scale || !B->tensor_scale || K % 256 ||
                               !aligned16(A->scales) || !aligned16(B->scales))) {
    set_error("%s: NVFP4 needs 16-byte aligned A and B scales, both tensor scales and K %% 256 == 0", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (M == 0) return MOE_OK;
  if (A->dtype == MOE_E2M1) {
    // codes [rows, K/2] bytes: the kernel walks K in bytes, 128 (= 256 elements) per stage
    const bool swn = epi == MOE_EPI_SWIGLU;
    CUtensorMap ta, tb, tsa, tsb;
    const uint64_t adims[2] = {static_cast<uint64_t>(K / 2), static_cast<uint64_t>(M)};
    const uint32_t abox[2] = {kBKBytes, kBM};
    const uint64_t bdims[3] = {static_cast<uint64_t>(K / 2), static_cast<uint64_t>(N), static_cast<uint64_t>(E)};
    const uint32_t bbox[3] = {kBKBytes, static_cast<uint32_t>(swn ? kBN / 2 : kBN), 1};
    const uint64_t sadims[2] = {static_cast<uint64_t>(K / 16), static_cast<uint64_t>(M)};
    const uint64_t sbdims[2] = {static_cast<uint64_t>(K / 16), static_cast<uint64_t>(N) * static_cast<uint64_t>(E)};
    const uint32_t sbox[2] = {16, kBM};
    if (!make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A->ptr, 2, adims, abox) ||
        !make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B->ptr, 3, bdims, bbox) ||
        !make_map(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A->scales, 2, sadims, sbox, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&tsb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B->scales, 2, sbdims, sbox, CU_TENSOR_MAP_SWIZZLE_NONE))
      return MOE_ERR_INVALID_ARG;
    Params p{offsets, M, N, K / 2, E, C, preact, nullptr, nullptr, dev_status, nullptr, nullptr,
             A->tensor_scale, B->tensor_scale};
    const bool f32o = c_dtype == MOE_F32;
    if (swn) return f32o ? launch<3, kFwd, kEpiSwiglu, float>(ta, tb, p, stream, sms, fn, &tsa, &tsb)
                         : launch<3, kFwd, kEpiSwiglu, uint16_t>(ta, tb, p, stream, sms, fn, &tsa, &tsb);
    return f32o ? launch<3, kFwd, kEpiNone, float>(ta, tb, p, stream, sms, fn, &tsa, &tsb)
                : launch<3, kFwd, kEpiNone, uint16_t>(ta, tb, p, stream, sms, fn, &tsa, &tsb);
  }
  const int eb = elem_bytes(A->dtype);
  const uint32_t bk = kBKBytes / eb;
  CUtensorMap ta, tb;
  const uint64_t adims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
  // bf16 operands, bf16 output, plain epilogue: the wide tile (256 A rows per stage)
  const uint32_t a_rows = (A->dtype == MOE_BF16 && c_dtype == MOE_BF16 && epi == MOE_EPI_NONE) ? kWideM : kBM;
  const uint32_t abox[2] = {bk, a_rows};
  const uint64_t bdims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(E)};
  const uint32_t bbox[3] = {bk, static_cast<uint32_t>(epi == MOE_EPI_SWIGLU ? kBN / 2 : kBN), 1};
  if (!make_map(&ta, map_type(A->dtype), eb, A->ptr, 2, adims, abox) ||
      !make_map(&tb, map_type(A->dtype), eb, B->ptr, 3, bdims, bbox))
    return MOE_ERR_INVALID_ARG;
  Params p{offsets, M, N, K, E, C, preact, nullptr, nullptr, dev_status};
  const bool sw = epi == MOE_EPI_SWIGLU;
  const bool f32 = c_dtype == MOE_F32;
  // bf16 C [M, n_out] is written by TMA from 32-row x 32-column staging boxes
  // (64-byte rows, 64-byte swizzle)
  CUtensorMap td = ta;
  if (!f32) {
    // MXFP8 operands store 16-column boxes (32-byte rows, 32-byte swizzle), the others 32-column ones
    const bool half_box = A->dtype == MOE_E4M3;
    const uint64_t cdims[2] = {static_cast<uint64_t>(sw ? N / 2 : N), static_cast<uint64_t>(M)};
    const uint32_t cbox[2] = {static_cast<uint32_t>(half_box ? 16 : kEpiRowBytes / 2), 32};
    if (!make_map(&td, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, 2, cdims, cbox,
                  half_box ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B))
      return MOE_ERR_INVALID_ARG;
  }
  if (A->dtype == MOE_E4M3) {
    // E8M0 scales, [rows, K/32] bytes, read 16 bytes (4 stages' worth) per row
    CUtensorMap tsa, tsb;
    const uint64_t sadims[2] = {static_cast<uint64_t>(K / 32), static_cast<uint64_t>(M)};
    const uint64_t sbdims[2] = {static_cast<uint64_t>(K / 32), static_cast<uint64_t>(N) * static_cast<uint64_t>(E)};
    const uint32_t sbox[2] = {16, kBM};
    if (!make_map(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A->scales, 2, sadims, sbox, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&tsb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B->scales, 2, sbdims, sbox, CU_TENSOR_MAP_SWIZZLE_NONE))
      return MOE_ERR_INVALID_ARG;
    if (sw) return f32 ? launch<2, kFwd, kEpiSwiglu, float>(ta, tb, p, stream, sms, fn, &tsa, &tsb)
                       : launch<2, kFwd, kEpiSwiglu, uint16_t>(ta, tb, p, stream, sms, fn, &tsa, &tsb, &td);
    return f32 ? launch<2, kFwd, kEpiNone, float>(ta, tb, p, stream, sms, fn, &tsa, &tsb)
               : launch<2, kFwd, kEpiNone, uint16_t>(ta, tb, p, stream, sms, fn, &tsa, &tsb, &td);
  }
  if (A->dtype == MOE_F32) {
    if (sw) return f32 ? launch<0, kFwd, kEpiSwiglu, float>(ta, tb, p, stream, sms, fn)
                       : launch<0, kFwd, kEpiSwiglu, uint16_t>(ta, tb, p, stream, sms, fn, nullptr, nullptr, &td);
    return f32 ? launch<0, kFwd, kEpiNone, float>(ta, tb, p, stream, sms, fn)
               : launch<0, kFwd, kEpiNone, uint16_t>(ta, tb, p, stream, sms, fn, nullptr, nullptr, &td);
  }
  if (sw) return f32 ? launch<1, kFwd, kEpiSwiglu, float>(ta, tb, p, stream, sms, fn)
                     : launch<1, kFwd, kEpiSwiglu, uint16_t>(ta, tb, p, stream, sms, fn, nullptr, nullptr, &td);
  return f32 ? launch<1, kFwd, kEpiNone, float>(ta, tb, p, stream, sms, fn)
             : launch<1, kFwd, kEpiNone, uint16_t>(ta, tb, p, stream, sms, fn, nullptr, nullptr, &td);
}

extern "C" moe_status_t moe_grouped_gemm_fwd_mxfp8_out(const moe_operand_t* A, const moe_operand_t* B,
                                                       const int32_t* offsets, int M, int N, int K, int E,
                                                       moe_epilogue_t epi, uint8_t* c_codes, uint8_t* c_scales,
                                                       int32_t* dev_status, cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_grouped_gemm_fwd_mxfp8_out");
  const char* fn = "moe_grouped_gemm_fwd_mxfp8_out";
  int sms = 0;
  moe_status_t st = common_checks(fn, A, B, offsets, M, N, K, E, c_codes, &sms);
  if (st != MOE_OK) return st;
  if ((epi != MOE_EPI_NONE && epi != MOE_EPI_SWIGLU) || (epi == MOE_EPI_SWIGLU && N % 64) ||
      (M > 0 && !c_scales)) {
    set_error("%s: epi NONE|SWIGLU (SWIGLU: N %% 64 == 0) and an output scale buffer", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (A->dtype != MOE_E4M3) {
    set_error("%s: MXFP8 (E4M3) operands only", fn);
    return MOE_ERR_UNSUPPORTED;
  }
  if (!A->scales || !B->scales || K % 512 || !aligned16(A->scales) || !aligned16(B->scales)) {
    set_error("%s: MXFP8 needs 16-byte aligned A and B scales and K %% 512 == 0", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (M == 0) return MOE_OK;
  const bool sw = epi == MOE_EPI_SWIGLU;
  const int n_out = sw ? N / 2 : N;
  CUtensorMap ta, tb, tsa, tsb, td;
  const uint64_t adims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
  const uint32_t abox[2] = {kBKBytes, kBM};
  const uint64_t bdims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(E)};
  const uint32_t bbox[3] = {kBKBytes, static_cast<uint32_t>(sw ? kBN / 2 : kBN), 1};
  const uint64_t sadims[2] = {static_cast<uint64_t>(K / 32), static_cast<uint64_t>(M)};
  const uint64_t sbdims[2] = {static_cast<uint64_t>(K / 32), static_cast<uint64_t>(N) * static_cast<uint64_t>(E)};
  const uint32_t sbox[2] = {16, kBM};
  // codes [M, n_out] are written by TMA from 32-row x 32-column staging boxes (32-byte swizzle)
  const uint64_t cdims[2] = {static_cast<uint64_t>(n_out), static_cast<uint64_t>(M)};
  const uint32_t cbox[2] = {32, 32};
  if (!make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A->ptr, 2, adims, abox) ||
      !make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B->ptr, 3, bdims, bbox) ||
      !make_map(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A->scales, 2, sadims, sbox, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map(&tsb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B->scales, 2, sbdims, sbox, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map(&td, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, c_codes, 2, cdims, cbox, CU_TENSOR_MAP_SWIZZLE_32B))
    return MOE_ERR_INVALID_ARG;
  Params p{offsets, M, N, K, E, c_codes, nullptr, nullptr, c_scales, dev_status};
  if (sw) return launch<2, kFwd, kEpiSwiglu, uint8_t>(ta, tb, p, stream, sms, fn, &tsa, &tsb, &td);
  return launch<2, kFwd, kEpiNone, uint8_t>(ta, tb, p, stream, sms, fn, &tsa, &tsb, &td);
}

extern "C" moe_status_t moe_grouped_gemm_dgrad(const moe_operand_t* dC, const moe_operand_t* B,
                                               const int32_t* offsets, int M, int N, int K, int E,
                                               moe_epilogue_t epi, const void* preact, void* dA,
                                               moe_dtype_t dA_dtype, int32_t* dev_status,
                                               cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_grouped_gemm_dgrad");
  const char* fn = "moe_grouped_gemm_dgrad";
  int sms = 0;
  moe_status_t st = common_checks(fn, dC, B, offsets, M, N, K, E, dA, &sms);
  if (st != MOE_OK) return st;
  if (dC->dtype != MOE_BF16 || dA_dtype != MOE_BF16) {
    set_error("%s: BF16 operands and output only", fn);
    return MOE_ERR_UNSUPPORTED;
  }
  if ((epi != MOE_EPI_NONE && epi != MOE_EPI_DSWIGLU) ||
      (epi == MOE_EPI_DSWIGLU && (!preact || !aligned16(preact)))) {
    set_error("%s: epi NONE|DSWIGLU (DSWIGLU needs an aligned preact [M, 2K])", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (M == 0) return MOE_OK;
  CUtensorMap ta, tb;
  const uint64_t adims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M)};
  const uint32_t abox[2] = {64, static_cast<uint32_t>(epi == MOE_EPI_DSWIGLU ? kBM : kWideM)};   // plain: wide tile
  const uint64_t bdims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(E)};
  const uint32_t bbox[3] = {64, kMnRows, 1};
  if (!make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dC->ptr, 2, adims, abox) ||
      !make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B->ptr, 3, bdims, bbox))
    return MOE_ERR_INVALID_ARG;
  Params p{offsets, M, N, K, E, dA, nullptr, preact, nullptr, dev_status};
  if (epi == MOE_EPI_DSWIGLU) return launch<1, kDgrad, kEpiDswiglu, uint16_t>(ta, tb, p, stream, sms, fn);
  // plain (wide tile): dA [M, K] is written by TMA from 32-row x 32-column staging boxes
  // (64-byte rows, 64-byte swizzle), as the forward output is
  CUtensorMap td;
  const uint64_t cdims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
  const uint32_t cbox[2] = {kEpiRowBytes / 2, 32};
  if (!make_map(&td, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dA, 2, cdims, cbox, CU_TENSOR_MAP_SWIZZLE_64B))
    return MOE_ERR_INVALID_ARG;
  return launch<1, kDgrad, kEpiNone, uint16_t>(ta, tb, p, stream, sms, fn, nullptr, nullptr, &td);
}

extern "C" moe_status_t moe_grouped_gemm_dgrad_mxfp8(const moe_operand_t* dC, const moe_operand_t* BT,
                                                     const int32_t* offsets, int M, int N, int K, int E,
                                                     moe_epilogue_t epi, const void* preact, void* dA,
                                                     int32_t* dev_status, cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_grouped_gemm_dgrad_mxfp8");
  // dA[R_e] = dC[R_e] @ B[e] with both operands quantised along the contraction dim N:
  // dC codes [M, N] (scales [M, N/32]) and B^T codes [E, K, N] (scales [E*K, N/32]).
  // That is the forward problem with N and K swapped, so the forward MXFP8 kernel runs it.
  const char* fn = "moe_grouped_gemm_dgrad_mxfp8";
  int sms = 0;
  moe_status_t st = common_checks(fn, dC, BT, offsets, M, N, K, E, dA, &sms);
  if (st != MOE_OK) return st;
  if (dC->dtype != MOE_E4M3) {
    set_error("%s: MXFP8 (E4M3) operands only", fn);
    return MOE_ERR_UNSUPPORTED;
  }
  if ((epi != MOE_EPI_NONE && epi != MOE_EPI_DSWIGLU) ||
      (epi == MOE_EPI_DSWIGLU && (!preact || !aligned16(preact))) || N % 512 || !dC->scales || !BT->scales ||
      !aligned16(dC->scales) || !aligned16(BT->scales)) {
    set_error("%s: epi NONE|DSWIGLU (DSWIGLU needs an aligned preact [M, 2K]), N %% 512 == 0, aligned scales", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (M == 0) return MOE_OK;
  CUtensorMap ta, tb, tsa, tsb, td;
  const uint64_t adims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M)};
  const uint32_t abox[2] = {kBKBytes, kBM};
  const uint64_t bdims[3] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K), static_cast<uint64_t>(E)};
  const uint32_t bbox[3] = {kBKBytes, kBN, 1};
  const uint64_t sadims[2] = {static_cast<uint64_t>(N / 32), static_cast<uint64_t>(M)};
  const uint64_t sbdims[2] = {static_cast<uint64_t>(N / 32), static_cast<uint64_t>(K) * static_cast<uint64_t>(E)};
  const uint32_t sbox[2] = {16, kBM};
  const uint64_t cdims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
  const uint32_t cbox[2] = {16, 32};   // 32-byte rows, 32-byte swizzle
  if (!make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, dC->ptr, 2, adims, abox) ||
      !make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, BT->ptr, 3, bdims, bbox) ||
      !make_map(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, dC->scales, 2, sadims, sbox, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map(&tsb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, BT->scales, 2, sbdims, sbox, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map(&td, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dA, 2, cdims, cbox, CU_TENSOR_MAP_SWIZZLE_32B))
    return MOE_ERR_INVALID_ARG;
  Params p{offsets, M, K, N, E, dA, nullptr, preact, nullptr, dev_status};
  if (epi == MOE_EPI_DSWIGLU) return launch<2, kFwd, kEpiDswiglu, uint16_t>(ta, tb, p, stream, sms, fn, &tsa, &tsb, &td);
  return launch<2, kFwd, kEpiNone, uint16_t>(ta, tb, p, stream, sms, fn, &tsa, &tsb, &td);
}

extern "C" moe_status_t moe_route_topk_gemm(const void* x, const void* w_router, moe_dtype_t dtype, int T,
                                            int d, int E, int k, int renormalize, float* logits,
                                            int32_t* topk_idx, float* topk_w, int32_t* counts,
                                            int32_t* dev_status, cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_route_topk_gemm");
  // logits = x . W_r^T on the tensor cores, top-k selection and softmax weights in
  // the GEMM epilogue: the logits need not make a round trip through memory.
  const char* fn = "moe_route_topk_gemm";
  if (T < 0 || d <= 0 || d % 32 || E < 1 || E > kBN || k < 1 || k > E || k > kTopkMax ||
      (dtype != MOE_BF16 && dtype != MOE_F32)) {
    set_error("%s: need T >= 0, d %% 32 == 0, 1 <= E <= %d, 1 <= k <= min(E, %d), BF16 or F32 (T=%d d=%d E=%d k=%d)",
              fn, kBN, kTopkMax, T, d, E, k);
    return MOE_ERR_INVALID_ARG;
  }
  if (!counts || (T > 0 && (!x || !w_router || !topk_idx || !topk_w)) || !aligned16(x) || !aligned16(w_router) ||
      !aligned16(logits)) {
    set_error("%s: null or misaligned pointer", fn);
    return MOE_ERR_INVALID_ARG;
  }
  int sms = 0;
  if (const moe_status_t dst = device_check(&sms); dst != MOE_OK) return dst;
  cudaError_t e = cudaMemsetAsync(counts, 0, static_cast<size_t>(E) * sizeof(int32_t), stream);
  if (e != cudaSuccess) {
    set_error("%s: cudaMemsetAsync: %s", fn, cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  if (T == 0) return MOE_OK;
  const int eb = elem_bytes(dtype);
  const uint32_t bk = kBKBytes / eb;
  CUtensorMap ta, tb;
  const uint64_t adims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(T)};
  const uint32_t abox[2] = {bk, kBM};
  const uint64_t bdims[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(E), 1};
  const int n_mma = ((E + 15) / 16) * 16;          // MMA width: E rounded up to 16
  const uint32_t bbox[3] = {bk, static_cast<uint32_t>(n_mma), 1};   // rows past E read as zeros
  if (!make_map(&ta, map_type(dtype), eb, x, 2, adims, abox) ||
      !make_map(&tb, map_type(dtype), eb, w_router, 3, bdims, bbox))
    return MOE_ERR_INVALID_ARG;
  // One CTA per tile (the epilogue stages the tile's logits in the operand stages),
  // or, when the tiles leave SMs idle, a cluster of `split` CTAs per tile, each
  // taking one run of the contraction (at least kMinSliceBlocks K blocks) and the
  // selection of 128 / split of its rows; every cluster owns exactly one tile.
  const int tiles = (T + kBM - 1) / kBM;
  const int kblocks = (d * eb + kBKBytes - 1) / kBKBytes;
  int split = 1;
  for (int c = kMaxSplit; c > 1; c /= 2)
    if (tiles * c <= sms && kblocks >= c * kMinSliceBlocks) {
      split = c;
      break;
    }
  Params p{nullptr, T, E, d, 1, logits, nullptr, nullptr, nullptr, dev_status, nullptr, nullptr, nullptr, nullptr,
           topk_idx, topk_w, counts, k, renormalize ? 1 : 0, n_mma, split};
  const int grid = tiles * split;
  if (dtype == MOE_F32) return launch<0, kFwd, kEpiTopk, float>(ta, tb, p, stream, grid, fn, nullptr, nullptr, nullptr, split);
  return launch<1, kFwd, kEpiTopk, float>(ta, tb, p, stream, grid, fn, nullptr, nullptr, nullptr, split);
}

extern "C" moe_status_t moe_grouped_gemm_wgrad(const moe_operand_t* A, const moe_operand_t* dC,
                                               const int32_t* offsets, int M, int N, int K, int E,
                                               int accumulate, void* dB, moe_dtype_t dB_dtype,
                                               int32_t* dev_status, cudaStream_t stream) {
  const moe::NvtxRange nvtx_range("moe_grouped_gemm_wgrad");
  const char* fn = "moe_grouped_gemm_wgrad";
  int sms = 0;
  moe_status_t st = common_checks(fn, A, dC, offsets, M, N, K, E, dB, &sms);
  if (st != MOE_OK) return st;
  if ((A->dtype != MOE_BF16 && A->dtype != MOE_E4M3) || (dB_dtype != MOE_BF16 && dB_dtype != MOE_F32)) {
    set_error("%s: BF16 or MXFP8 (E4M3) operands, BF16 or F32 output", fn);
    return MOE_ERR_UNSUPPORTED;
  }
  if (accumulate && dB_dtype != MOE_F32) {
    set_error("%s: accumulating needs an F32 dB (one rounding per element)", fn);
    return MOE_ERR_INVALID_ARG;
  }
  // dB [E, N, K] is written by TMA from 32-row staging boxes of 64-byte rows (64-byte
  // swizzle): 32 bf16 or 16 fp32 columns
  const bool f32 = dB_dtype == MOE_F32;
  CUtensorMap td;
  const uint64_t ddims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(E)};
  const uint32_t dbox[3] = {f32 ? 16u : 32u, 32, 1};
  if (!make_map(&td, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, f32 ? 4 : 2, dB, 3,
                ddims, dbox, CU_TENSOR_MAP_SWIZZLE_64B))
    return MOE_ERR_INVALID_ARG;
  if (A->dtype == MOE_E4M3) {
    // Both operands quantised column-wise (group-aware, along the rows), scales in
    // the tiled layout; read as 128 x 128 MN-major boxes (128-byte swizzle).
    if (N % 128 || K % 128 || (M > 0 && (!A->scales || !dC->scales)) || !aligned16(A->scales) ||
        !aligned16(dC->scales)) {
      set_error("%s: MXFP8 needs N %% 128 == 0, K %% 128 == 0 and 16-byte aligned tiled scales", fn);
      return MOE_ERR_INVALID_ARG;
    }
    CUtensorMap ta, tb;
    const uint64_t cdims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M > 0 ? M : 1)};
    const uint64_t adims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M > 0 ? M : 1)};
    const uint32_t box[2] = {128, kMxWgRows};
    const void* cptr = dC->ptr ? dC->ptr : dB;
    const void* aptr = A->ptr ? A->ptr : dB;
    if (!make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, cptr, 2, cdims, box) ||
        !make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, aptr, 2, adims, box))
      return MOE_ERR_INVALID_ARG;
    Params p{offsets, M, N, K, E, dB, nullptr, nullptr, nullptr, dev_status,
             static_cast<const uint8_t*>(dC->scales), static_cast<const uint8_t*>(A->scales)};
    p.accumulate = accumulate ? 1 : 0;
    if (f32) return launch<2, kWgrad, kEpiNone, float>(ta, tb, p, stream, sms, fn, nullptr, nullptr, &td);
    return launch<2, kWgrad, kEpiNone, uint16_t>(ta, tb, p, stream, sms, fn, nullptr, nullptr, &td);
  }
  CUtensorMap ta, tb;
  // The MMA's A operand is dC^T (rows n, contraction over the group's rows); its
  // B operand is A.  Both are read as 64 x 64 MN-major boxes.
  const uint64_t cdims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M > 0 ? M : 1)};
  const uint64_t adims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M > 0 ? M : 1)};
  const uint32_t box[2] = {64, kMnRows};
  const void* cptr = dC->ptr ? dC->ptr : dB;   // M == 0: never read, only a valid address
  const void* aptr = A->ptr ? A->ptr : dB;
  if (!make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cptr, 2, cdims, box) ||
      !make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, aptr, 2, adims, box))
    return MOE_ERR_INVALID_ARG;
  Params p{offsets, M, N, K, E, dB, nullptr, nullptr, nullptr, dev_status};
  p.accumulate = accumulate ? 1 : 0;
  if (f32) return launch<1, kWgrad, kEpiNone, float>(ta, tb, p, stream, sms, fn, nullptr, nullptr, &td);
  return launch<1, kWgrad, kEpiNone, uint16_t>(ta, tb, p, stream, sms, fn, nullptr, nullptr, &td);
}

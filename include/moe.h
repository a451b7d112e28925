/*
 * moe.h -- C ABI of libmoe: the single-GPU hot path of dropless Mixture-of-Experts
 * training on GB300 (sm_103a).
 *
 * The operations follow the dropless-MoE layer described in
 *   [1] "Accelerating Dropless MoE Training in JAX with NVIDIA Transformer Engine"
 *       (NVIDIA technical blog; zhiding.cn rewrite), and
 *   [3] a deep reading of arXiv 2603.07685 (paper-daily.com), "Method overview":
 *       Route -> Dispatch -> Compute -> Combine.
 * The pages give no formulas; where they leave a step open the plainest reading
 * is taken and stated next to the function.
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers owned by the caller unless stated otherwise.
 *     The library never allocates device memory; scratch comes from the caller
 *     (query the size with the matching *_workspace_size function).
 *   - Every call is asynchronous on `stream` (0 = legacy default stream).  No call
 *     synchronises the host or copies data back to it; per-expert counts and
 *     offsets live only on the device, so a whole layer can be captured in a
 *     CUDA graph ([1] "What dropless MoE needs": the CPU never learns the shapes).
 *   - Shapes (T tokens, d model dim, E experts, k experts per token, f expert
 *     hidden dim) are host ints.  Matrices are row-major and densely packed.
 *   - Host-side argument errors return a status and launch nothing; the message
 *     is kept in moe_last_error_string() (per thread).
 *   - `dev_status` (may be NULL) is a device int32 that kernels OR error bits
 *     into (MOE_DEV_*).  Kernels never trap; the caller reads the word when it
 *     wants to know.  Zero it once before use.
 *   - Calls on the same stream may reuse each other's outputs; calls that run
 *     concurrently must not share output or workspace buffers.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* bad shape, null or misaligned pointer, bad enum */
  MOE_ERR_UNSUPPORTED = 2, /* device is not sm_103 / dtype combination not built */
  MOE_ERR_CUDA = 3,        /* a CUDA call or kernel launch failed */
  MOE_ERR_WORKSPACE = 4    /* caller workspace too small */
} moe_status_t;

typedef enum {
  MOE_F32 = 0,  /* float32 storage (GEMMs run on the tensor cores as TF32) */
  MOE_BF16 = 1, /* bfloat16 */
  MOE_E4M3 = 2, /* MXFP8: FP8 E4M3 codes plus one E8M0 scale byte per 32 elements */
  MOE_E2M1 = 3  /* NVFP4: E2M1 codes two per byte, one E4M3 scale byte per 16 elements
                   and one fp32 tensor scale (moe_quantize_nvfp4) */
} moe_dtype_t;

typedef enum {
  MOE_EPI_NONE = 0,
  MOE_EPI_SWIGLU = 1,  /* forward GEMM1: out = silu(gate) * up                */
  MOE_EPI_DSWIGLU = 2  /* dgrad of GEMM2: out = d(gate, up) from dH and (G, U)  */
} moe_epilogue_t;

/* Device-side error bits OR-ed into *dev_status. */
#define MOE_DEV_NAN_LOGIT 1 /* a router logit was NaN (outside the router's domain) */
#define MOE_DEV_BAD_INDEX 2 /* an expert id / row index outside its range, or counts
                               inconsistent with topk_idx                        */
#define MOE_DEV_TIMEOUT 4   /* a bounded pipeline wait gave up; outputs are garbage */
#define MOE_DEV_ASSERT 8    /* a MOE_DEBUG build's device-side check failed; the
                               access it guards was skipped, outputs are garbage */

/* One GEMM operand.  For MOE_E4M3, `scales` points at the E8M0 bytes, one per 32
 * consecutive elements along the contraction dimension ([rows, K/32] row-major).
 * For MOE_E2M1, `ptr` holds the packed codes [rows, K/2], `scales` the E4M3 bytes
 * [rows, K/16] and `tensor_scale` the fp32 encode scale g of the tensor (as written
 * by moe_quantize_nvfp4).  Both are ignored (may be NULL) for the other dtypes. */
typedef struct {
  const void* ptr;
  moe_dtype_t dtype;
  const uint8_t* scales;
  const float* tensor_scale;
} moe_operand_t;

int moe_version(void);                    /* (major << 16) | (minor << 8) | patch */
const char* moe_last_error_string(void);  /* message of this thread's last error */

/* Diagnostic with no counterpart in the pages: exercises the failure path of the
 * bounded pipeline wait that every GEMM stage uses.  One CTA waits on a barrier
 * nothing arrives at; after limit_us microseconds (1 .. 2e6) the wait gives up,
 * ORs MOE_DEV_TIMEOUT into *dev_status and the kernel returns, leaving the CUDA
 * context usable.  Asynchronous on `stream`. */
moe_status_t moe_check_wait_timeout(int32_t* dev_status, int limit_us, cudaStream_t stream);

/* Diagnostic: whether this library is a MOE_DEBUG build (compiled with -DMOE_DEBUG).
 * Such a build adds device-side checks of the kernels' invariants (TMA coordinate
 * alignment and ranges, tile bounds, staging offsets) that OR MOE_DEV_ASSERT into
 * dev_status and skip the access they guard instead of trapping.  This call launches
 * one check that always fails: a debug build sets MOE_DEV_ASSERT in *dev_status, a
 * release build (whose checks compile to nothing) leaves it unchanged.  Asynchronous
 * on `stream`; *is_debug (host) receives 1 for a debug build, else 0. */
moe_status_t moe_debug_selftest(int32_t* dev_status, int* is_debug, cudaStream_t stream);

/* ---------------------------------------------------------------- route ----
 * Top-k expert selection with softmax routing weights ([1] opening section: a
 * learnable router activates the top-K experts of each token; [1] "Optimisation
 * 2": a fused router kernel assigns every token its experts before dispatch).
 *
 * logits    [T, E] float32.  -inf is allowed (a masked expert); NaN sets
 *           MOE_DEV_NAN_LOGIT.
 * topk_idx  [T, k] int32 out: slot j holds the j-th largest logit's expert;
 *           equal logits go to the lower expert id.
 * topk_w    [T, k] float32 out: renormalize != 0 -> softmax over the k selected
 *           logits (sums to 1); renormalize == 0 -> full-softmax probability of
 *           each selected expert.
 * counts    [E] int32 out: tokens routed to each expert (zeroed inside; the sum
 *           is T*k: dropless, nothing is dropped or padded).
 * Limits: 1 <= E <= 1024, 1 <= k <= min(E, 32), T >= 0.
 */
moe_status_t moe_route_topk(const float* logits, int T, int E, int k, int renormalize,
                            int32_t* topk_idx, float* topk_w, int32_t* counts,
                            int32_t* dev_status, cudaStream_t stream);

/* Router GEMM fused with the top-k selection ([1] "Optimisation 2": the fused
 * router kernel; [1] opening section: the router scores each token against every
 * expert).  logits = x . W_r^T on the tensor cores, then, in the GEMM epilogue,
 * the selection and weights of moe_route_topk on those fp32 logits (same rules:
 * value descending, lower expert id first on ties, -inf masked, NaN flagged).
 *   x         [T, d] in dtype (MOE_BF16, or MOE_F32 computed as TF32), 16-byte aligned.
 *   w_router  [E, d] in dtype.
 *   logits    [T, E] float32 out, or NULL (the logits then never reach memory;
 *             the router backward with renormalize == 0 needs them).
 *   topk_idx, topk_w, counts: as moe_route_topk (counts zeroed inside).
 * The MMA is E (rounded up to 16) columns wide; one 128-token tile per CTA, or,
 * when the tiles would leave SMs idle, per thread-block cluster of 2 or 4 CTAs that
 * split the contraction: the partial logits are summed in slice order through
 * distributed shared memory, so the logits are the same from call to call.
 * Limits: d % 32 == 0, 1 <= E <= 256, 1 <= k <= min(E, 8), T >= 0. */
moe_status_t moe_route_topk_gemm(const void* x, const void* w_router, moe_dtype_t dtype, int T, int d,
                                 int E, int k, int renormalize, float* logits, int32_t* topk_idx,
                                 float* topk_w, int32_t* counts, int32_t* dev_status,
                                 cudaStream_t stream);

/* ---------------------------------------------------------------- dispatch --
 * Local dispatch: reorder the T*k (token, slot) pairs into expert-contiguous
 * rows ([1] "Optimisation 2": dispatch rearranges tokens locally; Figure 3).
 * Rows are ordered by (expert, token), unpadded: expert e owns rows
 * [offsets[e], offsets[e+1]).
 *
 * x         [T, d] in x_dtype (MOE_F32 or MOE_BF16).
 * topk_idx  [T, k] int32 from moe_route_topk; counts [E] int32 likewise.
 * offsets   [E+1] int32 out: exclusive scan of counts, offsets[E] = T*k.
 * dest_row  [T, k] int32 out: row that pair (t, j) was written to.
 * src_pair  [T*k] int32 out: pair t*k+j held by each row (inverse of dest_row).
 * xp        [T*k, d] out, or NULL for the maps only.  xp_dtype == x_dtype copies
 *           rows bit-exactly; xp_dtype == MOE_E4M3 (x must be MOE_BF16 or
 *           MOE_F32, d % 32 == 0) quantises each row to MXFP8 on the way
 *           ([1] "What dropless MoE needs": group-aware MXFP8 quantisation; a
 *           row-wise 32-element block never spans two experts), writing codes
 *           to xp and E8M0 scales to xp_scales [T*k, d/32].
 * workspace moe_permute_workspace_size(T, k, E) bytes of device scratch.
 * Limits: E <= 1024, k <= 32, d % 8 == 0 (16-byte rows), 16-byte aligned rows.
 */
size_t moe_permute_workspace_size(int T, int k, int E);
moe_status_t moe_permute(const void* x, moe_dtype_t x_dtype, int T, int d,
                         const int32_t* topk_idx, int k, int E, const int32_t* counts,
                         int32_t* offsets, int32_t* dest_row, int32_t* src_pair,
                         void* xp, moe_dtype_t xp_dtype, uint8_t* xp_scales,
                         void* workspace, size_t workspace_bytes,
                         int32_t* dev_status, cudaStream_t stream);

/* Allocation-free variant of moe_permute.  The pages have no counterpart: it
 * exists for callers that cannot allocate device memory -- a plugin that is only
 * handed input and output pointers by the runtime that owns the allocator, a
 * serving process whose device memory is all reserved up front by its own pool,
 * or code that must not allocate while a stream is being captured.  Arguments,
 * layouts, outputs and errors are those of moe_permute, without the workspace.
 *
 * Scratch: a fixed 1 MiB array inside the library's own device memory (held on
 * every GPU that loads the library until the process exits).  The call needs
 * ceil(T / 256) * E int32 of it and returns MOE_ERR_WORKSPACE beyond 262144
 * (T = 65536 tokens with E = 1024 experts fits exactly).  It allocates nothing
 * and frees nothing.
 * All calls share the one array: calls whose kernels can overlap on the GPU
 * (other streams, other host threads) race and give wrong results -- serialise
 * them.  The first call in a CUDA context (normally once per device; again
 * after that device's primary context was reset) looks up the array's device
 * address; make that first call before any stream capture. */
moe_status_t moe_permute_noalloc(const void* x, moe_dtype_t x_dtype, int T, int d,
                                 const int32_t* topk_idx, int k, int E, const int32_t* counts,
                                 int32_t* offsets, int32_t* dest_row, int32_t* src_pair,
                                 void* xp, moe_dtype_t xp_dtype, uint8_t* xp_scales,
                                 int32_t* dev_status, cudaStream_t stream);

/* ---------------------------------------------------------------- quantise --
 * Group-aware MXFP8 quantisation ([1] "What dropless MoE needs" and
 * "Optimisation 1": MXFP8 block scaling of the expert matmuls; [3] contribution
 * 3: grouped quantisation for dynamic shapes).  Encoding per the OCP MX v1.0
 * definition: per block of 32 elements along a row, X = floor(log2 amax) - 8
 * clamped to [-127, 127] (an all-zero block gets X = 0), scale byte X + 127,
 * codes = round-to-nearest-even(v / 2^X) to E4M3, saturated to +-448.
 *
 * in     [rows, K] MOE_BF16 or MOE_F32; K % 32 == 0.
 * codes  [rows, K] uint8 out (both axes).
 * axis   0 = row-wise: blocks of 32 along a row (the forward operands);
 *        scales [rows, K/32] uint8 out.  Row-wise blocks lie inside one row and so
 *        inside one group; offsets may be NULL.
 *        1 = column-wise, group-aware (the operands that contract over rows, as in
 *        the weight gradient): blocks of 32 consecutive rows of one column that
 *        restart at every group start ([1] "grouped quantisation"); a group's last
 *        partial block is zero-padded (the padding has no codes).  offsets [E+1]
 *        (device, as from moe_permute) and 1 <= E <= 1024 required.  scales
 *        [n_blocks, K] uint8 out with group e's blocks from row sum over e' < e of
 *        ceil(count_e' / 32); the caller's buffer must hold ceil(rows/32) + E rows
 *        (the bound on n_blocks); rows past n_blocks are not written.
 *        2 = column-wise as axis 1 (same codes, same scale values), the scales laid
 *        out for the MXFP8 weight-gradient GEMM, which copies them into tensor
 *        memory as they are: group e's blocks taken four at a time (quads of 128
 *        rows), quad q of group e numbered Q = floor(offsets[e] / 128) + e + q; the
 *        scales of quad Q and columns [128c, 128c + 128) are one 512-byte tile at
 *        byte ((Q * K/128) + c) * 512, column m of the 128 and block j of the quad
 *        at (m % 32) * 16 + (m / 32) * 4 + j.  K % 128 == 0; the buffer must hold
 *        (ceil(rows/128) + E) * K/128 tiles; bytes of blocks past a group's last
 *        one are not written.
 * MOE_ERR_UNSUPPORTED for any other axis.
 */
moe_status_t moe_quantize_mxfp8_grouped(const void* in, moe_dtype_t in_dtype, int rows, int K,
                                        const int32_t* offsets, int E, int axis,
                                        uint8_t* codes, uint8_t* scales,
                                        cudaStream_t stream);

/* Column-wise, group-aware MXFP8 of the dispatched rows without materialising them
 * (MXFP8 training: the weight gradient of GEMM1 reads Xp column-wise, and nothing
 * else needs Xp in bf16 once the dispatch writes its row-wise MXFP8 form).  The
 * rows are Xp[r] = x[src_pair[r] / k], r < T*k, as moe_permute would write them;
 * the result equals moe_quantize_mxfp8_grouped (axis 1 or 2) of that Xp, bit for
 * bit ([1] "What dropless MoE needs": grouped quantisation of the expert inputs).
 *   x         [T, K] MOE_BF16 or MOE_F32 token rows, 16-byte aligned; K % 32 == 0
 *             (axis 2: K % 128 == 0).
 *   k         top-k (1..32); src_pair [T*k] and offsets [E+1] from moe_permute.
 *   row_w     optional [T*k] fp32 per-pair weights (the routing weights): the rows
 *             are then w[src_pair[r]] * x[src_pair[r] / k], the product taken in
 *             fp32 and rounded to x's dtype -- the dYp of moe_unpermute_combine_bwd,
 *             whose column-wise MXFP8 this gives without dYp being stored.
 *   axis      1 or 2, codes [T*k, K] and scales as for moe_quantize_mxfp8_grouped.
 *   dev_status  optional: a src_pair entry outside [0, T*k) sets MOE_DEV_BAD_INDEX
 *             and its row is quantised as zeros.
 * MOE_ERR_UNSUPPORTED for any other axis; T == 0 or K == 0 is a no-op. */
moe_status_t moe_quantize_mxfp8_gathered(const void* x, moe_dtype_t x_dtype, int T, int K, int k,
                                         const int32_t* src_pair, const float* row_w,
                                         const int32_t* offsets, int E,
                                         int axis, uint8_t* codes, uint8_t* scales,
                                         int32_t* dev_status, cudaStream_t stream);

/* Transposed row-wise MXFP8 of a batch of matrices, for weights that a gradient
 * contracts along their first dim (the data gradient contracts B [E, N, K] over N):
 *   in     [G, R, C] MOE_BF16 or MOE_F32, 16-byte aligned; R % 32 == 0, C % 8 == 0.
 *   codes  [G, C, R] uint8 out (E4M3): codes[g, c, r] encodes in[g, r, c].
 *   scales [G * C, R / 32] uint8 out (E8M0), blocks of 32 along R.
 * The result equals moe_quantize_mxfp8_grouped (axis 0) of each in[g]^T, bit for bit.
 * Stateless: no workspace; G, R or C == 0 is a no-op. */
moe_status_t moe_quantize_mxfp8_transposed(const void* in, moe_dtype_t in_dtype, int G, int R, int C,
                                           uint8_t* codes, uint8_t* scales, cudaStream_t stream);

/* NVFP4 quantisation ([3] contribution 3 names NVFP4 as the Blackwell FP4 recipe;
 * the encoding follows NVIDIA's published NVFP4 format): E2M1 elements, one E4M3
 * scale per 16 consecutive elements of a row, one fp32 scale for the tensor.  All
 * rounding that decides a code is fp32, in this order: g = 2688 / amax(tensor)
 * (1 for an all-zero tensor); s = E4M3_rn_sat((amax_block / 6) * g); code =
 * E2M1_rn_sat(v * (g / s)) (v * 0 when s decodes to 0); decoded v = e2m1 * s / g.
 *   in      [rows, K] MOE_BF16 or MOE_F32, 16-byte aligned; K % 16 == 0.
 *   codes   [rows, K/2] uint8 out, two codes per byte (element 2i in the low
 *           nibble), 8-byte aligned.
 *   scales  [rows, K/16] uint8 out (E4M3, sign bit clear).
 *   tensor_scale  float[2] device: [0] receives g; [1] is scratch for the amax.
 * A weight stack [E, N, K] is one tensor (rows = E*N): one g for all experts. */
moe_status_t moe_quantize_nvfp4(const void* in, moe_dtype_t in_dtype, int rows, int K, uint8_t* codes,
                                uint8_t* scales, float* tensor_scale, cudaStream_t stream);

/* Dispatch with NVFP4 rows: moe_permute's maps, and instead of bf16 rows the NVFP4
 * codes [T*k, d/2] and scales [T*k, d/16] of the permuted rows, bit-identical to
 * moe_quantize_nvfp4 of moe_permute's rows (the tensor amax of x is that of the
 * permuted rows: every token is routed).  x is read twice (its amax, then the
 * scatter); the bf16 rows are never written.  tensor_scale as moe_quantize_nvfp4.
 * d % 16 == 0; codes 4-byte aligned; workspace as moe_permute. */
moe_status_t moe_permute_nvfp4(const void* x, moe_dtype_t x_dtype, int T, int d, const int32_t* topk_idx,
                               int k, int E, const int32_t* counts, int32_t* offsets, int32_t* dest_row,
                               int32_t* src_pair, uint8_t* xp_codes, uint8_t* xp_scales, float* tensor_scale,
                               void* workspace, size_t workspace_bytes, int32_t* dev_status,
                               cudaStream_t stream);

/* ---------------------------------------------------------------- grouped GEMM
 * Ragged grouped GEMM ([1] "Optimisation 1": one kernel launch covers every
 * expert and computes only the valid token rows of each; the per-expert sizes
 * are read on the device, never copied to the host).  Persistent tcgen05/TMEM
 * kernel fed by TMA.  Rows of expert e are [offsets[e], offsets[e+1]); rows at
 * or beyond offsets[E] are not written.
 *
 * Forward: C[r, :] = A[r, :] . B[e]^T for r in expert e's rows.
 *   A [M, K] (A->dtype), B [E, N, K] (same dtype), accumulate in fp32.
 *   epi == MOE_EPI_NONE:   C [M, N] in c_dtype (MOE_BF16 or MOE_F32).
 *   epi == MOE_EPI_SWIGLU: N = 2f with rows 0..f-1 of B[e] the gate projection
 *     and f..2f-1 the up projection; C [M, f] = silu(A.Bg^T) * (A.Bu^T).  If
 *     preact != NULL the pre-activations [M, 2f] (gate | up) are stored too, in
 *     c_dtype, for the backward.
 * dtypes: F32 x F32 (TF32 tensor cores), BF16 x BF16, E4M3 x E4M3 (MXFP8 with
 *   E8M0 scales per 32 along K; both scale pointers required), E2M1 x E2M1
 *   (NVFP4: E4M3 scales per 16 along K and the two tensor scales; the product is
 *   multiplied by 1 / (g_A * g_B) before the epilogue; K % 256 == 0).
 * Limits: K % 32 == 0, N % 32 == 0 (SWIGLU: f % 32 == 0), E <= 1024,
 *   16-byte aligned pointers, M < 2^31.
 */
moe_status_t moe_grouped_gemm_fwd(const moe_operand_t* A, const moe_operand_t* B,
                                  const int32_t* offsets, int M, int N, int K, int E,
                                  moe_epilogue_t epi, void* C, moe_dtype_t c_dtype,
                                  void* preact, int32_t* dev_status, cudaStream_t stream);

/* Forward with MXFP8 output ([1] lists quantisation fused with the GEMM as
 * planned work; this is that fusion): as moe_grouped_gemm_fwd with E4M3 operands,
 * but the result (SWIGLU: H [M, f]; NONE: C [M, N]) leaves the epilogue quantised
 * row-wise to MXFP8, ready to be the A operand of the next forward GEMM.  Each
 * value is rounded to bf16 first, so codes and scales equal those of a bf16
 * result passed through moe_quantize_mxfp8_grouped.
 *   c_codes  [M, n_out] uint8 (E4M3), 16-byte aligned; c_scales [M, n_out / 32]
 *            uint8 (E8M0).  Rows outside every group are not written.
 * Limits as moe_grouped_gemm_fwd; A and B must be MOE_E4M3 (MOE_ERR_UNSUPPORTED
 * otherwise). */
moe_status_t moe_grouped_gemm_fwd_mxfp8_out(const moe_operand_t* A, const moe_operand_t* B,
                                            const int32_t* offsets, int M, int N, int K, int E,
                                            moe_epilogue_t epi, uint8_t* c_codes, uint8_t* c_scales,
                                            int32_t* dev_status, cudaStream_t stream);

/* Data gradient: dA[r, :] = dC[r, :] . B[e] for r in expert e's rows.
 *   dC [M, N], B [E, N, K] (both MOE_BF16 or both MOE_F32) -> dA [M, K] in dA_dtype.
 *   epi == MOE_EPI_DSWIGLU fuses the SwiGLU backward: the product is dH [M, K]
 *     and `preact` [M, 2K] holds the forward pre-activations (gate | up); the
 *     output is dA = [dG | dU] of shape [M, 2K] with
 *     dG = dH * U * s * (1 + G * (1 - s)), s = sigmoid(G), dU = dH * silu(G).
 * Limits as the forward. */
moe_status_t moe_grouped_gemm_dgrad(const moe_operand_t* dC, const moe_operand_t* B,
                                    const int32_t* offsets, int M, int N, int K, int E,
                                    moe_epilogue_t epi, const void* preact,
                                    void* dA, moe_dtype_t dA_dtype,
                                    int32_t* dev_status, cudaStream_t stream);

/* MXFP8 data gradient ([1] "Optimisation 1" with block-scaled operands; the
 * backward of the MXFP8 forward): dA[r, :] = dC[r, :] . B[e] for r in expert e's
 * rows, with both operands quantised along the contraction dim N.
 *   dC  MOE_E4M3 codes [M, N], scales [M, N/32] (moe_quantize_mxfp8_grouped, axis 0).
 *   BT  MOE_E4M3 codes [E, K, N] = B^T, scales [E*K, N/32]
 *       (moe_quantize_mxfp8_transposed of B [E, N, K]).
 *   dA  bf16 [M, K] (NONE) or [M, 2K] = [dG | dU] (DSWIGLU, with `preact` the
 *       bf16 forward pre-activations [M, 2K], formula as moe_grouped_gemm_dgrad).
 * Limits: N % 512 == 0, K % 32 == 0, E <= 1024, 16-byte aligned pointers and
 * scales; MOE_ERR_UNSUPPORTED unless both operands are MOE_E4M3. */
moe_status_t moe_grouped_gemm_dgrad_mxfp8(const moe_operand_t* dC, const moe_operand_t* BT,
                                          const int32_t* offsets, int M, int N, int K, int E,
                                          moe_epilogue_t epi, const void* preact, void* dA,
                                          int32_t* dev_status, cudaStream_t stream);

/* Weight gradient: dB[e] = dC[R_e]^T . A[R_e], a contraction over the ragged rows
 * R_e of each expert; an expert with no rows gets an exact zero gradient.
 *   A [M, K], dC [M, N], both MOE_BF16 -> dB [E, N, K] in dB_dtype (MOE_BF16 or
 *   MOE_F32, the fp32 accumulator as it is).
 *   Or both MOE_E4M3 ([1] "grouped quantisation": the blocks of 32 run down the
 *   contraction, restarting at each group): codes and tiled scales from
 *   moe_quantize_mxfp8_grouped axis 2 of A and of dC (scales required);
 *   N % 128 == 0 and K % 128 == 0.
 *   accumulate != 0 (dB_dtype MOE_F32 only, else MOE_ERR_INVALID_ARG): dB[e] +=
 *   the product instead, each element with one fp32 rounding of (dB + product), for
 *   gradients summed over several batches; an expert with no rows keeps its dB
 *   unchanged.  Each element belongs to one output tile, so a call adds to it once:
 *   the result does not depend on the order the tiles run in.
 * Limits as the forward. */
moe_status_t moe_grouped_gemm_wgrad(const moe_operand_t* A, const moe_operand_t* dC,
                                    const int32_t* offsets, int M, int N, int K, int E,
                                    int accumulate, void* dB, moe_dtype_t dB_dtype,
                                    int32_t* dev_status, cudaStream_t stream);

/* ---------------------------------------------------------------- combine ---
 * Weighted unpermute ([1] "Optimisation 2": combine routes expert outputs back
 * to the original token order and accumulates them; Figure 3).
 *   y[t] = sum_{j<k} w[t, j] * yp[dest_row[t, j]], summed in slot order in fp32,
 *   rounded once to y_dtype.  topk_w == NULL means unit weights (this is also
 *   the backward of dispatch: dx[t] = sum_j dxp[dest_row[t, j]]).
 *   yp [T*k, d] in dtype (MOE_BF16 / MOE_F32); y [T, d] in y_dtype.
 * Limits: d % 8 == 0, k <= 32. */
moe_status_t moe_unpermute_combine(const void* yp, moe_dtype_t dtype, int T, int d, int k,
                                   const int32_t* dest_row, const float* topk_w,
                                   void* y, moe_dtype_t y_dtype, int32_t* dev_status,
                                   cudaStream_t stream);

/* ---------------------------------------------------------------- capacity --
 * Capacity-based dispatch, the contrast case of [1] (first section: a fixed
 * per-expert capacity pads experts with fewer tokens and drops the tokens that
 * overflow the busy ones; dropless routing needs neither).  Not on the dropless
 * path: it exists to measure what padding and dropping cost.
 *
 * moe_permute_capacity: every expert e owns rows [e*C, (e+1)*C) of xp.  Its pairs,
 * in the dropless order (token ascending), fill its first min(count_e, C) rows; the
 * rest are zero; its pairs past the first C are dropped.
 *   x         [T, d] MOE_BF16 or MOE_F32 (rows a multiple of 16 bytes).
 *   topk_idx, counts: from moe_route_topk.
 *   offsets   [E+1] int32 out: e*C (uniform groups for the grouped GEMM).
 *   dest_row  [T, k] int32 out: the pair's row, or -1 when dropped.
 *   src_pair  [E*C] int32 out: the pair in each row, or -1 for padding.
 *   xp        [E*C, d] out, same dtype as x.
 *   workspace moe_permute_capacity_workspace_size(T, k, E) bytes of device scratch.
 * capacity C >= 0 (C = 0 drops everything).  Errors as moe_permute. */
size_t moe_permute_capacity_workspace_size(int T, int k, int E);
moe_status_t moe_permute_capacity(const void* x, moe_dtype_t x_dtype, int T, int d,
                                  const int32_t* topk_idx, int k, int E, int capacity,
                                  const int32_t* counts, int32_t* offsets, int32_t* dest_row,
                                  int32_t* src_pair, void* xp, void* workspace,
                                  size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream);

/* Combine for the capacity layout: as moe_unpermute_combine, with yp [rows, d]
 * (rows = E*C) and dest_row entries of -1 (dropped pairs) contributing nothing;
 * any other index outside [0, rows) sets MOE_DEV_BAD_INDEX. */
moe_status_t moe_unpermute_combine_capacity(const void* yp, moe_dtype_t dtype, int rows, int T, int d,
                                            int k, const int32_t* dest_row, const float* topk_w,
                                            void* y, moe_dtype_t y_dtype, int32_t* dev_status,
                                            cudaStream_t stream);

/* Backward of combine:
 *   dyp[dest_row[t, j]] = w[t, j] * dy[t]          (dyp [T*k, d] in dtype)
 *   dw[t, j] = sum_c dy[t, c] * yp[dest_row[t, j], c]   (dw [T, k] float32)
 *   dy [T, d] and yp [T*k, d] in dtype. */
moe_status_t moe_unpermute_combine_bwd(const void* dy, const void* yp, moe_dtype_t dtype,
                                       int T, int d, int k, const int32_t* dest_row,
                                       const float* topk_w, void* dyp, float* dw,
                                       int32_t* dev_status, cudaStream_t stream);

/* Backward of combine for the MXFP8 training step: as moe_unpermute_combine_bwd on
 * BF16 dy and yp (d % 32 == 0), with dYp written as its row-wise MXFP8 instead of in
 * BF16 -- codes [T*k, d] uint8 (16-byte aligned) and E8M0 scales [T*k, d/32] --
 * equal, bit for bit, to moe_quantize_mxfp8_grouped (axis 0) of the BF16 dYp that
 * moe_unpermute_combine_bwd would write ([1] "What dropless MoE needs": MXFP8
 * expert matmuls, quantisation fused with the producing kernel as future work).
 * dw as moe_unpermute_combine_bwd. */
moe_status_t moe_unpermute_combine_bwd_mxfp8(const void* dy, const void* yp, moe_dtype_t dtype, int T, int d,
                                             int k, const int32_t* dest_row, const float* topk_w,
                                             uint8_t* dyp_codes, uint8_t* dyp_scales, float* dw,
                                             int32_t* dev_status, cudaStream_t stream);

/* Backward of the routing weights with respect to the logits.
 *   renormalize != 0: dlogits[t, idx_j] = w_j (dw_j - sum_i w_i dw_i), 0 for
 *   unselected experts.  renormalize == 0: dlogits[t, e] = p_e (g_e - sum_i w_i dw_i)
 *   with p the full softmax of `logits` and g_e = dw_j where e = idx_j, else 0
 *   (`logits` is only read in this mode and may be NULL otherwise).
 *   dw, topk_w [T, k] float32; topk_idx [T, k]; dlogits [T, E] float32 out. */
moe_status_t moe_route_topk_bwd(const float* dw, const float* topk_w, const int32_t* topk_idx,
                                const float* logits, int T, int E, int k, int renormalize,
                                float* dlogits, int32_t* dev_status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */

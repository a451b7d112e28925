"""GB300-native (sm_103a) hot path of dropless Mixture-of-Experts training.

Route -> dispatch -> group-aware MXFP8 quantisation -> ragged grouped GEMM with
fused SwiGLU -> combine, and its backward (bf16, or every GEMM on MXFP8 operands),
as hand-written CUDA kernels behind the C ABI of include/moe.h (libmoe.so); also
an NVFP4 forward, the router GEMM fused with the top-k selection, and a
capacity-based (drop/pad) dispatch as the contrast to dropless routing.  This
package is the thin Python side:
``build`` compiles the library, ``binding`` exposes each C entry point under
the same name, ``layer`` chains them into a layer, ``workloads`` draws seeded
synthetic inputs.
"""

from .binding import (moe_check_wait_timeout, moe_debug_selftest, moe_grouped_gemm_dgrad, moe_grouped_gemm_dgrad_mxfp8,  # noqa: F401
                      moe_grouped_gemm_fwd, moe_grouped_gemm_fwd_mxfp8_out, moe_grouped_gemm_wgrad,
                      moe_permute, moe_permute_capacity, moe_permute_capacity_workspace_size,
                      moe_permute_noalloc, moe_permute_nvfp4, moe_permute_workspace_size,
                      moe_quantize_mxfp8_gathered, moe_quantize_mxfp8_grouped, moe_quantize_mxfp8_transposed,
                      moe_quantize_nvfp4, moe_route_topk, moe_route_topk_bwd, moe_route_topk_gemm,
                      moe_unpermute_combine, moe_unpermute_combine_bwd, moe_unpermute_combine_bwd_mxfp8,
                      moe_unpermute_combine_capacity,
                      moe_version, version)
from .layer import MoELayer  # noqa: F401

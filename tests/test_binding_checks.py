"""The Python binding's argument checks (no GPU needed: every check runs before a
pointer is taken, and a tensor that passes them but lives on the host is refused,
so there is no host path behind the binding)."""

import pytest
import torch

from ragged_grouped_gemm_topk_gb300 import binding as B

bf16, f32, i32, u8 = torch.bfloat16, torch.float32, torch.int32, torch.uint8


def test_combine_rejects_short_output_and_wrong_map_dtypes():
    yp = torch.zeros(8, 16, dtype=bf16)
    dest = torch.zeros(4, 2, dtype=i32)
    w = torch.zeros(4, 2, dtype=f32)
    with pytest.raises(ValueError, match="out: 48 elements, at least 64"):
        B.moe_unpermute_combine(yp, dest, w, out=torch.empty(3, 16, dtype=bf16))
    with pytest.raises(ValueError, match="dest_row: dtype"):
        B.moe_unpermute_combine(yp, dest.long(), w)
    with pytest.raises(ValueError, match="topk_w: dtype"):
        B.moe_unpermute_combine(yp, dest, w.double())
    with pytest.raises(ValueError, match="yp: 112 elements, at least 128"):
        B.moe_unpermute_combine(yp[:7], dest, w)
    with pytest.raises(ValueError, match="CUDA tensors"):            # valid, but on the host
        B.moe_unpermute_combine(yp, dest, w)


def test_route_rejects_non_fp32_logits_and_short_outputs():
    lg = torch.zeros(4, 8, dtype=f32)
    with pytest.raises(ValueError, match="logits: dtype"):
        B.moe_route_topk(lg.to(bf16), 2)
    with pytest.raises(ValueError, match="topk_idx"):
        B.moe_route_topk(lg, 2, topk_idx=torch.empty(4, 1, dtype=i32))
    with pytest.raises(ValueError, match="counts: dtype"):
        B.moe_route_topk(lg, 2, counts=torch.empty(8, dtype=torch.int64))
    with pytest.raises(ValueError, match="dev_status"):
        B.moe_route_topk(lg, 2, dev_status=torch.zeros(1, dtype=f32))
    with pytest.raises(ValueError, match="w_router: dtype"):
        B.moe_route_topk_gemm(torch.zeros(4, 32, dtype=bf16), torch.zeros(8, 32, dtype=f32), 2)


def test_gemm_rejects_short_scales_and_outputs():
    M, N, K, E = 64, 64, 512, 2
    A, Bw = torch.zeros(M, K, dtype=u8), torch.zeros(E, N, K, dtype=u8)
    As, Bs = torch.zeros(M, K // 32, dtype=u8), torch.zeros(E, N, K // 32, dtype=u8)
    off = torch.tensor([0, 32, 64], dtype=i32)
    with pytest.raises(ValueError, match="A_scales"):
        B.moe_grouped_gemm_fwd(A, Bw, off, A_scales=As[:10], B_scales=Bs)
    with pytest.raises(ValueError, match="B_scales"):
        B.moe_grouped_gemm_fwd(A, Bw, off, A_scales=As, B_scales=Bs[:1])
    with pytest.raises(ValueError, match="offsets"):
        B.moe_grouped_gemm_fwd(A, Bw, off[:2], A_scales=As, B_scales=Bs)
    with pytest.raises(ValueError, match="out"):
        B.moe_grouped_gemm_fwd(A, Bw, off, epi="swiglu", A_scales=As, B_scales=Bs,
                               out=torch.empty(M, N // 2 - 1, dtype=bf16))
    with pytest.raises(ValueError, match="preact"):
        B.moe_grouped_gemm_fwd(A, Bw, off, epi="swiglu", A_scales=As, B_scales=Bs,
                               preact=torch.empty(M, N, dtype=f32))
    with pytest.raises(ValueError, match="CUDA tensors"):
        B.moe_grouped_gemm_fwd(A, Bw, off, A_scales=As, B_scales=Bs)
    # NVFP4: scales per 16 elements of the unpacked K
    Aq, Bq = torch.zeros(M, K // 2, dtype=u8), torch.zeros(E, N, K // 2, dtype=u8)
    g = torch.ones(2, dtype=f32)
    with pytest.raises(ValueError, match="A_scales"):
        B.moe_grouped_gemm_fwd(Aq, Bq, off, A_scales=As, B_scales=torch.zeros(E, N, K // 16, dtype=u8),
                               A_tensor_scale=g, B_tensor_scale=g)
    with pytest.raises(ValueError, match="B_tensor_scale"):
        B.moe_grouped_gemm_fwd(Aq, Bq, off, A_scales=torch.zeros(M, K // 16, dtype=u8),
                               B_scales=torch.zeros(E, N, K // 16, dtype=u8), A_tensor_scale=g,
                               B_tensor_scale=g.double())


def test_wgrad_and_dgrad_check_their_buffers():
    M, K, N, E = 256, 128, 256, 2
    off = torch.tensor([0, 100, 256], dtype=i32)
    A, dC = torch.zeros(M, K, dtype=u8), torch.zeros(M, N, dtype=u8)
    tiles = lambda w: ((M + 127) // 128 + E) * (w // 128)     # noqa: E731
    sA, sC = torch.zeros(tiles(K), 512, dtype=u8), torch.zeros(tiles(N), 512, dtype=u8)
    with pytest.raises(ValueError, match="dC_scales"):
        B.moe_grouped_gemm_wgrad(A, dC, off, E, A_scales=sA, dC_scales=sA)
    with pytest.raises(ValueError, match="out"):
        B.moe_grouped_gemm_wgrad(A, dC, off, E, A_scales=sA, dC_scales=sC,
                                 out=torch.empty(E, N, K - 1, dtype=bf16))
    with pytest.raises(ValueError, match="accumulate"):                 # adds only into fp32
        B.moe_grouped_gemm_wgrad(A, dC, off, E, A_scales=sA, dC_scales=sC,
                                 out=torch.zeros(E, N, K, dtype=bf16), accumulate=True)
    with pytest.raises(ValueError, match="accumulate"):                 # and only into a given buffer
        B.moe_grouped_gemm_wgrad(A, dC, off, E, A_scales=sA, dC_scales=sC, accumulate=True)
    dCb, Wb = torch.zeros(M, N, dtype=bf16), torch.zeros(E, N, K, dtype=bf16)
    with pytest.raises(ValueError, match="preact"):
        B.moe_grouped_gemm_dgrad(dCb, Wb, off, epi="dswiglu", preact=torch.zeros(M, K, dtype=bf16))
    with pytest.raises(ValueError, match="CUDA tensors"):
        B.moe_grouped_gemm_dgrad(dCb, Wb, off, epi="dswiglu", preact=torch.zeros(M, 2 * K, dtype=bf16))


def test_operands_must_be_contiguous():
    A = torch.zeros(64, 128, dtype=bf16).t()                       # a transposed view
    with pytest.raises(ValueError, match="contiguous"):
        B._operand(A)


def test_quantisers_check_output_sizes():
    a = torch.zeros(64, 256, dtype=bf16)
    off = torch.tensor([0, 10, 64], dtype=i32)
    with pytest.raises(ValueError, match="scales"):
        B.moe_quantize_mxfp8_grouped(a, off, 2, axis=2, scales=torch.empty(1, 512, dtype=u8))
    with pytest.raises(ValueError, match="codes: dtype"):
        B.moe_quantize_mxfp8_grouped(a, codes=torch.empty(64, 256, dtype=bf16))
    with pytest.raises(ValueError, match="offsets: dtype"):
        B.moe_quantize_mxfp8_grouped(a, off.long(), 2, axis=1)
    with pytest.raises(ValueError, match="axis"):
        B.moe_quantize_mxfp8_grouped(a, axis=3)
    with pytest.raises(ValueError, match="tensor_scale"):
        B.moe_quantize_nvfp4(a, tensor_scale=torch.empty(1, dtype=f32))
    with pytest.raises(ValueError, match="scales"):
        B.moe_quantize_mxfp8_transposed(a.view(1, 64, 256), scales=torch.empty(10, dtype=u8))

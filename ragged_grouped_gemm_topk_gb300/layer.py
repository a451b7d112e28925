"""A dropless-MoE layer (route -> dispatch -> grouped MLP -> combine) on libmoe.

Route, dispatch, the two grouped GEMMs of the expert MLP and combine, in the
order of "Accelerating Dropless MoE Training in JAX with NVIDIA Transformer
Engine", Figure 3 (and the Route -> Dispatch -> Compute -> Combine stages of
the arXiv 2603.07685 reading, "Method overview").  All buffers are allocated
once, at construction, with the static size T*k for the permuted rows (exact
for dropless routing), so a forward (and backward) pass launches kernels only,
never reads a count on the host, and can be captured in one CUDA graph.
"""

from __future__ import annotations

import torch

from . import binding as B


class MoELayer:
    """Single-GPU MoE layer with SwiGLU experts.

    W1 [E, 2f, d] (gate rows then up rows) and W2 [E, d, f] in the compute dtype
    ("f32", "bf16"; "mxfp8" keeps bf16 master weights and quantises them once,
    at construction, to MXFP8 codes + E8M0 scales along the contraction dim).

    MXFP8 training quantises every GEMM operand along that GEMM's contraction:
    the forward and the data gradients read activations and gradients row-wise
    (the weights along d for GEMM1, along f for GEMM2, and along their output dim
    for the data gradients); the weight gradients read Xp, H, dYp and dGU
    column-wise, group-aware, with scales in the weight-gradient GEMM's tiled
    layout.  H, G|U and dGU are kept in bf16 between the GEMMs; Xp and dYp exist
    only in their two MXFP8 forms (Xp: the dispatch writes the row-wise one and the
    column-wise one is quantised from the token rows through the dispatch map; dYp
    = w * dy: the combine backward writes the row-wise one and the column-wise one
    is quantised from dy with the routing weights).
    """

    def __init__(self, T, d, E, k, f, W1, W2, *, dtype="bf16", renormalize=True, training=False,
                 w_router=None, keep_logits=False, accumulate_grads=False):
        """``w_router`` [E, d] (bf16, or fp32 for the fp32 layer) makes the layer score
        the tokens itself: ``forward(x)`` then runs the router GEMM fused with the
        top-k selection instead of taking logits.  With ``keep_logits`` (or when
        training without renormalisation, whose router backward needs them) the
        fused router also writes its fp32 logits to ``self.logits``.
        ``accumulate_grads`` (training): dW1 and dW2 are fp32 sums over the backward
        calls since construction or ``zero_grads()`` (gradients summed over several
        batches), each call's weight gradients added in by the GEMM itself."""
        self.T, self.d, self.E, self.k, self.f = T, d, E, k, f
        self.w_router = w_router
        keep = w_router is not None and (keep_logits or (training and not renormalize))
        self.logits = torch.empty(T, E, dtype=torch.float32, device=W1.device) if keep else None
        self.dtype, self.renormalize, self.training = dtype, renormalize, training
        dev = W1.device
        self.device = dev
        M = T * k
        self.M = M
        store = torch.float32 if dtype == "f32" else torch.bfloat16
        self.store = store
        i32 = dict(dtype=torch.int32, device=dev)
        self.W1, self.W2 = W1, W2
        self.topk_idx = torch.empty(T, k, **i32)
        self.topk_w = torch.empty(T, k, dtype=torch.float32, device=dev)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.dest_row = torch.empty(T, k, **i32)
        self.src_pair = torch.empty(M, **i32)
        self.workspace = torch.empty(B.moe_permute_workspace_size(T, k, E), dtype=torch.uint8, device=dev)
        self.dev_status = torch.zeros(1, **i32)
        # MXFP8: GEMM1 writes H straight as MXFP8 codes + scales (hq, hs)
        self.h = torch.empty(M, f, dtype=store, device=dev) if dtype != "mxfp8" or training else None
        self.yp = torch.empty(M, d, dtype=store, device=dev)
        self.y = torch.empty(T, d, dtype=store, device=dev)
        self.gu = torch.empty(M, 2 * f, dtype=store, device=dev) if training else None
        u8 = dict(dtype=torch.uint8, device=dev)
        if dtype == "nvfp4":
            if training:
                raise NotImplementedError("the NVFP4 layer is forward only")
            # each of W1, W2, Xp, H is one NVFP4 tensor (one fp32 tensor scale)
            self.W1q, self.W1s, self.W1g = B.moe_quantize_nvfp4(W1)
            self.W2q, self.W2s, self.W2g = B.moe_quantize_nvfp4(W2)
            self.xp = None                         # the dispatch writes NVFP4 rows only
            self.xq, self.xs = torch.empty(M, d // 2, **u8), torch.empty(M, d // 16, **u8)
            self.xg = torch.empty(2, dtype=torch.float32, device=dev)
            self.hq, self.hs = torch.empty(M, f // 2, **u8), torch.empty(M, f // 16, **u8)
            self.hg = torch.empty(2, dtype=torch.float32, device=dev)
        elif dtype == "mxfp8":
            self.xq = torch.empty(M, d, **u8)
            self.xs = torch.empty(M, d // 32, **u8)
            self.hq = torch.empty(M, f, **u8)
            self.hs = torch.empty(M, f // 32, **u8)
            self.W1q, self.W1s = B.moe_quantize_mxfp8_grouped(W1.reshape(E * 2 * f, d))
            self.W2q, self.W2s = B.moe_quantize_mxfp8_grouped(W2.reshape(E * d, f))
            self.W1q, self.W1s = self.W1q.view(E, 2 * f, d), self.W1s.view(E, 2 * f, d // 32)
            self.W2q, self.W2s = self.W2q.view(E, d, f), self.W2s.view(E, d, f // 32)
            self.xp = None        # training too: both MXFP8 forms of Xp come from x directly
        else:
            self.xp = torch.empty(M, d, dtype=store, device=dev)
        if dtype == "mxfp8" and training:
            # data gradients: the weights quantised along their output dim (W^T row-wise)
            self.W1t, self.W1ts = B.moe_quantize_mxfp8_transposed(W1)          # [E, d, 2f]
            self.W2t, self.W2ts = B.moe_quantize_mxfp8_transposed(W2)          # [E, f, d]

            def colwise(width):
                tiles = ((M + 127) // 128 + E) * (width // 128)
                return torch.empty(M, width, **u8), torch.empty(tiles, 512, **u8)
            # weight gradients: column-wise, group-aware operands (tiled scales)
            self.xcq, self.xcs = colwise(d)
            self.hcq, self.hcs = colwise(f)
            self.dycq, self.dycs = colwise(d)
            self.dgcq, self.dgcs = colwise(2 * f)
            # data gradients: row-wise dYp and dGU
            self.dyq, self.dys = torch.empty(M, d, **u8), torch.empty(M, d // 32, **u8)
            self.dgq, self.dgs = torch.empty(M, 2 * f, **u8), torch.empty(M, 2 * f // 32, **u8)
        if training:
            # MXFP8: dYp exists only as its two MXFP8 forms (from dy and the routing weights)
            self.dyp = torch.empty(M, d, dtype=store, device=dev) if dtype != "mxfp8" else None
            self.dw = torch.empty(T, k, dtype=torch.float32, device=dev)
            self.dgu = torch.empty(M, 2 * f, dtype=store, device=dev)
            self.dxp = torch.empty(M, d, dtype=store, device=dev)
            self.dx = torch.empty(T, d, dtype=store, device=dev)
            self.dlogits = torch.empty(T, E, dtype=torch.float32, device=dev)
            self.accumulate_grads = accumulate_grads
            if accumulate_grads:
                self.dW1 = torch.zeros(W1.shape, dtype=torch.float32, device=dev)
                self.dW2 = torch.zeros(W2.shape, dtype=torch.float32, device=dev)
            else:
                self.dW1 = torch.empty_like(W1)
                self.dW2 = torch.empty_like(W2)

    # ------------------------------------------------------------------ forward
    def route(self, logits, x=None):
        if logits is None:
            if self.w_router is None:
                raise ValueError("no logits and no router weights")
            B.moe_route_topk_gemm(x, self.w_router, self.k, self.renormalize, logits=self.logits,
                                  topk_idx=self.topk_idx, topk_w=self.topk_w, counts=self.counts,
                                  dev_status=self.dev_status)
        else:
            B.moe_route_topk(logits, self.k, self.renormalize, topk_idx=self.topk_idx,
                             topk_w=self.topk_w, counts=self.counts, dev_status=self.dev_status)

    def dispatch(self, x):
        if self.dtype == "nvfp4":
            B.moe_permute_nvfp4(x, self.topk_idx, self.counts, self.E, offsets=self.offsets,
                                dest_row=self.dest_row, src_pair=self.src_pair, codes=self.xq, scales=self.xs,
                                tensor_scale=self.xg, workspace=self.workspace, dev_status=self.dev_status)
        elif self.dtype == "mxfp8" and self.training:
            # row-wise MXFP8 rows from the dispatch, then the column-wise form for the
            # weight gradient gathered from the token rows (no bf16 Xp)
            B.moe_permute(x, self.topk_idx, self.counts, self.E, xp_dtype="mxfp8", offsets=self.offsets,
                          dest_row=self.dest_row, src_pair=self.src_pair, xp=self.xq,
                          xp_scales=self.xs, workspace=self.workspace, dev_status=self.dev_status)
            B.moe_quantize_mxfp8_gathered(x, self.src_pair, self.offsets, self.E, self.k, codes=self.xcq,
                                          scales=self.xcs, axis=2, dev_status=self.dev_status)
        elif self.dtype == "mxfp8":
            B.moe_permute(x, self.topk_idx, self.counts, self.E, xp_dtype="mxfp8", offsets=self.offsets,
                          dest_row=self.dest_row, src_pair=self.src_pair, xp=self.xq,
                          xp_scales=self.xs, workspace=self.workspace, dev_status=self.dev_status)
        else:
            B.moe_permute(x, self.topk_idx, self.counts, self.E, offsets=self.offsets,
                          dest_row=self.dest_row, src_pair=self.src_pair, xp=self.xp,
                          workspace=self.workspace, dev_status=self.dev_status)

    def expert_mlp(self, mark=None):
        """GEMM1 (+ SwiGLU), then GEMM2.  ``mark(name)``, when given, is called right
        after the kernels of GEMM1 are enqueued (timing hooks; nothing else)."""
        mark = mark or (lambda name: None)
        if self.dtype == "nvfp4":
            B.moe_grouped_gemm_fwd(self.xq, self.W1q, self.offsets, epi="swiglu", A_scales=self.xs,
                                   B_scales=self.W1s, A_tensor_scale=self.xg, B_tensor_scale=self.W1g,
                                   out=self.h, dev_status=self.dev_status)
            mark("gemm1")
            B.moe_quantize_nvfp4(self.h, codes=self.hq, scales=self.hs, tensor_scale=self.hg)
            B.moe_grouped_gemm_fwd(self.hq, self.W2q, self.offsets, A_scales=self.hs, B_scales=self.W2s,
                                   A_tensor_scale=self.hg, B_tensor_scale=self.W2g, out=self.yp,
                                   dev_status=self.dev_status)
        elif self.dtype == "mxfp8" and self.training:
            # GEMM1 keeps H and the pre-activations in bf16 for the backward
            B.moe_grouped_gemm_fwd(self.xq, self.W1q, self.offsets, epi="swiglu", A_scales=self.xs,
                                   B_scales=self.W1s, out=self.h, preact=self.gu, dev_status=self.dev_status)
            B.moe_quantize_mxfp8_grouped(self.h, codes=self.hq, scales=self.hs)
            B.moe_quantize_mxfp8_grouped(self.h, self.offsets, self.E, codes=self.hcq, scales=self.hcs, axis=2)
            mark("gemm1")
            B.moe_grouped_gemm_fwd(self.hq, self.W2q, self.offsets, A_scales=self.hs, B_scales=self.W2s,
                                   out=self.yp, dev_status=self.dev_status)
        elif self.dtype == "mxfp8":
            B.moe_grouped_gemm_fwd_mxfp8_out(self.xq, self.W1q, self.offsets, epi="swiglu", A_scales=self.xs,
                                             B_scales=self.W1s, codes=self.hq, scales=self.hs,
                                             dev_status=self.dev_status)
            mark("gemm1")
            B.moe_grouped_gemm_fwd(self.hq, self.W2q, self.offsets, A_scales=self.hs, B_scales=self.W2s,
                                   out=self.yp, dev_status=self.dev_status)
        else:
            B.moe_grouped_gemm_fwd(self.xp, self.W1, self.offsets, epi="swiglu", out=self.h,
                                   preact=self.gu, dev_status=self.dev_status)
            mark("gemm1")
            B.moe_grouped_gemm_fwd(self.h, self.W2, self.offsets, out=self.yp, dev_status=self.dev_status)

    def combine(self, out=None):
        y = self.y if out is None else out
        B.moe_unpermute_combine(self.yp, self.dest_row, self.topk_w, out=y,
                                dev_status=self.dev_status)
        return y

    def forward(self, x, logits=None, out=None):
        """y [T, d] (written to ``out`` when given, else to the layer's own buffer).
        Without ``logits`` the layer's router weights score the tokens."""
        self.route(logits, x)
        self.dispatch(x)
        self.expert_mlp()
        return self.combine(out)

    def launches_per_forward(self) -> int:
        """Kernels one forward enqueues: route (zero counts + top-k), dispatch (rank,
        scatter; NVFP4: the rank pass takes the tensor amax of x in the same launch),
        GEMM1 (MXFP8: with H quantised in its epilogue), GEMM2, combine; NVFP4 adds the
        amax and the quantisation of H; MXFP8 training adds the gathered column-wise
        quantisation of Xp and the row- and column-wise quantisation of H."""
        route = 1 if self.w_router is not None else 2     # fused router GEMM (counts zeroed by a memset)
        nv = 2 if self.dtype == "nvfp4" else 0            # amax + quantise of H
        return route + 2 + 2 + 1 + nv + (3 if self.dtype == "mxfp8" and self.training else 0)

    def launches_per_backward(self) -> int:
        """combine bwd, dgrad+dSwiGLU, wgrad, dgrad, wgrad, dispatch bwd, router bwd;
        MXFP8 adds the gathered column-wise quantisation of dYp (its row-wise form
        comes from the combine backward) and the row- and column-wise quantisation
        of dGU."""
        return 7 + (3 if self.dtype == "mxfp8" else 0)

    # ------------------------------------------------------------------ backward
    def zero_grads(self):
        """Reset the summed weight gradients (``accumulate_grads``) to zero."""
        if not self.training:
            raise RuntimeError("construct the layer with training=True")
        self.dW1.zero_()
        self.dW2.zero_()

    def backward(self, dy, logits=None, dx_out=None, mark=None):
        """Gradients of sum(y * dy) with respect to x, logits, W1 and W2 (after forward);
        dx goes to ``dx_out`` when given.  ``mark(name)``, when given, is called after
        each step's kernels are enqueued (combine_bwd, dgrad2, wgrad2, [quant_dgu],
        dgrad1, wgrad1, dispatch_bwd, route_bwd): timing hooks, nothing else."""
        if not self.training:
            raise RuntimeError("construct the layer with training=True")
        mark = mark or (lambda name: None)
        st = self.dev_status
        if self.dtype == "mxfp8":
            off, E = self.offsets, self.E
            # dYp = w * dy in its two MXFP8 forms: row-wise from the combine backward,
            # column-wise gathered from dy through the dispatch map
            B.moe_unpermute_combine_bwd_mxfp8(dy, self.yp, self.dest_row, self.topk_w, codes=self.dyq,
                                              scales=self.dys, dw=self.dw, dev_status=st)
            B.moe_quantize_mxfp8_gathered(dy, self.src_pair, off, E, self.k, row_w=self.topk_w, codes=self.dycq,
                                          scales=self.dycs, axis=2, dev_status=st)
            mark("combine_bwd")
            B.moe_grouped_gemm_dgrad_mxfp8(self.dyq, self.W2t, off, dC_scales=self.dys, BT_scales=self.W2ts,
                                           epi="dswiglu", preact=self.gu, out=self.dgu, dev_status=st)
            mark("dgrad2")
            B.moe_grouped_gemm_wgrad(self.hcq, self.dycq, off, E, A_scales=self.hcs, dC_scales=self.dycs,
                                     out=self.dW2, accumulate=self.accumulate_grads, dev_status=st)
            mark("wgrad2")
            B.moe_quantize_mxfp8_grouped(self.dgu, codes=self.dgq, scales=self.dgs)
            B.moe_quantize_mxfp8_grouped(self.dgu, off, E, codes=self.dgcq, scales=self.dgcs, axis=2)
            mark("quant_dgu")
            B.moe_grouped_gemm_dgrad_mxfp8(self.dgq, self.W1t, off, dC_scales=self.dgs, BT_scales=self.W1ts,
                                           out=self.dxp, dev_status=st)
            mark("dgrad1")
            B.moe_grouped_gemm_wgrad(self.xcq, self.dgcq, off, E, A_scales=self.xcs, dC_scales=self.dgcs,
                                     out=self.dW1, accumulate=self.accumulate_grads, dev_status=st)
            mark("wgrad1")
        else:
            B.moe_unpermute_combine_bwd(dy, self.yp, self.dest_row, self.topk_w, dyp=self.dyp, dw=self.dw,
                                        dev_status=st)
            mark("combine_bwd")
            B.moe_grouped_gemm_dgrad(self.dyp, self.W2, self.offsets, epi="dswiglu", preact=self.gu,
                                     out=self.dgu, dev_status=st)
            mark("dgrad2")
            B.moe_grouped_gemm_wgrad(self.h, self.dyp, self.offsets, self.E, out=self.dW2,
                                     accumulate=self.accumulate_grads, dev_status=st)
            mark("wgrad2")
            B.moe_grouped_gemm_dgrad(self.dgu, self.W1, self.offsets, out=self.dxp, dev_status=st)
            mark("dgrad1")
            B.moe_grouped_gemm_wgrad(self.xp, self.dgu, self.offsets, self.E, out=self.dW1,
                                     accumulate=self.accumulate_grads, dev_status=st)
            mark("wgrad1")
        dx = self.dx if dx_out is None else dx_out
        B.moe_unpermute_combine(self.dxp, self.dest_row, None, out=dx, dev_status=st)
        mark("dispatch_bwd")
        if logits is None:
            logits = self.logits          # the fused router's own (None is fine when renormalised)
        B.moe_route_topk_bwd(self.dw, self.topk_w, self.topk_idx, self.E, logits=logits,
                             renormalize=self.renormalize, out=self.dlogits, dev_status=st)
        mark("route_bwd")
        return dx, self.dlogits, self.dW1, self.dW2

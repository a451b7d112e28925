"""Python binding of libmoe: one function per C entry point, same names.

Argument marshalling only -- every step runs in the library's CUDA kernels.
Tensors must be CUDA tensors, contiguous, on the current device; calls are
enqueued on ``torch.cuda.current_stream()``.  Outputs are allocated with
torch when not passed in.  MXFP8 operands are uint8 code tensors plus uint8
E8M0 scale tensors.

The C ABI sees raw pointers only, so the sizes and element types it cannot check
are checked here before any pointer is taken: index maps and counts are int32,
routing weights, logits and tensor scales fp32, codes and scales uint8, and a
caller-supplied buffer holds at least the elements the call reads or writes
(it is used row-major from its first element).  A buffer that fails raises
ValueError and nothing is launched.
"""

from __future__ import annotations

import ctypes as C

import torch

from . import _lib
from ._lib import (MOE_BF16, MOE_DEV_BAD_INDEX, MOE_DEV_NAN_LOGIT, MOE_DEV_TIMEOUT,  # noqa: F401
                   MOE_E4M3, MOE_EPI_DSWIGLU, MOE_EPI_NONE, MOE_EPI_SWIGLU, MOE_F32, MoeError)

_DT = {torch.float32: MOE_F32, torch.bfloat16: MOE_BF16, torch.uint8: MOE_E4M3}
_EPI = {"none": MOE_EPI_NONE, "swiglu": MOE_EPI_SWIGLU, "dswiglu": MOE_EPI_DSWIGLU}
_I32, _F32, _U8 = torch.int32, torch.float32, torch.uint8


def _ptr(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("libmoe takes contiguous tensors")
    if not t.is_cuda:
        raise ValueError("libmoe takes CUDA tensors")
    return C.c_void_p(t.data_ptr())


def _need(t, name, dtype=None, numel=None):
    """Check a tensor the C side cannot check: element type and minimum size."""
    if t is None:
        return t
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name}: {t.numel()} elements, at least {numel} needed")
    return t


def _stream():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dt(t):
    try:
        return _DT[t.dtype]
    except KeyError:
        raise ValueError(f"unsupported dtype {t.dtype}") from None


def _operand(t, scales=None, tensor_scale=None):
    """A GEMM operand; uint8 codes are MXFP8 (E4M3), or NVFP4 (packed E2M1) when a
    tensor scale is given."""
    dt = _lib.MOE_E2M1 if tensor_scale is not None else _dt(t)
    addr = [p.value if p is not None else None for p in (_ptr(t), _ptr(scales), _ptr(tensor_scale))]
    return _lib.Operand(addr[0], dt, addr[1], addr[2])


def _maps(T, k, E, M, offsets=None, dest_row=None, src_pair=None, counts=None, topk_idx=None):
    _need(topk_idx, "topk_idx", _I32, T * k)
    _need(counts, "counts", _I32, E)
    _need(offsets, "offsets", _I32, E + 1)
    _need(dest_row, "dest_row", _I32, T * k)
    _need(src_pair, "src_pair", _I32, M)


def moe_version() -> int:
    return int(_lib.load().moe_version())


version = moe_version


def moe_route_topk(logits, k, renormalize=True, *, topk_idx=None, topk_w=None, counts=None,
                   dev_status=None):
    """logits [T,E] fp32 -> (topk_idx [T,k] int32, topk_w [T,k] fp32, counts [E] int32)."""
    T, E = logits.shape
    dev = logits.device
    _need(logits, "logits", _F32)
    _need(topk_w, "topk_w", _F32, T * k)
    _need(dev_status, "dev_status", _I32, 1)
    _maps(T, k, E, 0, topk_idx=topk_idx, counts=counts)
    topk_idx = topk_idx if topk_idx is not None else torch.empty(T, k, dtype=_I32, device=dev)
    topk_w = topk_w if topk_w is not None else torch.empty(T, k, dtype=_F32, device=dev)
    counts = counts if counts is not None else torch.empty(E, dtype=_I32, device=dev)
    _lib.call("moe_route_topk", _ptr(logits), T, E, k, int(bool(renormalize)), _ptr(topk_idx),
              _ptr(topk_w), _ptr(counts), _ptr(dev_status), _stream())
    return topk_idx, topk_w, counts


def moe_route_topk_gemm(x, w_router, k, renormalize=True, *, logits=None, want_logits=False, topk_idx=None,
                        topk_w=None, counts=None, dev_status=None):
    """Router GEMM fused with top-k: x [T,d], w_router [E,d] (bf16 or fp32) ->
    (topk_idx, topk_w, counts[, logits [T,E] fp32 when asked for])."""
    T, d = x.shape
    E, d2 = w_router.shape
    if d2 != d:
        raise ValueError("x and w_router disagree on d")
    _need(w_router, "w_router", x.dtype)
    _need(logits, "logits", _F32, T * E)
    _need(topk_w, "topk_w", _F32, T * k)
    _need(dev_status, "dev_status", _I32, 1)
    _maps(T, k, E, 0, topk_idx=topk_idx, counts=counts)
    dev = x.device
    topk_idx = topk_idx if topk_idx is not None else torch.empty(T, k, dtype=_I32, device=dev)
    topk_w = topk_w if topk_w is not None else torch.empty(T, k, dtype=_F32, device=dev)
    counts = counts if counts is not None else torch.empty(E, dtype=_I32, device=dev)
    if want_logits and logits is None:
        logits = torch.empty(T, E, dtype=_F32, device=dev)
    _lib.call("moe_route_topk_gemm", _ptr(x), _ptr(w_router), _dt(x), T, d, E, k, int(bool(renormalize)),
              _ptr(logits), _ptr(topk_idx), _ptr(topk_w), _ptr(counts), _ptr(dev_status), _stream())
    return (topk_idx, topk_w, counts, logits) if logits is not None else (topk_idx, topk_w, counts)


def moe_permute_workspace_size(T, k, E) -> int:
    return int(_lib.load().moe_permute_workspace_size(T, k, E))


def moe_permute(x, topk_idx, counts, E, *, xp_dtype=None, rows=True, offsets=None, dest_row=None,
                src_pair=None, xp=None, xp_scales=None, workspace=None, dev_status=None):
    """Dispatch x [T,d] into expert-contiguous rows.  xp_dtype: None (same as x) or
    "mxfp8" (fused row-wise MXFP8).  Returns a dict with offsets [E+1], dest_row
    [T,k], src_pair [T*k] (int32) and, if ``rows``, xp [T*k,d] (+ xp_scales)."""
    T, k = topk_idx.shape
    d = x.shape[1] if x is not None else 0
    dev = topk_idx.device
    M = T * k
    quant = xp_dtype == "mxfp8"
    _maps(T, k, E, M, offsets, dest_row, src_pair, counts, topk_idx)
    _need(dev_status, "dev_status", _I32, 1)
    if rows:
        _need(xp, "xp", _U8 if quant else x.dtype, M * d)
        _need(xp_scales, "xp_scales", _U8, M * (d // 32))
    offsets = offsets if offsets is not None else torch.empty(E + 1, dtype=_I32, device=dev)
    dest_row = dest_row if dest_row is not None else torch.empty(T, k, dtype=_I32, device=dev)
    src_pair = src_pair if src_pair is not None else torch.empty(M, dtype=_I32, device=dev)
    if rows:
        if xp is None:
            xp = torch.empty(M, d, dtype=_U8 if quant else x.dtype, device=dev)
        if quant and xp_scales is None:
            xp_scales = torch.empty(M, d // 32, dtype=_U8, device=dev)
    else:
        xp = None
    if workspace is None:
        workspace = torch.empty(moe_permute_workspace_size(T, k, E), dtype=_U8, device=dev)
    _lib.call("moe_permute", _ptr(x) if rows else None, _dt(x) if x is not None else MOE_BF16, T, d,
              _ptr(topk_idx), k, E, _ptr(counts), _ptr(offsets), _ptr(dest_row), _ptr(src_pair),
              _ptr(xp), MOE_E4M3 if quant else (_dt(x) if x is not None else MOE_BF16),
              _ptr(xp_scales), _ptr(workspace), workspace.numel() * workspace.element_size(),
              _ptr(dev_status), _stream())
    return dict(offsets=offsets, dest_row=dest_row, src_pair=src_pair, xp=xp, xp_scales=xp_scales)


def moe_permute_noalloc(x, topk_idx, counts, E, *, xp_dtype=None, offsets=None, dest_row=None, src_pair=None,
                        xp=None, xp_scales=None, dev_status=None):
    """moe_permute without a workspace (the library's fixed device scratch; at most
    ceil(T/256)*E <= 262144, and concurrent calls race).  Same outputs."""
    T, k = topk_idx.shape
    d = x.shape[1]
    dev = x.device
    M = T * k
    quant = xp_dtype == "mxfp8"
    _maps(T, k, E, M, offsets, dest_row, src_pair, counts, topk_idx)
    _need(dev_status, "dev_status", _I32, 1)
    _need(xp, "xp", _U8 if quant else x.dtype, M * d)
    _need(xp_scales, "xp_scales", _U8, M * (d // 32))
    offsets = offsets if offsets is not None else torch.empty(E + 1, dtype=_I32, device=dev)
    dest_row = dest_row if dest_row is not None else torch.empty(T, k, dtype=_I32, device=dev)
    src_pair = src_pair if src_pair is not None else torch.empty(M, dtype=_I32, device=dev)
    xp = xp if xp is not None else torch.empty(M, d, dtype=_U8 if quant else x.dtype, device=dev)
    if quant and xp_scales is None:
        xp_scales = torch.empty(M, d // 32, dtype=_U8, device=dev)
    _lib.call("moe_permute_noalloc", _ptr(x), _dt(x), T, d, _ptr(topk_idx), k, E, _ptr(counts), _ptr(offsets),
              _ptr(dest_row), _ptr(src_pair), _ptr(xp), MOE_E4M3 if quant else _dt(x), _ptr(xp_scales),
              _ptr(dev_status), _stream())
    return dict(offsets=offsets, dest_row=dest_row, src_pair=src_pair, xp=xp, xp_scales=xp_scales)


def moe_check_wait_timeout(limit_us, dev_status=None):
    """Run the bounded-wait failure path: returns the device status word (int32
    tensor) after a barrier wait of limit_us microseconds has given up."""
    _need(dev_status, "dev_status", _I32, 1)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=_I32, device=torch.cuda.current_device())
    _lib.call("moe_check_wait_timeout", _ptr(dev_status), int(limit_us), _stream())
    return dev_status


def moe_debug_selftest(dev_status=None):
    """(is_debug, status word): whether the loaded library is a MOE_DEBUG build, and
    the device status word after a device-side check that always fails (a debug
    build ORs MOE_DEV_ASSERT into it, a release build leaves it unchanged)."""
    _need(dev_status, "dev_status", _I32, 1)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=_I32, device=torch.cuda.current_device())
    flag = C.c_int(-1)
    _lib.call("moe_debug_selftest", _ptr(dev_status), C.byref(flag), _stream())
    return bool(flag.value), dev_status


def _colwise_scale_shape(rows, K, E, axis):
    return {0: (rows, K // 32), 1: ((rows + 31) // 32 + E, K),
            2: (((rows + 127) // 128 + E) * (K // 128), 512)}[axis]


def moe_quantize_mxfp8_grouped(inp, offsets=None, E=0, *, codes=None, scales=None, axis=0):
    """MXFP8 of inp [rows,K] (bf16/fp32) -> (codes u8 [rows,K], scales u8).
    axis 0: row-wise, scales [rows, K/32].  axis 1: column-wise and group-aware
    (offsets [E+1] required), scales [ceil(rows/32) + E, K] of which the first
    sum_e ceil(count_e/32) rows are written.  axis 2: as axis 1 with the scales in
    the weight-gradient GEMM's tiled layout, [(ceil(rows/128) + E) * K/128, 512]."""
    rows, K = inp.shape
    if axis not in (0, 1, 2):
        raise ValueError("axis must be 0, 1 or 2")
    shape = _colwise_scale_shape(rows, K, E, axis)
    _need(codes, "codes", _U8, rows * K)
    _need(scales, "scales", _U8, shape[0] * shape[1])
    _need(offsets, "offsets", _I32, E + 1 if axis else None)
    codes = codes if codes is not None else torch.empty(rows, K, dtype=_U8, device=inp.device)
    if scales is None:
        scales = torch.empty(*shape, dtype=_U8, device=inp.device)
    _lib.call("moe_quantize_mxfp8_grouped", _ptr(inp), _dt(inp), rows, K, _ptr(offsets), E, axis,
              _ptr(codes), _ptr(scales), _stream())
    return codes, scales


def moe_quantize_mxfp8_gathered(x, src_pair, offsets, E, k, *, row_w=None, codes=None, scales=None, axis=2,
                                dev_status=None):
    """Column-wise group-aware MXFP8 of the dispatched rows Xp[r] = x[src_pair[r] // k]
    (x [T, K] bf16/fp32; src_pair and offsets from moe_permute) without writing Xp:
    the codes [T*k, K] and scales of moe_quantize_mxfp8_grouped(Xp, offsets, E, axis).
    With row_w ([T, k] fp32 routing weights) the rows are w * x rounded to x's dtype:
    the dYp of the combine backward (x = dy)."""
    T, K = x.shape
    rows = T * k
    if axis not in (1, 2):
        raise ValueError("axis must be 1 or 2")
    shape = _colwise_scale_shape(rows, K, E, axis)
    _need(src_pair, "src_pair", _I32, rows)
    _need(row_w, "row_w", _F32, rows)
    _need(offsets, "offsets", _I32, E + 1)
    _need(codes, "codes", _U8, rows * K)
    _need(scales, "scales", _U8, shape[0] * shape[1])
    _need(dev_status, "dev_status", _I32, 1)
    codes = codes if codes is not None else torch.empty(rows, K, dtype=_U8, device=x.device)
    scales = scales if scales is not None else torch.empty(*shape, dtype=_U8, device=x.device)
    _lib.call("moe_quantize_mxfp8_gathered", _ptr(x), _dt(x), T, K, k, _ptr(src_pair), _ptr(row_w), _ptr(offsets),
              E, axis,
              _ptr(codes), _ptr(scales), _ptr(dev_status), _stream())
    return codes, scales


def moe_quantize_mxfp8_transposed(inp, *, codes=None, scales=None):
    """Row-wise MXFP8 of each inp[g]^T for inp [G,R,C] (bf16/fp32) -> (codes u8
    [G,C,R], scales u8 [G*C, R/32])."""
    G, R, Cc = inp.shape
    _need(codes, "codes", _U8, G * Cc * R)
    _need(scales, "scales", _U8, G * Cc * (R // 32))
    codes = codes if codes is not None else torch.empty(G, Cc, R, dtype=_U8, device=inp.device)
    scales = scales if scales is not None else torch.empty(G * Cc, R // 32, dtype=_U8, device=inp.device)
    _lib.call("moe_quantize_mxfp8_transposed", _ptr(inp), _dt(inp), G, R, Cc, _ptr(codes), _ptr(scales), _stream())
    return codes, scales


def moe_quantize_nvfp4(inp, *, codes=None, scales=None, tensor_scale=None):
    """NVFP4 of inp [rows, K] (bf16/fp32; a weight stack [E, N, K] as one tensor) ->
    (codes u8 [.., K/2] packed, scales u8 [.., K/16] E4M3, tensor_scale fp32 [2] with
    the encode scale g in element 0)."""
    K = inp.shape[-1]
    lead = inp.shape[:-1]
    rows = inp.numel() // K if K else 0
    _need(codes, "codes", _U8, rows * (K // 2))
    _need(scales, "scales", _U8, rows * (K // 16))
    _need(tensor_scale, "tensor_scale", _F32, 2)
    codes = codes if codes is not None else torch.empty(*lead, K // 2, dtype=_U8, device=inp.device)
    scales = scales if scales is not None else torch.empty(*lead, K // 16, dtype=_U8, device=inp.device)
    tensor_scale = tensor_scale if tensor_scale is not None else torch.empty(2, dtype=_F32, device=inp.device)
    _lib.call("moe_quantize_nvfp4", _ptr(inp), _dt(inp), rows, K, _ptr(codes), _ptr(scales), _ptr(tensor_scale),
              _stream())
    return codes, scales, tensor_scale


def moe_permute_nvfp4(x, topk_idx, counts, E, *, offsets=None, dest_row=None, src_pair=None, codes=None,
                      scales=None, tensor_scale=None, workspace=None, dev_status=None):
    """Dispatch with NVFP4 rows: a dict with offsets, dest_row, src_pair and the rows'
    codes [T*k, d/2], scales [T*k, d/16] and tensor_scale (fp32 [2], g in element 0)."""
    T, k = topk_idx.shape
    d = x.shape[1]
    dev = x.device
    i32 = dict(dtype=_I32, device=dev)
    M = T * k
    _maps(T, k, E, M, offsets, dest_row, src_pair, counts, topk_idx)
    _need(codes, "codes", _U8, M * (d // 2))
    _need(scales, "scales", _U8, M * (d // 16))
    _need(tensor_scale, "tensor_scale", _F32, 2)
    _need(dev_status, "dev_status", _I32, 1)
    offsets = offsets if offsets is not None else torch.empty(E + 1, **i32)
    dest_row = dest_row if dest_row is not None else torch.empty(T, k, **i32)
    src_pair = src_pair if src_pair is not None else torch.empty(M, **i32)
    codes = codes if codes is not None else torch.empty(M, d // 2, dtype=_U8, device=dev)
    scales = scales if scales is not None else torch.empty(M, d // 16, dtype=_U8, device=dev)
    tensor_scale = tensor_scale if tensor_scale is not None else torch.empty(2, dtype=_F32, device=dev)
    nbytes = moe_permute_workspace_size(T, k, E)
    workspace = workspace if workspace is not None else torch.empty(max(nbytes, 16), dtype=_U8, device=dev)
    _lib.call("moe_permute_nvfp4", _ptr(x), _dt(x), T, d, _ptr(topk_idx), k, E, _ptr(counts), _ptr(offsets),
              _ptr(dest_row), _ptr(src_pair), _ptr(codes), _ptr(scales), _ptr(tensor_scale), _ptr(workspace),
              workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream())
    return {"offsets": offsets, "dest_row": dest_row, "src_pair": src_pair, "codes": codes, "scales": scales,
            "tensor_scale": tensor_scale}


def _scaled_operands(A, B, A_scales, B_scales, M, N, K, E, A_tensor_scale=None, B_tensor_scale=None):
    """Scale buffers of a block-scaled A [M, K] and B [E, N, K] (K in elements); a
    missing one is left to the library, which rejects it."""
    blk = 16 if A_tensor_scale is not None else 32
    if A.dtype == _U8:
        _need(A_scales, "A_scales", _U8, M * (K // blk))
        _need(B_scales, "B_scales", _U8, E * N * (K // blk))
    _need(A_tensor_scale, "A_tensor_scale", _F32, 1)
    _need(B_tensor_scale, "B_tensor_scale", _F32, 1)


def moe_grouped_gemm_fwd(A, B, offsets, *, epi="none", A_scales=None, B_scales=None,
                         out_dtype=torch.bfloat16, out=None, preact=None, want_preact=False,
                         dev_status=None, A_tensor_scale=None, B_tensor_scale=None):
    """C = ragged A [M,K] . B[e]^T with B [E,N,K]; epi "swiglu" gives [M, N/2].
    NVFP4 (tensor scales given): A and B are packed codes [M, K/2] and [E, N, K/2]."""
    M, K = A.shape
    E, N, K2 = B.shape
    if A_tensor_scale is not None:
        K, K2 = 2 * K, 2 * K2
    if K2 != K:
        raise ValueError("A and B disagree on K")
    n_out = N // 2 if epi == "swiglu" else N
    _scaled_operands(A, B, A_scales, B_scales, M, N, K, E, A_tensor_scale, B_tensor_scale)
    _need(offsets, "offsets", _I32, E + 1)
    _need(out, "out", None, M * n_out)
    _need(preact, "preact", out.dtype if out is not None else out_dtype, M * N)
    _need(dev_status, "dev_status", _I32, 1)
    if out is None:
        out = torch.empty(M, n_out, dtype=out_dtype, device=A.device)
    if want_preact and preact is None:
        preact = torch.empty(M, N, dtype=out.dtype, device=A.device)
    a, b = _operand(A, A_scales, A_tensor_scale), _operand(B, B_scales, B_tensor_scale)
    _lib.call("moe_grouped_gemm_fwd", C.byref(a), C.byref(b), _ptr(offsets), M, N, K, E, _EPI[epi],
              _ptr(out), _dt(out), _ptr(preact), _ptr(dev_status), _stream())
    return (out, preact) if want_preact or preact is not None else out


def moe_grouped_gemm_fwd_mxfp8_out(A, B, offsets, *, epi="none", A_scales=None, B_scales=None, codes=None,
                                   scales=None, dev_status=None):
    """As moe_grouped_gemm_fwd on MXFP8 operands, with the result quantised to MXFP8
    in the epilogue: returns (codes [M, n_out] uint8, scales [M, n_out/32] uint8)."""
    M, K = A.shape
    E, N, K2 = B.shape
    if K2 != K:
        raise ValueError("A and B disagree on K")
    n_out = N // 2 if epi == "swiglu" else N
    _scaled_operands(A, B, A_scales, B_scales, M, N, K, E)
    _need(offsets, "offsets", _I32, E + 1)
    _need(codes, "codes", _U8, M * n_out)
    _need(scales, "scales", _U8, M * (n_out // 32))
    _need(dev_status, "dev_status", _I32, 1)
    if codes is None:
        codes = torch.empty(M, n_out, dtype=_U8, device=A.device)
    if scales is None:
        scales = torch.empty(M, n_out // 32, dtype=_U8, device=A.device)
    a, b = _operand(A, A_scales), _operand(B, B_scales)
    _lib.call("moe_grouped_gemm_fwd_mxfp8_out", C.byref(a), C.byref(b), _ptr(offsets), M, N, K, E, _EPI[epi],
              _ptr(codes), _ptr(scales), _ptr(dev_status), _stream())
    return codes, scales


def moe_grouped_gemm_dgrad(dC, B, offsets, *, epi="none", preact=None, out_dtype=torch.bfloat16,
                           out=None, dev_status=None):
    """dA = ragged dC [M,N] . B[e] with B [E,N,K]; epi "dswiglu" (with preact [M,2K])
    returns [dG | dU] of shape [M, 2K]."""
    M, N = dC.shape
    E, N2, K = B.shape
    if N2 != N:
        raise ValueError("dC and B disagree on N")
    width = 2 * K if epi == "dswiglu" else K
    _need(offsets, "offsets", _I32, E + 1)
    _need(preact, "preact", torch.bfloat16, M * 2 * K if epi == "dswiglu" else None)
    _need(out, "out", None, M * width)
    _need(dev_status, "dev_status", _I32, 1)
    if out is None:
        out = torch.empty(M, width, dtype=out_dtype, device=dC.device)
    a, b = _operand(dC), _operand(B)
    _lib.call("moe_grouped_gemm_dgrad", C.byref(a), C.byref(b), _ptr(offsets), M, N, K, E, _EPI[epi],
              _ptr(preact), _ptr(out), _dt(out), _ptr(dev_status), _stream())
    return out


def moe_grouped_gemm_dgrad_mxfp8(dC, BT, offsets, *, dC_scales, BT_scales, epi="none", preact=None, out=None,
                                 dev_status=None):
    """dA = ragged dC . B[e] on MXFP8 operands: dC codes [M,N], BT codes [E,K,N]
    (= B^T quantised along N); bf16 result [M,K], or [M,2K] = [dG | dU] with
    epi "dswiglu" and preact [M,2K]."""
    M, N = dC.shape
    E, K, N2 = BT.shape
    if N2 != N:
        raise ValueError("dC and BT disagree on N")
    width = 2 * K if epi == "dswiglu" else K
    _need(dC_scales, "dC_scales", _U8, M * (N // 32))
    _need(BT_scales, "BT_scales", _U8, E * K * (N // 32))
    _need(offsets, "offsets", _I32, E + 1)
    _need(preact, "preact", torch.bfloat16, M * 2 * K if epi == "dswiglu" else None)
    _need(out, "out", torch.bfloat16, M * width)
    _need(dev_status, "dev_status", _I32, 1)
    if out is None:
        out = torch.empty(M, width, dtype=torch.bfloat16, device=dC.device)
    a, b = _operand(dC, dC_scales), _operand(BT, BT_scales)
    _lib.call("moe_grouped_gemm_dgrad_mxfp8", C.byref(a), C.byref(b), _ptr(offsets), M, N, K, E, _EPI[epi],
              _ptr(preact), _ptr(out), _ptr(dev_status), _stream())
    return out


def moe_grouped_gemm_wgrad(A, dC, offsets, E, *, A_scales=None, dC_scales=None, out_dtype=torch.bfloat16,
                           out=None, accumulate=False, dev_status=None):
    """dB[e] = dC[R_e]^T . A[R_e] -> [E, N, K] (bf16 or fp32).  MXFP8: A and dC are
    codes from the tiled column-wise quantiser (axis 2), with their scale buffers.
    accumulate: dB[e] += the product, into the given fp32 ``out``."""
    if accumulate and (out is None or out.dtype != torch.float32):
        raise ValueError("accumulate needs an fp32 out tensor to add to")
    M, K = A.shape
    M2, N = dC.shape
    if M2 != M:
        raise ValueError("A and dC disagree on M")
    if A.dtype == _U8:
        sa, sc = _colwise_scale_shape(M, K, E, 2), _colwise_scale_shape(M, N, E, 2)
        _need(A_scales, "A_scales", _U8, sa[0] * sa[1])
        _need(dC_scales, "dC_scales", _U8, sc[0] * sc[1])
    _need(offsets, "offsets", _I32, E + 1)
    _need(out, "out", None, E * N * K)
    _need(dev_status, "dev_status", _I32, 1)
    if out is None:
        out = torch.empty(E, N, K, dtype=out_dtype, device=A.device)
    a, b = _operand(A, A_scales), _operand(dC, dC_scales)
    _lib.call("moe_grouped_gemm_wgrad", C.byref(a), C.byref(b), _ptr(offsets), M, N, K, E,
              1 if accumulate else 0, _ptr(out), _dt(out), _ptr(dev_status), _stream())
    return out


def moe_unpermute_combine(yp, dest_row, topk_w, *, out_dtype=None, out=None, dev_status=None):
    """y[t] = sum_j w[t,j] yp[dest_row[t,j]] (topk_w None = unit weights)."""
    T, k = dest_row.shape
    d = yp.shape[1]
    _need(yp, "yp", None, T * k * d)
    _need(dest_row, "dest_row", _I32)
    _need(topk_w, "topk_w", _F32, T * k)
    _need(out, "out", None, T * d)
    _need(dev_status, "dev_status", _I32, 1)
    if out is None:
        out = torch.empty(T, d, dtype=out_dtype or yp.dtype, device=yp.device)
    _lib.call("moe_unpermute_combine", _ptr(yp), _dt(yp), T, d, k, _ptr(dest_row), _ptr(topk_w),
              _ptr(out), _dt(out), _ptr(dev_status), _stream())
    return out


def moe_permute_capacity_workspace_size(T, k, E) -> int:
    return int(_lib.load().moe_permute_capacity_workspace_size(T, k, E))


def moe_permute_capacity(x, topk_idx, counts, E, capacity, *, offsets=None, dest_row=None, src_pair=None, xp=None,
                         workspace=None, dev_status=None):
    """Capacity-based dispatch (the contrast case): xp [E*C, d] with expert e's
    first min(count_e, C) tokens in rows [e*C, e*C + ...), zero padding after them,
    overflowing pairs dropped (dest_row -1).  Returns a dict like moe_permute."""
    T, k = topk_idx.shape
    d = x.shape[1]
    dev = x.device
    i32 = dict(dtype=_I32, device=dev)
    _maps(T, k, E, E * capacity, offsets, dest_row, src_pair, counts, topk_idx)
    _need(xp, "xp", x.dtype, E * capacity * d)
    _need(dev_status, "dev_status", _I32, 1)
    offsets = offsets if offsets is not None else torch.empty(E + 1, **i32)
    dest_row = dest_row if dest_row is not None else torch.empty(T, k, **i32)
    src_pair = src_pair if src_pair is not None else torch.empty(E * capacity, **i32)
    xp = xp if xp is not None else torch.empty(E * capacity, d, dtype=x.dtype, device=dev)
    nbytes = moe_permute_capacity_workspace_size(T, k, E)
    workspace = workspace if workspace is not None else torch.empty(max(nbytes, 16), dtype=_U8, device=dev)
    _lib.call("moe_permute_capacity", _ptr(x), _dt(x), T, d, _ptr(topk_idx), k, E, int(capacity), _ptr(counts),
              _ptr(offsets), _ptr(dest_row), _ptr(src_pair), _ptr(xp), _ptr(workspace),
              workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream())
    return {"offsets": offsets, "dest_row": dest_row, "src_pair": src_pair, "xp": xp}


def moe_unpermute_combine_capacity(yp, dest_row, topk_w, *, out_dtype=None, out=None, dev_status=None):
    """Combine of the capacity layout: dropped pairs (dest_row -1) contribute nothing."""
    T, k = dest_row.shape
    rows, d = yp.shape
    _need(dest_row, "dest_row", _I32)
    _need(topk_w, "topk_w", _F32, T * k)
    _need(out, "out", None, T * d)
    _need(dev_status, "dev_status", _I32, 1)
    if out is None:
        out = torch.empty(T, d, dtype=out_dtype or yp.dtype, device=yp.device)
    _lib.call("moe_unpermute_combine_capacity", _ptr(yp), _dt(yp), rows, T, d, k, _ptr(dest_row), _ptr(topk_w),
              _ptr(out), _dt(out), _ptr(dev_status), _stream())
    return out


def moe_unpermute_combine_bwd(dy, yp, dest_row, topk_w, *, dyp=None, dw=None, dev_status=None):
    """Backward of the combine: dyp [T*k, d] (row dest_row[t,j] = w[t,j] dy[t]) and
    dw [T,k] fp32 (= <dy[t], yp[dest_row[t,j]]>)."""
    T, k = dest_row.shape
    d = dy.shape[1]
    _need(yp, "yp", dy.dtype, T * k * d)
    _need(dest_row, "dest_row", _I32)
    _need(topk_w, "topk_w", _F32, T * k)
    _need(dyp, "dyp", dy.dtype, T * k * d)
    _need(dw, "dw", _F32, T * k)
    _need(dev_status, "dev_status", _I32, 1)
    if dyp is None:
        dyp = torch.empty(T * k, d, dtype=dy.dtype, device=dy.device)
    if dw is None:
        dw = torch.empty(T, k, dtype=_F32, device=dy.device)
    _lib.call("moe_unpermute_combine_bwd", _ptr(dy), _ptr(yp), _dt(dy), T, d, k, _ptr(dest_row),
              _ptr(topk_w), _ptr(dyp), _ptr(dw), _ptr(dev_status), _stream())
    return dyp, dw


def moe_unpermute_combine_bwd_mxfp8(dy, yp, dest_row, topk_w, *, codes=None, scales=None, dw=None,
                                    dev_status=None):
    """Backward of the combine with dYp written as its row-wise MXFP8 (bf16 dy and
    yp): (codes u8 [T*k, d], scales u8 [T*k, d/32], dw [T,k] fp32)."""
    T, k = dest_row.shape
    d = dy.shape[1]
    M = T * k
    _need(yp, "yp", dy.dtype, M * d)
    _need(dest_row, "dest_row", _I32)
    _need(topk_w, "topk_w", _F32, M)
    _need(codes, "codes", _U8, M * d)
    _need(scales, "scales", _U8, M * (d // 32))
    _need(dw, "dw", _F32, M)
    _need(dev_status, "dev_status", _I32, 1)
    codes = codes if codes is not None else torch.empty(M, d, dtype=_U8, device=dy.device)
    scales = scales if scales is not None else torch.empty(M, d // 32, dtype=_U8, device=dy.device)
    dw = dw if dw is not None else torch.empty(T, k, dtype=_F32, device=dy.device)
    _lib.call("moe_unpermute_combine_bwd_mxfp8", _ptr(dy), _ptr(yp), _dt(dy), T, d, k, _ptr(dest_row),
              _ptr(topk_w), _ptr(codes), _ptr(scales), _ptr(dw), _ptr(dev_status), _stream())
    return codes, scales, dw


def moe_route_topk_bwd(dw, topk_w, topk_idx, E, *, logits=None, renormalize=True, out=None,
                       dev_status=None):
    """Backward of the routing weights: dlogits [T,E] fp32 from dw [T,k]."""
    T, k = topk_idx.shape
    _need(dw, "dw", _F32, T * k)
    _need(topk_w, "topk_w", _F32, T * k)
    _need(topk_idx, "topk_idx", _I32)
    _need(logits, "logits", _F32, T * E)
    _need(out, "out", _F32, T * E)
    _need(dev_status, "dev_status", _I32, 1)
    if out is None:
        out = torch.empty(T, E, dtype=_F32, device=dw.device)
    _lib.call("moe_route_topk_bwd", _ptr(dw), _ptr(topk_w), _ptr(topk_idx), _ptr(logits), T, E, k,
              int(bool(renormalize)), _ptr(out), _ptr(dev_status), _stream())
    return out

"""Dropless-MoE layer on the CPU in float64: the definition the CUDA path is checked against.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this module;
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
use it.  It shares no code with the CUDA library and imports nothing from it.

Sources (cited by short name below):
[1] "Accelerating Dropless MoE Training in JAX with NVIDIA Transformer Engine"
    (zhiding.cn rewrite of the NVIDIA technical blog).  Sections used: the
    opening (learnable router picks the top-K experts per token), "How dropless
    MoE differs from capacity-based MoE" (every token is processed by every
    expert it chose; nothing is dropped or padded), "What dropless MoE needs"
    (kernels with data-dependent per-expert sizes the CPU never sees; Figure 3:
    router -> dispatch -> two grouped GEMMs over variable-length groups ->
    combine back into the original token order), "Optimisation 1: grouped GEMM"
    (one launch over all experts, computing only the valid token rows),
    "Optimisation 2: dispatch and combine" (dispatch = local rearrangement;
    combine = route results back and accumulate per token).
[3] Deep reading of arXiv 2603.07685 (paper-daily.com), "Method overview"
    (Route -> Dispatch -> Compute -> Combine).

The pages give no formulas.  Every step below is the plainest definition that
matches them; the readings (softmax scoring with renormalised top-k weights,
lower expert id wins ties, (expert, token) ordering of the permuted rows,
SwiGLU experts with gate rows first, routing weight applied in combine) are
stated where each function uses them.

Arrays are numpy; floating-point inputs are the exact stored values (bf16 or
fp32) widened to float64, and all arithmetic is float64.

Parity pins (tests/test_oracle_*.py): brute-force sorting for top-k and ties,
a counting-loop construction of the permutation, the dense masked-MoE formula,
E=1/k=1 reducing to a dense SwiGLU FFN in torch, equal counts against
torch.bmm, the permute/combine identities, torch float64 autograd and
gradcheck for the backward.
"""

from __future__ import annotations

import numpy as np

from . import mxfp8, nvfp4


# ----------------------------------------------------------------------------- route

def route_topk(logits: np.ndarray, k: int, renormalize: bool = True):
    """Top-k expert selection and routing weights ([1] opening paragraph: a learnable
    router activates the top-K experts of each token).

    Selection orders the experts of a token by (logit descending, expert id
    ascending) and keeps the first k, so slot j holds the j-th best expert.
    Weights are the softmax of the selected logits (``renormalize``), which is
    the full softmax restricted to the selection and rescaled to sum to one, or
    the full-softmax probabilities of the selected experts.

    Returns idx int32 [T,k], w float64 [T,k], counts int64 [E].
    """
    lg = np.asarray(logits)
    if lg.dtype != np.float32:
        raise TypeError("router logits are float32")
    if np.isnan(lg).any():
        raise ValueError("NaN logits are outside the router's domain")
    T, E = lg.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    l64 = lg.astype(np.float64)
    expert_ids = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((expert_ids, -l64), axis=-1)          # primary: -logit, then id
    idx = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(l64, idx.astype(np.int64), axis=1)
    # -inf marks a masked expert (no softmax mass).  A token whose experts are all
    # masked has no mass anywhere: its k slots (the lowest expert ids, by the
    # tie-break) get weight 0, so it contributes nothing to the combine.
    masked = np.isneginf(sel[:, :1])
    top = np.where(masked, 0.0, sel[:, :1])
    if renormalize:
        ex = np.where(masked, 0.0, np.exp(sel - top))
        w = ex / np.where(masked, 1.0, ex.sum(axis=1, keepdims=True))
    else:
        ex_all = np.where(masked, 0.0, np.exp(l64 - top))
        w = np.where(masked, 0.0, np.exp(sel - top)) / np.where(masked, 1.0, ex_all.sum(axis=1, keepdims=True))
    counts = np.bincount(idx.ravel(), minlength=E).astype(np.int64)
    return idx, w, counts


def router_logits(x: np.ndarray, w_router: np.ndarray) -> np.ndarray:
    """Router scores ([1] opening paragraph: a learnable router scores each token
    against every expert): logits[t, e] = <x[t], W_r[e]>, float64.  x [T,d],
    W_r [E,d] -> [T,E]."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(w_router, dtype=np.float64).T


# ----------------------------------------------------------------------------- dispatch

def permute_maps(idx: np.ndarray, E: int):
    """The permutation of the T*k (token, slot) pairs into expert-contiguous rows
    ([1] "Optimisation 2": dispatch rearranges tokens locally by expert).

    Pairs are ordered by (expert, token); a token picks an expert at most once,
    so the key is unique.  Rows of expert e are [offsets[e], offsets[e+1]),
    with no padding between groups.

    Returns offsets int64 [E+1] (exclusive scan of the counts), dest_row int64
    [T,k] (row of pair (t,j)) and src_pair int64 [T*k] (pair t*k+j stored in
    each row); dest_row and src_pair are inverse permutations.
    """
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    expert = idx.ravel()
    token = np.arange(T * k) // k
    src_pair = np.lexsort((token, expert))                     # primary: expert, then token
    dest_row = np.empty(T * k, dtype=np.int64)
    dest_row[src_pair] = np.arange(T * k)
    counts = np.bincount(expert, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    return offsets, dest_row.reshape(T, k), src_pair.astype(np.int64)


def permute(x: np.ndarray, src_pair: np.ndarray, k: int) -> np.ndarray:
    """Xp[r] = x[token of the pair stored in row r]."""
    return np.asarray(x, dtype=np.float64)[np.asarray(src_pair) // k]


# ----------------------------------------------------------------------------- compute

def grouped_gemm(A: np.ndarray, B: np.ndarray, offsets: np.ndarray) -> np.ndarray:
    """Ragged grouped GEMM ([1] "Optimisation 1": one call over all experts, each
    group computed at its own token count): C[R_e] = A[R_e] @ B[e]^T for the
    rows R_e = [offsets[e], offsets[e+1]).  A [M,K], B [E,N,K] -> C [M,N].
    Rows outside every group stay zero (there are none when offsets[E] = M)."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    E, N, K = B.shape
    C = np.zeros((A.shape[0], N))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            C[lo:hi] = A[lo:hi] @ B[e].T
    return C


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def swiglu(GU: np.ndarray) -> np.ndarray:
    """H = silu(G) * U with G the first f columns (gate) and U the last f (up)."""
    f = GU.shape[1] // 2
    G, U = GU[:, :f], GU[:, f:]
    return silu(G) * U


def expert_ffn(Xp, W1, W2, offsets):
    """The grouped MLP of [1] Figure 3: GEMM1 (gate+up), SwiGLU, GEMM2 (down)."""
    GU = grouped_gemm(Xp, W1, offsets)
    H = swiglu(GU)
    Yp = grouped_gemm(H, W2, offsets)
    return GU, H, Yp


# ----------------------------------------------------------------------------- combine

def combine(Yp: np.ndarray, dest_row: np.ndarray, w) -> np.ndarray:
    """y[t] = sum_j w[t,j] * Yp[dest_row[t,j]] ([1] "Optimisation 2": combine routes
    expert results back to the original token order and accumulates them).
    ``w=None`` means unit weights (the gradient of dispatch)."""
    Yp = np.asarray(Yp, dtype=np.float64)
    T, k = dest_row.shape
    y = np.zeros((T, Yp.shape[1]))
    for j in range(k):
        wj = 1.0 if w is None else np.asarray(w, dtype=np.float64)[:, j:j + 1]
        y += wj * Yp[dest_row[:, j]]
    return y


# ----------------------------------------------------------------------------- layer

def mx_roundtrip(a: np.ndarray) -> np.ndarray:
    """Values an MXFP8 operand carries: quantise row-wise along the last axis and
    dequantise exactly."""
    shp = a.shape
    a2 = np.asarray(a, dtype=np.float64).reshape(-1, shp[-1])
    return mxfp8.dequantize_rowwise(*mxfp8.quantize_rowwise(a2)).reshape(shp)


def nvfp4_roundtrip(a: np.ndarray) -> np.ndarray:
    """Values an NVFP4 operand carries: the whole array is one tensor (one fp32
    tensor scale), quantised row-wise along its last axis in blocks of 16."""
    shp = a.shape
    a2 = np.asarray(a, dtype=np.float32).reshape(-1, shp[-1])
    return nvfp4.dequantize(*nvfp4.quantize(a2)).reshape(shp)


def layer_forward(x, logits, W1, W2, k, renormalize=True, mxfp8_operands=False, nvfp4_operands=False):
    """Route -> dispatch -> grouped MLP -> combine ([3] "Method overview").

    With ``mxfp8_operands`` both GEMMs take MXFP8 operands (row-wise scales
    along the contraction): Xp, W1, H and W2 are each quantised and the GEMMs run
    on the exactly dequantised values.  ``nvfp4_operands`` does the same with
    NVFP4 (each of Xp, W1, H, W2 one tensor with its own tensor scale)."""
    E = W1.shape[0]
    idx, w, counts = route_topk(logits, k, renormalize)
    offsets, dest_row, src_pair = permute_maps(idx, E)
    Xp = permute(x, src_pair, k)
    if nvfp4_operands:
        Xq, W1q, W2q = nvfp4_roundtrip(Xp), nvfp4_roundtrip(W1), nvfp4_roundtrip(W2)
        GU = grouped_gemm(Xq, W1q, offsets)
        H = swiglu(GU)
        Yp = grouped_gemm(nvfp4_roundtrip(H), W2q, offsets)
    elif mxfp8_operands:
        Xq, W1q, W2q = mx_roundtrip(Xp), mx_roundtrip(W1), mx_roundtrip(W2)
        GU = grouped_gemm(Xq, W1q, offsets)
        H = swiglu(GU)
        Yp = grouped_gemm(mx_roundtrip(H), W2q, offsets)
    else:
        GU, H, Yp = expert_ffn(Xp, W1, W2, offsets)
    y = combine(Yp, dest_row, w)
    return dict(idx=idx, w=w, counts=counts, offsets=offsets, dest_row=dest_row,
                src_pair=src_pair, Xp=Xp, GU=GU, H=H, Yp=Yp, y=y)


# ----------------------------------------------------------------------------- capacity (contrast)

def permute_capacity(idx: np.ndarray, E: int, C: int):
    """Capacity-based dispatch, the contrast case of [1] (first section: a fixed
    per-expert capacity pads experts that get fewer tokens and drops the tokens
    that overflow).  Tokens are taken in order; each expert keeps its first C and
    drops the rest.  Expert e owns rows [e*C, (e+1)*C).

    Returns offsets [E+1] (= e*C), dest_row [T,k] (row, or -1 when dropped) and
    src_pair [E*C] (the pair t*k+j in each row, or -1 for padding)."""
    idx = np.asarray(idx)
    T, k = idx.shape
    dest = np.full((T, k), -1, dtype=np.int64)
    src = np.full(E * C, -1, dtype=np.int64)
    filled = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            if filled[e] < C:
                row = e * C + filled[e]
                dest[t, j] = row
                src[row] = t * k + j
            filled[e] += 1
    return np.arange(E + 1, dtype=np.int64) * C, dest, src


def permute_rows_capacity(x: np.ndarray, src_pair: np.ndarray, k: int) -> np.ndarray:
    """Rows of the capacity layout: the token of each kept pair, zeros for padding."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros((len(src_pair), x.shape[1]))
    kept = src_pair >= 0
    out[kept] = x[src_pair[kept] // k]
    return out


def combine_capacity(Yp: np.ndarray, dest_row: np.ndarray, w) -> np.ndarray:
    """y[t] = sum over the kept slots j of w[t,j] Yp[dest_row[t,j]]; dropped slots
    (dest_row -1) add nothing."""
    Yp = np.asarray(Yp, dtype=np.float64)
    T, k = dest_row.shape
    y = np.zeros((T, Yp.shape[1]))
    for j in range(k):
        kept = dest_row[:, j] >= 0
        wj = np.ones(T) if w is None else np.asarray(w, dtype=np.float64)[:, j]
        y[kept] += wj[kept, None] * Yp[dest_row[kept, j]]
    return y


def layer_forward_capacity(x, logits, W1, W2, k, C, renormalize=True):
    """The layer with capacity-based dispatch: route, keep each expert's first C
    tokens (zero-padded to C rows), the same SwiGLU experts over every row, combine
    the kept slots."""
    E = W1.shape[0]
    idx, w, counts = route_topk(logits, k, renormalize)
    offsets, dest_row, src_pair = permute_capacity(idx, E, C)
    Xp = permute_rows_capacity(x, src_pair, k)
    GU, H, Yp = expert_ffn(Xp, W1, W2, offsets)
    y = combine_capacity(Yp, dest_row, w)
    return dict(idx=idx, w=w, counts=counts, offsets=offsets, dest_row=dest_row, src_pair=src_pair,
                Xp=Xp, Yp=Yp, y=y)


# ----------------------------------------------------------------------------- backward

def combine_bwd(dy, Yp, dest_row, w):
    """Gradients of combine: dYp[dest_row[t,j]] = w[t,j] dy[t] and
    dw[t,j] = <dy[t], Yp[dest_row[t,j]]>."""
    dy = np.asarray(dy, dtype=np.float64)
    Yp = np.asarray(Yp, dtype=np.float64)
    T, k = dest_row.shape
    dYp = np.zeros_like(Yp)
    dw = np.zeros((T, k))
    for j in range(k):
        dYp[dest_row[:, j]] = np.asarray(w)[:, j:j + 1] * dy
        dw[:, j] = np.einsum("td,td->t", dy, Yp[dest_row[:, j]])
    return dYp, dw


def grouped_gemm_dgrad(dC, B, offsets):
    """Gradient of C = A B_e^T with respect to A: dA[R_e] = dC[R_e] @ B[e].
    dC [M,N], B [E,N,K] -> dA [M,K]."""
    dC = np.asarray(dC, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    dA = np.zeros((dC.shape[0], B.shape[2]))
    for e in range(B.shape[0]):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            dA[lo:hi] = dC[lo:hi] @ B[e]
    return dA


def grouped_gemm_wgrad(A, dC, offsets, E):
    """Gradient with respect to the expert weights: dB[e] = dC[R_e]^T @ A[R_e],
    a contraction over the ragged rows of each group; an empty group gives an
    exact zero gradient.  A [M,K], dC [M,N] -> dB [E,N,K]."""
    A = np.asarray(A, dtype=np.float64)
    dC = np.asarray(dC, dtype=np.float64)
    dB = np.zeros((E, dC.shape[1], A.shape[1]))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            dB[e] = dC[lo:hi].T @ A[lo:hi]
    return dB


def dswiglu(dH, GU):
    """Gradient of H = silu(G) * U:  dU = dH silu(G),
    dG = dH U sigma(G) (1 + G (1 - sigma(G)))."""
    f = GU.shape[1] // 2
    G, U = GU[:, :f], GU[:, f:]
    s = 1.0 / (1.0 + np.exp(-G))
    dG = dH * U * s * (1.0 + G * (1.0 - s))
    dU = dH * G * s
    return np.concatenate([dG, dU], axis=1)


def route_bwd(dw, w, idx, logits, renormalize=True):
    """Gradient of the routing weights with respect to the logits.

    Renormalised: the weights are a softmax over the selected logits, so
    dl_i = w_i (dw_i - sum_j w_j dw_j) on the selection and 0 elsewhere.
    Otherwise the weights are full-softmax probabilities p of the selected
    experts: dl_e = p_e (g_e - sum_j w_j dw_j) with g_e = dw_j if e = idx_j
    else 0.  The selection itself is piecewise constant and has no gradient."""
    dw = np.asarray(dw, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T, k = idx.shape
    E = logits.shape[1]
    inner = (w * dw).sum(axis=1, keepdims=True)
    dl = np.zeros((T, E))
    rows = np.arange(T)[:, None]
    if renormalize:
        dl[rows, idx] = w * (dw - inner)
    else:
        l64 = np.asarray(logits, dtype=np.float64)
        m = l64.max(axis=1, keepdims=True)
        masked = np.isneginf(m)                    # every expert masked: no probability mass
        p = np.where(masked, 0.0, np.exp(l64 - np.where(masked, 0.0, m)))
        p /= np.where(masked, 1.0, p.sum(axis=1, keepdims=True))
        g = np.zeros((T, E))
        g[rows, idx] = dw
        dl = p * (g - inner)
    return dl


def mx_roundtrip_dim1(W: np.ndarray) -> np.ndarray:
    """Values of a weight stack W [E, R, C] quantised along R (its output dim), as
    the data gradient reads it: blocks of 32 consecutive rows of one column."""
    Wt = np.ascontiguousarray(np.asarray(W, dtype=np.float64).transpose(0, 2, 1))
    return mx_roundtrip(Wt).transpose(0, 2, 1)


def mx_roundtrip_colwise(a: np.ndarray, offsets: np.ndarray) -> np.ndarray:
    """Values of a [rows, K] operand quantised column-wise and group-aware, as the
    weight gradient reads it (blocks of 32 rows restarting at each group)."""
    c, s = mxfp8.quantize_colwise_grouped(a, offsets)
    return mxfp8.dequantize_colwise_grouped(c, s, offsets)


def layer_backward(fwd, dy, x, logits, W1, W2, k, renormalize=True, mxfp8_operands=False):
    """The full backward of ``layer_forward``, returning dx, dlogits, dW1, dW2 and
    the intermediates dYp, dw, dGU, dXp.

    With ``mxfp8_operands`` every backward GEMM takes MXFP8 operands quantised
    along its own contraction dim ([1] "grouped quantisation"): the data
    gradients read dYp / dGU row-wise and W2 / W1 along their output dim; the
    weight gradients read H, dYp, Xp and dGU column-wise, group-aware."""
    E = W1.shape[0]
    offsets, dest_row = fwd["offsets"], fwd["dest_row"]
    dYp, dw = combine_bwd(dy, fwd["Yp"], dest_row, fwd["w"])
    if mxfp8_operands:
        dH = grouped_gemm_dgrad(mx_roundtrip(dYp), mx_roundtrip_dim1(W2), offsets)
        dGU = dswiglu(dH, fwd["GU"])
        dW2 = grouped_gemm_wgrad(mx_roundtrip_colwise(fwd["H"], offsets), mx_roundtrip_colwise(dYp, offsets),
                                 offsets, E)
        dXp = grouped_gemm_dgrad(mx_roundtrip(dGU), mx_roundtrip_dim1(W1), offsets)
        dW1 = grouped_gemm_wgrad(mx_roundtrip_colwise(fwd["Xp"], offsets), mx_roundtrip_colwise(dGU, offsets),
                                 offsets, E)
    else:
        dH = grouped_gemm_dgrad(dYp, W2, offsets)
        dGU = dswiglu(dH, fwd["GU"])
        dW2 = grouped_gemm_wgrad(fwd["H"], dYp, offsets, E)
        dXp = grouped_gemm_dgrad(dGU, W1, offsets)
        dW1 = grouped_gemm_wgrad(fwd["Xp"], dGU, offsets, E)
    dx = combine(dXp, dest_row, None)
    dlogits = route_bwd(dw, fwd["w"], fwd["idx"], logits, renormalize)
    return dict(dYp=dYp, dw=dw, dH=dH, dGU=dGU, dW2=dW2, dXp=dXp, dW1=dW1, dx=dx,
                dlogits=dlogits)


# ----------------------------------------------------------------------------- per-token form

def token_forward(x_t, logits_t, W1, W2, k, renormalize=True, mxfp8_operands=False):
    """Output of one token, y[t] = sum_j w_j FFN_{e_j}(x[t]); used to check
    large workloads on sampled tokens (a token's output depends only on its own
    activations, its logits and the weights of the experts it chose).
    W1/W2 may be callables e -> expert weights, so large weights can be fetched
    one expert at a time."""
    idx, w, _ = route_topk(np.asarray(logits_t, dtype=np.float32)[None, :], k, renormalize)
    get1 = W1 if callable(W1) else (lambda e: W1[e])
    get2 = W2 if callable(W2) else (lambda e: W2[e])
    xt = np.asarray(x_t, dtype=np.float64)[None, :]
    if mxfp8_operands:
        xt = mx_roundtrip(xt)
    y = np.zeros(xt.shape[1])
    for j in range(k):
        e = int(idx[0, j])
        w1, w2 = np.asarray(get1(e), np.float64), np.asarray(get2(e), np.float64)
        if mxfp8_operands:
            w1, w2 = mx_roundtrip(w1), mx_roundtrip(w2)
        h = swiglu(xt @ w1.T)
        if mxfp8_operands:
            h = mx_roundtrip(h)
        y += w[0, j] * (h @ w2.T)[0]
    return y


def token_backward(x_t, logits_t, dy_t, W1, W2, k, renormalize=True):
    """Backward of one token's output y[t] = sum_j w_j FFN_{e_j}(x[t]) with upstream
    gradient dy[t]: returns (dx[t], dlogits[t]).  The same steps as
    ``layer_backward`` restricted to one token (a token's gradients depend only on
    its own row, logits, upstream gradient and its experts' weights).  W1/W2 may be
    callables e -> expert weights."""
    lg = np.asarray(logits_t, dtype=np.float32)[None, :]
    idx, w, _ = route_topk(lg, k, renormalize)
    get1 = W1 if callable(W1) else (lambda e: W1[e])
    get2 = W2 if callable(W2) else (lambda e: W2[e])
    xt = np.asarray(x_t, dtype=np.float64)[None, :]
    dyt = np.asarray(dy_t, dtype=np.float64)[None, :]
    dx = np.zeros(xt.shape[1])
    dw = np.zeros((1, k))
    for j in range(k):
        e = int(idx[0, j])
        w1, w2 = np.asarray(get1(e), np.float64), np.asarray(get2(e), np.float64)
        GU = xt @ w1.T
        yp = swiglu(GU) @ w2.T
        dw[0, j] = float((dyt * yp).sum())
        dH = (w[0, j] * dyt) @ w2
        dx += (dswiglu(dH, GU) @ w1)[0]
    dl = route_bwd(dw, w, idx, lg, renormalize)[0]
    return dx, dl


def expert_backward_mxfp8(X_e, dYp_e, w1, w2):
    """Forward and backward of one expert on MXFP8 operands, from its own rows X_e
    [c, d] and upstream dYp_e [c, d]; w1 [2f, d], w2 [d, f].  Every quantisation
    of the layer's MXFP8 step is local to the expert: row-wise blocks lie in a row,
    the weights' blocks in the expert's own weights, and the column-wise blocks of
    the weight gradients restart at the group's first row, which is X_e's first.
    Returns GU, H, dGU, dXp, dW1, dW2 (the same values ``layer_backward`` with
    ``mxfp8_operands`` gives for this expert)."""
    X = np.asarray(X_e, dtype=np.float64)
    dY = np.asarray(dYp_e, dtype=np.float64)
    w1 = np.asarray(w1, dtype=np.float64)
    w2 = np.asarray(w2, dtype=np.float64)
    one = np.array([0, X.shape[0]])
    GU = mx_roundtrip(X) @ mx_roundtrip(w1).T
    H = swiglu(GU)
    dH = mx_roundtrip(dY) @ mx_roundtrip_dim1(w2[None])[0]
    dGU = dswiglu(dH, GU)
    dXp = mx_roundtrip(dGU) @ mx_roundtrip_dim1(w1[None])[0]
    dW2 = mx_roundtrip_colwise(dY, one).T @ mx_roundtrip_colwise(H, one)
    dW1 = mx_roundtrip_colwise(dGU, one).T @ mx_roundtrip_colwise(X, one)
    return dict(GU=GU, H=H, dGU=dGU, dXp=dXp, dW1=dW1, dW2=dW2)


def expert_wgrad_sampled(X_e, dYp_e, w1, w2, w1_rows, w2_cols):
    """Selected rows of dW1[e] and columns of dW2[e] for one expert, from its own
    rows X_e [c, d] and upstream dYp_e [c, d]; w1 [2f, d], w2 [d, f].

    Row n of dW1 = sum_r dGU[r, n] X_e[r]; dGU[:, n] needs only the gate/up
    columns n mod f of GU and column n mod f of dH = dYp_e w2.  Column c of dW2 =
    sum_r dYp_e[r] H[r, c]; H[:, c] needs gate/up columns c.  So each sampled row or
    column costs O(rows * d) and the full [c, 2f] intermediates are never formed."""
    X = np.asarray(X_e, dtype=np.float64)
    dY = np.asarray(dYp_e, dtype=np.float64)
    w1 = np.asarray(w1, dtype=np.float64)
    w2 = np.asarray(w2, dtype=np.float64)
    f = w2.shape[1]

    def cols(c):
        g = X @ w1[c]
        u = X @ w1[f + c]
        return g, u

    dw1 = np.zeros((len(w1_rows), X.shape[1]))
    for i, n in enumerate(w1_rows):
        c = int(n) % f
        g, u = cols(c)
        dh = dY @ w2[:, c]
        s = 1.0 / (1.0 + np.exp(-g))
        dgu = dh * u * s * (1.0 + g * (1.0 - s)) if n < f else dh * g * s
        dw1[i] = dgu @ X
    dw2 = np.zeros((w2.shape[0], len(w2_cols)))
    for i, c in enumerate(w2_cols):
        g, u = cols(int(c))
        h = silu(g) * u
        dw2[:, i] = dY.T @ h
    return dw1, dw2


def tokens_forward(x_rows, logits_rows, W1, W2, k, renormalize=True, mxfp8_operands=False):
    """``token_forward`` for several tokens at once, visiting each expert once: for
    expert e (ascending id), every (token, slot) routed to it adds w * FFN_e(x[t]).
    The same per-token sums as ``token_forward``; W1/W2 may be callables
    e -> expert weights, each called once per expert the tokens use (so a large
    layer's weights can be fetched one expert at a time)."""
    lg = np.asarray(logits_rows, dtype=np.float32)
    idx, w, _ = route_topk(lg, k, renormalize)
    get1 = W1 if callable(W1) else (lambda e: W1[e])
    get2 = W2 if callable(W2) else (lambda e: W2[e])
    X = np.asarray(x_rows, dtype=np.float64)
    if mxfp8_operands:
        X = mx_roundtrip(X)
    y = np.zeros_like(X)
    for e in np.unique(idx):
        w1, w2 = np.asarray(get1(int(e)), np.float64), np.asarray(get2(int(e)), np.float64)
        if mxfp8_operands:
            w1, w2 = mx_roundtrip(w1), mx_roundtrip(w2)
        t, j = np.nonzero(idx == e)
        h = swiglu(X[t] @ w1.T)
        if mxfp8_operands:
            h = mx_roundtrip(h)
        y[t] += w[t, j][:, None] * (h @ w2.T)
    return y


def tokens_backward(x_rows, logits_rows, dy_rows, W1, W2, k, renormalize=True):
    """``token_backward`` for several tokens at once, visiting each expert once:
    returns (dx [n, d], dlogits [n, E]).  W1/W2 may be callables e -> weights."""
    lg = np.asarray(logits_rows, dtype=np.float32)
    idx, w, _ = route_topk(lg, k, renormalize)
    get1 = W1 if callable(W1) else (lambda e: W1[e])
    get2 = W2 if callable(W2) else (lambda e: W2[e])
    X = np.asarray(x_rows, dtype=np.float64)
    dY = np.asarray(dy_rows, dtype=np.float64)
    dx = np.zeros_like(X)
    dw = np.zeros(idx.shape)
    for e in np.unique(idx):
        w1, w2 = np.asarray(get1(int(e)), np.float64), np.asarray(get2(int(e)), np.float64)
        t, j = np.nonzero(idx == e)
        GU = X[t] @ w1.T
        dw[t, j] = np.einsum("nd,nd->n", dY[t], swiglu(GU) @ w2.T)
        dH = (w[t, j][:, None] * dY[t]) @ w2
        np.add.at(dx, t, dswiglu(dH, GU) @ w1)
    return dx, route_bwd(dw, w, idx, lg, renormalize)

"""Pins for the oracle's grouped MLP, combine and backward (CPU only).

Pinned against: the dense masked-MoE formula (every expert applied to every
token, masked by the routing weights) written with torch float64 ops; a dense
SwiGLU FFN (E=1, k=1); torch.bmm when every expert has the same number of rows;
torch float64 autograd of the dense formula, itself checked by gradcheck
(finite differences).
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import moe


def _problem(T, d, E, k, f, seed, empty=()):
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    for e in empty:
        lg[:, e] -= 30.0
    x = rng.standard_normal((T, d))
    W1 = rng.standard_normal((E, 2 * f, d)) / np.sqrt(d)
    W2 = rng.standard_normal((E, d, f)) / np.sqrt(f)
    return lg, x, W1, W2


def _dense_masked_torch(x, logits, W1, W2, idx, renormalize=True):
    """y[t] = sum_e g[t,e] * FFN_e(x[t]) over ALL experts, with g the routing
    weights on the selected experts and 0 elsewhere.  Differentiable in torch."""
    T, E = logits.shape
    k = idx.shape[1]
    f = W2.shape[2]
    if renormalize:
        g_sel = torch.softmax(torch.gather(logits, 1, idx), dim=1)
    else:
        g_sel = torch.gather(torch.softmax(logits, dim=1), 1, idx)
    g = torch.zeros(T, E, dtype=logits.dtype).scatter(1, idx, g_sel)
    y = torch.zeros(T, W2.shape[1], dtype=x.dtype)
    for e in range(E):
        gu = x @ W1[e].T
        h = F.silu(gu[:, :f]) * gu[:, f:]
        y = y + g[:, e:e + 1] * (h @ W2[e].T)
    return y


@pytest.mark.parametrize("T,d,E,k,f,empty", [(40, 16, 6, 2, 12, (3,)), (25, 8, 4, 4, 8, ()),
                                             (30, 12, 8, 1, 10, (0, 5))])
def test_layer_equals_dense_masked_moe(T, d, E, k, f, empty):
    lg, x, W1, W2 = _problem(T, d, E, k, f, seed=T, empty=empty)
    fwd = moe.layer_forward(x, lg, W1, W2, k)
    idx = torch.from_numpy(fwd["idx"].astype(np.int64))
    want = _dense_masked_torch(torch.from_numpy(x), torch.from_numpy(lg.astype(np.float64)),
                               torch.from_numpy(W1), torch.from_numpy(W2), idx)
    np.testing.assert_allclose(fwd["y"], want.numpy(), rtol=1e-11, atol=1e-12)
    for e in empty:
        assert fwd["counts"][e] == 0


def test_single_expert_is_dense_swiglu_ffn():
    T, d, f = 33, 16, 20
    lg, x, W1, W2 = _problem(T, d, 1, 1, f, seed=11)
    fwd = moe.layer_forward(x, lg, W1, W2, 1)
    xt, w1, w2 = map(torch.from_numpy, (x, W1[0], W2[0]))
    want = (F.silu(xt @ w1[:f].T) * (xt @ w1[f:].T)) @ w2.T
    np.testing.assert_allclose(fwd["y"], want.numpy(), rtol=1e-12, atol=1e-13)
    assert (fwd["src_pair"] == np.arange(T)).all()


def test_equal_counts_is_bmm():
    E, per, K, N = 5, 7, 12, 9
    rng = np.random.default_rng(4)
    A = rng.standard_normal((E * per, K))
    B = rng.standard_normal((E, N, K))
    offsets = np.arange(E + 1) * per
    C = moe.grouped_gemm(A, B, offsets)
    want = torch.bmm(torch.from_numpy(A).view(E, per, K), torch.from_numpy(B).transpose(1, 2))
    np.testing.assert_allclose(C, want.reshape(E * per, N).numpy(), rtol=1e-13)
    dC = rng.standard_normal((E * per, N))
    dA = moe.grouped_gemm_dgrad(dC, B, offsets)
    np.testing.assert_allclose(dA, torch.bmm(torch.from_numpy(dC).view(E, per, N),
                                             torch.from_numpy(B)).reshape(E * per, K).numpy(),
                               rtol=1e-13)
    dB = moe.grouped_gemm_wgrad(A, dC, offsets, E)
    np.testing.assert_allclose(dB, torch.bmm(torch.from_numpy(dC).view(E, per, N).transpose(1, 2),
                                             torch.from_numpy(A).view(E, per, K)).numpy(),
                               rtol=1e-13)


def test_empty_group_zero_wgrad_and_untouched_rows():
    offsets = np.array([0, 3, 3, 8])
    rng = np.random.default_rng(6)
    A, dC = rng.standard_normal((8, 4)), rng.standard_normal((8, 5))
    dB = moe.grouped_gemm_wgrad(A, dC, offsets, 3)
    assert (dB[1] == 0).all()
    np.testing.assert_allclose(dB[0], dC[:3].T @ A[:3])


@pytest.mark.parametrize("renormalize", [True, False])
def test_backward_matches_torch_autograd(renormalize):
    T, d, E, k, f = 24, 10, 6, 3, 8
    lg, x, W1, W2 = _problem(T, d, E, k, f, seed=21, empty=(2,))
    rng = np.random.default_rng(22)
    dy = rng.standard_normal((T, d))
    fwd = moe.layer_forward(x, lg, W1, W2, k, renormalize)
    bwd = moe.layer_backward(fwd, dy, x, lg, W1, W2, k, renormalize)

    tx, tl, t1, t2 = (torch.from_numpy(a).clone().requires_grad_(True)
                      for a in (x, lg.astype(np.float64), W1, W2))
    idx = torch.from_numpy(fwd["idx"].astype(np.int64))
    y = _dense_masked_torch(tx, tl, t1, t2, idx, renormalize)
    np.testing.assert_allclose(fwd["y"], y.detach().numpy(), rtol=1e-11, atol=1e-12)
    (y * torch.from_numpy(dy)).sum().backward()
    for name, t in (("dx", tx), ("dlogits", tl), ("dW1", t1), ("dW2", t2)):
        np.testing.assert_allclose(bwd[name], t.grad.numpy(), rtol=1e-10, atol=1e-12, err_msg=name)
    assert (bwd["dW1"][2] == 0).all() and (bwd["dW2"][2] == 0).all()
    if renormalize:
        sel = np.zeros((T, E), dtype=bool)
        np.put_along_axis(sel, fwd["idx"].astype(np.int64), True, axis=1)
        assert (bwd["dlogits"][~sel] == 0).all()
        np.testing.assert_allclose(bwd["dlogits"].sum(axis=1), 0.0, atol=1e-12)


def test_dense_formula_gradcheck():
    """Finite differences pin the torch formula used above."""
    T, d, E, k, f = 5, 4, 3, 2, 3
    lg, x, W1, W2 = _problem(T, d, E, k, f, seed=3)
    idx, _, _ = moe.route_topk(lg, k)
    idx = torch.from_numpy(idx.astype(np.int64))
    args = tuple(torch.from_numpy(a).clone().requires_grad_(True)
                 for a in (x, lg.astype(np.float64), W1, W2))
    assert torch.autograd.gradcheck(lambda *a: _dense_masked_torch(*a, idx), args)


def test_dswiglu_against_autograd():
    rng = np.random.default_rng(8)
    GU = rng.standard_normal((7, 10)) * 3
    dH = rng.standard_normal((7, 5))
    t = torch.from_numpy(GU).requires_grad_(True)
    h = F.silu(t[:, :5]) * t[:, 5:]
    h.backward(torch.from_numpy(dH))
    np.testing.assert_allclose(moe.dswiglu(dH, GU), t.grad.numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(moe.swiglu(GU), h.detach().numpy(), rtol=1e-13)


def test_token_forward_matches_layer():
    T, d, E, k, f = 20, 8, 5, 2, 6
    lg, x, W1, W2 = _problem(T, d, E, k, f, seed=31)
    fwd = moe.layer_forward(x, lg, W1, W2, k)
    for t in (0, 7, 19):
        np.testing.assert_allclose(moe.token_forward(x[t], lg[t], W1, W2, k), fwd["y"][t],
                                   rtol=1e-12, atol=1e-13)


def test_mxfp8_layer_close_to_exact_layer():
    """MXFP8 operands perturb each element by at most 2^-4 relative; the layer
    output stays within a few percent, and the per-token form agrees exactly."""
    T, d, E, k, f = 40, 64, 4, 2, 32
    lg, x, W1, W2 = _problem(T, d, E, k, f, seed=41)
    exact = moe.layer_forward(x, lg, W1, W2, k)["y"]
    fwd = moe.layer_forward(x, lg, W1, W2, k, mxfp8_operands=True)
    rel = np.linalg.norm(fwd["y"] - exact) / np.linalg.norm(exact)
    assert 1e-3 < rel < 0.1
    for t in (0, 13, 39):
        np.testing.assert_allclose(moe.token_forward(x[t], lg[t], W1, W2, k, mxfp8_operands=True),
                                   fwd["y"][t], rtol=1e-12, atol=1e-13)


def test_token_backward_matches_layer_backward():
    T, d, E, k, f = 20, 8, 5, 2, 6
    lg, x, W1, W2 = _problem(T, d, E, k, f, seed=51)
    dy = np.random.default_rng(52).standard_normal((T, d))
    fwd = moe.layer_forward(x, lg, W1, W2, k)
    bwd = moe.layer_backward(fwd, dy, x, lg, W1, W2, k)
    for t in (0, 11, 19):
        dx, dl = moe.token_backward(x[t], lg[t], dy[t], W1, W2, k)
        np.testing.assert_allclose(dx, bwd["dx"][t], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(dl, bwd["dlogits"][t], rtol=1e-11, atol=1e-13)


def test_expert_wgrad_sampled_matches_full_wgrad():
    T, d, E, k, f = 30, 8, 4, 2, 6
    lg, x, W1, W2 = _problem(T, d, E, k, f, seed=61)
    dy = np.random.default_rng(62).standard_normal((T, d))
    fwd = moe.layer_forward(x, lg, W1, W2, k)
    bwd = moe.layer_backward(fwd, dy, x, lg, W1, W2, k)
    off = fwd["offsets"]
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        rows = [0, f - 1, f, 2 * f - 1]
        cols = [0, 3, f - 1]
        dw1, dw2 = moe.expert_wgrad_sampled(fwd["Xp"][lo:hi], bwd["dYp"][lo:hi], W1[e], W2[e], rows, cols)
        np.testing.assert_allclose(dw1, bwd["dW1"][e][rows], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(dw2, bwd["dW2"][e][:, cols], rtol=1e-11, atol=1e-13)


def _block_values(v, lo, hi):
    """Values of v[lo:hi] (one column of one group) under blocks of 32 starting at
    lo, each quantised by the row-wise quantiser as one zero-padded row."""
    from oracle import mxfp8
    out = np.zeros(hi - lo)
    for r0 in range(lo, hi, 32):
        r1 = min(r0 + 32, hi)
        blk = np.zeros((1, 32))
        blk[0, :r1 - r0] = v[r0:r1]
        out[r0 - lo:r1 - lo] = mxfp8.dequantize_rowwise(*mxfp8.quantize_rowwise(blk))[0, :r1 - r0]
    return out


def _row_values(v):
    from oracle import mxfp8
    return mxfp8.dequantize_rowwise(*mxfp8.quantize_rowwise(np.asarray(v, dtype=np.float64)[None, :]))[0]


def test_mxfp8_backward_elements_from_blockwise_quantisation():
    """Each MXFP8 backward GEMM, element by element: operands quantised along that
    GEMM's own contraction, built here one block at a time through the row-wise
    quantiser (pinned on its own) rather than through the layer's helpers."""
    T, d, E, k, f = 48, 64, 3, 2, 32
    lg, x, W1, W2 = _problem(T, d, E, k, f, seed=71)
    dy = np.random.default_rng(72).standard_normal((T, d))
    fwd = moe.layer_forward(x, lg, W1, W2, k, mxfp8_operands=True)
    bwd = moe.layer_backward(fwd, dy, x, lg, W1, W2, k, mxfp8_operands=True)
    off = fwd["offsets"]
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi - lo < 2:
            continue
        for i, j in ((0, 0), (d - 1, 5), (17, f - 1)):          # dW2[e][i, j]: contraction over the group's rows
            want = _block_values(bwd["dYp"][:, i], lo, hi) @ _block_values(fwd["H"][:, j], lo, hi)
            np.testing.assert_allclose(bwd["dW2"][e][i, j], want, rtol=1e-12, atol=1e-14)
        for m, c in ((0, 0), (2 * f - 1, d - 1), (f, 9)):       # dW1[e][m, c]
            want = _block_values(bwd["dGU"][:, m], lo, hi) @ _block_values(fwd["Xp"][:, c], lo, hi)
            np.testing.assert_allclose(bwd["dW1"][e][m, c], want, rtol=1e-12, atol=1e-14)
        for r in (lo, hi - 1):                                  # data gradients: contraction over d / 2f
            for j in (0, f - 1):
                want = _row_values(bwd["dYp"][r]) @ _row_values(W2[e][:, j])
                np.testing.assert_allclose(bwd["dH"][r, j], want, rtol=1e-12, atol=1e-14)
            for c in (0, d - 1):
                want = _row_values(bwd["dGU"][r]) @ _row_values(W1[e][:, c])
                np.testing.assert_allclose(bwd["dXp"][r, c], want, rtol=1e-12, atol=1e-14)


def test_mxfp8_backward_close_to_exact():
    """The MXFP8 gradients stay within the format's error of the exact ones: E4M3
    keeps 3 mantissa bits (about 3.6% rms relative error per quantised operand),
    and dx passes through two quantised data gradients, each with both operands
    quantised, after a quantised forward; a transposed operand or a wrong group
    would be off by order one."""
    T, d, E, k, f = 64, 64, 4, 2, 32
    lg, x, W1, W2 = _problem(T, d, E, k, f, seed=81)
    dy = np.random.default_rng(82).standard_normal((T, d))
    fwd = moe.layer_forward(x, lg, W1, W2, k)
    exact = moe.layer_backward(fwd, dy, x, lg, W1, W2, k)
    fwd_mx = moe.layer_forward(x, lg, W1, W2, k, mxfp8_operands=True)
    mx = moe.layer_backward(fwd_mx, dy, x, lg, W1, W2, k, mxfp8_operands=True)
    for name in ("dx", "dW1", "dW2", "dlogits"):
        err = np.linalg.norm(mx[name] - exact[name]) / np.linalg.norm(exact[name])
        assert 0 < err < 0.2, (name, err)


def test_nvfp4_layer_forward_close_to_exact_and_exact_on_representable_operands():
    """The NVFP4 layer stays within FP4's error of the exact one (E2M1 keeps one
    mantissa bit), and the round trip of a whole weight stack (one tensor scale
    across the experts) is the identity on representable values."""
    from oracle import nvfp4
    T, d, E, k, f = 48, 64, 4, 2, 32
    lg, x, W1, W2 = _problem(T, d, E, k, f, seed=91)
    exact = moe.layer_forward(x, lg, W1, W2, k)
    fp4 = moe.layer_forward(x, lg, W1, W2, k, nvfp4_operands=True)
    err = np.linalg.norm(fp4["y"] - exact["y"]) / np.linalg.norm(exact["y"])
    assert 0 < err < 0.35, err
    # representable weights: E2M1 values with a 6 in every 16-element block, so the
    # tensor scale is 448, every block scale 448 and every element maps to itself
    rng = np.random.default_rng(92)
    vals = np.array([0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    def rep(shape):
        a = rng.choice(vals, size=shape) * rng.choice([-1.0, 1.0], size=shape)
        a[..., ::16] = 6.0
        return a
    W1r, W2r = rep((E, 2 * f, d)), rep((E, d, f))
    assert np.array_equal(moe.nvfp4_roundtrip(W1r), W1r)
    assert np.array_equal(nvfp4.dequantize(*nvfp4.quantize(W2r.reshape(-1, f))).reshape(W2r.shape), W2r)


def test_expert_backward_mxfp8_matches_layer_backward():
    """The per-expert MXFP8 backward (used to check full-size layers expert by expert)
    equals the whole-layer MXFP8 backward restricted to each expert."""
    T, d, E, k, f = 60, 64, 4, 2, 32
    lg, x, W1, W2 = _problem(T, d, E, k, f, seed=101)
    dy = np.random.default_rng(102).standard_normal((T, d))
    fwd = moe.layer_forward(x, lg, W1, W2, k, mxfp8_operands=True)
    bwd = moe.layer_backward(fwd, dy, x, lg, W1, W2, k, mxfp8_operands=True)
    off = fwd["offsets"]
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        got = moe.expert_backward_mxfp8(fwd["Xp"][lo:hi], bwd["dYp"][lo:hi], W1[e], W2[e])
        np.testing.assert_allclose(got["GU"], fwd["GU"][lo:hi], rtol=1e-12, atol=1e-13)
        for name in ("dGU", "dXp"):
            np.testing.assert_allclose(got[name], bwd[name][lo:hi], rtol=1e-12, atol=1e-13, err_msg=name)
        np.testing.assert_allclose(got["dW1"], bwd["dW1"][e], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(got["dW2"], bwd["dW2"][e], rtol=1e-12, atol=1e-13)


def _mx_blockwise_row(v):
    """MXFP8 values of one row along its length, each 32-element block quantised on
    its own (a [1, 32] call of the row-wise quantiser, pinned separately)."""
    from oracle import mxfp8
    v = np.asarray(v, dtype=np.float64)
    out = np.empty_like(v)
    for b in range(0, v.size, 32):
        blk = v[None, b:b + 32]
        out[b:b + 32] = mxfp8.dequantize_rowwise(*mxfp8.quantize_rowwise(blk))[0]
    return out


def _fp32_tensor_scale(a):
    """NVFP4 tensor encode scale of a whole tensor, from its definition:
    fp32(2688 / fp32(amax)), 1 for an all-zero tensor."""
    amax = np.float32(np.abs(np.asarray(a, dtype=np.float32)).max())
    return np.float32(1.0) if amax == 0 else np.float32(np.float32(2688.0) / amax)


def _nv_blockwise_row(v, g):
    """NVFP4 values of one row, each 16-element block quantised on its own with the
    given tensor scale g (a [1, 16] call of the pinned NVFP4 quantiser)."""
    from oracle import nvfp4
    v = np.asarray(v, dtype=np.float32)
    out = np.empty(v.size)
    for b in range(0, v.size, 16):
        c, s, gg = nvfp4.quantize(v[None, b:b + 16], g=g)
        out[b:b + 16] = nvfp4.dequantize(c, s, gg)[0]
    return out


def _silu_mul_torch(g, u):
    return (F.silu(torch.from_numpy(np.asarray(g, dtype=np.float64))) *
            torch.from_numpy(np.asarray(u, dtype=np.float64))).numpy()


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_blockscaled_forward_elements_from_blockwise_quantisation(fmt):
    """Each block-scaled forward GEMM element by element, with its operands built
    here one block at a time: GU[r, n] = <q(Xp[r]), q(W1[e][n])>, H = silu(G) U
    (torch), Yp[r, c] = <q(H[r]), q(W2[e][c])>, y = sum_j w_j Yp[dest_row[t, j]].
    MXFP8 blocks are 32 elements with their own E8M0 scale; NVFP4 blocks are 16
    elements with an E4M3 scale under one fp32 tensor scale per tensor: one for
    Xp, one for the whole W1 stack (every expert), one for H, one for the whole W2
    stack."""
    T, d, E, k, f = 40, 64, 3, 2, 32
    lg, x, W1, W2 = _problem(T, d, E, k, f, seed=111)
    if fmt == "nvfp4":
        x, W1, W2 = (np.asarray(a, dtype=np.float32).astype(np.float64) for a in (x, W1, W2))
    fwd = moe.layer_forward(x, lg, W1, W2, k, mxfp8_operands=fmt == "mxfp8", nvfp4_operands=fmt == "nvfp4")
    off, src = fwd["offsets"], fwd["src_pair"]
    Xp = x[src // k]
    if fmt == "mxfp8":
        qx = qw1 = qh = qw2 = _mx_blockwise_row
    else:
        g_x, g_w1, g_w2 = _fp32_tensor_scale(Xp), _fp32_tensor_scale(W1), _fp32_tensor_scale(W2)
        qx = lambda v: _nv_blockwise_row(v, g_x)      # noqa: E731
        qw1 = lambda v: _nv_blockwise_row(v, g_w1)    # noqa: E731
        qw2 = lambda v: _nv_blockwise_row(v, g_w2)    # noqa: E731
    # GU and H of every row, from the blockwise operands
    GU = np.zeros((T * k, 2 * f))
    for e in range(E):
        for r in range(int(off[e]), int(off[e + 1])):
            xr = qx(Xp[r])
            GU[r] = [xr @ qw1(W1[e][n]) for n in range(2 * f)]
    np.testing.assert_allclose(fwd["GU"], GU, rtol=1e-12, atol=1e-13)
    H = _silu_mul_torch(GU[:, :f], GU[:, f:])
    np.testing.assert_allclose(fwd["H"], H, rtol=1e-12, atol=1e-13)
    if fmt == "nvfp4":
        g_h = _fp32_tensor_scale(H)
        qh = lambda v: _nv_blockwise_row(v, g_h)      # noqa: E731
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        for r in sorted({lo, (lo + hi) // 2, hi - 1} & set(range(lo, hi))):
            hr = qh(H[r])
            for c in (0, 7, d - 1):
                np.testing.assert_allclose(fwd["Yp"][r, c], hr @ qw2(W2[e][c]), rtol=1e-12, atol=1e-13)
    for t in (0, T // 2, T - 1):
        want = sum(fwd["w"][t, j] * fwd["Yp"][fwd["dest_row"][t, j]] for j in range(k))
        np.testing.assert_allclose(fwd["y"][t], want, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("mx", [False, True])
def test_tokens_forward_and_backward_match_layer(mx):
    """The expert-major forms (each expert's weights fetched once) give the layer's
    rows: forward with and without MXFP8 operands, backward (dx, dlogits)."""
    T, d, E, k, f = 30, 64, 5, 2, 32
    lg, x, W1, W2 = _problem(T, d, E, k, f, seed=121, empty=(1,))
    dy = np.random.default_rng(122).standard_normal((T, d))
    fwd = moe.layer_forward(x, lg, W1, W2, k, mxfp8_operands=mx)
    toks = np.array([0, 3, 17, 29])
    fetched = []
    def get1(e):
        fetched.append(e)
        return W1[e]
    y = moe.tokens_forward(x[toks], lg[toks], get1, lambda e: W2[e], k, mxfp8_operands=mx)
    np.testing.assert_allclose(y, fwd["y"][toks], rtol=1e-12, atol=1e-13)
    assert len(fetched) == len(set(fetched))
    if not mx:
        bwd = moe.layer_backward(fwd, dy, x, lg, W1, W2, k)
        dx, dl = moe.tokens_backward(x[toks], lg[toks], dy[toks], W1, W2, k)
        np.testing.assert_allclose(dx, bwd["dx"][toks], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(dl, bwd["dlogits"][toks], rtol=1e-11, atol=1e-13)

"""End-to-end parity of the whole layer (route -> dispatch -> grouped MLP ->
combine) on the seeded workloads, through MoELayer (the launch sequence the
benchmark times).

The tiny workload is checked in full against the float64 oracle.  The large
ones are checked in full for every integer output and on samples for the
floating ones: a token's output depends only on its own row, its logits and
its experts' weights, so the oracle evaluates sampled tokens one by one, and
sampled rows of each grouped GEMM stage for a set of experts (hottest, median,
smallest non-empty, and random ones).
"""

import numpy as np
import pytest
import torch

import ragged_grouped_gemm_topk_gb300 as moe_gpu
from ragged_grouped_gemm_topk_gb300 import workloads as W
from oracle import moe as om
from oracle import mxfp8 as omx
from _parity import TOL_BF16, TOL_MXFP8, f64, i64, logits_dev, need_gpu, rel_l2

pytestmark = pytest.mark.gpu


def _build(w, training=False):
    x = W.make_x(w, "cuda")
    W1 = W.make_w1(w, "cuda")
    W2 = W.make_w2(w, "cuda")
    lg = logits_dev(w)
    layer = moe_gpu.MoELayer(w.T, w.d, w.E, w.k, w.f, W1, W2, dtype=w.dtype,
                             renormalize=w.renormalize, training=training)
    return layer, x, W1, W2, lg


def test_tiny_fp32_full():
    need_gpu()
    w = W.BY_NAME["tiny-fp32"]
    layer, x, W1, W2, lg = _build(w)
    y = layer.forward(x, lg)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    ref = om.layer_forward(f64(x), lg.cpu().numpy(), f64(W1), f64(W2), w.k)
    assert (i64(layer.topk_idx) == ref["idx"]).all()
    assert (i64(layer.offsets) == ref["offsets"]).all()
    assert (i64(layer.dest_row) == ref["dest_row"]).all()
    assert (i64(layer.src_pair) == ref["src_pair"]).all()
    assert rel_l2(f64(layer.h), ref["H"]) < TOL_BF16
    assert rel_l2(f64(layer.yp), ref["Yp"]) < TOL_BF16
    assert rel_l2(f64(y), ref["y"]) < TOL_BF16


def _sample_experts(counts, rng, n_random=2):
    nz = np.nonzero(counts)[0]
    order = nz[np.argsort(counts[nz], kind="stable")]
    picks = {int(order[-1]), int(order[len(order) // 2]), int(order[0])}
    picks |= {int(e) for e in rng.choice(nz, size=min(n_random, len(nz)), replace=False)}
    return sorted(picks)


def _h_values(layer):
    """H as the layer holds it: bf16, or (MXFP8) decoded from its codes and scales."""
    if layer.dtype != "mxfp8":
        return f64(layer.h)
    return omx.dequantize_rowwise(layer.hq.cpu().numpy(), layer.hs.cpu().numpy())


def check_large_forward(w, layer, x, W1, W2, lg, n_tokens=16, rows_per_expert=12, seed=0):
    """Full integer parity + sampled float parity for a large workload."""
    rng = np.random.default_rng(seed)
    lg_h = lg.cpu().numpy()
    idx, wt, counts = om.route_topk(lg_h, w.k, w.renormalize)
    offsets, dest, src = om.permute_maps(idx, w.E)
    assert (i64(layer.topk_idx) == idx).all()
    assert np.abs(f64(layer.topk_w) - wt).max() <= 1e-6
    assert (i64(layer.counts) == counts).all()
    assert (i64(layer.offsets) == offsets).all()
    assert (i64(layer.dest_row) == dest).all()
    assert (i64(layer.src_pair) == src).all()
    mx = w.dtype == "mxfp8"
    tol = TOL_MXFP8 if mx else TOL_BF16
    cache = {}

    def get(e, which):
        if (e, which) not in cache:
            cache[(e, which)] = f64((W1 if which == 1 else W2)[e])
        return cache[(e, which)]

    # per-stage: sampled rows of GEMM1 (+SwiGLU) and GEMM2 for chosen experts
    h_got, h_want, y_got, y_want = [], [], [], []
    for e in _sample_experts(counts, rng):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        rows = np.sort(rng.choice(np.arange(lo, hi), size=min(rows_per_expert, hi - lo), replace=False))
        xr = f64(x[torch.from_numpy(src[rows] // w.k).cuda()])
        w1, w2 = get(e, 1), get(e, 2)
        if mx:
            xr, w1, w2 = om.mx_roundtrip(xr), om.mx_roundtrip(w1), om.mx_roundtrip(w2)
        h = om.swiglu(xr @ w1.T)
        yp = (om.mx_roundtrip(h) if mx else h) @ w2.T
        r = torch.from_numpy(rows).cuda()
        h_got.append(_h_values(layer)[rows] if mx else f64(layer.h[r]))
        h_want.append(om.mx_roundtrip(h) if mx else h)
        y_got.append(f64(layer.yp[r]))
        y_want.append(yp)
    assert rel_l2(np.concatenate(h_got), np.concatenate(h_want)) < tol
    assert rel_l2(np.concatenate(y_got), np.concatenate(y_want)) < tol

    # sampled tokens end to end (each routed expert's weights fetched once)
    cache.clear()
    toks = np.sort(rng.choice(w.T, size=n_tokens, replace=False))
    tt = torch.from_numpy(toks).cuda()
    got = f64(layer.y[tt])
    want = om.tokens_forward(f64(x[tt]), lg_h[toks], lambda e: f64(W1[e]), lambda e: f64(W2[e]),
                             w.k, w.renormalize, mxfp8_operands=mx)
    assert rel_l2(got, want) < tol


@pytest.mark.parametrize("name", ["mixtral-bf16", "qwen3-235b-bf16"])
def test_large_forward(name):
    need_gpu()
    w = W.BY_NAME[name]
    layer, x, W1, W2, lg = _build(w)
    layer.forward(x, lg)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    check_large_forward(w, layer, x, W1, W2, lg)


@pytest.mark.parametrize("w", [W.BY_NAME["qwen3-235b-bf16"].scaled(T=640, d=512, f=384, name="qwen-small"),
                               W.BY_NAME["dsv3-bf16-train"].scaled(T=256, d=256, f=128, name="dsv3-small"),
                               W.BY_NAME["mixtral-bf16"].scaled(T=300, d=128, f=448, name="mixtral-small")],
                         ids=lambda w: w.name)
def test_scaled_forward_full(w):
    """Reduced shapes checked in full (every output element)."""
    need_gpu()
    layer, x, W1, W2, lg = _build(w)
    y = layer.forward(x, lg)
    torch.cuda.synchronize()
    ref = om.layer_forward(f64(x), lg.cpu().numpy(), f64(W1), f64(W2), w.k)
    assert (i64(layer.src_pair) == ref["src_pair"]).all()
    assert rel_l2(f64(layer.h), ref["H"]) < TOL_BF16
    assert rel_l2(f64(layer.yp), ref["Yp"]) < TOL_BF16
    assert rel_l2(f64(y), ref["y"]) < TOL_BF16


def test_graph_replay_with_new_logits():
    """Capture the forward once; replaying with new logits changes the counts on
    the device only, and every replay still matches the oracle."""
    need_gpu()
    w = W.BY_NAME["qwen3-235b-bf16"].scaled(T=512, d=256, f=256, name="graph")
    layer, x, W1, W2, lg = _build(w)
    lg_buf = lg.clone()
    layer.forward(x, lg_buf)                 # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(x, lg_buf)
    for s in range(3):
        new = torch.from_numpy(np.random.default_rng(100 + s).standard_normal((w.T, w.E)).astype(np.float32) * (1 + s))
        lg_buf.copy_(new)
        g.replay()
        torch.cuda.synchronize()
        ref = om.layer_forward(f64(x), new.numpy(), f64(W1), f64(W2), w.k)
        assert (i64(layer.counts) == ref["counts"]).all()
        assert (i64(layer.src_pair) == ref["src_pair"]).all()
        assert rel_l2(f64(layer.y), ref["y"]) < TOL_BF16


@pytest.mark.parametrize("dtype", ["bf16", "mxfp8"])
def test_graph_replay_training_step(dtype):
    """The training step (forward + backward) captured once in one CUDA graph, as
    the benchmark times it, and replayed three times with new x, logits and dy
    written into the captured buffers: the routing (and the per-expert counts,
    some experts empty) changes on the device only, and after every replay each
    output matches the float64 oracle: maps bit-exact, y, dx, dlogits, dW1, dW2
    within the stated bound, experts without rows exactly zero."""
    import dataclasses
    need_gpu()
    base = W.BY_NAME["dsv3-mxfp8-train" if dtype == "mxfp8" else "dsv3-bf16-train"]
    w = base.scaled(T=512, E=64, d=512, f=512, name=f"graph-train-{dtype}")
    layer, x, W1, W2, lg = _build(w, training=True)
    x_buf, lg_buf, dy_buf = x.clone(), lg.clone(), W.make_dy(w, "cuda")
    tol = TOL_MXFP8 if dtype == "mxfp8" else TOL_BF16

    def step():
        layer.forward(x_buf, lg_buf)
        layer.backward(dy_buf, lg_buf)

    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()                                # warm-up outside capture
    stream.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    seen = set()
    for rep in range(3):
        wr = dataclasses.replace(w, seed=w.seed + 17 * (rep + 1))
        x_buf.copy_(W.make_x(wr, "cuda"))
        lg_buf.copy_(logits_dev(wr))
        dy_buf.copy_(W.make_dy(wr, "cuda"))
        g.replay()
        torch.cuda.synchronize()
        assert int(layer.dev_status.item()) == 0
        lg_h = lg_buf.cpu().numpy()
        mx = dtype == "mxfp8"
        ref = om.layer_forward(f64(x_buf), lg_h, f64(W1), f64(W2), w.k, mxfp8_operands=mx)
        bwd = om.layer_backward(ref, f64(dy_buf), f64(x_buf), lg_h, f64(W1), f64(W2), w.k, mxfp8_operands=mx)
        assert (i64(layer.counts) == ref["counts"]).all()
        assert (i64(layer.offsets) == ref["offsets"]).all()
        assert (i64(layer.dest_row) == ref["dest_row"]).all()
        assert (i64(layer.src_pair) == ref["src_pair"]).all()
        seen.add(tuple(ref["counts"].tolist()))
        for name, got, want in (("y", layer.y, ref["y"]), ("dx", layer.dx, bwd["dx"]),
                                ("dlogits", layer.dlogits, bwd["dlogits"]), ("dW1", layer.dW1, bwd["dW1"]),
                                ("dW2", layer.dW2, bwd["dW2"])):
            err = rel_l2(f64(got), want)
            assert err < tol, (rep, name, err)
        empty = np.nonzero(ref["counts"] == 0)[0]
        assert len(empty) > 0
        e_t = torch.from_numpy(empty).cuda()
        assert int(torch.count_nonzero(layer.dW1[e_t]).item()) == 0
        assert int(torch.count_nonzero(layer.dW2[e_t]).item()) == 0
    assert len(seen) == 3                     # the counts changed between replays


@pytest.mark.parametrize("dtype", ["bf16", "mxfp8"])
def test_accumulated_weight_gradients(dtype):
    """accumulate_grads: dW1 and dW2 are the fp32 sums of the weight gradients of every
    backward since construction (three batches with different routing, so different
    experts are empty in each) and start again from zero after zero_grads()."""
    import dataclasses
    need_gpu()
    base = W.BY_NAME["dsv3-mxfp8-train" if dtype == "mxfp8" else "dsv3-bf16-train"]
    w = base.scaled(T=384, E=32, d=512, f=512, name=f"acc-grads-{dtype}")   # MXFP8: K % 512 == 0
    W1, W2 = W.make_w1(w, "cuda"), W.make_w2(w, "cuda")
    layer = moe_gpu.MoELayer(w.T, w.d, w.E, w.k, w.f, W1, W2, dtype=w.dtype, renormalize=w.renormalize,
                             training=True, accumulate_grads=True)
    assert layer.dW1.dtype == torch.float32 and layer.dW2.dtype == torch.float32
    tol = TOL_MXFP8 if dtype == "mxfp8" else TOL_BF16
    mx = dtype == "mxfp8"
    sums = [0.0, 0.0]
    for b in range(4):
        if b == 3:
            layer.zero_grads()
            sums = [0.0, 0.0]
        wr = dataclasses.replace(w, seed=w.seed + 11 * (b + 1))
        x, lg, dy = W.make_x(wr, "cuda"), logits_dev(wr), W.make_dy(wr, "cuda")
        layer.forward(x, lg)
        layer.backward(dy, lg)
        torch.cuda.synchronize()
        assert int(layer.dev_status.item()) == 0
        lg_h = lg.cpu().numpy()
        ref = om.layer_forward(f64(x), lg_h, f64(W1), f64(W2), w.k, mxfp8_operands=mx)
        bwd = om.layer_backward(ref, f64(dy), f64(x), lg_h, f64(W1), f64(W2), w.k, mxfp8_operands=mx)
        sums = [sums[0] + bwd["dW1"], sums[1] + bwd["dW2"]]
        assert rel_l2(f64(layer.dW1), sums[0]) < tol, (b, "dW1")
        assert rel_l2(f64(layer.dW2), sums[1]) < tol, (b, "dW2")


@pytest.mark.parametrize("w", [W.BY_NAME["dsv3-bf16-train"].scaled(T=256, d=256, f=128, name="dsv3-train-small"),
                               W.BY_NAME["dsv3-bf16-train"].scaled(T=700, E=16, d=192, f=320, name="train-E16"),
                               W.BY_NAME["mixtral-bf16"].scaled(T=300, d=128, f=448, name="mixtral-train-small")],
                         ids=lambda w: w.name)
def test_scaled_backward_full(w):
    """Forward + backward of the layer against the float64 oracle, every element."""
    need_gpu()
    layer, x, W1, W2, lg = _build(w, training=True)
    dy = W.make_dy(w, "cuda")
    layer.forward(x, lg)
    dx, dlogits, dW1, dW2 = layer.backward(dy, lg)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    lg_h = lg.cpu().numpy()
    ref = om.layer_forward(f64(x), lg_h, f64(W1), f64(W2), w.k)
    bwd = om.layer_backward(ref, f64(dy), f64(x), lg_h, f64(W1), f64(W2), w.k)
    assert rel_l2(f64(layer.gu), ref["GU"]) < TOL_BF16
    assert rel_l2(f64(layer.dyp), bwd["dYp"]) < TOL_BF16
    assert rel_l2(f64(layer.dw), bwd["dw"]) < TOL_BF16
    assert rel_l2(f64(layer.dgu), bwd["dGU"]) < TOL_BF16
    assert rel_l2(f64(layer.dxp), bwd["dXp"]) < TOL_BF16
    assert rel_l2(f64(dW2), bwd["dW2"]) < TOL_BF16
    assert rel_l2(f64(dW1), bwd["dW1"]) < TOL_BF16
    assert rel_l2(f64(dx), bwd["dx"]) < TOL_BF16
    assert rel_l2(f64(dlogits), bwd["dlogits"]) < TOL_BF16
    empty = np.nonzero(ref["counts"] == 0)[0]
    for e in empty:
        assert (f64(dW1[e]) == 0).all() and (f64(dW2[e]) == 0).all()


def test_mxfp8_layer_scaled_full():
    """DeepSeek-V3-shaped MXFP8 layer at reduced size, every output element,
    against the oracle's own MXFP8 chain (it quantises X, W1, H and W2 itself)."""
    need_gpu()
    w = W.BY_NAME["dsv3-mxfp8"].scaled(T=400, d=512, f=512, name="dsv3-mx-small")
    layer, x, W1, W2, lg = _build(w)
    y = layer.forward(x, lg)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    ref = om.layer_forward(f64(x), lg.cpu().numpy(), f64(W1), f64(W2), w.k, mxfp8_operands=True)
    assert (i64(layer.src_pair) == ref["src_pair"]).all()
    # GEMM1 writes H as MXFP8: compare its dequantised values with the oracle's H
    # after the oracle's own MXFP8 round trip (what the oracle feeds GEMM2)
    assert rel_l2(_h_values(layer), om.mx_roundtrip(ref["H"])) < TOL_MXFP8
    assert rel_l2(f64(y), ref["y"]) < TOL_MXFP8


@pytest.mark.parametrize("w", [W.BY_NAME["dsv3-mxfp8"].scaled(T=256, d=512, f=512, name="dsv3-mx-train-small"),
                               W.BY_NAME["dsv3-mxfp8"].scaled(T=600, E=16, d=512, f=512, name="mx-train-E16")],
                         ids=lambda w: w.name)
def test_mxfp8_backward_scaled_full(w):
    """MXFP8 training step (forward and backward, every GEMM on MXFP8 operands
    quantised along its own contraction) against the oracle's MXFP8 chain, every
    element; experts without rows get exact zero weight gradients."""
    need_gpu()
    layer, x, W1, W2, lg = _build(w, training=True)
    dy = W.make_dy(w, "cuda")
    layer.forward(x, lg)
    dx, dlogits, dW1, dW2 = layer.backward(dy, lg)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    lg_h = lg.cpu().numpy()
    ref = om.layer_forward(f64(x), lg_h, f64(W1), f64(W2), w.k, mxfp8_operands=True)
    bwd = om.layer_backward(ref, f64(dy), f64(x), lg_h, f64(W1), f64(W2), w.k, mxfp8_operands=True)
    assert (i64(layer.src_pair) == ref["src_pair"]).all()
    assert rel_l2(f64(layer.gu), ref["GU"]) < TOL_MXFP8
    assert rel_l2(f64(layer.h), ref["H"]) < TOL_MXFP8
    # dYp exists only as MXFP8 (row-wise from the combine backward): its decoded values
    # against the oracle's dYp after the oracle's own row-wise round trip
    dyp_mx = omx.dequantize_rowwise(layer.dyq.cpu().numpy(), layer.dys.cpu().numpy())
    assert rel_l2(dyp_mx, om.mx_roundtrip(bwd["dYp"])) < TOL_MXFP8
    for name, got in (("dGU", layer.dgu), ("dXp", layer.dxp), ("dW2", dW2), ("dW1", dW1),
                      ("dx", dx), ("dlogits", dlogits)):
        err = rel_l2(f64(got), bwd[name])
        assert err < TOL_MXFP8, (name, err)
    for e in np.nonzero(ref["counts"] == 0)[0]:
        assert (f64(dW1[e]) == 0).all() and (f64(dW2[e]) == 0).all()


def test_mxfp8_layer_full_size_sampled():
    need_gpu()
    w = W.BY_NAME["dsv3-mxfp8"]
    layer, x, W1, W2, lg = _build(w)
    layer.forward(x, lg)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    check_large_forward(w, layer, x, W1, W2, lg, n_tokens=16, rows_per_expert=8)


def test_train_full_size_sampled():
    """The DeepSeek-V3-shaped training step at full size: integer outputs in full,
    forward on samples, dx / dlogits of sampled tokens, and sampled rows of dW1 /
    columns of dW2 for the hottest, median and smallest non-empty experts (the
    contraction over all of each expert's rows); empty experts exactly zero."""
    need_gpu()
    w = W.BY_NAME["dsv3-bf16-train"]
    layer, x, W1, W2, lg = _build(w, training=True)
    dy = W.make_dy(w, "cuda")
    layer.forward(x, lg)
    layer.backward(dy, lg)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    check_large_forward(w, layer, x, W1, W2, lg, n_tokens=16, rows_per_expert=8)

    rng = np.random.default_rng(5)
    lg_h = lg.cpu().numpy()
    idx, wt, counts = om.route_topk(lg_h, w.k)
    offsets, dest, src = om.permute_maps(idx, w.E)
    cache = {}

    def get(e, which):
        if (e, which) not in cache:
            cache[(e, which)] = f64((W1 if which == 1 else W2)[e])
        return cache[(e, which)]

    toks = np.sort(rng.choice(w.T, size=16, replace=False))
    tt = torch.from_numpy(toks).cuda()
    want_dx, want_dl = om.tokens_backward(f64(x[tt]), lg_h[toks], f64(dy[tt]), lambda e: f64(W1[e]),
                                          lambda e: f64(W2[e]), w.k)
    assert rel_l2(f64(layer.dx[tt]), want_dx) < TOL_BF16
    assert rel_l2(f64(layer.dlogits[tt]), want_dl) < TOL_BF16

    nz = np.nonzero(counts)[0]
    order = nz[np.argsort(counts[nz], kind="stable")]
    got1, want1, got2, want2 = [], [], [], []
    for e in (int(order[-1]), int(order[len(order) // 2]), int(order[0])):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        pairs = src[lo:hi]
        tok = torch.from_numpy(pairs // w.k).cuda()
        X_e = f64(x[tok])
        dYp_e = wt[pairs // w.k, pairs % w.k][:, None] * f64(dy[tok])
        rows = np.sort(rng.choice(2 * w.f, size=6, replace=False))
        cols = np.sort(rng.choice(w.f, size=6, replace=False))
        dw1, dw2 = om.expert_wgrad_sampled(X_e, dYp_e, get(e, 1), get(e, 2), rows, cols)
        got1.append(f64(layer.dW1[e][torch.from_numpy(rows).cuda()]))
        want1.append(dw1)
        got2.append(f64(layer.dW2[e][:, torch.from_numpy(cols).cuda()]))
        want2.append(dw2)
    assert rel_l2(np.concatenate(got1), np.concatenate(want1)) < TOL_BF16
    assert rel_l2(np.concatenate(got2, axis=1), np.concatenate(want2, axis=1)) < TOL_BF16
    empty = np.nonzero(counts == 0)[0]
    assert len(empty) > 0
    e_t = torch.from_numpy(empty).cuda()
    assert int(torch.count_nonzero(layer.dW1[e_t]).item()) == 0
    assert int(torch.count_nonzero(layer.dW2[e_t]).item()) == 0


def test_mxfp8_train_full_size_sampled():
    """The DeepSeek-V3-shaped MXFP8 training step at full size: maps in full, and for
    the median, the smallest non-empty and an upper-quartile expert the whole MXFP8
    chain of that expert (every quantisation in it is local to the expert) against
    dGU, dXp, dW1 and dW2; experts without rows get exact zero gradients."""
    need_gpu()
    w = W.BY_NAME["dsv3-mxfp8-train"]
    layer, x, W1, W2, lg = _build(w, training=True)
    dy = W.make_dy(w, "cuda")
    layer.forward(x, lg)
    layer.backward(dy, lg)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    lg_h = lg.cpu().numpy()
    idx, wt, counts = om.route_topk(lg_h, w.k)
    offsets, dest, src = om.permute_maps(idx, w.E)
    assert (i64(layer.offsets) == offsets).all() and (i64(layer.src_pair) == src).all()
    nz = np.nonzero(counts)[0]
    order = nz[np.argsort(counts[nz], kind="stable")]
    for e in (int(order[len(order) // 2]), int(order[0]), int(order[(3 * len(order)) // 4])):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        pairs = src[lo:hi]
        tok = torch.from_numpy(pairs // w.k).cuda()
        X_e = f64(x[tok])
        dYp_e = wt[pairs // w.k, pairs % w.k][:, None] * f64(dy[tok])
        ref = om.expert_backward_mxfp8(X_e, dYp_e, f64(W1[e]), f64(W2[e]))
        for name, got in (("dGU", layer.dgu[lo:hi]), ("dXp", layer.dxp[lo:hi]), ("dW1", layer.dW1[e]),
                          ("dW2", layer.dW2[e])):
            err = rel_l2(f64(got), ref[name])
            assert err < TOL_MXFP8, (e, hi - lo, name, err)
    e_t = torch.from_numpy(np.nonzero(counts == 0)[0]).cuda()
    assert int(torch.count_nonzero(layer.dW1[e_t]).item()) == 0
    assert int(torch.count_nonzero(layer.dW2[e_t]).item()) == 0

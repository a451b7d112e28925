"""Router GEMM fused with the top-k selection (moe_route_topk_gemm) against the
oracle: the fp32 logits the kernel computed are compared with the float64 product,
and the selection is checked bit-exactly against the oracle's selection on those
same fp32 logits (a selection decided by floating point is taken in the kernel's
precision on both sides)."""

import numpy as np
import pytest
import torch

import ragged_grouped_gemm_topk_gb300 as moe_gpu
from ragged_grouped_gemm_topk_gb300 import workloads as W
from oracle import moe as om
from _parity import f64, i64, need_gpu, rel_l2

pytestmark = pytest.mark.gpu


def _inputs(T, d, E, dtype, seed):
    x = W.make_matrix(T, d, seed=seed, dtype=dtype, device="cuda")
    Wr = W.make_matrix(E, d, seed=seed + 1, dtype=dtype, device="cuda", scale=d ** -0.5)
    return x, Wr


def _check(x, Wr, k, renorm, dtype):
    idx, w, counts, logits = moe_gpu.moe_route_topk_gemm(x, Wr, k, renorm, want_logits=True)
    lg = logits.cpu().numpy()
    want = om.router_logits(f64(x), f64(Wr))
    # bf16 products are exact in fp32 (only the accumulation rounds); tf32 rounds the inputs
    assert rel_l2(lg.astype(np.float64), want) < (1e-5 if dtype == torch.bfloat16 else 5e-3)
    ri, rw, rc = om.route_topk(lg, k, renorm)
    assert (i64(idx) == ri).all()
    assert np.abs(f64(w) - rw).max() <= 1e-6
    assert (i64(counts) == rc).all() and int(counts.sum()) == x.shape[0] * k
    return idx, w, counts


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "tf32"])
@pytest.mark.parametrize("renorm", [True, False], ids=["renorm", "full"])
@pytest.mark.parametrize("T,d,E,k", [(300, 256, 8, 2), (1000, 512, 64, 8), (257, 128, 256, 8),
                                     (130, 96, 100, 3), (64, 64, 1, 1)])
def test_route_topk_gemm_matches_oracle(T, d, E, k, dtype, renorm):
    need_gpu()
    x, Wr = _inputs(T, d, E, dtype, seed=T + d + E + k)
    idx, w, counts = _check(x, Wr, k, renorm, dtype)
    # without the logits output: the same selection and weights
    idx2, w2, c2 = moe_gpu.moe_route_topk_gemm(x, Wr, k, renorm)
    assert torch.equal(idx, idx2) and torch.equal(w, w2) and torch.equal(counts, c2)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "tf32"])
@pytest.mark.parametrize("renorm", [True, False], ids=["renorm", "full"])
@pytest.mark.parametrize("T,d,E,k", [(777, 2048, 96, 6), (2500, 1024, 160, 8), (50, 2048, 256, 8),
                                     (4100, 4096, 64, 4)])
def test_route_topk_gemm_split_contraction(T, d, E, k, dtype, renorm):
    """Tiles that leave SMs idle split their contraction over a cluster of 2 or 4 CTAs
    (the partial logits summed through distributed shared memory, each CTA selecting
    its share of the rows).  On 152 SMs: 777 x 2048 takes clusters of 4 (7 tiles, the
    last with 9 rows, so three CTAs of its cluster select nothing); 2500 x 1024 clusters
    of 2 in bf16 (16 K blocks) and of 4 in tf32 (68 rows in the last tile); 50 x 2048 one
    cluster of 4 over a single partial tile; 4100 x 4096 clusters of 4 (33 tiles, 4 rows
    in the last).  Clusters of 2 at the 8192-token DeepSeek-V3 size are tested below."""
    need_gpu()
    x, Wr = _inputs(T, d, E, dtype, seed=T + d + E + k + 1)
    idx, w, counts = _check(x, Wr, k, renorm, dtype)
    # the partials are summed in a fixed order: a second call is bit-identical
    idx2, w2, c2, lg2 = moe_gpu.moe_route_topk_gemm(x, Wr, k, renorm, want_logits=True)
    _, _, _, lg1 = moe_gpu.moe_route_topk_gemm(x, Wr, k, renorm, want_logits=True)
    assert torch.equal(idx, idx2) and torch.equal(w, w2) and torch.equal(counts, c2)
    assert torch.equal(lg1, lg2)


def test_route_topk_gemm_split_ties_and_nan():
    """Under a split contraction: bit-equal logits of duplicate router rows go to the
    lower expert id, and a NaN in a token owned by the second CTA of a cluster is
    flagged."""
    need_gpu()
    x, Wr = _inputs(200, 2048, 24, torch.bfloat16, seed=15)
    Wr[9] = Wr[2]
    Wr[17] = Wr[2]
    idx, _, _ = _check(x, Wr, 4, True, torch.bfloat16)
    i = i64(idx)
    for t, j in zip(*np.where(i == 9)):
        assert 2 in i[t, :j]
    for t, j in zip(*np.where(i == 17)):
        assert 2 in i[t, :j] and 9 in i[t, :j]
    x[190, 7] = float("nan")                  # tile 1, row 62: the second CTA's share
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe_gpu.moe_route_topk_gemm(x, Wr, 4, True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == moe_gpu.binding._lib.MOE_DEV_NAN_LOGIT


@pytest.mark.parametrize("renorm", [True, False], ids=["renorm", "full"])
def test_route_topk_gemm_deepseek_router_size(renorm):
    """The DeepSeek-V3 router shape (8192 tokens, d = 7168, E = 256, k = 8): 64 tiles,
    each contracted by a cluster of 2 CTAs whose 14 selecting warps share its rows."""
    need_gpu()
    x, Wr = _inputs(8192, 7168, 256, torch.bfloat16, seed=71)
    _check(x, Wr, 8, renorm, torch.bfloat16)


def test_route_topk_gemm_ties_go_to_lower_expert():
    """Duplicate router rows give bit-equal logits; the lower expert id wins."""
    need_gpu()
    x, Wr = _inputs(200, 128, 16, torch.bfloat16, seed=5)
    Wr[9] = Wr[2]
    Wr[12] = Wr[2]
    Wr[7] = Wr[0]
    idx, _, _ = _check(x, Wr, 4, True, torch.bfloat16)
    i = i64(idx)
    pos = {e: np.where(i == e) for e in (2, 9, 12)}
    # wherever 9 or 12 is selected, 2 is selected in an earlier slot
    for t, j in zip(*pos[9]):
        assert 2 in i[t, :j]
    for t, j in zip(*pos[12]):
        assert 2 in i[t, :j] and 9 in i[t, :j]


def test_route_topk_gemm_flags_nan_and_matches_route_topk():
    """A NaN in x makes that token's logits NaN: the status word is flagged.  On
    finite inputs the fused kernel equals moe_route_topk on its logits."""
    need_gpu()
    x, Wr = _inputs(128, 64, 32, torch.bfloat16, seed=9)
    idx, w, counts, logits = moe_gpu.moe_route_topk_gemm(x, Wr, 8, True, want_logits=True)
    i2, w2, c2 = moe_gpu.moe_route_topk(logits, 8, True)
    assert torch.equal(idx, i2) and torch.equal(counts, c2)
    assert (w - w2).abs().max().item() <= 1e-6
    x[5, 3] = float("nan")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe_gpu.moe_route_topk_gemm(x, Wr, 8, True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & moe_gpu.binding._lib.MOE_DEV_NAN_LOGIT


def test_route_topk_gemm_rejects_bad_args():
    need_gpu()
    x, Wr = _inputs(16, 64, 300, torch.bfloat16, seed=1)
    with pytest.raises(moe_gpu.binding.MoeError):
        moe_gpu.moe_route_topk_gemm(x, Wr, 2)            # E > 256
    x, Wr = _inputs(16, 64, 32, torch.bfloat16, seed=1)
    with pytest.raises(moe_gpu.binding.MoeError):
        moe_gpu.moe_route_topk_gemm(x, Wr, 9)            # k > 8


@pytest.mark.parametrize("renorm", [True, False], ids=["renorm", "full"])
def test_layer_with_router_weights(renorm):
    """A layer that scores its own tokens (fused router GEMM) equals the oracle's
    layer run on the logits that router produced; its backward gives the oracle's
    dlogits (the router backward reads the kept logits when not renormalised)."""
    need_gpu()
    w = W.BY_NAME["qwen3-235b-bf16"].scaled(T=320, E=32, d=256, f=192, name="router-layer")
    x = W.make_x(w, "cuda")
    W1, W2 = W.make_w1(w, "cuda"), W.make_w2(w, "cuda")
    Wr = W.make_matrix(w.E, w.d, seed=77, dtype=torch.bfloat16, device="cuda", scale=w.d ** -0.5)
    layer = moe_gpu.MoELayer(w.T, w.d, w.E, w.k, w.f, W1, W2, dtype="bf16", renormalize=renorm,
                             training=True, w_router=Wr, keep_logits=True)
    dy = W.make_dy(w, "cuda")
    y = layer.forward(x)
    dx, dlogits, dW1, dW2 = layer.backward(dy)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    lg = layer.logits.cpu().numpy()
    assert rel_l2(lg.astype(np.float64), om.router_logits(f64(x), f64(Wr))) < 1e-5
    ref = om.layer_forward(f64(x), lg, f64(W1), f64(W2), w.k, renorm)
    bwd = om.layer_backward(ref, f64(dy), f64(x), lg, f64(W1), f64(W2), w.k, renorm)
    assert (i64(layer.topk_idx) == ref["idx"]).all()
    assert rel_l2(f64(y), ref["y"]) < 1e-2
    assert rel_l2(f64(dlogits), bwd["dlogits"]) < 1e-2
    assert rel_l2(f64(dx), bwd["dx"]) < 1e-2

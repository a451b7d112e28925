"""Capacity-based dispatch (the contrast case to dropless routing) against the
oracle: maps and padded rows bit-exact, and the whole capacity-mode layer forward
(route -> capacity dispatch -> grouped GEMMs over E*C rows -> combine of the kept
slots) within the bf16 tolerance."""

import numpy as np
import pytest
import torch

import ragged_grouped_gemm_topk_gb300 as moe_gpu
from ragged_grouped_gemm_topk_gb300 import workloads as W
from oracle import moe as om
from _parity import TOL_BF16, f64, i64, logits_dev, need_gpu, rel_l2

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,T,E,k,C", [("qwen3-235b-bf16", 700, 32, 8, 150), ("mixtral-bf16", 300, 8, 2, 70),
                                          ("dsv3-mxfp8", 512, 64, 8, 0), ("qwen3-235b-bf16", 400, 16, 4, 1000)],
                         ids=["drops", "mixtral-drops", "zero-capacity", "no-drops"])
def test_capacity_dispatch_maps_and_rows(name, T, E, k, C):
    need_gpu()
    w = W.BY_NAME[name].scaled(T=T, E=E, k=k, d=256, f=128, name="cap")
    lg = logits_dev(w)
    x = W.make_x(w, "cuda").bfloat16()
    idx, wt, counts = moe_gpu.moe_route_topk(lg, k)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = moe_gpu.moe_permute_capacity(x, idx, counts, E, C, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    off, dest, src = om.permute_capacity(i64(idx), E, C)
    assert (i64(out["offsets"]) == off).all()
    assert (i64(out["dest_row"]) == dest).all()
    assert (i64(out["src_pair"]) == src).all()
    want = om.permute_rows_capacity(f64(x), src, k)
    assert np.array_equal(f64(out["xp"]), want)               # copies and zero padding, bit-exact


@pytest.mark.parametrize("C", [40, 0, 10_000], ids=["drops", "all-dropped", "no-drops"])
def test_capacity_layer_forward(C):
    """Capacity-mode forward against the oracle; with a capacity that drops
    nothing it equals the dropless layer."""
    need_gpu()
    w = W.BY_NAME["qwen3-235b-bf16"].scaled(T=256, E=16, d=256, f=192, name="cap-layer")
    lg = logits_dev(w)
    x = W.make_x(w, "cuda")
    W1, W2 = W.make_w1(w, "cuda"), W.make_w2(w, "cuda")
    idx, wt, counts = moe_gpu.moe_route_topk(lg, w.k)
    m = moe_gpu.moe_permute_capacity(x, idx, counts, w.E, C)
    rows = w.E * C
    y = torch.zeros(w.T, w.d, dtype=torch.bfloat16, device="cuda")
    if rows > 0:
        h = moe_gpu.moe_grouped_gemm_fwd(m["xp"], W1, m["offsets"], epi="swiglu")
        yp = moe_gpu.moe_grouped_gemm_fwd(h, W2, m["offsets"])
    else:
        yp = torch.empty(0, w.d, dtype=torch.bfloat16, device="cuda")
    moe_gpu.moe_unpermute_combine_capacity(yp, m["dest_row"], wt, out=y)
    torch.cuda.synchronize()
    ref = om.layer_forward_capacity(f64(x), lg.cpu().numpy(), f64(W1), f64(W2), w.k, C)
    if C == 0:
        assert (f64(y) == 0).all()
    else:
        assert rel_l2(f64(y), ref["y"]) < TOL_BF16
    if C == 10_000:
        dropless = om.layer_forward(f64(x), lg.cpu().numpy(), f64(W1), f64(W2), w.k)
        assert np.allclose(ref["y"], dropless["y"], rtol=1e-12, atol=1e-12)


def test_combine_capacity_flags_bad_rows_but_not_drops():
    need_gpu()
    yp = torch.randn(10, 64, device="cuda").bfloat16()
    dest = torch.tensor([[0, -1], [9, 3]], dtype=torch.int32, device="cuda")
    w = torch.ones(2, 2, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = moe_gpu.moe_unpermute_combine_capacity(yp, dest, w, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(y[0], yp[0]) and rel_l2(f64(y[1]), f64(yp[9]) + f64(yp[3])) < 1e-2
    dest[0, 1] = 10                                   # past the rows: flagged
    moe_gpu.moe_unpermute_combine_capacity(yp, dest, w, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & moe_gpu.binding._lib.MOE_DEV_BAD_INDEX

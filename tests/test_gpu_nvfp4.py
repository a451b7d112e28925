"""NVFP4 on the GPU against the NVFP4 oracle: the quantiser bit-exact (codes,
scales and the fp32 tensor scale), including the hand-worked blocks."""

import os

import numpy as np
import pytest
import torch

import ragged_grouped_gemm_topk_gb300 as moe_gpu
from ragged_grouped_gemm_topk_gb300 import workloads as W
from oracle import nvfp4 as o4
from _parity import f64, need_gpu

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_blocks.txt")


def _check_quant(t):
    codes, scales, ts = moe_gpu.moe_quantize_nvfp4(t)
    c, s, g = o4.quantize(t.float().cpu().numpy().reshape(-1, t.shape[-1]))
    assert ts[0].item() == float(g)
    assert (scales.cpu().numpy().reshape(s.shape) == s).all()
    assert (codes.cpu().numpy().reshape(c.shape) == c).all()
    return codes, scales, ts, (c, s, g)


def test_quantize_nvfp4_golden_blocks():
    need_gpu()
    vals = [l.split()[1:] for l in open(GOLDEN) if l.startswith("values")][0]
    t = torch.tensor([float(v) for v in vals], dtype=torch.float32, device="cuda")[None, :]
    codes, scales, ts, _ = _check_quant(t)
    assert ts[0].item() == 448.0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("rows,K", [(1, 16), (37, 64), (300, 512), (64, 7168)])
def test_quantize_nvfp4_bit_exact(dtype, rows, K):
    need_gpu()
    t = W.make_matrix(rows, K, seed=rows + K, dtype=dtype, device="cuda", scale=3.0)
    if rows > 10:
        t[3] *= 2.0 ** -14                           # tiny rows: subnormal E4M3 block scales
        t[4, :16] = 0                                # an all-zero block
        t[5, 1] = -0.0
        t[6] *= 2.0 ** 6                             # the tensor's amax comes from here
    _check_quant(t)


def test_quantize_nvfp4_weight_stack_and_zero_tensor():
    need_gpu()
    Wt = W.make_matrix(4 * 96, 256, seed=7, dtype=torch.bfloat16, device="cuda").view(4, 96, 256)
    codes, scales, ts, _ = _check_quant(Wt)
    assert codes.shape == (4, 96, 128) and scales.shape == (4, 96, 16)
    z = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    codes, scales, ts, _ = _check_quant(z)
    assert ts[0].item() == 1.0 and int(codes.sum()) == 0 and int(scales.sum()) == 0


# ----------------------------------------------------------------------------- NVFP4 grouped GEMM

from oracle import moe as om  # noqa: E402
from _parity import ragged_offsets, rel_l2  # noqa: E402

COUNTS = {"mixed": [0, 1, 130, 257, 3, 128, 0, 64], "singles": [1] * 37, "one-expert": [700],
          "many-tiles": [5200, 0, 5100]}      # with 2+ column tiles: more tiles than SMs


def _mats(M, K, N, E, seed):
    A = W.make_matrix(M, K, seed=seed, dtype=torch.bfloat16, device="cuda")
    B = W.make_matrix(E * N, K, seed=seed + 1, dtype=torch.bfloat16, device="cuda", scale=K ** -0.5).view(E, N, K)
    Aq, As, Ag, (ca, sa, ga) = _check_quant(A)
    Bq, Bs, Bg, (cb, sb, gb) = _check_quant(B)
    A_deq = o4.dequantize(ca, sa, ga)
    B_deq = o4.dequantize(cb, sb, gb).reshape(E, N, K)
    return (Aq, As, Ag, A_deq), (Bq, Bs, Bg, B_deq)


@pytest.mark.parametrize("counts", ["mixed", "singles", "one-expert", "many-tiles"], ids=str)
@pytest.mark.parametrize("K,N", [(256, 256), (512, 320), (1024, 64)])
def test_fwd_nvfp4_plain(counts, K, N):
    """C = A . B[e]^T on NVFP4 operands against the oracle on the same decoded
    values (only the fp32 accumulation and the bf16 store round); rows outside
    every group untouched."""
    need_gpu()
    cnt = COUNTS[counts]
    E = len(cnt)
    rows = int(sum(cnt))
    M = rows + 2
    (Aq, As, Ag, A_deq), (Bq, Bs, Bg, B_deq) = _mats(M, K, N, E, seed=K + N + 41)
    off = ragged_offsets(cnt)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe_gpu.moe_grouped_gemm_fwd(Aq, Bq, off, A_scales=As, B_scales=Bs, A_tensor_scale=Ag, B_tensor_scale=Bg, out=C)
    want = om.grouped_gemm(A_deq, B_deq, off.cpu().numpy())
    got = f64(C)
    assert np.isnan(got[rows:]).all()
    err = rel_l2(got[:rows], want[:rows])
    assert err < 1e-2, err


@pytest.mark.parametrize("counts", ["mixed", "singles", "many-tiles"], ids=str)
@pytest.mark.parametrize("K,f", [(256, 128), (512, 96), (768, 288)])
def test_fwd_nvfp4_swiglu(counts, K, f):
    need_gpu()
    cnt = COUNTS[counts]
    E = len(cnt)
    M = int(sum(cnt))
    (Aq, As, Ag, A_deq), (Bq, Bs, Bg, B_deq) = _mats(M, K, 2 * f, E, seed=K + f + 43)
    off = ragged_offsets(cnt)
    H, GU = moe_gpu.moe_grouped_gemm_fwd(Aq, Bq, off, epi="swiglu", A_scales=As, B_scales=Bs, A_tensor_scale=Ag,
                                         B_tensor_scale=Bg, out_dtype=torch.float32, want_preact=True)
    gu = om.grouped_gemm(A_deq, B_deq, off.cpu().numpy())
    assert rel_l2(f64(GU), gu) < 1e-3                      # fp32 out: the accumulation rounding only
    assert rel_l2(f64(H), om.swiglu(gu)) < 1e-3
    Hb = moe_gpu.moe_grouped_gemm_fwd(Aq, Bq, off, epi="swiglu", A_scales=As, B_scales=Bs, A_tensor_scale=Ag,
                                      B_tensor_scale=Bg)
    assert rel_l2(f64(Hb), om.swiglu(gu)) < 1e-2


def test_fwd_nvfp4_requires_k_multiple_of_256_and_scales():
    need_gpu()
    (Aq, As, Ag, _), (Bq, Bs, Bg, _) = _mats(64, 512, 64, 2, seed=3)
    off = ragged_offsets([32, 32])
    with pytest.raises(moe_gpu.binding.MoeError, match="256"):
        moe_gpu.moe_grouped_gemm_fwd(Aq[:, :64].contiguous(), Bq[:, :, :64].contiguous(), off,
                                     A_scales=As[:, :8].contiguous(), B_scales=Bs[:, :, :8].contiguous(),
                                     A_tensor_scale=Ag, B_tensor_scale=Bg)
    with pytest.raises(moe_gpu.binding.MoeError):
        moe_gpu.moe_grouped_gemm_fwd(Aq, Bq, off, A_scales=As, B_scales=None, A_tensor_scale=Ag, B_tensor_scale=Bg)


# ----------------------------------------------------------------------------- NVFP4 layer

from _parity import i64, logits_dev  # noqa: E402


def test_nvfp4_layer_scaled():
    """DeepSeek-V3-shaped NVFP4 layer at reduced size: maps exact; H (the GPU's own
    bf16 H) quantised bit-exactly as the oracle quantises it; the output against the
    oracle's NVFP4 chain (which quantises its own float64 H: the two H tensor scales
    differ in their last bits, so a few codes differ)."""
    need_gpu()
    w = W.BY_NAME["dsv3-nvfp4"].scaled(T=400, d=512, f=512, name="fp4-small")
    x, W1, W2, lg = W.make_x(w, "cuda"), W.make_w1(w, "cuda"), W.make_w2(w, "cuda"), logits_dev(w)
    layer = moe_gpu.MoELayer(w.T, w.d, w.E, w.k, w.f, W1, W2, dtype="nvfp4", renormalize=w.renormalize)
    y = layer.forward(x, lg)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    ref = om.layer_forward(f64(x), lg.cpu().numpy(), f64(W1), f64(W2), w.k, nvfp4_operands=True)
    assert (i64(layer.src_pair) == ref["src_pair"]).all()
    c, s, g = o4.quantize(layer.h.float().cpu().numpy())
    assert layer.hg[0].item() == float(g)
    assert (layer.hs.cpu().numpy() == s).all() and (layer.hq.cpu().numpy() == c).all()
    assert rel_l2(f64(y), ref["y"]) < 5e-2


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("T,d,E,k", [(300, 256, 8, 2), (1000, 512, 64, 8), (77, 48, 4, 3), (300, 4368, 16, 4),
                                     (200, 6144, 32, 8), (600, 256, 1024, 4)])
def test_permute_nvfp4_equals_permute_then_quantize(dtype, T, d, E, k):
    """The fused NVFP4 dispatch writes, bit for bit, the NVFP4 of the rows moe_permute
    writes (and the same maps), which the quantiser tests pin to the oracle.  Beside
    the small rows: rows over several staging segments of the scatter, the last partial
    with 273-byte scale rows (d = 4368) or all whole (d = 6144), and E = 1024 (the rank
    pass, which shares its launch with the tensor amax, then needs 64 KB of shared
    memory)."""
    need_gpu()
    w = W.BY_NAME["qwen3-235b-bf16"].scaled(T=T, E=E, k=k, d=d, name="fp4-perm")
    x = W.make_x(w, "cuda").to(dtype)
    idx, wt, counts = moe_gpu.moe_route_topk(logits_dev(w), k)
    ref = moe_gpu.moe_permute(x, idx, counts, E)
    rc, rs, rg = moe_gpu.moe_quantize_nvfp4(ref["xp"])
    out = moe_gpu.moe_permute_nvfp4(x, idx, counts, E)
    for key in ("offsets", "dest_row", "src_pair"):
        assert torch.equal(out[key], ref[key]), key
    assert out["tensor_scale"][0].item() == rg[0].item()
    assert torch.equal(out["codes"], rc) and torch.equal(out["scales"], rs)


def test_nvfp4_layer_full_size_by_stage():
    """The DeepSeek-V3-shaped NVFP4 layer at full size, stage by stage on samples: the
    tensor scale of Xp (from the amax of x) and the codes of sampled Xp rows; W1 and W2
    codes of sampled experts (their tensor scale from the amax of the whole stack);
    sampled rows of H and Yp against the oracle on the decoded operands; and H
    re-quantised by the oracle from the GPU's bf16 H (its tensor scale from all of H)."""
    need_gpu()
    w = W.BY_NAME["dsv3-nvfp4"]
    x, W1, W2, lg = W.make_x(w, "cuda"), W.make_w1(w, "cuda"), W.make_w2(w, "cuda"), logits_dev(w)
    layer = moe_gpu.MoELayer(w.T, w.d, w.E, w.k, w.f, W1, W2, dtype="nvfp4", renormalize=w.renormalize)
    layer.forward(x, lg)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    rng = np.random.default_rng(17)
    idx, wt, counts = om.route_topk(lg.cpu().numpy(), w.k)
    offsets, dest, src = om.permute_maps(idx, w.E)
    assert (i64(layer.src_pair) == src).all()
    gx = o4.tensor_scale(x.float().cpu().numpy())
    assert layer.xg[0].item() == float(gx)
    rows = np.sort(rng.choice(w.M, size=64, replace=False))
    c, s, _ = o4.quantize(x[torch.from_numpy(src[rows] // w.k).cuda()].float().cpu().numpy(), gx)
    r_t = torch.from_numpy(rows).cuda()
    assert (layer.xq[r_t].cpu().numpy() == c).all() and (layer.xs[r_t].cpu().numpy() == s).all()
    # the weight stacks' tensor scales from their amax (a torch reduction of the inputs)
    g1 = np.float32(2688.0) / np.float32(W1.abs().max().float().item())
    g2 = np.float32(2688.0) / np.float32(W2.abs().max().float().item())
    assert layer.W1g[0].item() == float(g1) and layer.W2g[0].item() == float(g2)
    h_all = layer.h.float().cpu().numpy()
    gh = o4.tensor_scale(h_all)
    assert layer.hg[0].item() == float(gh)
    nz = np.nonzero(counts)[0]
    order = nz[np.argsort(counts[nz], kind="stable")]
    got_h, want_h, got_y, want_y = [], [], [], []
    for e in (int(order[-1]), int(order[len(order) // 2]), int(order[0])):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        c1, s1, _ = o4.quantize(W1[e].float().cpu().numpy(), g1)
        assert (layer.W1q[e].cpu().numpy() == c1).all() and (layer.W1s[e].cpu().numpy() == s1).all()
        c2, s2, _ = o4.quantize(W2[e].float().cpu().numpy(), g2)
        assert (layer.W2q[e].cpu().numpy() == c2).all() and (layer.W2s[e].cpu().numpy() == s2).all()
        rr = np.sort(rng.choice(np.arange(lo, hi), size=min(8, hi - lo), replace=False))
        rr_t = torch.from_numpy(rr).cuda()
        xa = o4.dequantize(layer.xq[rr_t].cpu().numpy(), layer.xs[rr_t].cpu().numpy(), gx)
        gu = xa @ o4.dequantize(c1, s1, g1).T
        got_h.append(h_all[rr])
        want_h.append(om.swiglu(gu))
        hc, hs, _ = o4.quantize(h_all[rr], gh)                      # the oracle's own quantisation of H
        assert (layer.hq[rr_t].cpu().numpy() == hc).all() and (layer.hs[rr_t].cpu().numpy() == hs).all()
        got_y.append(f64(layer.yp[rr_t]))
        want_y.append(o4.dequantize(hc, hs, gh) @ o4.dequantize(c2, s2, g2).T)
    assert rel_l2(np.concatenate(got_h), np.concatenate(want_h)) < 1e-2
    assert rel_l2(np.concatenate(got_y), np.concatenate(want_y)) < 1e-2

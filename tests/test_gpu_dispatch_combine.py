"""GPU parity: routing, dispatch (plain and fused MXFP8), quantisation, combine,
combine backward and router backward against the float64 oracle.

Integers (expert ids, counts, offsets, both permutation maps) and MXFP8
bytes must match bit-exactly; routing weights within 1e-6; floating outputs
within the bound their arithmetic allows.
"""

import numpy as np
import pytest
import torch

import ragged_grouped_gemm_topk_gb300 as moe_gpu
from ragged_grouped_gemm_topk_gb300 import workloads as W
from oracle import moe as om
from oracle import mxfp8 as omx
from _parity import TOL_W, f64, i64, logits_dev, need_gpu, rel_l2

pytestmark = pytest.mark.gpu

# Full-size routing/dispatch for every workload (integer work is cheap to check
# in full), plus reduced shapes with awkward sizes.
ROUTE_CASES = [w.name for w in W.WORKLOADS]
SMALL = [
    W.WORKLOADS[0].scaled(T=1, name="T1"),
    W.WORKLOADS[0].scaled(T=257, E=5, k=3, d=40, name="ragged-T257"),
    W.WORKLOADS[2].scaled(T=1000, E=128, k=8, d=64, name="zipf-E128"),
    W.WORKLOADS[3].scaled(T=300, E=256, k=8, d=96, name="zipf-E256-empty"),
    W.WORKLOADS[0].scaled(T=64, E=1, k=1, d=32, name="E1"),
    W.WORKLOADS[0].scaled(T=50, E=6, k=6, d=32, name="k=E"),
    W.WORKLOADS[0].scaled(T=77, E=1000, k=32, d=32, name="E1000-k32"),
    W.WORKLOADS[0].scaled(T=300, E=1024, k=8, d=32, name="E1024-k8"),
]


def _route_check(w, renormalize=True):
    lg = logits_dev(w)
    idx, wt, counts = moe_gpu.moe_route_topk(lg, w.k, renormalize)
    o_idx, o_w, o_counts = om.route_topk(lg.cpu().numpy(), w.k, renormalize)
    assert (i64(idx) == o_idx).all()
    assert np.abs(f64(wt) - o_w).max() <= TOL_W
    assert (i64(counts) == o_counts).all()
    return lg, idx, wt, counts, o_idx


@pytest.mark.parametrize("name", ROUTE_CASES)
def test_route_full_size(name):
    need_gpu()
    _route_check(W.BY_NAME[name])


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("renormalize", [True, False])
def test_route_small(w, renormalize):
    need_gpu()
    _route_check(w, renormalize)


def test_route_ties_and_masked():
    need_gpu()
    lg = torch.tensor([[1, 3, 2, 3], [0, 0, 0, 0], [-np.inf, 5, -np.inf, -np.inf]],
                      dtype=torch.float32).cuda()
    idx, wt, counts = moe_gpu.moe_route_topk(lg, 2)
    assert idx.cpu().tolist() == [[1, 3], [0, 1], [1, 0]]
    got = wt.cpu().numpy()
    np.testing.assert_allclose(got[:2], 0.5, atol=TOL_W)
    assert got[2, 0] == 1.0 and got[2, 1] == 0.0
    assert counts.cpu().tolist() == [2, 3, 0, 1]


def test_route_nan_flags_status():
    need_gpu()
    lg = torch.zeros(4, 8, device="cuda")
    lg[2, 3] = float("nan")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe_gpu.moe_route_topk(lg, 2, dev_status=st)
    assert int(st.item()) & moe_gpu.binding.MOE_DEV_NAN_LOGIT


def _dispatch_check(w, x, quant=False):
    lg, idx, wt, counts, o_idx = _route_check(w)
    out = moe_gpu.moe_permute(x, idx, counts, w.E, xp_dtype="mxfp8" if quant else None)
    o_off, o_dest, o_src = om.permute_maps(o_idx, w.E)
    assert (i64(out["offsets"]) == o_off).all()
    assert (i64(out["dest_row"]) == o_dest).all()
    assert (i64(out["src_pair"]) == o_src).all()
    return out, (o_off, o_dest, o_src), idx, wt


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_permute_rows_bit_exact(w):
    need_gpu()
    x = W.make_x(w, "cuda")
    out, (o_off, o_dest, o_src), _, _ = _dispatch_check(w, x)
    want = x.cpu()[torch.from_numpy(o_src // w.k)]
    assert torch.equal(out["xp"].cpu().view(torch.int16) if x.dtype == torch.bfloat16 else out["xp"].cpu(),
                       want.view(torch.int16) if x.dtype == torch.bfloat16 else want)


@pytest.mark.parametrize("name", ["mixtral-bf16", "qwen3-235b-bf16", "dsv3-bf16-train"])
def test_permute_full_size(name):
    need_gpu()
    w = W.BY_NAME[name]
    x = W.make_x(w, "cuda")
    out, (o_off, o_dest, o_src), _, _ = _dispatch_check(w, x)
    # the copied rows: every row equals its source token's row, bit for bit
    src_tok = torch.from_numpy(o_src // w.k).cuda()
    assert torch.equal(out["xp"].view(torch.int16), x.view(torch.int16)[src_tok])


@pytest.mark.parametrize("w", [SMALL[1].scaled(d=64, name="ragged-T257-d64"), SMALL[3],
                               W.WORKLOADS[3].scaled(T=512, name="dsv3-T512")],
                         ids=lambda w: w.name)
def test_permute_fused_mxfp8_bit_exact(w):
    need_gpu()
    x = W.make_x(w, "cuda").to(torch.bfloat16)
    out, (o_off, o_dest, o_src), _, _ = _dispatch_check(w, x, quant=True)
    xo = f64(x)[o_src // w.k]
    codes, scales = omx.quantize_rowwise(xo)
    assert (out["xp"].cpu().numpy() == codes).all()
    assert (out["xp_scales"].cpu().numpy() == scales).all()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("d", [4192, 6144])
def test_permute_fused_mxfp8_segments(d, dtype):
    """Rows longer than one staging segment of the quantising scatter (2048 bf16 or 1024
    fp32 elements): d = 4192 ends in a partial segment and has 131-byte scale rows (copied
    out byte by byte), d = 6144 is whole segments with 16-byte copies throughout."""
    need_gpu()
    w = W.WORKLOADS[3].scaled(T=200, E=32, k=4, d=d, name="mx-seg")
    x = W.make_x(w, "cuda").to(dtype)
    out, (o_off, o_dest, o_src), _, _ = _dispatch_check(w, x, quant=True)
    codes, scales = omx.quantize_rowwise(f64(x)[o_src // w.k])
    assert (out["xp"].cpu().numpy() == codes).all()
    assert (out["xp_scales"].cpu().numpy() == scales).all()


def test_permute_mxfp8_rejects_width_not_multiple_of_32():
    need_gpu()
    w = SMALL[1]                                     # d = 40
    x = W.make_x(w, "cuda").to(torch.bfloat16)
    lg = logits_dev(w)
    idx, wt, counts = moe_gpu.moe_route_topk(lg, w.k)
    with pytest.raises(moe_gpu.binding.MoeError, match="d % 32"):
        moe_gpu.moe_permute(x, idx, counts, w.E, xp_dtype="mxfp8")


def test_permute_fused_mxfp8_full_dsv3():
    need_gpu()
    w = W.BY_NAME["dsv3-mxfp8"]
    x = W.make_x(w, "cuda")
    out, (o_off, o_dest, o_src), _, _ = _dispatch_check(w, x, quant=True)
    # quantisation is row-wise: check a seeded sample of 2048 rows in full
    rows = np.random.default_rng(0).choice(w.M, 2048, replace=False)
    xo = f64(x[torch.from_numpy(o_src[rows] // w.k).cuda()])
    codes, scales = omx.quantize_rowwise(xo)
    r = torch.from_numpy(rows).cuda()
    assert (out["xp"][r].cpu().numpy() == codes).all()
    assert (out["xp_scales"][r].cpu().numpy() == scales).all()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantize_rowwise_bit_exact(dtype):
    need_gpu()
    a = W.make_matrix(333, 2048, seed=5, dtype=dtype, device="cuda")
    a[7, 64:96] = 0                                     # an all-zero block
    a[8] *= 1e-30 if dtype == torch.float32 else 1.0   # tiny magnitudes
    a[9, :32] = 448.0 * 2.0 ** 20                       # saturation boundary
    a[10, 0] = -0.0
    if dtype == torch.float32:
        a[11, :32] = 1e-40                              # subnormal block maximum
    codes, scales = moe_gpu.moe_quantize_mxfp8_grouped(a)
    c, s = omx.quantize_rowwise(f64(a))
    assert (codes.cpu().numpy() == c).all()
    assert (scales.cpu().numpy() == s).all()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("counts,K", [([0, 1, 130, 257, 3, 128, 0, 64], 2048),   # empty, single, partial blocks
                                      ([33] * 5, 544),                            # strip tail (544 = 512 + 32)
                                      ([0, 0, 700], 32),                          # leading empty groups
                                      ([31, 32, 0, 65, 1], 96),
                                      ([1] * 300, 64)],                           # many one-row groups
                         ids=["mixed", "K544", "lead-empty", "edges", "singles"])
def test_quantize_colwise_grouped_bit_exact(dtype, counts, K):
    """Column-wise group-aware MXFP8 (blocks of 32 rows restarting per group, the
    last one zero-padded) against the oracle: codes and every written scale row
    bit-exact; scale rows past the blocks untouched."""
    need_gpu()
    rows = int(sum(counts))
    a = W.make_matrix(rows, K, seed=len(counts) + K, dtype=dtype, device="cuda")
    if rows > 40:
        a[3:6, :] = 0                                     # zero rows inside a block
        a[40, 0] = 448.0 * 2.0 ** 20                      # saturation boundary
        a[41, 1] = -0.0
    off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device="cuda")
    E = len(counts)
    cap = (rows + 31) // 32 + E
    codes = torch.full((rows, K), 0x5A, dtype=torch.uint8, device="cuda")
    scales = torch.full((cap, K), 0xA5, dtype=torch.uint8, device="cuda")
    moe_gpu.moe_quantize_mxfp8_grouped(a, off, E, codes=codes, scales=scales, axis=1)
    c, sc = omx.quantize_colwise_grouped(f64(a), off.cpu().numpy())
    assert (codes.cpu().numpy() == c).all()
    n = sc.shape[0]
    assert (scales[:n].cpu().numpy() == sc).all()
    assert (scales[n:] == 0xA5).all()


def tiled_scale_index(offsets, K):
    """Byte index, in the tiled column-wise scale layout, of every (block row, column)
    of the compact layout, block rows numbered group by group."""
    idx = []
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        for b in range((hi - lo + 31) // 32):
            quad = lo // 128 + e + b // 4
            m = np.arange(K)
            idx.append((quad * (K // 128) + m // 128) * 512 + (m % 32) * 16 + ((m % 128) // 32) * 4 + b % 4)
    return np.array(idx, dtype=np.int64).reshape(-1, K)


@pytest.mark.parametrize("counts,K", [([0, 1, 130, 257, 3, 128, 0, 64], 256),
                                      ([1] * 300, 128),
                                      ([0, 0, 700], 384),
                                      ([127, 129, 0, 256, 31], 512)],
                         ids=["mixed", "singles", "lead-empty", "quad-edges"])
def test_quantize_colwise_tiled_scales(counts, K):
    """Axis 2: the codes of axis 1, and each scale byte at its place in the tiled
    layout equal to the oracle's; bytes outside every group's blocks untouched."""
    need_gpu()
    rows = int(sum(counts))
    a = W.make_matrix(rows, K, seed=len(counts) + K + 1, dtype=torch.bfloat16, device="cuda")
    off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device="cuda")
    E = len(counts)
    codes = torch.full((rows, K), 0x5A, dtype=torch.uint8, device="cuda")
    tiles = ((rows + 127) // 128 + E) * (K // 128)
    scales = torch.full((tiles, 512), 0xA5, dtype=torch.uint8, device="cuda")
    moe_gpu.moe_quantize_mxfp8_grouped(a, off, E, codes=codes, scales=scales, axis=2)
    c, sc = omx.quantize_colwise_grouped(f64(a), off.cpu().numpy())
    assert (codes.cpu().numpy() == c).all()
    idx = tiled_scale_index(off.cpu().numpy(), K)
    flat = scales.cpu().numpy().reshape(-1)
    assert len(np.unique(idx)) == idx.size and idx.max() < flat.size      # distinct places, in the buffer
    assert (flat[idx] == sc).all()
    rest = np.ones(flat.size, dtype=bool)
    rest[idx.reshape(-1)] = False
    assert (flat[rest] == 0xA5).all()


def test_quantize_colwise_needs_offsets():
    need_gpu()
    a = W.make_matrix(64, 64, seed=1, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe_gpu.binding.MoeError):
        moe_gpu.moe_quantize_mxfp8_grouped(a, None, 0, axis=1)


GATHER_CASES = [SMALL[1].scaled(d=128, name="ragged-T257"), SMALL[2].scaled(d=128, name="zipf-E128"),
                SMALL[3].scaled(d=256, name="zipf-E256-empty"), SMALL[6].scaled(d=128, name="E1000-k32"),
                W.WORKLOADS[3].scaled(T=512, name="dsv3-T512")]


@pytest.mark.parametrize("w", GATHER_CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("axis", [1, 2])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_quantize_gathered_colwise_bit_exact(w, axis, dtype):
    """Column-wise MXFP8 of the dispatched rows read through src_pair equals the
    oracle's column-wise quantisation of its own permuted rows, codes and every
    scale byte; the status word stays clear."""
    need_gpu()
    x = W.make_x(w, "cuda").to(dtype)
    out, (o_off, o_dest, o_src), _, _ = _dispatch_check(w, x)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales = moe_gpu.moe_quantize_mxfp8_gathered(x, out["src_pair"], out["offsets"], w.E, w.k, axis=axis,
                                                        dev_status=st)
    c, sc = omx.quantize_colwise_grouped(f64(x)[o_src // w.k], o_off)
    assert (codes.cpu().numpy() == c).all()
    if axis == 1:
        assert (scales[:sc.shape[0]].cpu().numpy() == sc).all()
    else:
        idx = tiled_scale_index(o_off, w.d)
        assert (scales.cpu().numpy().reshape(-1)[idx] == sc).all()
    assert int(st.item()) == 0


def test_quantize_gathered_colwise_full_dsv3_sampled():
    """Full DeepSeek-V3 training size (T=16384, k=8, d=7168): the codes and tiled
    scales of sampled column strips of every group's first and last block."""
    need_gpu()
    w = W.BY_NAME["dsv3-mxfp8-train"]
    x = W.make_x(w, "cuda").to(torch.bfloat16)
    out, (o_off, o_dest, o_src), _, _ = _dispatch_check(w, x)
    codes, scales = moe_gpu.moe_quantize_mxfp8_gathered(x, out["src_pair"], out["offsets"], w.E, w.k, axis=2)
    cols = np.array([0, 1, 127, 128, 3583, 5000, 7167])
    rng = np.random.default_rng(7)
    groups = [e for e in range(w.E) if o_off[e + 1] > o_off[e]]
    for e in rng.choice(groups, size=12, replace=False):
        lo, hi = int(o_off[e]), int(o_off[e + 1])
        for r0 in sorted({lo, lo + ((hi - lo - 1) // 32) * 32}):
            r1 = min(r0 + 32, hi)
            blk = f64(x[torch.from_numpy(o_src[r0:r1] // w.k).cuda()][:, torch.from_numpy(cols).cuda()])
            c, sc = omx.quantize_colwise_grouped(blk, np.array([0, r1 - r0]))
            assert (codes[r0:r1][:, torch.from_numpy(cols).cuda()].cpu().numpy() == c).all()
            b = (r0 - lo) // 32
            quad = lo // 128 + e + b // 4
            flat = scales.view(-1)
            pos = (quad * (w.d // 128) + cols // 128) * 512 + (cols % 32) * 16 + ((cols % 128) // 32) * 4 + b % 4
            assert (flat[torch.from_numpy(pos).cuda()].cpu().numpy() == sc[0]).all()


def test_quantize_gathered_flags_bad_pair_index():
    """A src_pair entry outside [0, T*k) sets MOE_DEV_BAD_INDEX and its row reads as
    zeros (the kernel checks the index before the load)."""
    need_gpu()
    w = SMALL[1].scaled(d=64, name="ragged-T257")
    x = W.make_x(w, "cuda").to(torch.bfloat16)
    out, (o_off, o_dest, o_src), _, _ = _dispatch_check(w, x)
    src = out["src_pair"].clone()
    src[5] = w.T * w.k + 3
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, _ = moe_gpu.moe_quantize_mxfp8_gathered(x, src, out["offsets"], w.E, w.k, axis=1, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & moe_gpu.binding.MOE_DEV_BAD_INDEX
    assert (codes[5] == 0).all()


def _combine_bound(yp64, dest, w):
    """|fp32 sum of k products rounded once to bf16 - exact| <= 2^-8 * sum_j |w_j yp_j|."""
    T, k = dest.shape
    mag = np.zeros((T, yp64.shape[1]))
    for j in range(k):
        mag += np.abs(w[:, j:j + 1] * yp64[dest[:, j]])
    return 2.0 ** -8 * mag + 1e-30


@pytest.mark.parametrize("w", SMALL + [W.BY_NAME["qwen3-235b-bf16"], W.BY_NAME["dsv3-bf16-train"]],
                         ids=lambda w: w.name)
def test_combine(w):
    need_gpu()
    lg, idx, wt, counts, o_idx = _route_check(w)
    out = moe_gpu.moe_permute(None, idx, counts, w.E, rows=False)
    yp = W.make_matrix(w.M, w.d, seed=77, dtype=w.torch_dtype, device="cuda")
    y = moe_gpu.moe_unpermute_combine(yp, out["dest_row"], wt)
    o_w = om.route_topk(lg.cpu().numpy(), w.k)[1]
    o_dest = om.permute_maps(o_idx, w.E)[1]
    yp64 = f64(yp)
    want = om.combine(yp64, o_dest, o_w)
    got = f64(y)
    assert (np.abs(got - want) <= _combine_bound(yp64, o_dest, o_w) + 1e-6 * np.abs(want)).all()
    assert rel_l2(got, want) < 4e-3


@pytest.mark.parametrize("k", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("d", [8, 2056])
@pytest.mark.parametrize("dt_in,dt_out", [(torch.bfloat16, torch.bfloat16), (torch.bfloat16, torch.float32),
                                          (torch.float32, torch.bfloat16), (torch.float32, torch.float32)],
                         ids=["bf16-bf16", "bf16-f32", "f32-bf16", "f32-f32"])
def test_combine_each_k_width_and_dtype(k, d, dt_in, dt_out):
    """Every specialised k (1, 2, 4, 8) and the general loop (k=3), a one-chunk row
    (d=8) and a row one chunk past a work item (d=2056 bf16), all dtype pairs."""
    need_gpu()
    T = 97
    rng = np.random.default_rng(1000 + 10 * k + d)
    dest = rng.permutation(T * k).reshape(T, k).astype(np.int64)
    wts = rng.uniform(0.05, 1.0, size=(T, k))
    yp = W.make_matrix(T * k, d, seed=79, dtype=dt_in, device="cuda")
    got = f64(moe_gpu.moe_unpermute_combine(yp, torch.from_numpy(dest).to(torch.int32).cuda(),
                                            torch.from_numpy(wts).float().cuda(), out_dtype=dt_out))
    w32 = wts.astype(np.float32).astype(np.float64)
    yp64 = f64(yp)
    want = om.combine(yp64, dest, w32)
    mag = _combine_bound(yp64, dest, w32) * 2.0 ** 8
    ulp = 2.0 ** -8 if dt_out == torch.bfloat16 else 2.0 ** -23
    assert (np.abs(got - want) <= (ulp + k * 2.0 ** -24) * mag + 1e-30).all()


@pytest.mark.parametrize("k", [1, 2, 4, 8])
def test_combine_of_permute_identity_bit_exact(k):
    """k=1 with unit weights, or w = 1/k: combine(permute(x)) == x exactly."""
    need_gpu()
    w = W.WORKLOADS[2].scaled(T=999, E=16, k=k, d=256, name=f"id-k{k}")
    x = W.make_x(w, "cuda")
    lg = logits_dev(w)
    idx, wt, counts = moe_gpu.moe_route_topk(lg, k)
    out = moe_gpu.moe_permute(x, idx, counts, w.E)
    ones = torch.full_like(wt, 1.0 / k)
    y = moe_gpu.moe_unpermute_combine(out["xp"], out["dest_row"], ones)
    assert torch.equal(y.view(torch.int16), x.view(torch.int16))
    if k == 1:
        y1 = moe_gpu.moe_unpermute_combine(out["xp"], out["dest_row"], None)
        assert torch.equal(y1.view(torch.int16), x.view(torch.int16))


@pytest.mark.parametrize("w", [SMALL[1], SMALL[2], W.BY_NAME["dsv3-bf16-train"].scaled(T=2048, name="dsv3-T2048")],
                         ids=lambda w: w.name)
def test_combine_bwd(w):
    need_gpu()
    lg, idx, wt, counts, o_idx = _route_check(w)
    out = moe_gpu.moe_permute(None, idx, counts, w.E, rows=False)
    yp = W.make_matrix(w.M, w.d, seed=78, dtype=w.torch_dtype, device="cuda")
    dy = W.make_dy(w, "cuda")
    dyp, dw = moe_gpu.moe_unpermute_combine_bwd(dy, yp, out["dest_row"], wt)
    o_w = om.route_topk(lg.cpu().numpy(), w.k)[1]
    o_dest = om.permute_maps(o_idx, w.E)[1]
    want_dyp, want_dw = om.combine_bwd(f64(dy), f64(yp), o_dest, o_w)
    assert rel_l2(f64(dyp), want_dyp) < 4e-3
    assert rel_l2(f64(dw), want_dw) < 1e-5


def _dyp_case(w, seed):
    """Seeded inputs of the MXFP8 combine backward: the oracle's own maps (from its
    routing of the workload's logits), seeded routing weights, dy and yp; and the
    dYp the bf16 combine backward stores, w * dy in fp32 rounded to bf16 (the
    precision in which the kernel takes the value its codes come from)."""
    o_idx = om.route_topk(W.make_logits(w), w.k)[0]
    o_off, o_dest, o_src = om.permute_maps(o_idx, w.E)
    rng = np.random.default_rng(seed)
    w32 = rng.uniform(0.05, 1.0, size=(w.T, w.k)).astype(np.float32)
    dy = W.make_matrix(w.T, w.d, seed=seed + 1, dtype=torch.bfloat16, device="cuda")
    yp = W.make_matrix(w.M, w.d, seed=seed + 2, dtype=torch.bfloat16, device="cuda")
    prod = (torch.from_numpy(w32)[:, :, None] * dy.cpu().float()[:, None, :]).to(torch.bfloat16)
    dyp = torch.empty(w.M, w.d, dtype=torch.bfloat16)
    dyp[torch.from_numpy(o_dest.reshape(-1))] = prod.reshape(-1, w.d)
    dev = {"dest_row": torch.from_numpy(o_dest.astype(np.int32)).cuda(),
           "src_pair": torch.from_numpy(o_src.astype(np.int32)).cuda(),
           "offsets": torch.from_numpy(o_off.astype(np.int32)).cuda(),
           "topk_w": torch.from_numpy(w32).cuda()}
    return dy, yp, w32, (o_off, o_dest, o_src), f64(dyp), dev


MX_BWD_CASES = [SMALL[1].scaled(d=64, name="ragged-T257"), SMALL[3].scaled(d=256, name="zipf-E256-empty"),
                SMALL[2].scaled(d=384, name="zipf-E128-d384"),          # a partly filled second 32-chunk step
                W.BY_NAME["dsv3-bf16-train"].scaled(T=1024, name="dsv3-T1024")]


@pytest.mark.parametrize("w", MX_BWD_CASES, ids=lambda w: w.name)
def test_combine_bwd_mxfp8_bit_exact(w):
    """Row-wise MXFP8 of dYp from the combine backward equals the oracle's row-wise
    quantisation of the bf16 dYp, codes and scales bit for bit; dw as the bf16 path."""
    need_gpu()
    dy, yp, w32, (o_off, o_dest, o_src), dyp64, dev = _dyp_case(w, seed=31)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales, dw = moe_gpu.moe_unpermute_combine_bwd_mxfp8(dy, yp, dev["dest_row"], dev["topk_w"],
                                                                dev_status=st)
    c, sc = omx.quantize_rowwise(dyp64)
    assert (codes.cpu().numpy() == c).all()
    assert (scales.cpu().numpy() == sc).all()
    want_dw = om.combine_bwd(f64(dy), f64(yp), o_dest, w32.astype(np.float64))[1]
    assert rel_l2(f64(dw), want_dw) < 1e-5
    assert int(st.item()) == 0


@pytest.mark.parametrize("w", MX_BWD_CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("axis", [1, 2])
def test_quantize_gathered_weighted_is_colwise_of_dyp(w, axis):
    """Column-wise MXFP8 gathered from dy with the routing weights equals the
    oracle's column-wise quantisation of the bf16 dYp, codes and scales."""
    need_gpu()
    if axis == 2 and w.d % 128:
        pytest.skip("tiled scales need d % 128 == 0")
    dy, yp, w32, (o_off, o_dest, o_src), dyp64, dev = _dyp_case(w, seed=41)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales = moe_gpu.moe_quantize_mxfp8_gathered(dy, dev["src_pair"], dev["offsets"], w.E, w.k,
                                                        row_w=dev["topk_w"], axis=axis, dev_status=st)
    c, sc = omx.quantize_colwise_grouped(dyp64, o_off)
    assert (codes.cpu().numpy() == c).all()
    if axis == 1:
        assert (scales[:sc.shape[0]].cpu().numpy() == sc).all()
    else:
        idx = tiled_scale_index(o_off, w.d)
        assert (scales.cpu().numpy().reshape(-1)[idx] == sc).all()
    assert int(st.item()) == 0


def test_combine_bwd_mxfp8_rejects_bad_args():
    need_gpu()
    w = SMALL[1].scaled(d=40, name="d40")
    dy, yp = torch.zeros(w.T, 40, dtype=torch.bfloat16, device="cuda"), torch.zeros(w.M, 40, dtype=torch.bfloat16,
                                                                                     device="cuda")
    dest = torch.zeros(w.T, w.k, dtype=torch.int32, device="cuda")
    wt = torch.ones(w.T, w.k, dtype=torch.float32, device="cuda")
    with pytest.raises(moe_gpu.binding.MoeError, match="32"):                 # d % 32
        moe_gpu.moe_unpermute_combine_bwd_mxfp8(dy, yp, dest, wt)
    with pytest.raises(moe_gpu.binding.MoeError):                             # fp32 input
        moe_gpu.moe_unpermute_combine_bwd_mxfp8(torch.zeros(w.T, 64, device="cuda"),
                                                torch.zeros(w.M, 64, device="cuda"), dest, wt)


@pytest.mark.parametrize("renormalize", [True, False])
def test_route_bwd(renormalize):
    need_gpu()
    w = W.WORKLOADS[3].scaled(T=700, name="rb")
    lg = logits_dev(w)
    idx, wt, counts = moe_gpu.moe_route_topk(lg, w.k, renormalize)
    dw = W.make_matrix(w.T, w.k, seed=3, dtype=torch.float32, device="cuda")
    dl = moe_gpu.moe_route_topk_bwd(dw, wt, idx, w.E, logits=lg, renormalize=renormalize)
    o_idx, o_w, _ = om.route_topk(lg.cpu().numpy(), w.k, renormalize)
    want = om.route_bwd(f64(dw), o_w, o_idx, lg.cpu().numpy(), renormalize)
    got = f64(dl)
    assert np.abs(got - want).max() < 1e-5
    if renormalize:
        sel = np.zeros_like(want, dtype=bool)
        np.put_along_axis(sel, o_idx.astype(np.int64), True, axis=1)
        assert (got[~sel] == 0).all()


@pytest.mark.parametrize("renormalize", [True, False])
def test_route_fully_masked_token(renormalize):
    """A token with every expert masked (-inf) gets the lowest expert ids with
    weight 0 and a zero router gradient, like the oracle; the other tokens of the
    batch are routed as usual."""
    need_gpu()
    w = W.WORKLOADS[2].scaled(T=96, E=40, k=4, name="masked")
    lg = logits_dev(w)
    lg[5] = -float("inf")
    lg[70, 3:] = -float("inf")            # only three experts left for k = 4
    idx, wt, counts = moe_gpu.moe_route_topk(lg, w.k, renormalize)
    o_idx, o_w, o_counts = om.route_topk(lg.cpu().numpy(), w.k, renormalize)
    assert (i64(idx) == o_idx).all() and (i64(counts) == o_counts).all()
    got = f64(wt)
    assert not np.isnan(got).any() and (got[5] == 0).all() and got[70, 3] == 0
    assert np.abs(got - o_w).max() <= TOL_W
    dw = W.make_matrix(w.T, w.k, seed=4, dtype=torch.float32, device="cuda")
    dl = f64(moe_gpu.moe_route_topk_bwd(dw, wt, idx, w.E, logits=lg, renormalize=renormalize))
    want = om.route_bwd(f64(dw), o_w, o_idx, lg.cpu().numpy(), renormalize)
    assert not np.isnan(dl).any() and (dl[5] == 0).all()
    assert np.abs(dl - want).max() < 1e-5

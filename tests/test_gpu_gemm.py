"""GPU parity of the ragged grouped GEMM (tcgen05) against the float64 oracle.

Ragged groups with empty experts, single rows, exact tile multiples and tails,
several K blocks and column tiles, partial last column tiles, TF32 and BF16,
with and without the fused SwiGLU epilogue.  Rows beyond offsets[E] must stay
untouched.
"""

import numpy as np
import pytest
import torch

import ragged_grouped_gemm_topk_gb300 as moe_gpu
from ragged_grouped_gemm_topk_gb300 import workloads as W
from oracle import moe as om
from _parity import TOL_BF16, f64, need_gpu, ragged_offsets, rel_l2

pytestmark = pytest.mark.gpu

COUNTS = {
    "mixed": [0, 1, 130, 257, 3, 128, 0, 64],
    "one-expert": [700],
    "all-in-last": [0, 0, 0, 385],
    "singles": [1] * 37,
}


def _mats(M, K, N, E, dtype, seed):
    A = W.make_matrix(M, K, seed=seed, dtype=dtype, device="cuda")
    B = W.make_matrix(E * N, K, seed=seed + 1, dtype=dtype, device="cuda", scale=K ** -0.5).view(E, N, K)
    return A, B


@pytest.mark.parametrize("counts", list(COUNTS), ids=str)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "tf32"])
@pytest.mark.parametrize("K,N", [(256, 512), (1024, 320), (96, 64)])
def test_fwd_plain(counts, dtype, K, N):
    need_gpu()
    cnt = COUNTS[counts]
    E = len(cnt)
    M = int(sum(cnt)) + 5                      # 5 trailing rows outside every group
    A, B = _mats(M, K, N, E, dtype, seed=K + N)
    off = ragged_offsets(cnt)
    C = torch.full((M, N), float("nan"), dtype=dtype, device="cuda")
    moe_gpu.moe_grouped_gemm_fwd(A, B, off, out=C)
    want = om.grouped_gemm(f64(A), f64(B), off.cpu().numpy())
    got = f64(C)
    rows = int(sum(cnt))
    assert np.isnan(got[rows:]).all(), "rows past offsets[E] were written"
    err = rel_l2(got[:rows], want[:rows])
    assert err < TOL_BF16, err


@pytest.mark.parametrize("counts", ["mixed", "singles"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "tf32"])
@pytest.mark.parametrize("K,f", [(256, 256), (512, 160), (64, 32)])
def test_fwd_swiglu(counts, dtype, K, f):
    need_gpu()
    cnt = COUNTS[counts]
    E = len(cnt)
    M = int(sum(cnt))
    A, B = _mats(M, K, 2 * f, E, dtype, seed=K + f)
    off = ragged_offsets(cnt)
    H, GU = moe_gpu.moe_grouped_gemm_fwd(A, B, off, epi="swiglu", out_dtype=dtype, want_preact=True)
    GU_want = om.grouped_gemm(f64(A), f64(B), off.cpu().numpy())
    H_want = om.swiglu(GU_want)
    assert rel_l2(f64(GU), GU_want) < TOL_BF16
    assert rel_l2(f64(H), H_want) < TOL_BF16
    H2 = moe_gpu.moe_grouped_gemm_fwd(A, B, off, epi="swiglu", out_dtype=dtype)
    assert torch.equal(H2, H)


def test_fwd_empty_rows_and_zero_M():
    need_gpu()
    A, B = _mats(0, 64, 64, 3, torch.bfloat16, seed=1)
    off = ragged_offsets([0, 0, 0])
    C = moe_gpu.moe_grouped_gemm_fwd(A, B, off)
    assert C.shape == (0, 64)
    # all experts empty but rows allocated: nothing is written
    A, B = _mats(40, 64, 64, 3, torch.bfloat16, seed=2)
    C = torch.full((40, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    moe_gpu.moe_grouped_gemm_fwd(A, B, off, out=C)
    assert (C == 7.0).all()


def test_fwd_rejects_bad_shapes():
    need_gpu()
    A, B = _mats(16, 48, 64, 2, torch.bfloat16, seed=3)
    with pytest.raises(moe_gpu.binding.MoeError):
        moe_gpu.moe_grouped_gemm_fwd(A, B, ragged_offsets([8, 8]))          # K % 32 != 0
    A, B = _mats(16, 64, 64, 2, torch.bfloat16, seed=3)
    with pytest.raises(moe_gpu.binding.MoeError):
        moe_gpu.moe_grouped_gemm_fwd(A, B.float(), ragged_offsets([8, 8]))  # mixed dtypes


def test_fwd_bad_offsets_flag_status():
    need_gpu()
    A, B = _mats(64, 64, 64, 2, torch.bfloat16, seed=4)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    off = torch.tensor([0, 40, 100], dtype=torch.int32, device="cuda")     # past M
    C = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    moe_gpu.moe_grouped_gemm_fwd(A, B, off, out=C, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & moe_gpu.binding.MOE_DEV_BAD_INDEX


# ----------------------------------------------------------------------------- backward GEMMs

@pytest.mark.parametrize("counts", ["mixed", "singles", "all-in-last"], ids=str)
@pytest.mark.parametrize("N,K", [(256, 512), (96, 320), (1024, 64)])
def test_dgrad_plain(counts, N, K):
    """dA = dC . B[e]: contraction over N (B read MN-major), output width K."""
    need_gpu()
    cnt = COUNTS[counts]
    E = len(cnt)
    M = int(sum(cnt)) + 3
    dC = W.make_matrix(M, N, seed=N + K, dtype=torch.bfloat16, device="cuda")
    B = W.make_matrix(E * N, K, seed=N + K + 1, dtype=torch.bfloat16, device="cuda",
                      scale=N ** -0.5).view(E, N, K)
    off = ragged_offsets(cnt)
    dA = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe_gpu.moe_grouped_gemm_dgrad(dC, B, off, out=dA)
    want = om.grouped_gemm_dgrad(f64(dC), f64(B), off.cpu().numpy())
    got = f64(dA)
    rows = int(sum(cnt))
    assert np.isnan(got[rows:]).all()
    assert rel_l2(got[:rows], want[:rows]) < TOL_BF16


@pytest.mark.parametrize("counts", ["mixed", "singles"], ids=str)
@pytest.mark.parametrize("d,f", [(256, 256), (512, 96), (128, 1024)])
def test_dgrad_dswiglu(counts, d, f):
    """GEMM2 data gradient with the SwiGLU backward fused: [dG | dU] from dYp, W2 and G|U."""
    need_gpu()
    cnt = COUNTS[counts]
    E = len(cnt)
    M = int(sum(cnt))
    dyp = W.make_matrix(M, d, seed=d + f, dtype=torch.bfloat16, device="cuda")
    W2 = W.make_matrix(E * d, f, seed=d + f + 1, dtype=torch.bfloat16, device="cuda",
                       scale=f ** -0.5).view(E, d, f)
    GU = W.make_matrix(M, 2 * f, seed=d + f + 2, dtype=torch.bfloat16, device="cuda", scale=2.0)
    off = ragged_offsets(cnt)
    dGU = moe_gpu.moe_grouped_gemm_dgrad(dyp, W2, off, epi="dswiglu", preact=GU)
    dH = om.grouped_gemm_dgrad(f64(dyp), f64(W2), off.cpu().numpy())
    want = om.dswiglu(dH, f64(GU))
    assert dGU.shape == (M, 2 * f)
    assert rel_l2(f64(dGU), want) < TOL_BF16


@pytest.mark.parametrize("counts", ["mixed", "singles", "all-in-last", "one-expert"], ids=str)
@pytest.mark.parametrize("N,K", [(256, 512), (160, 96), (64, 1024)])
def test_wgrad(counts, N, K):
    """dB[e] = dC[R_e]^T A[R_e]: a contraction over each group's ragged rows; empty
    groups give exact zeros; rows of neighbouring groups never leak in."""
    need_gpu()
    cnt = COUNTS[counts]
    E = len(cnt)
    M = int(sum(cnt)) + 7                     # trailing rows outside every group
    A = W.make_matrix(M, K, seed=N + K, dtype=torch.bfloat16, device="cuda")
    dC = W.make_matrix(M, N, seed=N + K + 3, dtype=torch.bfloat16, device="cuda")
    A[int(sum(cnt)):] = 1e4                   # poison the rows no group owns
    off = ragged_offsets(cnt)
    dB = torch.full((E, N, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe_gpu.moe_grouped_gemm_wgrad(A, dC, off, E, out=dB)
    want = om.grouped_gemm_wgrad(f64(A), f64(dC), off.cpu().numpy(), E)
    got = f64(dB)
    for e in range(E):
        if cnt[e] == 0:
            assert (got[e] == 0).all() and not np.signbit(got[e]).any(), f"expert {e} not exactly zero"
    assert not np.isnan(got).any()
    assert rel_l2(got, want) < TOL_BF16


def _check_fp32_and_accumulate(call, want, cnt, E, N, K, tol):
    """fp32 dB: the fp32 accumulator as it is, empty groups exact +0.  Accumulating:
    dB + the product with one fp32 rounding (bit for bit the fp32 sum of the old dB and
    the fp32 result), empty groups keep their values; a second call adds it again."""
    dB = torch.full((E, N, K), float("nan"), dtype=torch.float32, device="cuda")
    call(dB, False)
    got = f64(dB)
    for e in range(E):
        if cnt[e] == 0:
            assert (got[e] == 0).all() and not np.signbit(got[e]).any(), f"expert {e} not exactly zero"
    assert not np.isnan(got).any()
    assert rel_l2(got, want) < tol
    old = W.make_matrix(E * N, K, seed=N + K + 77, dtype=torch.float32, device="cuda").view(E, N, K)
    acc = old.clone()
    call(acc, True)
    torch.cuda.synchronize()
    assert torch.equal(acc, old + dB)
    for e in range(E):
        if cnt[e] == 0:
            assert torch.equal(acc[e], old[e]), f"expert {e} changed"
    call(acc, True)
    assert rel_l2(f64(acc), f64(old) + 2 * want) < tol


@pytest.mark.parametrize("counts", ["mixed", "singles", "one-expert"], ids=str)
@pytest.mark.parametrize("N,K", [(256, 512), (160, 96)])
def test_wgrad_fp32_and_accumulate(counts, N, K):
    """The weight gradient into an fp32 dB, written or added to (gradients summed over
    several batches), bf16 operands; rows no group owns are poisoned."""
    need_gpu()
    cnt = COUNTS[counts]
    E = len(cnt)
    M = int(sum(cnt)) + 7
    A = W.make_matrix(M, K, seed=N + K + 5, dtype=torch.bfloat16, device="cuda")
    dC = W.make_matrix(M, N, seed=N + K + 6, dtype=torch.bfloat16, device="cuda")
    A[int(sum(cnt)):] = 1e4
    off = ragged_offsets(cnt)
    want = om.grouped_gemm_wgrad(f64(A), f64(dC), off.cpu().numpy(), E)
    # bf16 products are exact in fp32: only the fp32 accumulation rounds
    _check_fp32_and_accumulate(lambda out, a: moe_gpu.moe_grouped_gemm_wgrad(A, dC, off, E, out=out, accumulate=a),
                               want, cnt, E, N, K, 2e-5)


def test_wgrad_accumulate_rejects_bf16_output():
    need_gpu()
    off = ragged_offsets([32, 32])
    A = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    dB = torch.zeros(2, 64, 64, dtype=torch.bfloat16, device="cuda")
    lib = moe_gpu.binding._lib
    a, b = moe_gpu.binding._operand(A), moe_gpu.binding._operand(A)
    import ctypes
    st = lib.load().moe_grouped_gemm_wgrad(ctypes.byref(a), ctypes.byref(b), ctypes.c_void_p(off.data_ptr()), 64, 64,
                                           64, 2, 1, ctypes.c_void_p(dB.data_ptr()), lib.MOE_BF16, None, None)
    assert st == lib.MOE_ERR_INVALID_ARG


# ----------------------------------------------------------------------------- MXFP8 forward

from oracle import mxfp8 as omx  # noqa: E402
from _parity import TOL_MXFP8  # noqa: E402


def _quantize(t):
    """Row-wise MXFP8 on the GPU; the oracle quantises the same values itself and
    the codes must agree bit for bit."""
    rows = t.reshape(-1, t.shape[-1])
    codes, scales = moe_gpu.moe_quantize_mxfp8_grouped(rows)
    c, s = omx.quantize_rowwise(f64(rows))
    assert (codes.cpu().numpy() == c).all() and (scales.cpu().numpy() == s).all()
    return codes.view(t.shape), scales.view(*t.shape[:-1], t.shape[-1] // 32), omx.dequantize_rowwise(c, s)


@pytest.mark.parametrize("counts", ["mixed", "singles", "one-expert"], ids=str)
@pytest.mark.parametrize("K,N", [(512, 256), (1024, 320), (2048, 64), (512, 192), (512, 448)])
def test_fwd_mxfp8_plain(counts, K, N):
    need_gpu()
    cnt = COUNTS[counts]
    E = len(cnt)
    M = int(sum(cnt)) + 2
    A, B = _mats(M, K, N, E, torch.bfloat16, seed=K + N + 7)
    Aq, As, A_deq = _quantize(A)
    Bq, Bs, B_deq = _quantize(B)
    off = ragged_offsets(cnt)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe_gpu.moe_grouped_gemm_fwd(Aq, Bq, off, A_scales=As, B_scales=Bs, out=C)
    want = om.grouped_gemm(A_deq, B_deq.reshape(E, N, K), off.cpu().numpy())
    got = f64(C)
    rows = int(sum(cnt))
    assert np.isnan(got[rows:]).all()
    err = rel_l2(got[:rows], want[:rows])
    assert err < TOL_MXFP8 and err < 1e-2, err       # same quantised inputs: only fp32/bf16 rounding


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_fwd_mxfp8_plain_many_tiles_per_cta(out_dtype):
    """Several tiles per persistent CTA (462 tiles of 128 x 256 for 152 SMs), so the
    accumulator, the scale slots and the staging boxes are reused many times; a
    partial last column tile; an empty and a one-row group."""
    need_gpu()
    cnt = [3000, 0, 1, 2900, 130, 2000]
    E, K, N = len(cnt), 512, 1568 + 96
    M = int(sum(cnt))
    A, B = _mats(M, K, N, E, torch.bfloat16, seed=77)
    Aq, As, A_deq = _quantize(A)
    Bq, Bs, B_deq = _quantize(B)
    off = ragged_offsets(cnt)
    C = torch.empty((M, N), dtype=out_dtype, device="cuda")
    moe_gpu.moe_grouped_gemm_fwd(Aq, Bq, off, A_scales=As, B_scales=Bs, out=C)
    want = om.grouped_gemm(A_deq, B_deq.reshape(E, N, K), off.cpu().numpy())
    err = rel_l2(f64(C), want)
    assert err < 1e-2, err
    for e in range(E):                                    # every group on its own
        lo, hi = int(off[e]), int(off[e + 1])
        if hi > lo:
            assert rel_l2(f64(C[lo:hi]), want[lo:hi]) < 1e-2, e


@pytest.mark.parametrize("counts", ["mixed", "singles"], ids=str)
@pytest.mark.parametrize("K,f", [(512, 128), (1024, 256), (512, 96), (512, 288)])
def test_fwd_mxfp8_swiglu(counts, K, f):
    need_gpu()
    cnt = COUNTS[counts]
    E = len(cnt)
    M = int(sum(cnt))
    A, B = _mats(M, K, 2 * f, E, torch.bfloat16, seed=K + f + 9)
    Aq, As, A_deq = _quantize(A)
    Bq, Bs, B_deq = _quantize(B)
    off = ragged_offsets(cnt)
    H = moe_gpu.moe_grouped_gemm_fwd(Aq, Bq, off, epi="swiglu", A_scales=As, B_scales=Bs)
    want = om.swiglu(om.grouped_gemm(A_deq, B_deq.reshape(E, 2 * f, K), off.cpu().numpy()))
    assert rel_l2(f64(H), want) < 1e-2


@pytest.mark.parametrize("f", [96, 160])
def test_fwd_mxfp8_swiglu_f32_out_and_preact(f):
    """fp32 H and the pre-activation G|U store, across a partial last column tile."""
    need_gpu()
    cnt = COUNTS["mixed"]
    E = len(cnt)
    M, K = int(sum(cnt)), 512
    A, B = _mats(M, K, 2 * f, E, torch.bfloat16, seed=f + 11)
    Aq, As, A_deq = _quantize(A)
    Bq, Bs, B_deq = _quantize(B)
    off = ragged_offsets(cnt)
    H, GU = moe_gpu.moe_grouped_gemm_fwd(Aq, Bq, off, epi="swiglu", A_scales=As, B_scales=Bs,
                                         out_dtype=torch.float32, want_preact=True)
    gu = om.grouped_gemm(A_deq, B_deq.reshape(E, 2 * f, K), off.cpu().numpy())
    # same quantised inputs, fp32 out: only the tensor core's accumulation rounding
    assert rel_l2(f64(GU), gu) < 1e-3
    assert rel_l2(f64(H), om.swiglu(gu)) < 1e-3


@pytest.mark.parametrize("counts", ["mixed", "singles", "one-expert"], ids=str)
@pytest.mark.parametrize("epi,K,N", [("swiglu", 512, 256), ("swiglu", 1024, 576), ("none", 512, 320),
                                     ("none", 512, 64)], ids=["swiglu-f128", "swiglu-f288", "none-N320", "none-N64"])
def test_fwd_mxfp8_out(counts, epi, K, N):
    """GEMM with the result quantised to MXFP8 in its epilogue: codes and scales
    equal, bit for bit, the bf16 result of the same GEMM passed through the row-wise
    quantiser (itself pinned bit-exactly against the oracle's quantiser); the
    decoded values match the oracle's result on the same quantised operands."""
    need_gpu()
    cnt = COUNTS[counts]
    E = len(cnt)
    M = int(sum(cnt)) + 2
    rows = int(sum(cnt))
    A, B = _mats(M, K, N, E, torch.bfloat16, seed=K + N + 13)
    Aq, As, A_deq = _quantize(A)
    Bq, Bs, B_deq = _quantize(B)
    off = ragged_offsets(cnt)
    n_out = N // 2 if epi == "swiglu" else N
    codes = torch.full((M, n_out), 0xAB, dtype=torch.uint8, device="cuda")
    scales = torch.full((M, n_out // 32), 0xCD, dtype=torch.uint8, device="cuda")
    moe_gpu.moe_grouped_gemm_fwd_mxfp8_out(Aq, Bq, off, epi=epi, A_scales=As, B_scales=Bs, codes=codes,
                                           scales=scales)
    C = moe_gpu.moe_grouped_gemm_fwd(Aq, Bq, off, epi=epi, A_scales=As, B_scales=Bs)
    cq, cs = moe_gpu.moe_quantize_mxfp8_grouped(C[:rows].contiguous())
    assert torch.equal(codes[:rows], cq) and torch.equal(scales[:rows], cs)
    assert (codes[rows:] == 0xAB).all() and (scales[rows:] == 0xCD).all()     # rows outside every group
    want = om.grouped_gemm(A_deq, B_deq.reshape(E, N, K), off.cpu().numpy())
    if epi == "swiglu":
        want = om.swiglu(want)
    got = omx.dequantize_rowwise(codes[:rows].cpu().numpy(), scales[:rows].cpu().numpy())
    assert rel_l2(got, want[:rows]) < TOL_MXFP8


def test_fwd_mxfp8_out_rejects_bf16_operands():
    need_gpu()
    A, B = _mats(64, 512, 64, 2, torch.bfloat16, seed=3)
    with pytest.raises(moe_gpu.binding.MoeError):
        moe_gpu.moe_grouped_gemm_fwd_mxfp8_out(A, B, ragged_offsets([32, 32]))


def test_fwd_mxfp8_requires_scales_and_k_multiple_of_512():
    need_gpu()
    A, B = _mats(64, 256, 64, 2, torch.bfloat16, seed=1)
    Aq, As, _ = _quantize(A)
    Bq, Bs, _ = _quantize(B)
    with pytest.raises(moe_gpu.binding.MoeError, match="512"):
        moe_gpu.moe_grouped_gemm_fwd(Aq, Bq, ragged_offsets([32, 32]), A_scales=As, B_scales=Bs)


# ----------------------------------------------------------------------------- MXFP8 data gradient

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("G,R,C", [(3, 64, 40), (2, 512, 264), (1, 32, 8), (4, 96, 1024)])
def test_quantize_transposed(dtype, G, R, C):
    """Codes and scales of B^T equal the oracle's row-wise quantiser on each B[g]^T,
    bit for bit (C spans several 256-column tiles and a partial one)."""
    need_gpu()
    x = W.make_matrix(G * R, C, seed=G + R + C, dtype=dtype, device="cuda", scale=3.0).view(G, R, C)
    codes, scales = moe_gpu.moe_quantize_mxfp8_transposed(x)
    assert codes.shape == (G, C, R) and scales.shape == (G * C, R // 32)
    xt = f64(x).transpose(0, 2, 1).reshape(G * C, R)
    c, s = omx.quantize_rowwise(xt)
    assert (codes.cpu().numpy().reshape(G * C, R) == c).all()
    assert (scales.cpu().numpy() == s).all()


def test_quantize_transposed_rejects_bad_shapes():
    need_gpu()
    x = torch.zeros(2, 48, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe_gpu.binding.MoeError):
        moe_gpu.moe_quantize_mxfp8_transposed(x)          # R % 32 != 0


def _dgrad_mx_operands(M, N, K, E, seed):
    """dC [M,N] and B [E,N,K] in bf16, their MXFP8 forms along N, and the values
    the quantised operands decode to."""
    dC = W.make_matrix(M, N, seed=seed, dtype=torch.bfloat16, device="cuda")
    B = W.make_matrix(E * N, K, seed=seed + 1, dtype=torch.bfloat16, device="cuda", scale=N ** -0.5).view(E, N, K)
    dCq, dCs, dC_deq = _quantize(dC)
    BTq, BTs = moe_gpu.moe_quantize_mxfp8_transposed(B)
    c, s = omx.quantize_rowwise(f64(B).transpose(0, 2, 1).reshape(E * K, N))
    assert (BTq.cpu().numpy().reshape(E * K, N) == c).all() and (BTs.cpu().numpy() == s).all()
    B_deq = omx.dequantize_rowwise(c, s).reshape(E, K, N).transpose(0, 2, 1)   # [E, N, K]
    return dCq, dCs, dC_deq, BTq, BTs, B_deq


@pytest.mark.parametrize("counts", ["mixed", "singles", "all-in-last"], ids=str)
@pytest.mark.parametrize("N,K", [(512, 256), (1024, 96), (512, 320)])
def test_dgrad_mxfp8_plain(counts, N, K):
    """dA = dC . B[e] on MXFP8 operands quantised along N; rows outside every group
    untouched."""
    need_gpu()
    cnt = COUNTS[counts]
    E = len(cnt)
    M = int(sum(cnt)) + 3
    rows = int(sum(cnt))
    dCq, dCs, dC_deq, BTq, BTs, B_deq = _dgrad_mx_operands(M, N, K, E, seed=N + K + 21)
    off = ragged_offsets(cnt)
    dA = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe_gpu.moe_grouped_gemm_dgrad_mxfp8(dCq, BTq, off, dC_scales=dCs, BT_scales=BTs, out=dA)
    want = om.grouped_gemm_dgrad(dC_deq, B_deq, off.cpu().numpy())
    got = f64(dA)
    assert np.isnan(got[rows:]).all()
    err = rel_l2(got[:rows], want[:rows])
    assert err < TOL_MXFP8 and err < 1e-2, err        # same quantised inputs: only fp32/bf16 rounding


@pytest.mark.parametrize("counts", ["mixed", "singles"], ids=str)
@pytest.mark.parametrize("d,f", [(512, 256), (1024, 96), (512, 288)])
def test_dgrad_mxfp8_dswiglu(counts, d, f):
    """GEMM2 data gradient on MXFP8 operands with the SwiGLU backward fused."""
    need_gpu()
    cnt = COUNTS[counts]
    E = len(cnt)
    M = int(sum(cnt))
    dCq, dCs, dC_deq, BTq, BTs, B_deq = _dgrad_mx_operands(M, d, f, E, seed=d + f + 23)
    GU = W.make_matrix(M, 2 * f, seed=d + f + 25, dtype=torch.bfloat16, device="cuda", scale=2.0)
    off = ragged_offsets(cnt)
    dGU = moe_gpu.moe_grouped_gemm_dgrad_mxfp8(dCq, BTq, off, dC_scales=dCs, BT_scales=BTs, epi="dswiglu",
                                               preact=GU)
    dH = om.grouped_gemm_dgrad(dC_deq, B_deq, off.cpu().numpy())
    want = om.dswiglu(dH, f64(GU))
    assert dGU.shape == (M, 2 * f)
    assert rel_l2(f64(dGU), want) < 1e-2


def test_dgrad_mxfp8_rejects_bad_args():
    need_gpu()
    dCq, dCs, _, BTq, BTs, _ = _dgrad_mx_operands(64, 512, 64, 2, seed=5)
    off = ragged_offsets([32, 32])
    with pytest.raises(moe_gpu.binding.MoeError, match="512"):     # N % 512
        moe_gpu.moe_grouped_gemm_dgrad_mxfp8(dCq[:, :256].contiguous(), BTq[:, :, :256].contiguous(), off,
                                             dC_scales=dCs[:, :8].contiguous(), BT_scales=BTs[:, :8].contiguous())
    with pytest.raises(moe_gpu.binding.MoeError):                  # bf16 operands
        dC = torch.zeros(64, 512, dtype=torch.bfloat16, device="cuda")
        B = torch.zeros(2, 64, 512, dtype=torch.bfloat16, device="cuda")
        moe_gpu.moe_grouped_gemm_dgrad_mxfp8(dC, B, off, dC_scales=None, BT_scales=None)


# ----------------------------------------------------------------------------- MXFP8 weight gradient

def _colwise_tiled(t, off, E):
    """Tiled column-wise MXFP8 of t on the GPU and the values the oracle's own
    column-wise quantisation of t decodes to (codes bit-exact with the oracle)."""
    codes, scales = moe_gpu.moe_quantize_mxfp8_grouped(t, off, E, axis=2)
    c, sc = omx.quantize_colwise_grouped(f64(t), off.cpu().numpy())
    rows = int(off[-1])                       # rows no group owns get no codes
    assert (codes[:rows].cpu().numpy() == c[:rows]).all()
    return codes, scales, omx.dequantize_colwise_grouped(c, sc, off.cpu().numpy())


@pytest.mark.parametrize("counts", ["mixed", "singles", "all-in-last", "one-expert"], ids=str)
@pytest.mark.parametrize("N,K", [(256, 512), (128, 384), (384, 128)])
def test_wgrad_mxfp8(counts, N, K):
    """dB[e] = dC[R_e]^T A[R_e] on column-wise group-aware MXFP8 operands (blocks of
    32 down the contraction, restarting at each group): the oracle's result on the
    same quantised values; empty groups exact zeros; rows no group owns never read."""
    need_gpu()
    cnt = COUNTS[counts]
    E = len(cnt)
    rows = int(sum(cnt))
    M = rows + 7
    A = W.make_matrix(M, K, seed=N + K + 31, dtype=torch.bfloat16, device="cuda")
    dC = W.make_matrix(M, N, seed=N + K + 33, dtype=torch.bfloat16, device="cuda")
    off = ragged_offsets(cnt)
    Aq, As, A_deq = _colwise_tiled(A, off, E)
    Cq, Cs, C_deq = _colwise_tiled(dC, off, E)
    Aq[rows:] = 0x7E                          # poison the rows no group owns (448)
    dB = torch.full((E, N, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe_gpu.moe_grouped_gemm_wgrad(Aq, Cq, off, E, A_scales=As, dC_scales=Cs, out=dB)
    want = om.grouped_gemm_wgrad(A_deq, C_deq, off.cpu().numpy(), E)
    got = f64(dB)
    for e in range(E):
        if cnt[e] == 0:
            assert (got[e] == 0).all() and not np.signbit(got[e]).any(), f"expert {e} not exactly zero"
    assert not np.isnan(got).any()
    err = rel_l2(got, want)
    assert err < TOL_MXFP8 and err < 1e-2, err       # same quantised inputs: only fp32/bf16 rounding


@pytest.mark.parametrize("counts", ["mixed", "singles"], ids=str)
def test_wgrad_mxfp8_fp32_and_accumulate(counts):
    """The MXFP8 weight gradient into an fp32 dB, written or added to."""
    need_gpu()
    N, K = 256, 384
    cnt = COUNTS[counts]
    E = len(cnt)
    rows = int(sum(cnt))
    A = W.make_matrix(rows + 7, K, seed=N + K + 41, dtype=torch.bfloat16, device="cuda")
    dC = W.make_matrix(rows + 7, N, seed=N + K + 43, dtype=torch.bfloat16, device="cuda")
    off = ragged_offsets(cnt)
    Aq, As, A_deq = _colwise_tiled(A, off, E)
    Cq, Cs, C_deq = _colwise_tiled(dC, off, E)
    Aq[rows:] = 0x7E
    want = om.grouped_gemm_wgrad(A_deq, C_deq, off.cpu().numpy(), E)
    _check_fp32_and_accumulate(lambda out, a: moe_gpu.moe_grouped_gemm_wgrad(Aq, Cq, off, E, A_scales=As,
                                                                             dC_scales=Cs, out=out, accumulate=a),
                               want, cnt, E, N, K, 1e-4)


def test_wgrad_mxfp8_rejects_bad_shapes_and_missing_scales():
    need_gpu()
    off = ragged_offsets([32, 32])
    A = torch.zeros(64, 96, dtype=torch.uint8, device="cuda")
    dC = torch.zeros(64, 128, dtype=torch.uint8, device="cuda")
    s = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe_gpu.binding.MoeError, match="128"):                 # K % 128
        moe_gpu.moe_grouped_gemm_wgrad(A, dC, off, 2, A_scales=s, dC_scales=s)
    A = torch.zeros(64, 128, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe_gpu.binding.MoeError):                             # no scales
        moe_gpu.moe_grouped_gemm_wgrad(A, dC, off, 2)

"""The oracle's pins must catch plausible mistakes: plant each one in the
oracle (on the CPU, via monkeypatch) and check that a pin test fails."""

import numpy as np
import pytest

from oracle import moe, mxfp8
import test_oracle_ffn_backward as ffn_pins
import test_oracle_mxfp8 as mx_pins
import test_oracle_route_permute as route_pins


def _swapped_swiglu(GU):
    f = GU.shape[1] // 2
    return moe.silu(GU[:, f:]) * GU[:, :f]


def _dswiglu_missing_term(dH, GU):
    f = GU.shape[1] // 2
    G, U = GU[:, :f], GU[:, f:]
    s = 1.0 / (1.0 + np.exp(-G))
    return np.concatenate([dH * U * s, dH * G * s], axis=1)


_real_route = moe.route_topk


def _route_ties_to_higher_id(logits, k, renormalize=True):
    T, E = logits.shape
    flipped = logits[:, ::-1].copy()
    idx, w, counts = _real_route(flipped, k, renormalize)
    return (E - 1 - idx).astype(np.int32), w, counts[::-1].copy()


def _permute_unstable(idx, E):
    offsets, dest, src = moe_permute_real(idx, E)
    T, k = idx.shape
    src2 = src.copy()
    for e in range(E):
        src2[offsets[e]:offsets[e + 1]] = src[offsets[e]:offsets[e + 1]][::-1]
    dest2 = np.empty(T * k, dtype=np.int64)
    dest2[src2] = np.arange(T * k)
    return offsets, dest2.reshape(T, k), src2


moe_permute_real = moe.permute_maps


def _encode_ties_away(y):
    y = np.asarray(y, dtype=np.float64)
    mag = np.abs(y)
    hi = np.minimum(np.searchsorted(mxfp8.E4M3_POS, mag, side="left"), 0x7E)
    lo = np.maximum(hi - 1, 0)
    pick_hi = (mxfp8.E4M3_POS[hi] - mag) <= (mag - mxfp8.E4M3_POS[lo])
    code = np.where(pick_hi, hi, lo)
    code = np.where(mag >= 448, 0x7E, code)
    return (code | np.where(np.signbit(y), 0x80, 0)).astype(np.uint8)


def _wgrad_transposed(A, dC, offsets, E):
    """dB[e] = A_e^T dC_e instead of dC_e^T A_e (operands swapped)."""
    out = np.zeros((E, A.shape[1], dC.shape[1]))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        out[e] = A[lo:hi].T @ dC[lo:hi]
    return out


@pytest.mark.parametrize("target,attr,fake,check", [
    (moe, "swiglu", _swapped_swiglu,
     lambda: ffn_pins.test_layer_equals_dense_masked_moe(40, 16, 6, 2, 12, (3,))),
    (moe, "dswiglu", _dswiglu_missing_term,
     lambda: ffn_pins.test_backward_matches_torch_autograd(True)),
    (moe, "route_topk", _route_ties_to_higher_id,
     lambda: route_pins.test_route_bruteforce(64, 8, 2, True)),
    (moe, "permute_maps", _permute_unstable,
     lambda: route_pins.test_permutation_against_counting_loop(50, 8, 2)),
    (mxfp8, "e4m3_encode", _encode_ties_away,
     lambda: mx_pins.test_e4m3_matches_torch_cast_in_range()),
    (moe, "grouped_gemm_wgrad", _wgrad_transposed,
     lambda: ffn_pins.test_equal_counts_is_bmm()),
], ids=["swiglu-swapped", "dswiglu-term", "tie-break", "unstable-permute", "ties-away",
        "wgrad-rows"])
def test_pins_catch_planted_mistake(monkeypatch, target, attr, fake, check):
    monkeypatch.setattr(target, attr, fake)
    with pytest.raises(AssertionError):
        check()


def test_pins_catch_scale_exponent_off_by_one(monkeypatch):
    real = mxfp8.shared_exponent
    monkeypatch.setattr(mxfp8, "shared_exponent", lambda a: real(a) + 1)
    with pytest.raises(AssertionError):
        mx_pins.test_shared_exponent_closed_form(1.0, 119)
    with pytest.raises(AssertionError):
        mx_pins.test_quantize_rowwise_properties()


def _dequant_colwise_next_scale(codes, scales, offsets):
    """Each block decoded with the scale row of the block after it."""
    rolled = np.concatenate([scales[1:], scales[:1]], axis=0)
    return _real_dequant_colwise(codes, rolled, offsets)


_real_dequant_colwise = mxfp8.dequantize_colwise_grouped


@pytest.mark.parametrize("target,attr,fake,check", [
    (moe, "mx_roundtrip_colwise", lambda a, offsets: moe.mx_roundtrip(a),
     lambda: ffn_pins.test_mxfp8_backward_elements_from_blockwise_quantisation()),
    (moe, "mx_roundtrip_dim1", lambda W: moe.mx_roundtrip(W),
     lambda: ffn_pins.test_mxfp8_backward_elements_from_blockwise_quantisation()),
    (mxfp8, "dequantize_colwise_grouped", _dequant_colwise_next_scale,
     lambda: mx_pins.test_colwise_dequantize_matches_transposed_rowwise()),
], ids=["wgrad-operands-row-wise", "dgrad-weights-wrong-dim", "colwise-scale-row"])
def test_mxfp8_backward_pins_catch_planted_mistake(monkeypatch, target, attr, fake, check):
    monkeypatch.setattr(target, attr, fake)
    with pytest.raises(AssertionError):
        check()


from oracle import nvfp4  # noqa: E402
import test_oracle_nvfp4 as fp4_pins  # noqa: E402

_real_e2m1 = nvfp4.e2m1_encode


def _e2m1_ties_away(y):
    y = np.asarray(y, dtype=np.float64)
    mag = np.abs(y)
    code = np.argmin(np.abs(mag[..., None] - nvfp4.E2M1_POS[::-1]), axis=-1)
    code = (7 - code).astype(np.uint8)                        # on a tie the larger magnitude wins
    code = np.where(mag >= 6, 7, code)
    return (code | np.where(np.signbit(y), 0x8, 0)).astype(np.uint8)


def _quantize_swapped_nibbles(a, g=None):
    c, s, gg = _real_quantize(a, g)
    return ((c >> 4) | (c << 4)).astype(np.uint8), s, gg


_real_quantize = nvfp4.quantize


@pytest.mark.parametrize("attr,fake,check", [
    ("e2m1_encode", _e2m1_ties_away, lambda: fp4_pins.test_e2m1_midpoints_round_to_even_and_saturate()),
    ("quantize", _quantize_swapped_nibbles, lambda: fp4_pins.test_golden_blocks()),
    ("TENSOR_NUM", np.float32(448.0), lambda: fp4_pins.test_golden_blocks()),
], ids=["e2m1-ties-away", "nibbles-swapped", "tensor-scale-448"])
def test_nvfp4_pins_catch_planted_mistake(monkeypatch, attr, fake, check):
    monkeypatch.setattr(nvfp4, attr, fake)
    with pytest.raises(AssertionError):
        check()


_real_capacity = moe.permute_capacity


def _capacity_keeps_last(idx, E, C):
    """Keeps each expert's last C tokens instead of its first C."""
    T, k = np.asarray(idx).shape
    rev = np.asarray(idx)[::-1]
    off, dest, src = _real_capacity(rev, E, C)
    dest = dest[::-1].copy()
    src = np.where(src >= 0, (T - 1 - src // k) * k + src % k, -1)
    return off, dest, src


@pytest.mark.parametrize("attr,fake,check", [
    # features paired in reverse order (x[t, d-1-i] with W_r[e, i])
    ("router_logits", lambda x, w: np.asarray(x, dtype=np.float64)[:, ::-1] @ np.asarray(w, dtype=np.float64).T,
     lambda: route_pins.test_router_logits_bruteforce_and_one_hot()),
    ("permute_capacity", _capacity_keeps_last,
     lambda: route_pins.test_capacity_keeps_first_tokens_and_drops_the_rest()),
], ids=["router-reversed-features", "capacity-keeps-last"])
def test_router_and_capacity_pins_catch_planted_mistake(monkeypatch, attr, fake, check):
    monkeypatch.setattr(moe, attr, fake)
    with pytest.raises(AssertionError):
        check()


_real_layer_forward = moe.layer_forward


def _layer_forward_variant(h_quantised=True, w1_scale_per_expert=False):
    """The oracle's block-scaled forward with one step changed: H fed to GEMM2
    unquantised, or W1 given one NVFP4 tensor scale per expert instead of one for
    the stack."""
    def fwd(x, logits, W1, W2, k, renormalize=True, mxfp8_operands=False, nvfp4_operands=False):
        out = _real_layer_forward(x, logits, W1, W2, k, renormalize)
        rt = moe.nvfp4_roundtrip if nvfp4_operands else moe.mx_roundtrip
        off = out["offsets"]
        if w1_scale_per_expert:
            W1q = np.stack([rt(W1[e]) for e in range(W1.shape[0])])
        else:
            W1q = rt(W1)
        GU = moe.grouped_gemm(rt(out["Xp"]), W1q, off)
        H = moe.swiglu(GU)
        Yp = moe.grouped_gemm(rt(H) if h_quantised else H, rt(W2), off)
        out.update(GU=GU, H=H, Yp=Yp, y=moe.combine(Yp, out["dest_row"], out["w"]))
        return out
    return fwd


@pytest.mark.parametrize("fake,fmt", [
    (_layer_forward_variant(h_quantised=False), "nvfp4"),
    (_layer_forward_variant(w1_scale_per_expert=True), "nvfp4"),
    (_layer_forward_variant(h_quantised=False), "mxfp8"),
], ids=["nvfp4-h-unquantised", "nvfp4-w1-scale-per-expert", "mxfp8-h-unquantised"])
def test_blockscaled_forward_pins_catch_planted_mistake(monkeypatch, fake, fmt):
    monkeypatch.setattr(moe, "layer_forward", fake)
    with pytest.raises(AssertionError):
        ffn_pins.test_blockscaled_forward_elements_from_blockwise_quantisation(fmt)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_blockscaled_forward_variant_without_mistake_passes(monkeypatch, fmt):
    """The rebuilt forward with no step changed passes the same pin, so the
    failures above come from the planted step alone."""
    monkeypatch.setattr(moe, "layer_forward", _layer_forward_variant())
    ffn_pins.test_blockscaled_forward_elements_from_blockwise_quantisation(fmt)

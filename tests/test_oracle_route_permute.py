"""Pins for the oracle's routing and dispatch (CPU only).

Each check comes from somewhere other than the oracle itself: hand-worked
golden rows, brute-force sorting with Python's ``sorted``, a sequential
counting construction of the permutation, scipy's softmax, and identities that
hold exactly in floating point.
"""

import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import moe

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows():
    rows = []
    for line in open(os.path.join(GOLDEN, "route_tiny.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, lg, ids, ws = [p.strip() for p in line.split("|")]
        rows.append((int(k), np.array(lg.split(), dtype=np.float32),
                     [int(v) for v in ids.split()], [float(v) for v in ws.split()]))
    return rows


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: f"k{r[0]}")
def test_route_golden(row):
    k, lg, ids, ws = row
    idx, w, counts = moe.route_topk(lg[None, :], k)
    assert idx[0].tolist() == ids
    np.testing.assert_allclose(w[0], ws, atol=1e-7, rtol=0)
    assert counts.sum() == k


def _rand_logits(rng, T, E, ties):
    if ties:   # small integer logits force many exact ties
        return rng.integers(-3, 4, size=(T, E)).astype(np.float32)
    return rng.standard_normal((T, E)).astype(np.float32)


@pytest.mark.parametrize("T,E,k,ties", [(64, 8, 2, True), (64, 8, 2, False), (40, 16, 5, True),
                                        (33, 32, 8, True), (17, 6, 6, False), (50, 5, 1, True)])
def test_route_bruteforce(T, E, k, ties):
    rng = np.random.default_rng(T * 131 + E)
    lg = _rand_logits(rng, T, E, ties)
    idx, w, counts = moe.route_topk(lg, k)
    for t in range(T):
        want = sorted(range(E), key=lambda e: (-float(lg[t, e]), e))[:k]
        assert idx[t].tolist() == want
        sel = np.array([float(lg[t, e]) for e in want])
        np.testing.assert_allclose(w[t], scipy.special.softmax(sel), rtol=1e-13)
    assert counts.tolist() == np.bincount(idx.ravel(), minlength=E).tolist()
    assert counts.sum() == T * k
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-14)
    assert (np.diff(np.take_along_axis(lg, idx.astype(np.int64), 1), axis=1) <= 0).all()


def test_route_k1_weight_exactly_one():
    lg = np.random.default_rng(1).standard_normal((100, 12)).astype(np.float32)
    _, w, _ = moe.route_topk(lg, 1)
    assert (w == 1.0).all()


def test_route_k_equals_E_is_full_softmax():
    lg = np.random.default_rng(2).standard_normal((30, 7)).astype(np.float32)
    idx, w, _ = moe.route_topk(lg, 7)
    full = scipy.special.softmax(lg.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(full, idx.astype(np.int64), 1), rtol=1e-13)


def test_route_not_renormalized_is_full_softmax_probability():
    lg = np.random.default_rng(3).standard_normal((30, 16)).astype(np.float32)
    idx, w, _ = moe.route_topk(lg, 4, renormalize=False)
    full = scipy.special.softmax(lg.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(full, idx.astype(np.int64), 1), rtol=1e-13)
    assert (w.sum(axis=1) < 1.0).all()


def test_route_masked_experts():
    lg = np.array([[-np.inf, 0.0, -np.inf, 1.0]], dtype=np.float32)
    idx, w, _ = moe.route_topk(lg, 3)
    assert idx[0].tolist() == [3, 1, 0]        # -inf ties go to the lower id
    assert w[0, 2] == 0.0


@pytest.mark.parametrize("renormalize", [True, False])
def test_route_fully_masked_token_has_zero_weights(renormalize):
    """A token whose experts are all masked has no softmax mass: its slots hold the
    lowest expert ids (every logit ties) with weight exactly 0, and its router
    gradient is 0; the other tokens are unaffected (same as routed alone)."""
    lg = np.array([[-np.inf] * 5, [0.5, -np.inf, 2.0, 1.0, -1.0]], dtype=np.float32)
    idx, w, counts = moe.route_topk(lg, 3, renormalize)
    assert idx[0].tolist() == [0, 1, 2]
    assert (w[0] == 0.0).all() and not np.isnan(w).any()
    idx1, w1, _ = moe.route_topk(lg[1:], 3, renormalize)
    assert (idx[1] == idx1[0]).all() and (w[1] == w1[0]).all()
    assert counts.tolist() == [2, 1, 2, 1, 0]
    dl = moe.route_bwd(np.ones((2, 3)), w, idx, lg, renormalize)
    assert (dl[0] == 0.0).all() and not np.isnan(dl).any()
    dl1 = moe.route_bwd(np.ones((1, 3)), w1, idx1, lg[1:], renormalize)
    np.testing.assert_array_equal(dl[1], dl1[0])


def _counting_permutation(idx, E):
    """Sequential construction: visit tokens in order and hand each (token, slot)
    the next free row of its expert's group."""
    T, k = idx.shape
    counts = [0] * E
    for t in range(T):
        for j in range(k):
            counts[int(idx[t, j])] += 1
    start = [0] * (E + 1)
    for e in range(E):
        start[e + 1] = start[e] + counts[e]
    nxt = list(start[:E])
    dest = np.zeros((T, k), dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            dest[t, j] = nxt[e]
            nxt[e] += 1
    return np.array(start), dest


@pytest.mark.parametrize("T,E,k", [(50, 8, 2), (64, 16, 8), (31, 5, 1), (20, 3, 3), (1, 4, 2)])
def test_permutation_against_counting_loop(T, E, k):
    rng = np.random.default_rng(T + 7 * E)
    lg = _rand_logits(rng, T, E, ties=False)
    lg[:, 0] -= 10.0                      # expert 0 left empty
    idx, _, counts = moe.route_topk(lg, k)
    offsets, dest, src = moe.permute_maps(idx, E)
    want_off, want_dest = _counting_permutation(idx, E)
    assert offsets.tolist() == want_off.tolist()
    assert (dest == want_dest).all()
    # inverse maps, stability and group membership
    assert (dest.ravel()[src] == np.arange(T * k)).all()
    assert offsets[-1] == T * k and (np.diff(offsets) == counts).all()
    for e in range(E):
        toks = src[offsets[e]:offsets[e + 1]] // k
        assert (np.diff(toks) > 0).all()
        assert (idx.ravel()[src[offsets[e]:offsets[e + 1]]] == e).all()


def test_empty_and_single_expert_groups():
    idx = np.array([[2, 0], [2, 1], [0, 2]], dtype=np.int32)
    offsets, dest, src = moe.permute_maps(idx, 4)
    assert offsets.tolist() == [0, 2, 3, 6, 6]
    assert src.tolist() == [1, 4, 3, 0, 2, 5]
    assert dest.tolist() == [[3, 0], [4, 2], [1, 5]]


@pytest.mark.parametrize("k", [1, 2, 8])
def test_combine_of_permute_is_identity(k):
    """Unit weights with k=1, or uniform weights 1/k for k a power of two, make
    combine(permute(x)) reproduce x exactly when x carries few significant bits
    (bf16 values: the partial sums j*x/k then need at most 8+3 bits)."""
    T, E, d = 40, 16, 24
    rng = np.random.default_rng(k)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    x = torch.from_numpy(rng.standard_normal((T, d))).to(torch.bfloat16).double().numpy()
    idx, _, _ = moe.route_topk(lg, k)
    offsets, dest, src = moe.permute_maps(idx, E)
    xp = moe.permute(x, src, k)
    w = np.full((T, k), 1.0 / k)
    assert (moe.combine(xp, dest, w) == x).all()
    if k == 1:
        assert (moe.combine(xp, dest, None) == x).all()


def test_router_logits_bruteforce_and_one_hot():
    """logits[t, e] = sum_i x[t, i] W_r[e, i]: a triple loop on a tiny case, and a
    one-hot token reads out one column of W_r (a transposed W_r would read a row)."""
    rng = np.random.default_rng(31)
    x = rng.standard_normal((5, 7))
    Wr = rng.standard_normal((3, 7))
    got = moe.router_logits(x, Wr)
    for t in range(5):
        for e in range(3):
            assert abs(got[t, e] - sum(x[t, i] * Wr[e, i] for i in range(7))) < 1e-12
    onehot = np.zeros((1, 7))
    onehot[0, 4] = 1.0
    assert np.array_equal(moe.router_logits(onehot, Wr)[0], Wr[:, 4])


def test_capacity_keeps_first_tokens_and_drops_the_rest():
    """Each expert keeps exactly min(count, C) pairs, those of its C lowest token
    ids (checked against a sort of the routed tokens), at rows e*C.. in token
    order; the other pairs are dropped; every row is used at most once."""
    rng = np.random.default_rng(41)
    T, E, k, C = 60, 6, 2, 7
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[:, 1] += 3.0                                          # an overloaded expert
    idx, _, counts = moe.route_topk(lg, k)
    offsets, dest, src = moe.permute_capacity(idx, E, C)
    assert np.array_equal(offsets, np.arange(E + 1) * C)
    for e in range(E):
        toks = sorted(t for t in range(T) for j in range(k) if idx[t, j] == e)
        keep = toks[:C]
        rows = [dest[t, j] for t in range(T) for j in range(k) if idx[t, j] == e and dest[t, j] >= 0]
        assert len(rows) == min(counts[e], C)
        assert sorted(rows) == list(range(e * C, e * C + len(keep)))
        assert [src[r] // k for r in range(e * C, e * C + len(keep))] == keep
        assert (src[e * C + len(keep):(e + 1) * C] == -1).all()
    assert counts[1] > C and (dest == -1).sum() == sum(max(int(c) - C, 0) for c in counts)


def test_capacity_large_enough_is_dropless_and_zero_drops_everything():
    """C >= the largest count: nothing is dropped and combine(permute(x)) = x for
    k=1; C = 0: every pair is dropped and the combine is zero."""
    rng = np.random.default_rng(42)
    T, E = 50, 5
    lg = rng.standard_normal((T, E)).astype(np.float32)
    idx, w, counts = moe.route_topk(lg, 1)
    x = rng.standard_normal((T, 8))
    C = int(counts.max())
    _, dest, src = moe.permute_capacity(idx, E, C)
    assert (dest >= 0).all()
    np.testing.assert_array_equal(moe.combine_capacity(moe.permute_rows_capacity(x, src, 1), dest, w), x)
    _, dest0, src0 = moe.permute_capacity(idx, E, 0)
    assert (dest0 == -1).all() and len(src0) == 0
    assert (moe.combine_capacity(np.zeros((0, 8)), dest0, w) == 0).all()

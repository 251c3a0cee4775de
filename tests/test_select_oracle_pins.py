"""Pins for the fp64 route-producer oracle (qsa page, select_qsa_token_ids).

Each test ties the oracle to something other than itself: a hand-derived
fixture (tests/golden/route_producer_small.json), a closed form of the block
score, brute-force best subsets, the dense-causal special case, the row
structure the page fixes (complete blocks, the causal tail, -1 fill, padding
rows), the visibility boundary and shard consistency of
query_position_offset.  A dropped relu or scale, a sign or off-by-one in the
visible-block count, a reversed tie order or a misplaced tail fails one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    with open(os.path.join(GOLDEN, "route_producer_small.json")) as f:
        return json.load(f)


def test_golden_hand_derived_example():
    g = _golden()
    q = np.array(g["index_queries"], float)
    k = np.array(g["compressed_keys"], float)
    sc = oracle.index_scores(q, k, g["compress_ratio"])
    for t, want in g["scores_b0"].items():
        np.testing.assert_array_equal(sc[0, int(t)], want)
    ids = oracle.select_qsa_token_ids(q, k, g["sequence_lengths"], g["token_budget"], g["compress_ratio"])
    np.testing.assert_array_equal(ids, np.array(g["ids"]))


def test_score_closed_form():
    """q[t,h] = a_h * u and k[blk] = b_blk * u + w_blk with w_blk orthogonal to
    u: dot = a_h b_blk |u|^2, so score = sum_h relu(a_h b_blk) |u|^2 / sqrt(D)."""
    rng = np.random.default_rng(1)
    D, H, c, NB = 16, 5, 4, 6
    u = np.zeros(D)
    u[:3] = rng.standard_normal(3)
    a = np.array([1.5, -2.0, 0.25, -0.5, 3.0])
    b = rng.standard_normal(NB) * 2
    w = np.zeros((NB, D))
    w[:, 3:] = rng.standard_normal((NB, D - 3))
    S = NB * c
    q = np.broadcast_to((a[:, None] * u[None, :])[None, None], (1, S, H, D)).copy()
    k = (b[:, None] * u[None, :] + w)[None]
    sc = oracle.index_scores(q, k, c)
    uu = float(u @ u)
    for t in range(S):
        nvis = (t + 1) // c
        for blk in range(NB):
            if blk < nvis:
                want = sum(max(0.0, ah * b[blk] * uu) for ah in a) / math.sqrt(D)
                assert sc[0, t, blk] == pytest.approx(want, rel=1e-12, abs=1e-12)
            else:
                assert sc[0, t, blk] == -np.inf


def test_brute_force_best_subset():
    """With distinct scores the chosen blocks are the subset of size
    floor(budget / c) with the largest score sum, found by enumeration."""
    rng = np.random.default_rng(2)
    c, budget = 3, 9  # three blocks per row
    B, S_q, NB = 2, 27, 9
    sc = rng.standard_normal((B, S_q, NB))
    lens = np.array([S_q, S_q])
    ids = oracle.select_ids(sc, lens, budget, c)
    n_best = budget // c
    for b in range(B):
        for t in range(S_q):
            nvis = (t + 1) // c
            row = ids[b, t]
            got = sorted({int(x) // c for x in row[row >= 0] if x < nvis * c})
            if nvis <= n_best:
                assert got == list(range(nvis))
                continue
            best = max(itertools.combinations(range(nvis), n_best), key=lambda s: sum(sc[b, t, j] for j in s))
            assert got == sorted(best)


def test_ties_go_to_the_lower_block():
    c, budget, NB = 2, 6, 10
    S_q = NB * c
    sc = np.zeros((1, S_q, NB))
    sc[0, :, 7] = 1.0  # one clear winner, the rest tied at 0
    ids = oracle.select_ids(sc, [S_q], budget, c)
    row = ids[0, S_q - 1]  # ten complete blocks, no tail; three best
    assert list(row) == [0, 1, 2, 3, 14, 15, -1]
    sc[0, :, 0] = -1.0  # a lower score loses to later zeros
    row = oracle.select_ids(sc, [S_q], budget, c)[0, S_q - 1]
    assert list(row) == [2, 3, 4, 5, 14, 15, -1]


def test_visibility_boundary():
    """Block m-1 becomes visible exactly at position c*m - 1, never earlier."""
    c, budget, D, H = 4, 4, 8, 2  # one best block per row
    NB = 6
    S = NB * c
    k = np.zeros((1, NB, D))
    k[0, :, 1] = 1.0
    k[0, :, 0] = np.arange(NB)  # later blocks score higher for q ~ e_0
    q = np.zeros((1, S, H, D))
    q[..., 0] = 1.0
    ids = oracle.select_qsa_token_ids(q, k, [S], budget, c)
    for t in range(S):
        nvis = (t + 1) // c
        row = ids[0, t]
        blocks = sorted({int(x) // c for x in row[row >= 0] if x < nvis * c})
        assert blocks == ([nvis - 1] if nvis >= 1 else [])
        if t == c * 3 - 2:
            assert 2 not in blocks
        if t == c * 3 - 1:
            assert blocks == [2]


@pytest.mark.parametrize("c,budget", [(4, 16), (4, 18), (3, 6), (1, 5)])
def test_row_structure(c, budget):
    rng = np.random.default_rng(3 + c + budget)
    B, S_q, H, D = 2, 61, 3, 8
    NB = S_q // c
    q = rng.standard_normal((B, S_q, H, D))
    k = rng.standard_normal((B, NB, D))
    lens = np.array([S_q, 45])
    ids = oracle.select_qsa_token_ids(q, k, lens, budget, c)
    W = budget + c - 1
    assert ids.shape == (B, S_q, W)
    n_best = budget // c
    for b in range(B):
        for t in range(S_q):
            row = ids[b, t]
            if t >= lens[b]:
                assert (row == -1).all()
                continue
            nvis = (t + 1) // c
            valid = row[row >= 0]
            n = valid.size
            assert (row[n:] == -1).all()
            assert (np.diff(valid) > 0).all()
            assert valid.max() <= t
            want_n = min(n_best, nvis) * c + (t + 1 - nvis * c)
            assert n == want_n
            # the causal tail: every token of the incomplete block
            np.testing.assert_array_equal(valid[valid >= nvis * c], np.arange(nvis * c, t + 1))
            # whole blocks only
            blocks, counts = np.unique(valid[valid < nvis * c] // c, return_counts=True)
            assert (counts == c).all()
            if nvis <= n_best:  # dense causal row
                np.testing.assert_array_equal(valid, np.arange(t + 1))


def test_query_position_offset_matches_the_full_sequence():
    """A shard of local rows at offset o gets the rows of positions o.. of the
    unsharded call against the same global keys."""
    rng = np.random.default_rng(4)
    c, budget, H, D = 4, 12, 2, 8
    S = 64
    NB = S // c
    q = rng.standard_normal((1, S, H, D))
    k = rng.standard_normal((1, NB, D))
    full = oracle.select_qsa_token_ids(q, k, [S], budget, c)
    for o in (16, 32, 48):
        part = oracle.select_qsa_token_ids(q[:, o:o + 16], k, [S], budget, c, offset=o)
        np.testing.assert_array_equal(part, full[:, o:o + 16])
    # a logical length inside the shard pads the rows past it
    part = oracle.select_qsa_token_ids(q[:, 32:48], k, [40], budget, c, offset=32)
    np.testing.assert_array_equal(part[:, :8], full[:, 32:40])
    assert (part[:, 8:] == -1).all()


def test_bad_shapes_rejected():
    q = np.zeros((1, 9, 1, 4))
    k = np.zeros((1, 2, 4))  # 2 blocks of 4 cover positions < 11
    oracle.index_scores(q, k, 4)
    with pytest.raises(RuntimeError):
        oracle.index_scores(np.zeros((1, 12, 1, 4)), k, 4)
    with pytest.raises(RuntimeError):
        oracle.index_scores(q, k, 4, offset=4)

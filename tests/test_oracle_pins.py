"""Pins for the fp64 CPU oracle, against facts fixed by the pages and by mathematics.

Each test ties the oracle to something other than itself: torch's dense
scaled_dot_product_attention with a boolean mask, its causal mode, hand-derived
closed forms (tests/golden), invariance under duplicates and permutation,
brute-force route sets, central finite differences and exact identities of the
gradients.  A dropped term, a wrong sign or head index, or a transposed operand
anywhere in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _random_problem(rng, B, S_q, S_kv, Hq, Hkv, D, K, p_empty=0.0, dtype=np.int64):
    q = rng.standard_normal((B, S_q, Hq, D))
    k = rng.standard_normal((B, S_kv, Hkv, D))
    v = rng.standard_normal((B, S_kv, Hkv, D))
    routes = rng.integers(-3, S_kv + 3, size=(B, S_q, K)).astype(dtype)
    empty = rng.random((B, S_q)) < p_empty
    routes[empty] = -1
    return q, k, v, routes


def _membership(routes, S_kv):
    """Dense boolean membership [B, S_q, S_kv] by brute force (python sets)."""
    B, S_q, K = routes.shape
    m = np.zeros((B, S_q, S_kv), bool)
    for b in range(B):
        for i in range(S_q):
            for x in set(int(t) for t in routes[b, i]):
                if 0 <= x < S_kv:
                    m[b, i, x] = True
    return m


def _dense_reference(q, k, v, routes, scale):
    """torch fp64 dense attention with a boolean mask; K/V heads expanded so that
    query head h reads KV head h // G."""
    B, S_q, Hq, D = q.shape
    S_kv, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    mask = torch.from_numpy(_membership(routes, S_kv))[:, None]  # [B,1,S_q,S_kv]
    qt = torch.from_numpy(q).permute(0, 2, 1, 3)
    kt = torch.from_numpy(k).repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
    vt = torch.from_numpy(v).repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
    o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    scores = torch.matmul(qt, kt.transpose(-1, -2)) * scale
    lse = torch.logsumexp(scores.masked_fill(~mask, float("-inf")), dim=-1)  # [B,Hq,S_q]
    return o.permute(0, 2, 1, 3).numpy(), lse.numpy(), mask[:, 0].numpy()


@pytest.mark.parametrize("B,S_q,S_kv,Hq,Hkv,D,K", [
    (1, 16, 16, 4, 2, 4, 8),
    (2, 24, 40, 4, 1, 8, 12),
    (1, 8, 64, 8, 8, 256, 20),
    (1, 12, 20, 6, 3, 16, 5),
])
def test_forward_equals_dense_masked_attention(B, S_q, S_kv, Hq, Hkv, D, K):
    rng = np.random.default_rng(B * 1000 + S_kv + D)
    q, k, v, routes = _random_problem(rng, B, S_q, S_kv, Hq, Hkv, D, K)
    scale = 0.37
    o, lse = oracle.forward(q, k, v, routes, scale)
    o_ref, lse_ref, mask = _dense_reference(q, k, v, routes, scale)
    rows = mask.any(-1)  # SDPA yields NaN on rows with no key; those are checked elsewhere
    assert rows.sum() > 0
    np.testing.assert_allclose(o[rows], o_ref[rows], rtol=1e-12, atol=1e-12)
    lse_t = np.transpose(lse, (0, 2, 1))
    lse_ref_t = np.transpose(lse_ref, (0, 2, 1))
    np.testing.assert_allclose(lse_t[rows], lse_ref_t[rows], rtol=1e-12, atol=1e-12)


def test_all_prior_tokens_equals_causal_attention():
    rng = np.random.default_rng(7)
    S, Hq, Hkv, D = 24, 4, 2, 8
    q = rng.standard_normal((1, S, Hq, D))
    k = rng.standard_normal((1, S, Hkv, D))
    v = rng.standard_normal((1, S, Hkv, D))
    K = S + 6
    routes = np.full((1, S, K), -1, np.int64)
    for i in range(S):
        ids = list(range(i + 1)) + [i, 0, S + 5]  # prior tokens, plus a duplicate pair and an invalid ID
        rng.shuffle(ids)
        routes[0, i, :len(ids)] = ids
    scale = 1.0 / math.sqrt(D)
    o, _ = oracle.forward(q, k, v, routes, scale)
    qt = torch.from_numpy(q).permute(0, 2, 1, 3)
    kt = torch.from_numpy(k).repeat_interleave(Hq // Hkv, dim=2).permute(0, 2, 1, 3)
    vt = torch.from_numpy(v).repeat_interleave(Hq // Hkv, dim=2).permute(0, 2, 1, 3)
    ref = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale).permute(0, 2, 1, 3).numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)


def test_single_route_returns_that_value_row():
    rng = np.random.default_rng(11)
    B, S_q, S_kv, Hq, Hkv, D = 1, 6, 9, 4, 2, 16
    q = rng.standard_normal((B, S_q, Hq, D))
    k = rng.standard_normal((B, S_kv, Hkv, D))
    v = rng.standard_normal((B, S_kv, Hkv, D))
    dout = rng.standard_normal((B, S_q, Hq, D))
    js = [0, 3, 8, 5, 5, 1]  # each row routes to exactly one key (padded with -1 / invalid / the same key)
    routes = np.array([[[j, -1, j, S_kv + 1] for j in js]], np.int64)
    scale = 0.5
    o, lse = oracle.forward(q, k, v, routes, scale)
    dq, dk, dv = oracle.backward(q, k, v, routes, dout, scale)
    G = Hq // Hkv
    for i, j in enumerate(js):
        for h in range(Hq):
            g = h // G
            assert np.array_equal(o[0, i, h], v[0, j, g])  # P = 1 exactly
            assert lse[0, h, i] == pytest.approx(scale * float(np.dot(q[0, i, h], k[0, j, g])), abs=1e-13)
    assert np.all(dq == 0.0)  # dS = P (dP - Delta) = dP - dP = 0
    assert np.all(dk == 0.0)
    for j in range(S_kv):
        for g in range(Hkv):
            expect = sum(dout[0, i, h] for i, jj in enumerate(js) if jj == j for h in range(g * G, (g + 1) * G))
            np.testing.assert_allclose(dv[0, j, g], expect if np.ndim(expect) else np.zeros(D), atol=1e-13)


def test_two_route_golden():
    with open(os.path.join(GOLDEN, "two_route_softmax.json")) as f:
        g = json.load(f)
    q, k, v, dout = (np.array(g[n], np.float64) for n in ("q", "k", "v", "dout"))
    routes = np.array(g["routes"], np.int64)
    e = g["expect"]
    ids, counts = oracle.route_sets(routes, k.shape[1])
    assert ids.tolist() == e["ids"] and counts.tolist() == e["counts"]
    o, lse = oracle.forward(q, k, v, routes, g["scale"])
    dq, dk, dv = oracle.backward(q, k, v, routes, dout, g["scale"])
    for got, name in ((o, "o"), (lse, "lse"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        np.testing.assert_allclose(got, np.array(e[name]), rtol=1e-14, atol=1e-14, err_msg=name)


def test_route_validity_golden():
    with open(os.path.join(GOLDEN, "route_validity.json")) as f:
        g = json.load(f)
    routes = np.array([[r["routes"] for r in g["rows"]]], np.int64)
    ids, counts = oracle.route_sets(routes, g["S_kv"])
    for i, r in enumerate(g["rows"]):
        n = len(r["ids"])
        assert counts[0, i] == n
        assert ids[0, i, :n].tolist() == r["ids"]
        assert np.all(ids[0, i, n:] == -1)


def test_route_sets_brute_force():
    rng = np.random.default_rng(5)
    B, S_q, K, S_kv = 3, 50, 40, 37
    routes = rng.integers(-5, S_kv + 5, size=(B, S_q, K)).astype(np.int64)
    specials = np.array([2**40 + 1, 2**62, -(2**63), 2**63 - 1, 2**32 + 2, -1], np.int64)
    mask = rng.random(routes.shape) < 0.1
    routes[mask] = rng.choice(specials, size=mask.sum())
    ids, counts = oracle.route_sets(routes, S_kv)
    for b in range(B):
        for i in range(S_q):
            expect = sorted(set(int(x) for x in routes[b, i] if 0 <= int(x) < S_kv))
            assert counts[b, i] == len(expect)
            assert ids[b, i, :len(expect)].tolist() == expect
            assert np.all(ids[b, i, len(expect):] == -1)


def test_duplicates_and_order_do_not_matter():
    rng = np.random.default_rng(13)
    B, S_q, S_kv, Hq, Hkv, D, K = 2, 10, 30, 4, 2, 8, 12
    q, k, v, routes = _random_problem(rng, B, S_q, S_kv, Hq, Hkv, D, K)
    dout = rng.standard_normal(q.shape)
    # Same route sets: permuted slots, extra duplicates, extra invalid values, wider rows.
    wide = np.concatenate([routes, routes[:, :, :5], np.full((B, S_q, 3), -9), np.full((B, S_q, 2), 2**41)], axis=2)
    perm = np.argsort(rng.random(wide.shape), axis=2)
    wide = np.take_along_axis(wide, perm, 2)
    a = oracle.forward(q, k, v, routes, 0.3) + oracle.backward(q, k, v, routes, dout, 0.3)
    b = oracle.forward(q, k, v, wide, 0.3) + oracle.backward(q, k, v, wide, dout, 0.3)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_empty_rows_zero_output_and_gradients():
    rng = np.random.default_rng(17)
    B, S_q, S_kv, Hq, Hkv, D, K = 1, 12, 16, 4, 1, 8, 6
    q, k, v, routes = _random_problem(rng, B, S_q, S_kv, Hq, Hkv, D, K)
    empty = [2, 7, 11]
    routes[0, empty] = [-1, -5, S_kv, 2**40, -1, S_kv + 9]
    dout = rng.standard_normal(q.shape)
    o, lse = oracle.forward(q, k, v, routes, 0.25)
    dq, dk, dv = oracle.backward(q, k, v, routes, dout, 0.25)
    assert np.all(o[0, empty] == 0.0)
    assert np.all(np.isneginf(lse[0, :, empty]))
    assert np.all(dq[0, empty] == 0.0)
    # An empty row contributes nothing to dK/dV: changing its Q and dO changes nothing.
    q2, d2 = q.copy(), dout.copy()
    q2[0, empty] = 100.0
    d2[0, empty] = -50.0
    _, dk2, dv2 = oracle.backward(q2, k, v, routes, d2, 0.25)
    assert np.array_equal(dk, dk2) and np.array_equal(dv, dv2)


def test_gradients_match_central_finite_differences():
    rng = np.random.default_rng(19)
    B, S_q, S_kv, Hq, Hkv, D, K = 1, 8, 8, 4, 2, 4, 6
    q, k, v, routes = _random_problem(rng, B, S_q, S_kv, Hq, Hkv, D, K, p_empty=0.1)
    dout = rng.standard_normal(q.shape)
    scale = 0.7
    dq, dk, dv = oracle.backward(q, k, v, routes, dout, scale)

    def loss(q_, k_, v_):
        o, _ = oracle.forward(q_, k_, v_, routes, scale)
        return float(np.sum(o * dout))

    eps = 1e-6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        args = [q, k, v]
        fd = np.zeros_like(grad)
        base = args[which]
        for idx in np.ndindex(base.shape):
            plus, minus = base.copy(), base.copy()
            plus[idx] += eps
            minus[idx] -= eps
            a = list(args)
            a[which] = plus
            lp = loss(*a)
            a[which] = minus
            fd[idx] = (lp - loss(*a)) / (2 * eps)
        err = np.max(np.abs(fd - grad)) / max(np.max(np.abs(grad)), 1e-30)
        assert err < 1e-6, (which, err)


def test_gradient_identities_and_untouched_keys():
    """sum_j dS_j = 0 per (row, head), hence sum_j dK_j = 0; sum_j dV_j equals the
    sum of dO over the group's non-empty rows; unrouted keys get exact zeros."""
    rng = np.random.default_rng(23)
    B, S_q, S_kv, Hq, Hkv, D, K = 2, 20, 40, 8, 2, 16, 10
    q, k, v, routes = _random_problem(rng, B, S_q, S_kv, Hq, Hkv, D, K, p_empty=0.2)
    routes[routes >= 30] = -1  # keys 30..39 are never routed
    dout = rng.standard_normal(q.shape)
    _, counts = oracle.route_sets(routes, S_kv)
    _, dk, dv = oracle.backward(q, k, v, routes, dout, 0.2)
    G = Hq // Hkv
    for b in range(B):
        for g in range(Hkv):
            np.testing.assert_allclose(dk[b, :, g].sum(0), 0.0, atol=1e-12)
            live = counts[b] > 0
            expect = dout[b, live][:, g * G:(g + 1) * G].sum((0, 1))
            np.testing.assert_allclose(dv[b, :, g].sum(0), expect, atol=1e-11)
    assert np.all(dk[:, 30:] == 0.0) and np.all(dv[:, 30:] == 0.0)


def test_listed_keys_equal_full_backward():
    rng = np.random.default_rng(29)
    B, S_q, S_kv, Hq, Hkv, D, K = 2, 16, 24, 4, 2, 8, 9
    q, k, v, routes = _random_problem(rng, B, S_q, S_kv, Hq, Hkv, D, K)
    dout = rng.standard_normal(q.shape)
    dq, dk, dv = oracle.backward(q, k, v, routes, dout, 0.4)
    keys = np.array([0, 5, 23, 24 + 3, 24 + 17], np.int64)
    dq2, dk2, dv2 = oracle.backward(q, k, v, routes, dout, 0.4, keys=keys)
    assert np.array_equal(dq, dq2)
    flat_dk = dk.reshape(B * S_kv, Hkv, D)
    flat_dv = dv.reshape(B * S_kv, Hkv, D)
    assert np.array_equal(dk2, flat_dk[keys]) and np.array_equal(dv2, flat_dv[keys])


def test_int32_wrap_threshold_stated_on_the_pages():
    """flex_qsa _membership_flat_offset: a square 46341-token sequence already
    puts B * S_q * kv_length past 2^31, so offsets need int64."""
    assert 46341 * 46341 > 2**31 - 1 > 46340 * 46340

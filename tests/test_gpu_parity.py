"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on
the same seeded inputs.  Route sets must match bit for bit; O, dQ, dK, dV within
|gpu - ref| <= 2e-2 |ref| + 2e-2; LSE within 1e-3 absolute, -inf where the
oracle has -inf."""
import numpy as np
import pytest

import oracle
from route_sparse_gqa_gb300 import workloads as W
from tests.qsa_testlib import assert_close, assert_lse_close, f64, run_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def _full_compare(q, k, v, do, routes, scale, S_kv, fp32=False, transform=None):
    out = run_library(q, k, v, do, routes, scale, fp32_dkdv=fp32, transform=transform)
    ids_ref, counts_ref = oracle.route_sets(routes, S_kv)
    assert np.array_equal(out["counts"], counts_ref)
    assert np.array_equal(out["ids"], ids_ref)
    qd, kd, vd, dod = f64(q), f64(k), f64(v), f64(do)
    o_ref, lse_ref = oracle.forward(qd, kd, vd, routes, scale)
    dq_ref, dk_ref, dv_ref = oracle.backward(qd, kd, vd, routes, dod, scale)
    assert_close("O", out["o"], o_ref)
    assert_lse_close(out["lse"], lse_ref)
    assert_close("dQ", out["dq"], dq_ref)
    assert_close("dK", out["dk"], dk_ref)
    assert_close("dV", out["dv"], dv_ref)
    if fp32:
        assert_close("dK fp32", out["dk32"], dk_ref)
        assert_close("dV fp32", out["dv32"], dv_ref)
    return out


def test_tiny_causal_rows_workload():
    c = W.make_case(0)
    w = c.workload
    out = _full_compare(c.q, c.k, c.v, c.do, c.routes, w.softmax_scale, w.S_kv, fp32=True)
    assert np.all(out["o"][0, 240:] == 0) and np.all(out["dq"][0, 240:] == 0)


def _random_case(seed, B, S_q, S_kv, Hq, Hkv, K, pattern="random", dtype=np.int32, p_empty=0.1, D=256):
    rng = np.random.default_rng(seed)
    q = W.bf16_normal(rng, (B, S_q, Hq, D))
    k = W.bf16_normal(rng, (B, S_kv, Hkv, D))
    v = W.bf16_normal(rng, (B, S_kv, Hkv, D))
    do = W.bf16_normal(rng, (B, S_q, Hq, D))
    if pattern == "random":
        routes = rng.integers(-2, S_kv + 2, size=(B, S_q, K)).astype(np.int64)
    elif pattern == "blocks":
        routes = np.stack([W._block_routes(rng, np.arange(S_q) % S_kv, np.zeros(S_q, np.int64), 7, K)
                           for _ in range(B)])
    elif pattern == "dense":  # every key, shuffled, plus padding
        base = np.tile(np.arange(S_kv), (B, S_q, 1))
        routes = np.concatenate([base, np.full((B, S_q, K - S_kv), -1)], axis=2)
        routes = np.take_along_axis(routes, np.argsort(rng.random(routes.shape), axis=2), 2)
    else:
        raise ValueError(pattern)
    routes[rng.random((B, S_q)) < p_empty] = -1
    if dtype == np.int64:
        huge = rng.random(routes.shape) < 0.05
        routes[huge] = rng.integers(2**40, 2**62, size=huge.sum())
        routes[rng.random(routes.shape) < 0.02] = 2**32 + 5  # would alias id 5 if narrowed first
    return q, k, v, do, routes.astype(dtype)


@pytest.mark.parametrize("B,S_q,S_kv,Hq,Hkv,K,pattern,dtype", [
    (1, 100, 300, 16, 2, 50, "random", np.int32),    # G=8, ragged last tile, S_q != S_kv
    (2, 70, 70, 8, 2, 40, "blocks", np.int64),       # G=4
    (1, 50, 130, 32, 2, 64, "random", np.int64),     # G=16
    (1, 33, 50, 2, 2, 20, "random", np.int32),       # G=1
    (1, 40, 64, 12, 2, 24, "random", np.int32),      # G=6
    (1, 64, 40, 16, 2, 48, "dense", np.int32),       # S_kv < one chunk, every key routed
    (2, 130, 700, 16, 2, 300, "blocks", np.int32),   # several chunks per tile
    (1, 17, 2000, 16, 2, 1, "random", np.int32),     # K = 1
])
def test_small_shapes(B, S_q, S_kv, Hq, Hkv, K, pattern, dtype):
    q, k, v, do, routes = _random_case(B * 7 + S_q + K, B, S_q, S_kv, Hq, Hkv, K, pattern, dtype)
    _full_compare(q, k, v, do, routes, 1.0 / 16, S_kv)


@pytest.mark.parametrize("D,Hq,Hkv,det", [
    (128, 16, 2, False),  # G = 8 at D = 128: the tile path
    (128, 8, 2, True),    # G = 4 at D = 128: the tile path, deterministic backward
    (64, 8, 8, False),    # G = 1 (MHA-shaped) at D = 64: the warp-level path
    (128, 6, 2, True),    # G = 3: the warp-level path, deterministic backward
])
def test_other_head_dims(D, Hq, Hkv, det):
    """Head dims 64 and 128 (the pages fix 256): D = 128 with G dividing 128 on the
    tile path, the rest on the warp-level path."""
    B, S_q, S_kv, K = 2, 60, 150, 40
    q, k, v, do, routes = _random_case(D + Hq, B, S_q, S_kv, Hq, Hkv, K, D=D)
    scale = 1.0 / np.sqrt(D)
    out = run_library(q, k, v, do, routes, scale, fp32_dkdv=True, deterministic=det)
    ids_ref, counts_ref = oracle.route_sets(routes, S_kv)
    assert np.array_equal(out["ids"], ids_ref)
    qd, kd, vd, dod = f64(q), f64(k), f64(v), f64(do)
    o_ref, lse_ref = oracle.forward(qd, kd, vd, routes, scale)
    dq_ref, dk_ref, dv_ref = oracle.backward(qd, kd, vd, routes, dod, scale)
    assert_close("O", out["o"], o_ref)
    assert_lse_close(out["lse"], lse_ref)
    assert_close("dQ", out["dq"], dq_ref)
    assert_close("dK", out["dk"], dk_ref)
    assert_close("dV", out["dv"], dv_ref)
    assert_close("dK fp32", out["dk32"], dk_ref)


def test_maximum_route_slots():
    """K = 16384 route slots (the library's maximum) with duplicates and invalid
    values, over 20000 keys: the uncached route-row path and tiles of ~300 chunks."""
    rng = np.random.default_rng(16384)
    B, S_q, S_kv, Hq, Hkv, K = 1, 20, 20000, 16, 2, 16384
    q = W.bf16_normal(rng, (B, S_q, Hq, 256))
    k = W.bf16_normal(rng, (B, S_kv, Hkv, 256))
    v = W.bf16_normal(rng, (B, S_kv, Hkv, 256))
    do = W.bf16_normal(rng, (B, S_q, Hq, 256))
    routes = rng.integers(-5, S_kv + 5, size=(B, S_q, K)).astype(np.int32)
    routes[0, 3] = -1  # an empty row
    _full_compare(q, k, v, do, routes, 1.0 / 16, S_kv)


def test_all_rows_empty():
    q, k, v, do, routes = _random_case(3, 1, 40, 64, 16, 2, 8, p_empty=1.0)
    out = _full_compare(q, k, v, do, routes, 0.1, 64)
    assert np.all(out["o"] == 0) and np.all(np.isneginf(out["lse"]))
    assert np.all(out["dq"] == 0) and np.all(out["dk"] == 0) and np.all(out["dv"] == 0)


def test_strided_inputs():
    """Q/K/V as views with non-dense strides and routes as a transposed view."""
    import torch

    q, k, v, do, routes = _random_case(11, 2, 48, 96, 16, 2, 32, "random", np.int64)

    def transform(qt, kt, vt, rt):
        qw = torch.zeros(qt.shape[0], qt.shape[1], qt.shape[2] + 8, 256, dtype=qt.dtype, device=qt.device)
        qw[:, :, 3:3 + qt.shape[2]] = qt
        kw = torch.zeros(kt.shape[0], kt.shape[1] * 2, kt.shape[2], 256, dtype=kt.dtype, device=kt.device)
        kw[:, ::2] = kt
        rT = rt.transpose(1, 2).contiguous().transpose(1, 2)
        return qw[:, :, 3:3 + qt.shape[2]], kw[:, ::2], vt, rT

    _full_compare(q, k, v, do, routes, 0.0625, 96, transform=transform)


def test_scale_default_and_scale_changes_result():
    import torch

    import route_sparse_gqa_gb300 as qsa
    from tests.qsa_testlib import bf16_to_device

    q, k, v, _, routes = _random_case(5, 1, 20, 40, 16, 2, 10)
    dev = torch.device("cuda:0")
    qt, kt, vt = (bf16_to_device(x, dev) for x in (q, k, v))
    rt = torch.from_numpy(routes).to(dev)
    o_default = qsa.qsa_attention(qt, kt, vt, rt)
    o_16 = qsa.qsa_attention(qt, kt, vt, rt, 1.0 / 16)
    o_1 = qsa.qsa_attention(qt, kt, vt, rt, 1.0)
    assert torch.equal(o_default, o_16)
    assert not torch.equal(o_default, o_1)


def test_invalid_arguments_raise():
    import torch

    import route_sparse_gqa_gb300 as qsa

    dev = torch.device("cuda:0")
    q = torch.zeros(1, 8, 16, 256, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(1, 8, 2, 256, dtype=torch.bfloat16, device=dev)
    r = torch.zeros(1, 8, 4, dtype=torch.int32, device=dev)
    with pytest.raises(qsa.QSAError, match="INVALID"):
        qsa.qsa_attention(q, k, k, r, -1.0)
    with pytest.raises(qsa.QSAError, match="INVALID"):
        qsa.qsa_attention(q[:, :, :15], k, k, r)  # Hq not a multiple of Hkv
    with pytest.raises(qsa.QSAError, match="UNSUPPORTED"):
        qsa.qsa_attention(q.float(), k, k, r)
    with pytest.raises(qsa.QSAError, match="UNSUPPORTED"):
        qsa.qsa_attention(q[..., :96], k[..., :96], k[..., :96], r)  # head dim 96
    with pytest.raises(qsa.QSAError, match="INVALID"):
        qsa.qsa_attention(q, k, k[:, :4], r)


def test_autograd_matches_explicit_backward():
    import torch

    import route_sparse_gqa_gb300 as qsa
    from tests.qsa_testlib import bf16_to_device

    q, k, v, do, routes = _random_case(9, 1, 30, 60, 16, 2, 12)
    dev = torch.device("cuda:0")
    qt, kt, vt, dot = (bf16_to_device(x, dev) for x in (q, k, v, do))
    rt = torch.from_numpy(routes).to(dev)
    qt.requires_grad_(True), kt.requires_grad_(True), vt.requires_grad_(True)
    o = qsa.qsa_attention(qt, kt, vt, rt)
    o.backward(dot)
    plan = qsa.preprocess(qt.detach(), kt.detach(), vt.detach(), rt)
    o2, lse2 = qsa.forward(plan, qt.detach(), kt.detach(), vt.detach())
    dq, dk, dv = qsa.backward(plan, qt.detach(), kt.detach(), vt.detach(), o2, lse2, dot)
    assert torch.equal(o.detach(), o2)
    for a, b in ((qt.grad, dq), (kt.grad, dk), (vt.grad, dv)):
        assert torch.allclose(a.float(), b.float(), rtol=1e-2, atol=1e-2)


def test_route_sets_wide_and_narrow_ranges():
    """Rows whose ids span a huge key range (sorted by the bitonic fallback) next
    to narrow rows (sorted through the shared-memory byte map): bit-exact."""
    import torch

    import route_sparse_gqa_gb300 as qsa

    rng = np.random.default_rng(31)
    S_q, S_kv, K = 24, 1_500_000, 96
    routes = rng.integers(-4, S_kv + 4, size=(1, S_q, K)).astype(np.int64)
    routes[0, ::3] = rng.integers(1000, 1200, size=(S_q // 3 + (S_q % 3 > 0), K))  # narrow rows
    routes[0, 1::5, :10] = 2**45 + 3
    routes[0, 7] = -1
    dev = torch.device("cuda:0")
    q = torch.zeros(1, S_q, 16, 256, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(1, S_kv, 2, 256, dtype=torch.bfloat16, device=dev)
    plan = qsa.preprocess(q, k, k, torch.from_numpy(routes).to(dev))
    ids, counts = plan.route_sets()
    ids_ref, counts_ref = oracle.route_sets(routes, S_kv)
    assert np.array_equal(counts.cpu().numpy(), counts_ref)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)


def _rows_at_sort_boundaries(rng, K):
    """Route rows whose valid ids span exactly the key ranges where route_rows changes
    method: byte map up to 16384 keys, 65536-key bitmap windows up to 8 windows, bitonic
    sort beyond; with contiguous 64-id runs, repeats, invalid values and empty rows."""
    rows = []
    for lo, span in ((5, 16383), (100, 16384), (0, 65535), (7, 65536), (3, 524287), (3, 524288), (11, 200_000)):
        r = rng.integers(lo, lo + span + 1, size=K)
        r[0], r[1] = lo, lo + span  # the range's ends
        r[2:6] = r[6:10]  # repeats
        r[10] = -1
        r[11] = 2**40 + 5  # invalid, outside int32
        rows.append(r)
    for span in (8000, 200_000):  # runs of 64 consecutive ids, in generation order
        starts = rng.choice(span // 64, size=(K + 63) // 64, replace=False) * 64 + 17
        rows.append((starts[:, None] + np.arange(64)[None, :]).reshape(-1)[:K])
    rows.append(np.full(K, -1))
    rows.append(np.full(K, 2**40))
    return np.stack(rows).astype(np.int64)


@pytest.mark.parametrize("K", [96, 2600])  # route slots kept in registers / re-read for every window
def test_route_sets_at_sort_method_boundaries(K):
    """Every sort path of the route preprocessing and the range edges between them:
    bit-exact against the oracle's route sets."""
    import torch

    import route_sparse_gqa_gb300 as qsa

    rng = np.random.default_rng(77 + K)
    routes = _rows_at_sort_boundaries(rng, K)[None]
    S_q, S_kv = routes.shape[1], 600_000
    dev = torch.device("cuda:0")
    q = torch.zeros(1, S_q, 16, 256, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(1, S_kv, 2, 256, dtype=torch.bfloat16, device=dev)
    plan = qsa.preprocess(q, k, k, torch.from_numpy(routes).to(dev))
    ids, counts = plan.route_sets()
    ids_ref, counts_ref = oracle.route_sets(routes, S_kv)
    assert np.array_equal(counts.cpu().numpy(), counts_ref)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)


@pytest.mark.parametrize("K", [96, 2176, 2177])
def test_route_sets_presorted_rows(K):
    """Rows that arrive sorted (as the route producer writes them), and rows that only nearly are (a repeat,
    an invalid slot before a valid one, descending ids, an id at S_kv, out-of-range and huge tails): bit-exact
    against the oracle's route sets with and without the rows-sorted flag (which copies sorted rows through
    and must sort the others as usual), on both sides of route_rows' register-row limit (17 x 128 slots)."""
    import torch

    import route_sparse_gqa_gb300 as qsa

    rng = np.random.default_rng(91 + K)
    S_kv = 50_000
    n_valid = min(K - 8, 1500)
    rows = []
    for kind in range(8):
        ids = np.sort(rng.choice(S_kv, size=n_valid, replace=False)).astype(np.int64)
        r = np.full(K, -1, np.int64)
        r[:n_valid] = ids
        if kind == 1:  # out-of-range tail after the sorted valid ids (invalid, still after them)
            r[n_valid:] = S_kv + rng.integers(0, 5, size=K - n_valid)
        elif kind == 2:  # a repeat
            r[n_valid // 2] = r[n_valid // 2 - 1]
        elif kind == 3:  # an invalid slot before a valid one
            r[n_valid // 3] = -5
        elif kind == 4:  # descending
            r[:n_valid] = ids[::-1]
        elif kind == 5:  # id S_kv (invalid) in the middle of the valid run
            r[n_valid // 4] = S_kv
        elif kind == 6:  # empty row
            r[:] = -1
        elif kind == 7:  # huge int64 tail
            r[n_valid:] = 2**40 + 1
        rows.append(r)
    routes = np.stack(rows)[None]
    S_q = routes.shape[1]
    dev = torch.device("cuda:0")
    q = torch.zeros(1, S_q, 16, 256, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(1, S_kv, 2, 256, dtype=torch.bfloat16, device=dev)
    for dtype in (np.int64, np.int32):
        rt = routes.astype(dtype) if dtype == np.int64 else np.where(routes > 2**31 - 1, -1, routes).astype(np.int32)
        ids_ref, counts_ref = oracle.route_sets(rt, S_kv)
        for hint in (False, True):  # QSA_ROUTES_SORTED: sorted rows copied through, the others sorted as usual
            plan = qsa.preprocess(q, k, k, torch.from_numpy(rt).to(dev), routes_sorted=hint)
            ids, counts = plan.route_sets()
            assert np.array_equal(counts.cpu().numpy(), counts_ref), (dtype, hint)
            assert np.array_equal(ids.cpu().numpy(), ids_ref), (dtype, hint)


def test_repeated_calls_share_one_workspace():
    """The tile and key-major kernels take their work from queues whose counters
    live in the workspace and are reset by the last CTA of every launch.  Calls
    repeated on one plan must therefore give the same results: O and LSE bit for
    bit (each forward item is computed by one CTA in a fixed order), dQ, dK and
    dV within the tolerance (fp32 reductions in any order), all matching the
    oracle; a work-item count below the SM count and one far above it are both
    exercised."""
    import torch

    import route_sparse_gqa_gb300 as qsa
    from tests.qsa_testlib import bf16_to_device

    dev = torch.device("cuda:0")
    for seed, (B, S_q, S_kv, Hq, Hkv, K) in ((41, (1, 40, 96, 16, 2, 24)), (42, (2, 1200, 700, 16, 2, 40))):
        q, k, v, do, routes = _random_case(seed, B, S_q, S_kv, Hq, Hkv, K)
        qt, kt, vt, dot = (bf16_to_device(x, dev) for x in (q, k, v, do))
        rt = torch.from_numpy(routes).to(dev)
        plan = qsa.preprocess(qt, kt, vt, rt, 1.0 / 16)
        outs = []
        for _ in range(3):
            o, lse = qsa.forward(plan, qt, kt, vt)
            dq, dk, dv = qsa.backward(plan, qt, kt, vt, o, lse, dot)
            outs.append([x.float().cpu().numpy() for x in (o, lse, dq, dk, dv)])
        plan.device_status()
        for later in outs[1:]:
            for name, a, b in zip(("O", "LSE"), outs[0][:2], later[:2]):
                assert np.array_equal(a, b, equal_nan=True), f"{name} differs between repeated calls"
            for name, a, b in zip(("dQ", "dK", "dV"), outs[0][2:], later[2:]):
                assert_close(name + " repeat", b.astype(np.float64), a.astype(np.float64))
        qd, kd, vd, dod = f64(q), f64(k), f64(v), f64(do)
        o_ref, lse_ref = oracle.forward(qd, kd, vd, routes, 1.0 / 16)
        dq_ref, dk_ref, dv_ref = oracle.backward(qd, kd, vd, routes, dod, 1.0 / 16)
        last = outs[-1]
        assert_close("O", last[0].astype(np.float64), o_ref)
        assert_lse_close(last[1].astype(np.float64), lse_ref)
        assert_close("dQ", last[2].astype(np.float64), dq_ref)
        assert_close("dK", last[3].astype(np.float64), dk_ref)
        assert_close("dV", last[4].astype(np.float64), dv_ref)

"""The deterministic backward (qsa_backward_deterministic): dK/dV summed as
fixed-point integers, so repeated runs give bitwise identical gradients, and the
gradients match the fp64 oracle within the usual tolerance
(|gpu - ref| <= 2e-2 |ref| + 2e-2).  Covers the tile path (G = 4, 8) and the
warp-level path (G = 3), and the full right-padded workload, where thousands of
CTAs add into the same keys in an order that changes from run to run."""
import numpy as np
import pytest

import oracle
from route_sparse_gqa_gb300 import workloads as W
from tests.qsa_testlib import assert_close, f64, run_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def _random_case(seed, B, S_q, S_kv, Hq, Hkv, K):
    rng = np.random.default_rng(seed)
    q = W.bf16_normal(rng, (B, S_q, Hq, 256))
    k = W.bf16_normal(rng, (B, S_kv, Hkv, 256))
    v = W.bf16_normal(rng, (B, S_kv, Hkv, 256))
    do = W.bf16_normal(rng, (B, S_q, Hq, 256))
    routes = rng.integers(-2, S_kv + 2, size=(B, S_q, K)).astype(np.int32)
    routes[:, -3:] = -1  # a few empty rows
    return q, k, v, do, routes


@pytest.mark.parametrize("shape", [
    (1, 96, 300, 4, 1, 40),    # tile path, G = 4
    (2, 64, 200, 16, 2, 64),   # tile path, G = 8
    (1, 50, 120, 6, 2, 30),    # warp-level path, G = 3
])
def test_deterministic_backward_matches_oracle_and_repeats_bitwise(shape):
    B, S_q, S_kv, Hq, Hkv, K = shape
    q, k, v, do, routes = _random_case(sum(shape), *shape)
    scale = 0.0625
    a = run_library(q, k, v, do, routes, scale, fp32_dkdv=True, deterministic=True)
    b = run_library(q, k, v, do, routes, scale, fp32_dkdv=True, deterministic=True)
    for name in ("dq", "dk", "dv", "dk32", "dv32"):
        assert np.array_equal(a[name], b[name]), name
    dq_ref, dk_ref, dv_ref = oracle.backward(f64(q), f64(k), f64(v), routes, f64(do), scale)
    assert_close("dQ", a["dq"], dq_ref)
    assert_close("dK", a["dk"], dk_ref)
    assert_close("dV", a["dv"], dv_ref)
    assert_close("dK fp32", a["dk32"], dk_ref)
    assert_close("dV fp32", a["dv32"], dv_ref)


def test_deterministic_backward_full_right_padded_workload():
    case = W.make_case(1)
    w = case.workload
    runs = [run_library(case.q, case.k, case.v, case.do, case.routes, w.softmax_scale, fp32_dkdv=True,
                        deterministic=True) for _ in range(2)]
    for name in ("dq", "dk", "dv", "dk32", "dv32"):
        assert np.array_equal(runs[0][name], runs[1][name]), name
    # Against the fp32-atomic backward (same sums, other rounding): within the tolerance.
    fast = run_library(case.q, case.k, case.v, case.do, case.routes, w.softmax_scale, fp32_dkdv=True)
    assert_close("dK det vs fp32", runs[0]["dk32"], fast["dk32"], rtol=1e-3, atol=1e-3)
    assert_close("dV det vs fp32", runs[0]["dv32"], fast["dv32"], rtol=1e-3, atol=1e-3)
    # And against the oracle on sampled late keys of batch row 0.
    rng = np.random.default_rng(5)
    keys = np.sort(rng.choice(np.arange(3500, 4096), size=6, replace=False))
    flat = keys  # batch row 0
    _, dk_ref, dv_ref = oracle.backward(f64(case.q), f64(case.k), f64(case.v), case.routes, f64(case.do),
                                        w.softmax_scale, keys=flat)
    assert_close("dK sampled", runs[0]["dk32"][0, keys], dk_ref)
    assert_close("dV sampled", runs[0]["dv32"][0, keys], dv_ref)

"""GPU parity of each kernel path on its own.  Problems that both the tile and
the key-major kernels accept (G a power of two from 8 to 64, D = 256 or 128)
pick a path on the device from the preprocessed routes; the test hooks
QSA_DEBUG_FORWARD_PATH / QSA_DEBUG_BACKWARD_PATH (= "tile" or "keymajor") force
one, so every path is compared with the fp64 oracle on every shape here,
whatever the choice would have been: ragged tiles and groups, S_q != S_kv, a
key range ending inside a chunk, empty rows, int64 routes with huge values,
several batch rows, whole-block and scattered routes, and chunks whose reverse
lists span several work items and query windows."""
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


def _case(seed, B, S_q, S_kv, Hq, Hkv, K, D, pattern, dtype):
    rng = np.random.default_rng(seed)
    q = W.bf16_normal(rng, (B, S_q, Hq, D))
    k = W.bf16_normal(rng, (B, S_kv, Hkv, D))
    v = W.bf16_normal(rng, (B, S_kv, Hkv, D))
    do = W.bf16_normal(rng, (B, S_q, Hq, D))
    if pattern == "random":
        routes = rng.integers(-2, S_kv + 2, size=(B, S_q, K)).astype(np.int64)
    else:  # causal whole blocks (the workloads' structure)
        routes = np.stack([W._block_routes(rng, np.arange(S_q) % S_kv, np.zeros(S_q, np.int64), 9, K)
                           for _ in range(B)])
    routes[rng.random((B, S_q)) < 0.08] = -1
    if dtype == np.int64:
        huge = rng.random(routes.shape) < 0.03
        routes[huge] = rng.integers(2**40, 2**62, size=huge.sum())
    return q, k, v, do, routes.astype(dtype)


SHAPES = [
    # seed, B, S_q, S_kv, Hq, Hkv, K, D, pattern, dtype
    (71, 1, 100, 300, 16, 2, 50, 256, "random", np.int32),    # G = 8, ragged last group, S_kv ends mid-chunk
    (76, 2, 300, 520, 16, 2, 448, 256, "blocks", np.int64),   # two batch rows, lists over several work items
    (73, 1, 90, 200, 32, 2, 40, 256, "random", np.int32),     # G = 16
    (74, 1, 120, 256, 16, 2, 64, 128, "blocks", np.int32),    # D = 128
    (78, 1, 70, 260, 64, 2, 60, 128, "random", np.int32),     # G = 32 (four queries per group), D = 128
    (79, 2, 50, 200, 64, 1, 40, 256, "random", np.int64),    # G = 64 (two queries per group)
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"G{s[4] // s[5]}-D{s[7]}-{s[8]}" for s in SHAPES])
@pytest.mark.parametrize("fwd,bwd", [("tile", "keymajor"), ("keymajor", "tile"), ("keymajor", "keymajor")])
def test_each_path_matches_oracle(shape, fwd, bwd, monkeypatch):
    seed, B, S_q, S_kv, Hq, Hkv, K, D, pattern, dtype = shape
    monkeypatch.setenv("QSA_DEBUG_FORWARD_PATH", fwd)
    monkeypatch.setenv("QSA_DEBUG_BACKWARD_PATH", bwd)
    q, k, v, do, routes = _case(seed, B, S_q, S_kv, Hq, Hkv, K, D, pattern, dtype)
    scale = 1.0 / np.sqrt(D)
    out = run_library(q, k, v, do, routes, scale, fp32_dkdv=True)
    qd, kd, vd, dod = f64(q), f64(k), f64(v), f64(do)
    o_ref, lse_ref = oracle.forward(qd, kd, vd, routes, scale)
    dq_ref, dk_ref, dv_ref = oracle.backward(qd, kd, vd, routes, dod, scale)
    assert_close("O", out["o"], o_ref)
    assert_lse_close(out["lse"], lse_ref)
    assert_close("dQ", out["dq"], dq_ref)
    assert_close("dK", out["dk"], dk_ref)
    assert_close("dV", out["dv"], dv_ref)
    assert_close("dK fp32", out["dk32"], dk_ref)
    assert_close("dV fp32", out["dv32"], dv_ref)


def test_keymajor_forward_repeats_within_rounding_and_deterministic_flag(monkeypatch):
    """The key-major forward sums each row's output over work items in fp32 in the order they finish:
    repeated calls agree within the tolerance (and with the oracle).  With the deterministic-forward flag the
    preprocessing picks the tile forward even when the key-major one is forced by the test hook, so repeated
    calls, and with the deterministic backward the whole step, agree bit for bit."""
    import torch

    import route_sparse_gqa_gb300 as qsa
    from tests.qsa_testlib import bf16_to_device

    monkeypatch.setenv("QSA_DEBUG_FORWARD_PATH", "keymajor")
    q, k, v, do, routes = _case(80, 1, 600, 1500, 16, 2, 700, 256, "blocks", np.int32)
    dev = torch.device("cuda:0")
    qt, kt, vt, dot = (bf16_to_device(x, dev) for x in (q, k, v, do))
    rt = torch.from_numpy(routes).to(dev)
    o_ref, lse_ref = oracle.forward(f64(q), f64(k), f64(v), routes, 0.0625)
    for det in (False, True):
        plan = qsa.preprocess(qt, kt, vt, rt, 0.0625, deterministic_forward=det)
        runs = []
        for _ in range(3):
            o, lse = qsa.forward(plan, qt, kt, vt)
            grads = qsa.backward(plan, qt, kt, vt, o, lse, dot, deterministic=det)
            runs.append([x.float().cpu().numpy() for x in (o, lse, *grads)])
        plan.device_status()
        for later in runs[1:]:
            for name, a, b in zip(("O", "LSE", "dQ", "dK", "dV"), runs[0], later):
                if det:
                    assert np.array_equal(a, b, equal_nan=True), f"{name} differs between repeated calls"
                elif name == "LSE":
                    assert_lse_close(b.astype(np.float64), a.astype(np.float64))
                else:
                    assert_close(name + " repeat", b.astype(np.float64), a.astype(np.float64))
        assert_close("O", runs[-1][0].astype(np.float64), o_ref)
        assert_lse_close(runs[-1][1].astype(np.float64), lse_ref)


def test_keymajor_forward_deterministic_backward(monkeypatch):
    """The key-major forward followed by the bitwise reproducible backward on the key-major path: two
    runs agree bit for bit and match the oracle."""
    monkeypatch.setenv("QSA_DEBUG_FORWARD_PATH", "keymajor")
    monkeypatch.setenv("QSA_DEBUG_BACKWARD_PATH", "keymajor")
    q, k, v, do, routes = _case(75, 1, 200, 400, 16, 2, 96, 256, "blocks", np.int32)
    runs = [run_library(q, k, v, do, routes, 0.0625, deterministic=True) for _ in range(2)]
    for name in ("dq", "dk", "dv"):
        assert np.array_equal(runs[0][name], runs[1][name]), f"{name} differs between runs"
    qd, kd, vd, dod = f64(q), f64(k), f64(v), f64(do)
    dq_ref, dk_ref, dv_ref = oracle.backward(qd, kd, vd, routes, dod, 0.0625)
    assert_close("dQ", runs[0]["dq"], dq_ref)
    assert_close("dK", runs[0]["dk"], dk_ref)
    assert_close("dV", runs[0]["dv"], dv_ref)


@pytest.mark.parametrize("mode", ["bound", "forced-max", "large-logits"])
def test_keymajor_forward_reference(mode, monkeypatch):
    """The key-major forward's exponent reference: the Cauchy-Schwarz bound (unit-variance inputs keep every
    row's gap well under the limit), the row-max pass forced by the test hook QSA_DEBUG_FORWARD_MAXPASS, and
    queries scaled by 4 (exact in BF16), whose logits spread beyond the bound's limit so the row-max
    pass runs on its own."""
    monkeypatch.setenv("QSA_DEBUG_FORWARD_PATH", "keymajor")
    if mode == "forced-max":
        monkeypatch.setenv("QSA_DEBUG_FORWARD_MAXPASS", "1")
    q, k, v, do, routes = _case(77, 1, 180, 350, 16, 2, 120, 256, "blocks", np.int32)
    if mode == "large-logits":
        q = W.bf16_bits_from_f32(W.bf16_bits_to_f32(q) * np.float32(4.0))
    scale = 1.0 / 16
    out = run_library(q, k, v, do, routes, scale, fp32_dkdv=True)
    qd, kd, vd, dod = f64(q), f64(k), f64(v), f64(do)
    o_ref, lse_ref = oracle.forward(qd, kd, vd, routes, scale)
    assert_close("O", out["o"], o_ref)
    assert_lse_close(out["lse"], lse_ref)
    if mode == "large-logits":
        # Forward only: the backward's Delta = <dO, O> reads the BF16 output, and with logits this sharp
        # that rounding alone moves dK past the parity tolerance (whichever forward made O).
        return
    dq_ref, dk_ref, dv_ref = oracle.backward(qd, kd, vd, routes, dod, scale)
    assert_close("dQ", out["dq"], dq_ref)
    assert_close("dK", out["dk"], dk_ref)
    assert_close("dV", out["dv"], dv_ref)

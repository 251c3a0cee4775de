"""Full-size parity on the five workloads (and the D = 128 / G = 1 variants), run through the same C-ABI calls the
benchmark times.  The oracle cannot redo a full step of the large workloads in
seconds, so:

* route sets are compared bit for bit on EVERY row;
* O, LSE and dQ on sampled rows (first, last, empty, random), each recomputed
  by the oracle from its own inputs;
* dK and dV on sampled keys, recomputed from every row that routes to them:
  keys late in the sequence (few routing rows) and the hottest ones -- the
  first routed key (block 0, routed by thousands of rows on the long
  workloads: the most reductions and the most work items per chunk), the two
  keys with the most routing rows, and the last routed key (the last rows'
  own block; past 2^31 bytes of K/V on the long-K/V workload);
* properties that hold at any size on the whole output: sum_j dK_j = 0 and
  sum_j dV_j = sum of dO over the group's non-empty rows (fp32 accumulators),
  and exact zeros for keys no row routes to.
"""
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


def _sample_rows(rng, counts_b, n):
    S = counts_b.shape[0]
    rows = {0, S - 1}
    empty = np.nonzero(counts_b == 0)[0]
    if empty.size:
        rows.update(rng.choice(empty, size=min(4, empty.size), replace=False).tolist())
    rows.update(rng.choice(S, size=n, replace=False).tolist())
    return np.array(sorted(rows))


def _sample_keys(rng, ids_b, counts_b, S_kv, n):
    """Keys late in the sequence (few routing rows, so the oracle stays fast),
    the first and the last routed key (block 0 and the highest key), the two
    keys the most rows route to (the most reductions: block 0 again, or on the
    packed workload the first blocks of the longest documents), plus one
    never-routed key if there is one."""
    used = np.zeros(S_kv, bool)
    valid = ids_b[ids_b >= 0]
    used[valid] = True
    cand = np.nonzero(used)[0]
    late = cand[cand >= cand.max() - 512] if cand.size else cand
    keys = set(rng.choice(late, size=min(n, late.size), replace=False).tolist())
    if cand.size:
        keys.update((int(cand[0]), int(cand[-1])))
        hot = np.bincount(valid, minlength=S_kv)
        keys.update(int(x) for x in np.argsort(-hot, kind="stable")[:2])
    keys = np.array(sorted(keys), dtype=np.int64)
    unused = np.nonzero(~used)[0]
    return keys, unused


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5, 6])
def test_workload_full_size(index):
    case = W.make_case(index)
    w = case.workload
    out = run_library(case.q, case.k, case.v, case.do, case.routes, w.softmax_scale, fp32_dkdv=True)
    ids_ref, counts_ref = oracle.route_sets(case.routes, w.S_kv)
    assert np.array_equal(out["counts"], counts_ref)
    assert np.array_equal(out["ids"], ids_ref)
    rng = np.random.default_rng(100 + index)
    G = w.Hq // w.Hkv
    for b in range(w.B):
        kd, vd = f64(case.k[b:b + 1]), f64(case.v[b:b + 1])
        rows = _sample_rows(rng, counts_ref[b], 24)
        qd, dod, r = f64(case.q[b:b + 1, rows]), f64(case.do[b:b + 1, rows]), case.routes[b:b + 1, rows]
        o_ref, lse_ref = oracle.forward(qd, kd, vd, r, w.softmax_scale)
        dq_ref, _, _ = oracle.backward(qd, kd, vd, r, dod, w.softmax_scale, keys=np.zeros(0, np.int64))
        assert_close(f"O b{b}", out["o"][b:b + 1, rows], o_ref)
        assert_lse_close(out["lse"][b:b + 1, :, rows], lse_ref)
        assert_close(f"dQ b{b}", out["dq"][b:b + 1, rows], dq_ref)

        keys, unused = _sample_keys(rng, ids_ref[b], counts_ref[b], w.S_kv, 12)
        hit = np.nonzero(np.isin(ids_ref[b], keys).any(axis=1))[0]
        qd, dod, r = f64(case.q[b:b + 1, hit]), f64(case.do[b:b + 1, hit]), case.routes[b:b + 1, hit]
        _, dk_ref, dv_ref = oracle.backward(qd, kd, vd, r, dod, w.softmax_scale, keys=keys)
        assert_close(f"dK b{b}", out["dk"][b, keys], dk_ref)
        assert_close(f"dV b{b}", out["dv"][b, keys], dv_ref)
        assert_close(f"dK fp32 b{b}", out["dk32"][b, keys], dk_ref)
        assert_close(f"dV fp32 b{b}", out["dv32"][b, keys], dv_ref)
        if unused.size:
            assert np.all(out["dk32"][b, unused] == 0) and np.all(out["dv32"][b, unused] == 0)

        live = counts_ref[b] > 0
        do_b = f64(case.do[b])
        for g in range(w.Hkv):
            dk_sum = out["dk32"][b, :, g].sum(0)
            scale_k = np.abs(out["dk32"][b, :, g]).sum(0) + 1.0
            assert np.all(np.abs(dk_sum) <= 1e-3 * scale_k), f"sum dK b{b} g{g}"
            dv_sum = out["dv32"][b, :, g].sum(0)
            expect = do_b[live][:, g * G:(g + 1) * G].sum((0, 1))
            scale_v = np.abs(do_b[live][:, g * G:(g + 1) * G]).sum((0, 1)) + 1.0
            assert np.all(np.abs(dv_sum - expect) <= 1e-3 * scale_v), f"sum dV b{b} g{g}"


_ORACLE_CACHE = {}


@pytest.mark.parametrize("fwd", ["auto", "keymajor"])
def test_right_padded_workload_every_element(fwd, monkeypatch):
    """Every output element of the right-padded workload against the full oracle
    (forward and backward, ~15 s of oracle time, computed once).  Short tiles there (two chunks)
    end their items right after their first PV, which exposes any barrier-phase
    mistake between the PV and the epilogue that sampled rows can miss.  Run with
    the forward the device chooses (the tile forward here) and with the key-major
    forward forced."""
    if fwd != "auto":
        monkeypatch.setenv("QSA_DEBUG_FORWARD_PATH", fwd)
    case = W.make_case(1)
    w = case.workload
    out = run_library(case.q, case.k, case.v, case.do, case.routes, w.softmax_scale, fp32_dkdv=True)
    if not _ORACLE_CACHE:
        qd, kd, vd, dod = f64(case.q), f64(case.k), f64(case.v), f64(case.do)
        _ORACLE_CACHE["fwd"] = oracle.forward(qd, kd, vd, case.routes, w.softmax_scale)
        _ORACLE_CACHE["bwd"] = oracle.backward(qd, kd, vd, case.routes, dod, w.softmax_scale)
    o_ref, lse_ref = _ORACLE_CACHE["fwd"]
    dq_ref, dk_ref, dv_ref = _ORACLE_CACHE["bwd"]
    assert_close("O", out["o"], o_ref)
    assert_lse_close(out["lse"], lse_ref)
    assert_close("dQ", out["dq"], dq_ref)
    assert_close("dK", out["dk"], dk_ref)
    assert_close("dV", out["dv"], dv_ref)
    assert_close("dK fp32", out["dk32"], dk_ref)
    assert_close("dV fp32", out["dv32"], dv_ref)

"""Failure detection without a GPU fault.

The tile kernels bound every pipeline wait.  The host-side test hook
QSA_DEBUG_WAIT_LIMIT_NS=0 makes those waits run out almost at once; the
kernels must then record QSA_ERR_TIMEOUT in the workspace status word, drain
their in-flight copies and MMAs, free their TMEM and return, leaving the CUDA
context usable: the next normal call on the same process must match the oracle.
"""
import numpy as np
import pytest

import oracle
from route_sparse_gqa_gb300 import workloads as W
from tests.qsa_testlib import assert_close, assert_lse_close, bf16_to_device, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def _case():
    rng = np.random.default_rng(77)
    B, S_q, S_kv, Hq, Hkv, K = 1, 256, 2048, 16, 2, 512  # ~32 chunks per tile, 32 work items
    q = W.bf16_normal(rng, (B, S_q, Hq, 256))
    k = W.bf16_normal(rng, (B, S_kv, Hkv, 256))
    v = W.bf16_normal(rng, (B, S_kv, Hkv, 256))
    do = W.bf16_normal(rng, (B, S_q, Hq, 256))
    routes = rng.integers(-1, S_kv, size=(B, S_q, K)).astype(np.int32)
    return q, k, v, do, routes


@pytest.mark.parametrize("which", ["forward", "backward"])
def test_forced_wait_timeout_is_reported_and_context_survives(which, monkeypatch):
    import torch

    import route_sparse_gqa_gb300 as qsa

    dev = torch.device("cuda:0")
    qb, kb, vb, dob, routes_np = _case()
    q, k, v, do = (bf16_to_device(x, dev) for x in (qb, kb, vb, dob))
    routes = torch.from_numpy(routes_np).to(dev)
    plan = qsa.preprocess(q, k, v, routes, 0.0625)
    o, lse = qsa.forward(plan, q, k, v) if which == "backward" else (None, None)
    plan.device_status()  # clean so far

    monkeypatch.setenv("QSA_DEBUG_WAIT_LIMIT_NS", "0")
    if which == "forward":
        qsa.forward(plan, q, k, v)
    else:
        qsa.backward(plan, q, k, v, o, lse, do)
    monkeypatch.delenv("QSA_DEBUG_WAIT_LIMIT_NS")
    with pytest.raises(qsa.QSAError) as err:
        plan.device_status()
    assert err.value.status == 5, err.value  # QSA_ERR_TIMEOUT
    plan.device_status()  # reading cleared the word

    # The context is still usable and a normal run is correct.
    o2, lse2 = qsa.forward(plan, q, k, v)
    dq2, _, _ = qsa.backward(plan, q, k, v, o2, lse2, do)
    plan.device_status()
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.forward(f64(qb), f64(kb), f64(vb), routes_np, 0.0625)
    dq_ref, _, _ = oracle.backward(f64(qb), f64(kb), f64(vb), routes_np, f64(dob), 0.0625,
                                   keys=np.zeros(0, np.int64))
    assert_close("O", o2.float().cpu().numpy().astype(np.float64), o_ref)
    assert_lse_close(lse2.cpu().numpy().astype(np.float64), lse_ref)
    assert_close("dQ", dq2.float().cpu().numpy().astype(np.float64), dq_ref)

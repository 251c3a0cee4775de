"""qsa_forward_no_alloc: preprocessing + forward without any device allocation.

It exists for callers that cannot allocate device memory while they run (code
inside a framework that owns all device memory, such as an inference engine
plugin's enqueue, or a latency-critical loop that cannot take an allocation's
implicit synchronisation).  Its scratch is a fixed 32 MiB device array inside
libqsa.  This test calls it through the C ABI twice in a row on different
problems, so the second call runs on the array the first one left behind, and
checks both against the allocating qsa_preprocess + qsa_forward path at the
parity tolerances.  It also checks that an oversize problem is refused before
any device work.  It sits in its own file so pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

from route_sparse_gqa_gb300 import _abi
from route_sparse_gqa_gb300 import workloads as W
from tests.qsa_testlib import assert_close, assert_lse_close, bf16_to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build()
    return _abi.load()


def _inputs(index_or_seed):
    if index_or_seed == 0:
        c = W.make_case(0)
        return c.q, c.k, c.v, c.routes, c.workload.softmax_scale
    rng = np.random.default_rng(index_or_seed)
    B, S_q, S_kv, Hq, Hkv, K = 2, 75, 333, 16, 2, 90  # ragged last tile, int64 routes with huge values
    q = W.bf16_normal(rng, (B, S_q, Hq, 256))
    k = W.bf16_normal(rng, (B, S_kv, Hkv, 256))
    v = W.bf16_normal(rng, (B, S_kv, Hkv, 256))
    r = rng.integers(-3, S_kv + 3, size=(B, S_q, K)).astype(np.int64)
    r[rng.random(r.shape) < 0.05] = 2**41 + 7
    r[rng.random((B, S_q)) < 0.1] = -1
    return q, k, v, r, 0.07


def test_no_alloc_forward_matches_allocating_path(lib):
    import torch

    import route_sparse_gqa_gb300 as qsa

    dev = torch.device("cuda:0")
    for case in (0, 12345):  # two calls in a row on the shared scratch
        qb, kb, vb, routes_np, scale = _inputs(case)
        q, k, v = (bf16_to_device(x, dev) for x in (qb, kb, vb))
        routes = torch.from_numpy(routes_np).to(dev)
        plan = qsa.preprocess(q, k, v, routes, scale)
        o_ref, lse_ref = qsa.forward(plan, q, k, v)

        p = plan.problem
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        stream = torch.cuda.current_stream(dev).cuda_stream
        _abi.check(lib.qsa_forward_no_alloc(ctypes.byref(p), routes.data_ptr(), q.data_ptr(), k.data_ptr(),
                                            v.data_ptr(), o.data_ptr(), lse.data_ptr(), stream))
        torch.cuda.synchronize()
        assert_close("O", o.float().cpu().numpy().astype(np.float64), o_ref.float().cpu().numpy().astype(np.float64))
        assert_lse_close(lse.cpu().numpy().astype(np.float64), lse_ref.cpu().numpy().astype(np.float64))


def test_no_alloc_rejects_oversize_problem(lib):
    p = _abi.Problem()
    p.B, p.S_q, p.S_kv, p.Hq, p.Hkv, p.D, p.K = 1, 32768, 32768, 32, 4, 256, 2048
    p.route_bits, p.softmax_scale = 32, 0.0625
    for f, (S, H) in (("q_stride", (32768, 32)), ("k_stride", (32768, 4)), ("v_stride", (32768, 4))):
        arr = getattr(p, f)
        arr[0], arr[1], arr[2], arr[3] = S * H * 256, H * 256, 256, 1
    p.r_stride[0], p.r_stride[1], p.r_stride[2] = 32768 * 2048, 2048, 1
    st = lib.qsa_forward_no_alloc(ctypes.byref(p), None, None, None, None, None, None, None)
    assert st == 2  # QSA_ERR_UNSUPPORTED
    assert b"32 MiB" in lib.qsa_last_error()

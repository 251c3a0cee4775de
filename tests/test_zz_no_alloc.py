"""qsa_forward_no_alloc: preprocessing + forward without any device allocation.

It exists for callers that cannot allocate device memory while they run (code
inside a framework that owns all device memory, such as an inference engine
plugin's enqueue, or a latency-critical loop that cannot take an allocation's
implicit synchronisation).  Its scratch is a fixed 32 MiB device array inside
libqsa.  These tests call it through the C ABI on several problems in a row, so
later calls run on the array earlier ones left behind, and check each call
against the fp64 oracle and against the allocating qsa_preprocess +
qsa_forward path at the parity tolerances; they cover the tile kernels (G = 8),
the warp-level kernels (G = 3) and a ragged problem with int64 routes.  They
also check that a warm call leaves the device's free memory unchanged, that a
device-side failure of a call is reported by qsa_read_no_alloc_status, and that
an oversize problem is refused before any device work.  This file sits last in
pytest's collection order.
"""
import ctypes

import numpy as np
import pytest

import oracle
from route_sparse_gqa_gb300 import _abi
from route_sparse_gqa_gb300 import workloads as W
from tests.qsa_testlib import assert_close, assert_lse_close, bf16_to_device, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build()
    return _abi.load()


def _inputs(kind):
    if kind == "tiny":
        c = W.make_case(0)
        return c.q, c.k, c.v, c.routes, c.workload.softmax_scale
    rng = np.random.default_rng(12345 if kind == "ragged" else 777)
    if kind == "ragged":  # G = 8, ragged last tile, int64 routes with huge values
        B, S_q, S_kv, Hq, Hkv, K = 2, 75, 333, 16, 2, 90
    else:  # G = 3: the warp-level kernels on the same array
        B, S_q, S_kv, Hq, Hkv, K = 1, 40, 200, 6, 2, 30
    q = W.bf16_normal(rng, (B, S_q, Hq, 256))
    k = W.bf16_normal(rng, (B, S_kv, Hkv, 256))
    v = W.bf16_normal(rng, (B, S_kv, Hkv, 256))
    r = rng.integers(-3, S_kv + 3, size=(B, S_q, K)).astype(np.int64)
    r[rng.random(r.shape) < 0.05] = 2**41 + 7
    r[rng.random((B, S_q)) < 0.1] = -1
    return q, k, v, r, 0.07


def _no_alloc(lib, plan, routes, q, k, v, o, lse):
    import torch

    stream = torch.cuda.current_stream(q.device).cuda_stream
    p = plan.problem
    return lib.qsa_forward_no_alloc(ctypes.byref(p), routes.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                    o.data_ptr(), lse.data_ptr(), stream)


def test_no_alloc_forward_matches_oracle_and_allocating_path(lib):
    import torch

    import route_sparse_gqa_gb300 as qsa

    dev = torch.device("cuda:0")
    for kind in ("tiny", "ragged", "g3", "tiny"):  # calls in a row on the shared array
        qb, kb, vb, routes_np, scale = _inputs(kind)
        q, k, v = (bf16_to_device(x, dev) for x in (qb, kb, vb))
        routes = torch.from_numpy(routes_np).to(dev)
        plan = qsa.preprocess(q, k, v, routes, scale)
        o_ref, lse_ref = qsa.forward(plan, q, k, v)
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        _abi.check(_no_alloc(lib, plan, routes, q, k, v, o, lse))
        _abi.check(lib.qsa_read_no_alloc_status(torch.cuda.current_stream(dev).cuda_stream))
        got_o = o.float().cpu().numpy().astype(np.float64)
        got_lse = lse.cpu().numpy().astype(np.float64)
        assert_close("O vs allocating path", got_o, o_ref.float().cpu().numpy().astype(np.float64))
        assert_lse_close(got_lse, lse_ref.cpu().numpy().astype(np.float64))
        oo, ll = oracle.forward(f64(qb), f64(kb), f64(vb), routes_np, scale)
        assert_close("O vs oracle", got_o, oo)
        assert_lse_close(got_lse, ll)


def test_no_alloc_forward_keymajor_path(lib, monkeypatch):
    """The same on the key-major forward (forced by the test hook) on the static array: reverse lists,
    key norm bound, output pass and final division all in its forward part."""
    import torch

    import route_sparse_gqa_gb300 as qsa

    monkeypatch.setenv("QSA_DEBUG_FORWARD_PATH", "keymajor")
    dev = torch.device("cuda:0")
    qb, kb, vb, routes_np, scale = _inputs("ragged")
    q, k, v = (bf16_to_device(x, dev) for x in (qb, kb, vb))
    routes = torch.from_numpy(routes_np).to(dev)
    plan = qsa.preprocess(q, k, v, routes, scale)
    o = torch.full((q.shape[0], q.shape[1], q.shape[2], q.shape[3]), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((q.shape[0], q.shape[2], q.shape[1]), float("nan"), dtype=torch.float32, device=dev)
    for _ in range(2):
        _abi.check(_no_alloc(lib, plan, routes, q, k, v, o, lse))
        _abi.check(lib.qsa_read_no_alloc_status(torch.cuda.current_stream(dev).cuda_stream))
        oo, ll = oracle.forward(f64(qb), f64(kb), f64(vb), routes_np, scale)
        assert_close("O (key-major, no alloc)", o.float().cpu().numpy().astype(np.float64), oo)
        assert_lse_close(lse.cpu().numpy().astype(np.float64), ll)


def test_no_alloc_call_allocates_nothing(lib):
    import torch

    import route_sparse_gqa_gb300 as qsa

    dev = torch.device("cuda:0")
    qb, kb, vb, routes_np, scale = _inputs("ragged")
    q, k, v = (bf16_to_device(x, dev) for x in (qb, kb, vb))
    routes = torch.from_numpy(routes_np).to(dev)
    plan = qsa.preprocess(q, k, v, routes, scale)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((q.shape[0], q.shape[2], q.shape[1]), dtype=torch.float32, device=dev)
    _abi.check(_no_alloc(lib, plan, routes, q, k, v, o, lse))  # warm: kernels loaded, limits set
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    for _ in range(3):
        _abi.check(_no_alloc(lib, plan, routes, q, k, v, o, lse))
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"


def test_no_alloc_reports_device_failures(lib, monkeypatch):
    """A bounded wait made to run out (the QSA_DEBUG_WAIT_LIMIT_NS=0 test hook, read at launch) is
    reported by qsa_read_no_alloc_status, and the next call on the same context is correct again."""
    import torch

    import route_sparse_gqa_gb300 as qsa

    dev = torch.device("cuda:0")
    qb, kb, vb, routes_np, scale = _inputs("ragged")
    q, k, v = (bf16_to_device(x, dev) for x in (qb, kb, vb))
    routes = torch.from_numpy(routes_np).to(dev)
    plan = qsa.preprocess(q, k, v, routes, scale)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((q.shape[0], q.shape[2], q.shape[1]), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    monkeypatch.setenv("QSA_DEBUG_WAIT_LIMIT_NS", "0")
    _abi.check(_no_alloc(lib, plan, routes, q, k, v, o, lse))
    assert lib.qsa_read_no_alloc_status(stream) == 5  # QSA_ERR_TIMEOUT
    monkeypatch.delenv("QSA_DEBUG_WAIT_LIMIT_NS")
    _abi.check(_no_alloc(lib, plan, routes, q, k, v, o, lse))
    _abi.check(lib.qsa_read_no_alloc_status(stream))
    oo, ll = oracle.forward(f64(qb), f64(kb), f64(vb), routes_np, scale)
    assert_close("O after a reported failure", o.float().cpu().numpy().astype(np.float64), oo)
    assert_lse_close(lse.cpu().numpy().astype(np.float64), ll)


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

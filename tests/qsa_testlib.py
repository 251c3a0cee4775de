"""Helpers shared by the parity tests: move workload bytes to the GPU, run the
library through its binding, and compare with the fp64 oracle at the stated
tolerances (|gpu - ref| <= 2e-2 |ref| + 2e-2 for O, dQ, dK, dV; LSE within 1e-3
absolute, -inf exactly where the oracle has -inf; route sets bit-exact)."""
from __future__ import annotations

import numpy as np

from route_sparse_gqa_gb300 import workloads as W

RTOL = 2e-2
ATOL = 2e-2
LSE_ATOL = 1e-3


def bf16_to_device(bits: np.ndarray, device):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def f64(bits: np.ndarray) -> np.ndarray:
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def run_library(case_q, case_k, case_v, case_do, routes_np, scale, device="cuda:0", fp32_dkdv=False,
                transform=None, deterministic=False):
    """Runs preprocess, forward and backward; returns numpy outputs (float64 /
    int32) and the plan.  ``transform`` may rewrap the device tensors (to test
    strided inputs)."""
    import torch

    import route_sparse_gqa_gb300 as qsa

    dev = torch.device(device)
    q, k, v, do = (bf16_to_device(x, dev) for x in (case_q, case_k, case_v, case_do))
    routes = torch.from_numpy(np.ascontiguousarray(routes_np)).to(dev)
    if transform is not None:
        q, k, v, routes = transform(q, k, v, routes)
    plan = qsa.preprocess(q, k, v, routes, scale)
    o, lse = qsa.forward(plan, q, k, v)
    res = qsa.backward(plan, q, k, v, o, lse, do, fp32_dkdv=fp32_dkdv, deterministic=deterministic)
    ids, counts = plan.route_sets()
    plan.device_status()
    torch.cuda.synchronize()
    out = {
        "o": o.float().cpu().numpy().astype(np.float64),
        "lse": lse.cpu().numpy().astype(np.float64),
        "dq": res[0].float().cpu().numpy().astype(np.float64),
        "dk": res[1].float().cpu().numpy().astype(np.float64),
        "dv": res[2].float().cpu().numpy().astype(np.float64),
        "ids": ids.cpu().numpy(),
        "counts": counts.cpu().numpy(),
    }
    if fp32_dkdv:
        out["dk32"] = res[3].cpu().numpy().astype(np.float64)
        out["dv32"] = res[4].cpu().numpy().astype(np.float64)
    return out


def assert_close(name: str, got: np.ndarray, ref: np.ndarray, rtol=RTOL, atol=ATOL):
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    err = np.abs(got - ref)
    bad = err > rtol * np.abs(ref) + atol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{name}: {bad.sum()} of {bad.size} elements outside |d| <= {rtol}|ref| + {atol}; "
                             f"first {idx.tolist()}: got {got[bad][:5]} ref {ref[bad][:5]}; "
                             f"max err {err.max():.4g}")


def assert_lse_close(got: np.ndarray, ref: np.ndarray):
    assert got.shape == ref.shape
    ninf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), ninf), "-inf LSE entries differ"
    fin = ~ninf
    if fin.any():
        err = np.abs(got[fin] - ref[fin])
        assert err.max() <= LSE_ATOL, f"LSE max abs err {err.max():.3g} > {LSE_ATOL}"

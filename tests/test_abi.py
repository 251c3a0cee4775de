"""The C-ABI library builds, loads without a GPU, exports every symbol include/qsa.h
declares, and rejects bad problems with the documented status codes before any
device work (CPU only)."""
import ctypes
import math
import os
import re
import subprocess

import pytest

from route_sparse_gqa_gb300 import _abi, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "qsa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _abi.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"QSA_API\s+[\w\s\*]*?\b(qsa_\w+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_symbols() == sorted(_abi.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _abi.LIB_PATH], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\bT\s+(qsa_\w+)$", out.stdout, re.M))
    for name in declared_symbols():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_header_compiles_as_c():
    src = f'#include "{HEADER}"\nint main(void) {{ qsa_problem p; (void)p; return (int)QSA_OK; }}\n'
    r = subprocess.run(["gcc", "-x", "c", "-std=c99", "-fsyntax-only", "-I/usr/local/cuda/include", "-"],
                       input=src, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def good_problem(**kw):
    p = _abi.Problem()
    B, S_q, S_kv, Hq, Hkv, D, K = 2, 100, 300, 16, 2, 256, 50
    p.B, p.S_q, p.S_kv, p.Hq, p.Hkv, p.D, p.K = B, S_q, S_kv, Hq, Hkv, D, K
    p.route_bits = 32
    p.softmax_scale = 1.0 / 16
    for f, (S, H) in (("q_stride", (S_q, Hq)), ("k_stride", (S_kv, Hkv)), ("v_stride", (S_kv, Hkv))):
        arr = getattr(p, f)
        arr[0], arr[1], arr[2], arr[3] = S * H * D, H * D, D, 1
    p.r_stride[0], p.r_stride[1], p.r_stride[2] = S_q * K, K, 1
    for k, v in kw.items():
        if k.endswith("_stride"):
            arr = getattr(p, k)
            for i, x in enumerate(v):
                arr[i] = x
        else:
            setattr(p, k, v)
    return p


@pytest.mark.parametrize("kw,status", [
    ({}, 0),
    ({"B": 0}, 1),
    ({"K": 0}, 1),
    ({"S_kv": -3}, 1),
    ({"Hq": 15}, 1),
    ({"softmax_scale": 0.0}, 1),
    ({"softmax_scale": -1.0}, 1),
    ({"softmax_scale": math.inf}, 1),
    ({"softmax_scale": math.nan}, 1),
    ({"route_bits": 16}, 1),
    ({"D": 128}, 2),
    ({"S_kv": 2**31}, 2),
    ({"K": 16385}, 2),
    ({"q_stride": (100 * 16 * 256, 16 * 256, 256, 2)}, 2),
    ({"k_stride": (300 * 2 * 256, 2 * 256, 260, 1)}, 2),
])
def test_problem_validation(lib, kw, status):
    p = good_problem(**kw)
    got = lib.qsa_check_problem(ctypes.byref(p))
    assert got == status, lib.qsa_last_error()
    n = lib.qsa_workspace_bytes(ctypes.byref(p))
    assert (n > 0) == (status == 0)
    if status:
        assert lib.qsa_last_error().decode()


def test_workspace_size_covers_int64_sized_problems(lib):
    # B*S_q*S_kv = 2^32 (context-parallel shape): sizes are computed in 64 bits.
    p = good_problem(B=1, S_q=32768, S_kv=131072, K=2048,
                     q_stride=(32768 * 16 * 256, 16 * 256, 256, 1),
                     k_stride=(131072 * 2 * 256, 2 * 256, 256, 1), v_stride=(131072 * 2 * 256, 2 * 256, 256, 1),
                     r_stride=(32768 * 2048, 2048, 1))
    n = lib.qsa_workspace_bytes(ctypes.byref(p))
    assert n > 32768 * 2048 * 4  # at least the sorted route rows
    assert n < 8 * 2**30


def test_host_side_errors_need_no_device(lib):
    p = good_problem()
    assert lib.qsa_preprocess(ctypes.byref(p), None, None, 0, None) == 1  # null workspace
    assert lib.qsa_forward(ctypes.byref(p), ctypes.c_void_p(256), 0, None, None, None, None, None, None) == 3
    assert lib.qsa_forward(ctypes.byref(p), ctypes.c_void_p(257), 1 << 40, None, None, None, None, None, None) == 1
    for code in range(7):
        assert lib.qsa_status_string(code).decode().startswith("QSA_")


def test_binding_fails_loudly_without_gpu_tensors(lib):
    import torch

    import route_sparse_gqa_gb300 as qsa

    q = torch.zeros(1, 4, 2, 256, dtype=torch.bfloat16)
    k = torch.zeros(1, 4, 1, 256, dtype=torch.bfloat16)
    r = torch.zeros(1, 4, 3, dtype=torch.int32)
    with pytest.raises(qsa.QSAError, match="CUDA tensor"):
        qsa.qsa_attention(q, k, k, r)

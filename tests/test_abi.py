"""The C-ABI library builds, loads without a GPU, exports every symbol
include/qsa.h and include/qsa_route.h declare, and rejects bad problems with the
documented status codes before any device work (CPU only)."""
import ctypes
import glob
import math
import os
import re
import subprocess

import pytest

from route_sparse_gqa_gb300 import _abi, build

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADER = os.path.join(INCLUDE, "qsa.h")
HEADERS = sorted(glob.glob(os.path.join(INCLUDE, "*.h")))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _abi.load()


def declared_symbols():
    text = "".join(open(h).read() for h in HEADERS)
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
    src = (f'#include "{HEADER}"\n#include "{os.path.join(INCLUDE, "qsa_route.h")}"\n'
           'int main(void) { qsa_problem p; qsa_route_problem r; (void)p; (void)r; return (int)QSA_OK; }\n')
    r = subprocess.run(["gcc", "-x", "c", "-std=c99", "-fsyntax-only", "-I/usr/local/cuda/include", "-"],
                       input=src, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_problem_struct_layout_matches_the_header(tmp_path):
    """The binding's ctypes structs have the C structs' sizes and field offsets."""
    fields = [f for f, _ in _abi.Problem._fields_]
    src = (f'#include <stdio.h>\n#include <stddef.h>\n#include "{HEADER}"\nint main(void) {{\n'
           '  printf("%zu", sizeof(qsa_problem));\n' +
           "".join(f'  printf(" %zu", offsetof(qsa_problem, {f}));\n' for f in fields) + '  return 0;\n}\n')
    exe = tmp_path / "layout"
    r = subprocess.run(["gcc", "-x", "c", "-std=c99", "-I/usr/local/cuda/include", "-o", str(exe), "-"],
                       input=src, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert got[0] == ctypes.sizeof(_abi.Problem)
    assert got[1:] == [getattr(_abi.Problem, f).offset for f in fields]


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
    ({"flags": 1}, 0),
    ({"flags": 2}, 0),
    ({"flags": 3}, 0),
    ({"flags": 4}, 1),
    ({"D": 128, "q_stride": (100 * 16 * 128, 16 * 128, 128, 1), "k_stride": (300 * 2 * 128, 2 * 128, 128, 1),
      "v_stride": (300 * 2 * 128, 2 * 128, 128, 1)}, 0),
    ({"D": 96}, 2),
    ({"D": 512}, 2),
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


def good_route_problem(**kw):
    p = _abi.RouteProblem()
    B, S_q, H, D, c = 2, 100, 32, 128, 4
    p.B, p.S_q, p.H_index, p.D_index, p.n_blocks = B, S_q, H, D, S_q // c
    p.token_budget, p.compress_ratio, p.query_position_offset = 64, c, 0
    p.q_stride[0], p.q_stride[1], p.q_stride[2], p.q_stride[3] = S_q * H * D, H * D, D, 1
    p.k_stride[0], p.k_stride[1], p.k_stride[2] = (S_q // c) * D, D, 1
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
    ({"H_index": 1}, 0),
    ({"H_index": 128, "D_index": 64}, 0),
    ({"token_budget": 0}, 0),
    ({"n_blocks": 0, "S_q": 3}, 0),
    ({"query_position_offset": 3}, 0),     # positions up to 102 < 25 * 4 + 3
    ({"query_position_offset": 4}, 1),     # position 103 lies past the global sequence
    ({"B": 0}, 1),
    ({"compress_ratio": 0}, 1),
    ({"token_budget": -1}, 1),
    ({"query_position_offset": -1}, 1),
    ({"H_index": 24}, 2),
    ({"H_index": 256}, 2),
    ({"D_index": 256}, 2),
    ({"D_index": 96}, 2),
    ({"n_blocks": 600_000_000}, 2),         # token IDs past int32
    ({"q_stride": (100 * 32 * 128, 32 * 128, 128, 2)}, 2),
    ({"k_stride": (25 * 128, 132, 1)}, 2),
])
def test_route_problem_validation(lib, kw, status):
    p = good_route_problem(**kw)
    got = lib.qsa_route_check_problem(ctypes.byref(p))
    assert got == status, lib.qsa_last_error()
    n = lib.qsa_route_workspace_bytes(ctypes.byref(p))
    assert (n > 0) == (status == 0)
    w = lib.qsa_route_width(ctypes.byref(p))
    assert w == (p.token_budget + p.compress_ratio - 1 if status == 0 else 0)
    if status == 0:
        assert n >= 512 + p.B * p.S_q * p.n_blocks * 4


def test_route_host_side_errors_need_no_device(lib):
    p = good_route_problem()
    assert lib.qsa_select_token_ids(ctypes.byref(p), None, None, None, None, 0, None, None) == 1  # null tensors
    one = ctypes.c_void_p(1 << 20)
    assert lib.qsa_select_token_ids(ctypes.byref(p), one, one, one, ctypes.c_void_p(256), 0, one, None) == 3
    assert lib.qsa_index_scores(ctypes.byref(p), one, one, one, ctypes.c_void_p(257), 1 << 30, one, None) == 1
    assert lib.qsa_select_from_scores(ctypes.byref(p), one, one, None, 512, one, None) == 1  # null workspace

"""fp64 CPU oracle for route-set sparse GQA attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it and fails loudly when its own extension is
missing; there is no CPU fallback.

The arithmetic lives in ``qsa_oracle.c`` (plain C, every sum in double).  This
module only compiles that file with gcc and marshals numpy arrays to it.  It is
independent of the CUDA path: no shared code, headers or helpers.

Functions follow the NeMo-AutoModel Qwen3.8-Flash-Next pages:

* :func:`route_sets` -- fa4_qsa ``_preprocess`` (duplicates collapse; invalid
  IDs, large int64 included, are discarded before indexing) and flex_qsa
  ``_routes_to_membership`` (negative / out-of-range entries are padding).
* :func:`forward` -- flex_qsa module docstring ("each query row attends exactly
  to its route IDs"; all -1 rows give zero output), qsa
  ``_gathered_qsa_gqa_attention_chunk`` (grouped queries ``[B,Q,Hkv,G,D]``).
* :func:`backward` -- fa4_qsa ``fa4_sparse_gqa_attention`` (first-order
  gradients; empty rows have zero query gradients) and flex_qsa (zero gradients
  for padding rows).
* :func:`index_scores`, :func:`select_ids`, :func:`select_qsa_token_ids` -- qsa
  ``select_qsa_token_ids`` (compressed-block relu-sum scores, top
  ``token_budget / compress_ratio`` blocks, expansion, causal tail, -1 fill);
  the arithmetic is in ``qsa_select_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsa_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "qsa_select_oracle.c")]
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libqsa_oracle.so")
_lock = threading.Lock()
_lib = None


class _Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("B", "S_q", "S_kv", "Hq", "Hkv", "D", "K")]


class _SelectShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("B", "S_q", "H", "D", "NB", "budget", "c", "offset")]


def build(force: bool = False) -> str:
    """Compile the oracle's C files into ``oracle/_build/libqsa_oracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(f) for f in _SRCS)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", *_SRCS, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p = ctypes.c_void_p
            lib.qsa_oracle_route_sets.argtypes = [ctypes.POINTER(_Shape), p, p, p]
            lib.qsa_oracle_forward.argtypes = [ctypes.POINTER(_Shape), p, p, p, p, ctypes.c_double, p, p]
            lib.qsa_oracle_backward.argtypes = [ctypes.POINTER(_Shape), p, p, p, p, p, ctypes.c_double, p,
                                                ctypes.c_int64, p, p, p]
            lib.qsa_oracle_index_scores.argtypes = [ctypes.POINTER(_SelectShape), p, p, p]
            lib.qsa_oracle_select_ids.argtypes = [ctypes.POINTER(_SelectShape), p, p, p]
            for f in (lib.qsa_oracle_route_sets, lib.qsa_oracle_forward, lib.qsa_oracle_backward,
                      lib.qsa_oracle_index_scores, lib.qsa_oracle_select_ids):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _shape(q, k, routes) -> _Shape:
    B, S_q, Hq, D = q.shape
    Bk, S_kv, Hkv, Dk = k.shape
    Br, S_r, K = routes.shape
    if (Bk, Dk) != (B, D) or (Br, S_r) != (B, S_q):
        raise ValueError(f"shape mismatch: q{q.shape} k{k.shape} routes{routes.shape}")
    return _Shape(B, S_q, S_kv, Hq, Hkv, D, K)


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def route_sets(routes: np.ndarray, S_kv: int):
    """Sorted unique valid IDs per row (int32 ``[B,S_q,K]``, tail -1) and counts ``[B,S_q]``."""
    r = np.ascontiguousarray(routes, dtype=np.int64)
    B, S_q, K = r.shape
    s = _Shape(B, S_q, S_kv, 1, 1, 1, K)
    ids = np.empty((B, S_q, K), np.int32)
    counts = np.empty((B, S_q), np.int32)
    _check(_load().qsa_oracle_route_sets(ctypes.byref(s), _ptr(r), _ptr(ids), _ptr(counts)), "route_sets")
    return ids, counts


def forward(q, k, v, routes, scale: float):
    """O ``[B,S_q,Hq,D]`` and natural-log LSE ``[B,Hq,S_q]`` in float64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    r = np.ascontiguousarray(routes, dtype=np.int64)
    s = _shape(q, k, r)
    o = np.empty(q.shape, np.float64)
    lse = np.empty((s.B, s.Hq, s.S_q), np.float64)
    _check(_load().qsa_oracle_forward(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(_f64(v)), _ptr(r), float(scale),
                                      _ptr(o), _ptr(lse)), "forward")
    return o, lse


def backward(q, k, v, routes, dout, scale: float, keys=None):
    """dQ for every row, and dK/dV for every key (``keys=None``) or for the listed
    flat keys ``b * S_kv + j`` (then shaped ``[n_keys, Hkv, D]``)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    r = np.ascontiguousarray(routes, dtype=np.int64)
    s = _shape(q, k, r)
    dq = np.empty(q.shape, np.float64)
    if keys is None:
        n_keys, kp = -1, None
        dk = np.empty(k.shape, np.float64)
    else:
        kk = np.ascontiguousarray(keys, dtype=np.int64).reshape(-1)
        n_keys, kp = kk.size, _ptr(kk)
        dk = np.empty((kk.size, s.Hkv, s.D), np.float64)
    dv = np.empty_like(dk)
    _check(_load().qsa_oracle_backward(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(r), _ptr(dout),
                                       float(scale), _ptr(dq), n_keys, kp, _ptr(dk), _ptr(dv)), "backward")
    return dq, dk, dv


def route_width(token_budget: int, compress_ratio: int) -> int:
    """Slots per row of the route producer's output: ``token_budget + compress_ratio - 1``."""
    return int(token_budget) + int(compress_ratio) - 1


def index_scores(q, k, compress_ratio: int, offset: int = 0) -> np.ndarray:
    """Block scores ``[B,S_q,NB]`` (float64, -inf where the block is not visible).

    ``q``: index queries ``[B,S_q,H,D]``; ``k``: compressed keys ``[B,NB,D]`` or
    ``[B,NB,1,D]``; ``offset``: global position of local query row zero."""
    q = _f64(q)
    k = _f64(k)
    if k.ndim == 4:
        k = k.reshape(k.shape[0], k.shape[1], k.shape[3])
    B, S_q, H, D = q.shape
    if k.shape[0] != B or k.shape[2] != D:
        raise ValueError(f"shape mismatch: q{q.shape} k{k.shape}")
    NB = k.shape[1]
    s = _SelectShape(B, S_q, H, D, NB, 0, int(compress_ratio), int(offset))
    out = np.empty((B, S_q, NB), np.float64)
    _check(_load().qsa_oracle_index_scores(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(out)), "index_scores")
    return out


def select_ids(scores, sequence_lengths, token_budget: int, compress_ratio: int, offset: int = 0) -> np.ndarray:
    """Route rows int32 ``[B,S_q,token_budget+compress_ratio-1]`` from block scores ``[B,S_q,NB]``.

    Only the visible blocks of each row are read; higher score wins, the lower
    block index breaks ties."""
    sc = _f64(scores)
    B, S_q, NB = sc.shape
    lens = np.ascontiguousarray(sequence_lengths, dtype=np.int64).reshape(-1)
    if lens.size != B:
        raise ValueError("sequence_lengths must have B entries")
    s = _SelectShape(B, S_q, 1, 1, NB, int(token_budget), int(compress_ratio), int(offset))
    ids = np.empty((B, S_q, route_width(token_budget, compress_ratio)), np.int32)
    _check(_load().qsa_oracle_select_ids(ctypes.byref(s), _ptr(sc), _ptr(lens), _ptr(ids)), "select_ids")
    return ids


def select_qsa_token_ids(q, k, sequence_lengths, token_budget: int, compress_ratio: int, offset: int = 0):
    """Scores then selection: the route producer end to end, in fp64."""
    sc = index_scores(q, k, compress_ratio, offset)
    return select_ids(sc, sequence_lengths, token_budget, compress_ratio, offset)


def omp_threads() -> int:
    """Threads OpenMP will use (OMP_NUM_THREADS if set, else the usable cores)."""
    env = os.environ.get("OMP_NUM_THREADS")
    if env:
        return int(env)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1

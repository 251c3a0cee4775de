"""PyTorch binding of libqsa: route-set sparse GQA attention on GB300.

Argument marshalling only -- PyTorch supplies device memory and the current
stream; preprocessing, forward and backward all run in libqsa's CUDA kernels.
There is no CPU path and no fallback: CPU tensors, non-BF16 tensors or an
unbuilt library raise.

The call signature follows ``flex_sparse_gqa_attention`` /
``fa4_sparse_gqa_attention`` on the NeMo-AutoModel Qwen3.8-Flash-Next pages:
``query [B,S_q,Hq,D]``, ``key``/``value [B,S_kv,Hkv,D]`` (BF16, D = 256; also 128, and 64 on the warp-level kernels),
``selected_token_ids [B,S_q,K]`` signed int32/int64 in K/V coordinates (-1 and
out-of-range IDs are padding, duplicates count once), ``softmax_scale``
defaulting to ``1/sqrt(D)``.  The output is an independent BF16 tensor.
"""
from __future__ import annotations

import dataclasses
import math

import torch

from . import _abi
from ._abi import QSAError

_INVALID, _UNSUPPORTED = 1, 2


def _stream_handle(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _attn_operand(t: torch.Tensor) -> torch.Tensor:
    # fa4_sparse_gqa_attention: arbitrary strides accepted, non-unit final strides copied.
    if t.stride(-1) != 1 or any(s % 8 for s in t.stride()[:-1]) or t.data_ptr() % 16:
        t = t.contiguous()
    return t


def _check_inputs(query, key, value, routes):
    for name, t in (("query", query), ("key", key), ("value", value), ("selected_token_ids", routes)):
        if not isinstance(t, torch.Tensor):
            raise QSAError(_INVALID, f"{name} must be a tensor")
        if not t.is_cuda:
            raise QSAError(_UNSUPPORTED, f"{name} must be a CUDA tensor (there is no CPU path)")
    if query.dim() != 4 or key.dim() != 4 or value.dim() != 4 or routes.dim() != 3:
        raise QSAError(_INVALID, "expected query/key/value [B,S,H,D] and selected_token_ids [B,S_q,K]")
    for name, t in (("query", query), ("key", key), ("value", value)):
        if t.dtype != torch.bfloat16:
            raise QSAError(_UNSUPPORTED, f"{name} must be bfloat16 (got {t.dtype})")
    if routes.dtype not in (torch.int32, torch.int64):
        raise QSAError(_INVALID, f"selected_token_ids must be int32 or int64 (got {routes.dtype})")
    if key.shape != value.shape:
        raise QSAError(_INVALID, f"value shape {tuple(value.shape)} differs from key shape {tuple(key.shape)}")
    B, S_q, Hq, D = query.shape
    if key.shape[0] != B or key.shape[3] != D or routes.shape[0] != B or routes.shape[1] != S_q:
        raise QSAError(_INVALID, f"shape mismatch: query {tuple(query.shape)} key {tuple(key.shape)} "
                                 f"ids {tuple(routes.shape)}")
    if not (query.device == key.device == value.device == routes.device):
        raise QSAError(_INVALID, "all tensors must be on the same device")


def make_problem(query, key, value, routes, softmax_scale, routes_sorted: bool = False,
                 deterministic_forward: bool = False) -> _abi.Problem:
    B, S_q, Hq, D = query.shape
    _, S_kv, Hkv, _ = key.shape
    p = _abi.Problem()
    p.B, p.S_q, p.S_kv, p.Hq, p.Hkv, p.D, p.K = B, S_q, S_kv, Hq, Hkv, D, routes.shape[2]
    p.route_bits = 64 if routes.dtype == torch.int64 else 32
    p.softmax_scale = float(softmax_scale)
    for field, t in (("q_stride", query), ("k_stride", key), ("v_stride", value)):
        arr = getattr(p, field)
        for i, s in enumerate(t.stride()):
            arr[i] = s
    for i, s in enumerate(routes.stride()):
        p.r_stride[i] = s
    p.flags = (_abi.ROUTES_SORTED if routes_sorted else 0) | (_abi.DETERMINISTIC_FORWARD if deterministic_forward else 0)
    return p


def resolve_scale(softmax_scale, D: int) -> float:
    s = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    if not math.isfinite(s) or s <= 0.0:
        raise QSAError(_INVALID, f"softmax_scale must be finite and positive (got {softmax_scale})")
    return s


@dataclasses.dataclass
class RoutePlan:
    """Preprocessed routes (the library's workspace) for one problem.  Reused by
    the forward and backward calls on the same routes."""
    problem: _abi.Problem
    workspace: torch.Tensor

    @property
    def nbytes(self) -> int:
        return self.workspace.numel()

    def route_sets(self):
        """(ids [B,S_q,K] int32 ascending unique valid IDs then -1, counts [B,S_q] int32)."""
        p = self.problem
        dev = self.workspace.device
        ids = torch.empty((p.B, p.S_q, p.K), dtype=torch.int32, device=dev)
        counts = torch.empty((p.B, p.S_q), dtype=torch.int32, device=dev)
        _abi.check(_abi.load().qsa_copy_route_sets(p, self.workspace.data_ptr(), self.nbytes, ids.data_ptr(),
                                                   counts.data_ptr(), _stream_handle(dev)))
        return ids, counts

    def device_status(self) -> None:
        """Synchronises and raises if a kernel reported a timeout or a failed check."""
        _abi.check(_abi.load().qsa_read_device_status(self.workspace.data_ptr(), _stream_handle(self.workspace.device)))


def preprocess(query, key, value, selected_token_ids, softmax_scale=None, routes_sorted: bool = False,
               deterministic_forward: bool = False) -> RoutePlan:
    """Route preprocessing.  routes_sorted: the rows' valid IDs already ascend with invalid slots last (as
    select_qsa_token_ids returns them); rows found so are copied through (the result is the same either way).
    deterministic_forward: the forward's O and LSE bitwise reproducible (the tile kernels run)."""
    _check_inputs(query, key, value, selected_token_ids)
    scale = resolve_scale(softmax_scale, query.shape[-1])
    lib = _abi.load()
    p = make_problem(query, key, value, selected_token_ids, scale, routes_sorted, deterministic_forward)
    _abi.check(lib.qsa_check_problem(p))
    n = lib.qsa_workspace_bytes(p)
    ws = torch.empty(n, dtype=torch.uint8, device=query.device)
    _abi.check(lib.qsa_preprocess(p, selected_token_ids.data_ptr(), ws.data_ptr(), n, _stream_handle(query.device)))
    return RoutePlan(p, ws)


def forward(plan: RoutePlan, query, key, value):
    """Returns (O [B,S_q,Hq,D] bf16, LSE [B,Hq,S_q] fp32)."""
    p = plan.problem
    query, key, value = _attn_operand(query), _attn_operand(key), _attn_operand(value)
    pp = make_problem(query, key, value, _RouteShape(p), p.softmax_scale)
    o = torch.empty((p.B, p.S_q, p.Hq, p.D), dtype=torch.bfloat16, device=query.device)
    lse = torch.empty((p.B, p.Hq, p.S_q), dtype=torch.float32, device=query.device)
    _abi.check(_abi.load().qsa_forward(pp, plan.workspace.data_ptr(), plan.nbytes, query.data_ptr(), key.data_ptr(),
                                       value.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                       _stream_handle(query.device)))
    return o, lse


def backward(plan: RoutePlan, query, key, value, out, lse, grad_out, fp32_dkdv: bool = False,
             deterministic: bool = False):
    """Returns (dQ, dK, dV) in bf16, plus the fp32 dK/dV sums when fp32_dkdv.

    ``deterministic`` selects the bitwise reproducible backward (dK/dV summed as
    fixed-point integers, ``qsa_backward_deterministic``)."""
    p = plan.problem
    query, key, value = _attn_operand(query), _attn_operand(key), _attn_operand(value)
    pp = make_problem(query, key, value, _RouteShape(p), p.softmax_scale)
    out = out.contiguous()
    grad_out = grad_out.to(torch.bfloat16).contiguous()
    lse = lse.contiguous()
    dev = query.device
    dq = torch.empty((p.B, p.S_q, p.Hq, p.D), dtype=torch.bfloat16, device=dev)
    dk = torch.empty((p.B, p.S_kv, p.Hkv, p.D), dtype=torch.bfloat16, device=dev)
    dv = torch.empty_like(dk)
    dk32 = dv32 = None
    if fp32_dkdv:
        dk32 = torch.empty((p.B, p.S_kv, p.Hkv, p.D), dtype=torch.float32, device=dev)
        dv32 = torch.empty_like(dk32)
    lib = _abi.load()
    entry = lib.qsa_backward_deterministic if deterministic else lib.qsa_backward
    _abi.check(entry(
        pp, plan.workspace.data_ptr(), plan.nbytes, query.data_ptr(), key.data_ptr(), value.data_ptr(),
        out.data_ptr(), lse.data_ptr(), grad_out.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
        dk32.data_ptr() if dk32 is not None else None, dv32.data_ptr() if dv32 is not None else None,
        _stream_handle(dev)))
    if fp32_dkdv:
        return dq, dk, dv, dk32, dv32
    return dq, dk, dv


class _RouteShape:
    """Stands in for the routes tensor when rebuilding a problem from a plan."""

    def __init__(self, p: _abi.Problem):
        self.shape = (p.B, p.S_q, p.K)
        self.dtype = torch.int64 if p.route_bits == 64 else torch.int32
        self._stride = tuple(p.r_stride)

    def stride(self):
        return self._stride


class _QSAFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, query, key, value, routes, softmax_scale, deterministic):
        plan = preprocess(query, key, value, routes, softmax_scale, deterministic_forward=deterministic)
        o, lse = forward(plan, query, key, value)
        ctx.save_for_backward(query, key, value, o, lse)
        ctx.plan = plan
        ctx.deterministic = deterministic
        return o

    @staticmethod
    def backward(ctx, grad_out):
        query, key, value, o, lse = ctx.saved_tensors
        dq, dk, dv = backward(ctx.plan, query, key, value, o, lse, grad_out, deterministic=ctx.deterministic)
        return dq, dk, dv, None, None, None


def qsa_attention(query, key, value, selected_token_ids, softmax_scale=None, deterministic: bool = False):
    """Exact route-set sparse GQA attention; differentiable in query/key/value
    (first order).  Returns BF16 ``[B,S_q,Hq,D]``.  ``deterministic`` makes the
    forward and the backward bitwise reproducible."""
    return _QSAFunction.apply(query, key, value, selected_token_ids, softmax_scale, deterministic)


def qsa_attention_with_lse(query, key, value, selected_token_ids, softmax_scale=None):
    """Forward only: (O bf16 [B,S_q,Hq,D], LSE fp32 [B,Hq,S_q] natural log, RoutePlan)."""
    plan = preprocess(query, key, value, selected_token_ids, softmax_scale)
    o, lse = forward(plan, query, key, value)
    return o, lse, plan

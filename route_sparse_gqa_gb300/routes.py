"""PyTorch binding of libqsa's route producer (include/qsa_route.h).

``select_qsa_token_ids`` follows the NeMo-AutoModel Qwen3.8-Flash-Next qsa
page: ``index_queries [B,S_query,H_index,D_index]`` and ``compressed_keys
[B,floor(S_global/compress_ratio),1,D_index]`` (BF16), ``sequence_lengths [B]``
(right padding), ``token_budget`` and ``compress_ratio``.  It returns int32
global token IDs ``[B,S_query,token_budget+compress_ratio-1]``: the best
``token_budget // compress_ratio`` visible blocks expanded to tokens, then the
incomplete causal tail, then -1 -- ascending within each row, so the result is
already the sorted route set ``qsa_attention`` consumes.

Argument marshalling only: scoring and selection run in libqsa's CUDA kernels;
CPU tensors or an unbuilt library raise.
"""
from __future__ import annotations

import ctypes

import torch

from . import _abi
from ._abi import QSAError

_INVALID, _UNSUPPORTED = 1, 2


def _stream_handle(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _operand(t: torch.Tensor) -> torch.Tensor:
    if t.stride(-1) != 1 or any(s % 8 for s in t.stride()[:-1]) or t.data_ptr() % 16:
        t = t.contiguous()
    return t


def _problem(index_queries, compressed_keys, token_budget, compress_ratio, query_position_offset,
             global_sequence_length):
    for name, t in (("index_queries", index_queries), ("compressed_keys", compressed_keys)):
        if not isinstance(t, torch.Tensor):
            raise QSAError(_INVALID, f"{name} must be a tensor")
        if not t.is_cuda:
            raise QSAError(_UNSUPPORTED, f"{name} must be a CUDA tensor (there is no CPU path)")
        if t.dtype != torch.bfloat16:
            raise QSAError(_UNSUPPORTED, f"{name} must be bfloat16 (got {t.dtype})")
    if index_queries.dim() != 4:
        raise QSAError(_INVALID, "index_queries must be [B, S_query, H_index, D_index]")
    if compressed_keys.dim() == 4:
        if compressed_keys.shape[2] != 1:
            raise QSAError(_INVALID, "compressed_keys must have one head: [B, blocks, 1, D_index]")
        compressed_keys = compressed_keys[:, :, 0]
    if compressed_keys.dim() != 3:
        raise QSAError(_INVALID, "compressed_keys must be [B, blocks, 1, D_index] or [B, blocks, D_index]")
    B, S_q, H, D = index_queries.shape
    if compressed_keys.shape[0] != B or compressed_keys.shape[2] != D:
        raise QSAError(_INVALID, f"shape mismatch: index_queries {tuple(index_queries.shape)} "
                                 f"compressed_keys {tuple(compressed_keys.shape)}")
    n_blocks = compressed_keys.shape[1]
    if global_sequence_length is not None and int(global_sequence_length) // int(compress_ratio) != n_blocks:
        raise QSAError(_INVALID, f"compressed_keys has {n_blocks} blocks, expected "
                                 f"floor({global_sequence_length} / {compress_ratio})")
    q = _operand(index_queries)
    k = _operand(compressed_keys)
    p = _abi.RouteProblem()
    p.B, p.S_q, p.H_index, p.D_index, p.n_blocks = B, S_q, H, D, n_blocks
    p.token_budget, p.compress_ratio = int(token_budget), int(compress_ratio)
    p.query_position_offset = int(query_position_offset)
    for i, s in enumerate(q.stride()):
        p.q_stride[i] = s
    for i, s in enumerate(k.stride()):
        p.k_stride[i] = s
    _abi.check(_abi.load().qsa_route_check_problem(ctypes.byref(p)))
    return p, q, k


def _lengths(sequence_lengths, B, device):
    if not isinstance(sequence_lengths, torch.Tensor):
        sequence_lengths = torch.as_tensor(sequence_lengths)
    lens = sequence_lengths.to(device=device, dtype=torch.int64).reshape(-1).contiguous()
    if lens.numel() != B:
        raise QSAError(_INVALID, f"sequence_lengths has {lens.numel()} entries, expected {B}")
    return lens


def _workspace(p, device, full: bool) -> torch.Tensor:
    n = _abi.load().qsa_route_workspace_bytes(ctypes.byref(p)) if full else 512
    return torch.empty(n, dtype=torch.uint8, device=device)


def select_qsa_token_ids(index_queries, compressed_keys, sequence_lengths, token_budget: int, compress_ratio: int,
                         query_chunk_size: int | None = None, query_position_offset: int = 0,
                         global_sequence_length: int | None = None) -> torch.Tensor:
    """Route rows int32 ``[B, S_query, token_budget + compress_ratio - 1]``.

    ``query_chunk_size`` splits the query rows into separate library calls
    (bounding the fp32 score workspace to ``rows x blocks``); the result does
    not depend on it.  ``None`` scores every row in one call."""
    p, q, k = _problem(index_queries, compressed_keys, token_budget, compress_ratio, query_position_offset,
                       global_sequence_length)
    dev = q.device
    lens = _lengths(sequence_lengths, p.B, dev)
    W = p.token_budget + p.compress_ratio - 1
    ids = torch.empty((p.B, p.S_q, W), dtype=torch.int32, device=dev)
    lib = _abi.load()
    stream = _stream_handle(dev)
    S_q = p.S_q
    chunk = S_q if query_chunk_size is None else max(1, min(int(query_chunk_size), S_q))
    if chunk == S_q:
        ws = _workspace(p, dev, True)
        _abi.check(lib.qsa_select_token_ids(ctypes.byref(p), q.data_ptr(), k.data_ptr(), lens.data_ptr(),
                                            ws.data_ptr(), ws.numel(), ids.data_ptr(), stream))
        return ids
    # Chunks are separate batch-strided calls: rows [r0, r1) of every batch row.
    out = torch.empty((p.B, chunk, W), dtype=torch.int32, device=dev)
    ws = None
    for r0 in range(0, S_q, chunk):
        rows = min(chunk, S_q - r0)
        pc, qc, kc = _problem(q[:, r0:r0 + rows], k, token_budget, compress_ratio,
                              int(query_position_offset) + r0, global_sequence_length)
        need = lib.qsa_route_workspace_bytes(ctypes.byref(pc))
        if ws is None or ws.numel() < need:
            ws = torch.empty(need, dtype=torch.uint8, device=dev)
        _abi.check(lib.qsa_select_token_ids(ctypes.byref(pc), qc.data_ptr(), kc.data_ptr(), lens.data_ptr(),
                                            ws.data_ptr(), ws.numel(), out.data_ptr(), stream))
        ids[:, r0:r0 + rows].copy_(out.view(-1)[:p.B * rows * W].view(p.B, rows, W))
    return ids


def index_scores(index_queries, compressed_keys, sequence_lengths, compress_ratio: int,
                 query_position_offset: int = 0) -> torch.Tensor:
    """Block scores fp32 ``[B, S_query, blocks]`` (sum over heads of relu(q . k) / sqrt(D)).

    Entries of blocks a row cannot see, and of padding rows, are NaN."""
    p, q, k = _problem(index_queries, compressed_keys, 0, compress_ratio, query_position_offset, None)
    dev = q.device
    lens = _lengths(sequence_lengths, p.B, dev)
    scores = torch.full((p.B, p.S_q, p.n_blocks), float("nan"), dtype=torch.float32, device=dev)
    ws = _workspace(p, dev, False)
    _abi.check(_abi.load().qsa_index_scores(ctypes.byref(p), q.data_ptr(), k.data_ptr(), lens.data_ptr(),
                                            ws.data_ptr(), ws.numel(), scores.data_ptr(), _stream_handle(dev)))
    return scores


def select_from_scores(scores, sequence_lengths, token_budget: int, compress_ratio: int,
                       query_position_offset: int = 0) -> torch.Tensor:
    """Route rows from fp32 block scores ``[B, S_query, blocks]`` (selection and expansion only)."""
    if not isinstance(scores, torch.Tensor) or not scores.is_cuda or scores.dtype != torch.float32:
        raise QSAError(_UNSUPPORTED, "scores must be a float32 CUDA tensor (there is no CPU path)")
    if scores.dim() != 3:
        raise QSAError(_INVALID, "scores must be [B, S_query, blocks]")
    sc = scores.contiguous()
    B, S_q, NB = sc.shape
    p = _abi.RouteProblem()
    p.B, p.S_q, p.H_index, p.D_index, p.n_blocks = B, S_q, 1, 64, NB
    p.token_budget, p.compress_ratio = int(token_budget), int(compress_ratio)
    p.query_position_offset = int(query_position_offset)
    p.q_stride[0], p.q_stride[1], p.q_stride[2], p.q_stride[3] = S_q * 64, 64, 64, 1
    p.k_stride[0], p.k_stride[1], p.k_stride[2] = NB * 64, 64, 1
    lib = _abi.load()
    _abi.check(lib.qsa_route_check_problem(ctypes.byref(p)))
    dev = sc.device
    lens = _lengths(sequence_lengths, B, dev)
    ids = torch.empty((B, S_q, p.token_budget + p.compress_ratio - 1), dtype=torch.int32, device=dev)
    ws = _workspace(p, dev, False)
    _abi.check(lib.qsa_select_from_scores(ctypes.byref(p), sc.data_ptr(), lens.data_ptr(), ws.data_ptr(),
                                          ws.numel(), ids.data_ptr(), _stream_handle(dev)))
    return ids

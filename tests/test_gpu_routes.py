"""GPU parity of the route producer (qsa page, select_qsa_token_ids) against the
fp64 CPU oracle on the same seeded inputs.

* Selection from given fp32 scores is integer work decided on fp32 values, so
  both sides decide on the same fp32 numbers (the oracle reads them widened
  exactly to fp64) and the route rows must match bit for bit, ties included.
* Scores: |gpu - ref| <= 2^-17 A + 1e-6 |ref| per entry, A = sum_h sum_d
  |q_hd k_d| / sqrt(D).  Products of BF16 inputs are exact in fp32; 2^-17
  covers the fp32 accumulation of D <= 128 terms (at most D ulps of the
  magnitude sum, 2^-24 each) with room for the tensor core's summation order;
  1e-6 |ref| covers the fp32 relu-sum over heads and the final scaling.
* End to end (scores then selection on the GPU): where the fp64 scores leave
  no doubt the rows are unique; elsewhere several rows are correct.  Every row
  must have the exact structure (chosen blocks whole and ascending, the causal
  tail, -1 fill, padding rows), and the chosen blocks must be a valid top-k of
  the fp64 scores: no unchosen block may beat a chosen one by more than twice
  the score tolerance.
"""
import numpy as np
import pytest

import oracle
from route_sparse_gqa_gb300 import workloads as W
from tests.qsa_testlib import bf16_to_device, f64

pytestmark = pytest.mark.gpu

EPS_ACC = 2.0 ** -17
EPS_REL = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def _dev():
    import torch

    return torch.device("cuda:0")


def _score_tol(qd, kd, ref):
    """Per-entry tolerance [B, S_q, NB] of the fp32 scores (module docstring)."""
    B, S_q, H, D = qd.shape
    kk = np.abs(kd.reshape(kd.shape[0], kd.shape[1], kd.shape[-1]))
    a = np.empty(ref.shape, np.float64)
    for b in range(B):
        for r0 in range(0, S_q, 256):
            r1 = min(S_q, r0 + 256)
            m = np.abs(qd[b, r0:r1]).reshape(-1, D) @ kk[b].T
            a[b, r0:r1] = m.reshape(r1 - r0, H, -1).sum(1)
    a /= np.sqrt(D)
    fin = np.where(np.isfinite(ref), np.abs(ref), 0.0)
    return EPS_ACC * a + EPS_REL * fin + 1e-30


def _row_structure(ids, lens, budget, c, offset, NB):
    """Vectorised checks that hold at any size: count, ascending IDs, tail, -1 fill, padding."""
    B, S_q, W_ = ids.shape
    assert W_ == budget + c - 1
    t = np.arange(S_q)[None, :] + offset
    tg = np.broadcast_to(t, (B, S_q))
    live = tg < np.asarray(lens)[:, None]
    nvis = np.minimum((tg + 1) // c, NB)
    n_best = budget // c
    want = np.where(live, np.minimum(nvis, n_best) * c + (tg + 1 - nvis * c), 0)
    valid = ids >= 0
    n = valid.sum(-1)
    assert np.array_equal(n, want), "slot counts differ"
    # valid slots first, then -1 only
    pos = np.arange(W_)[None, None, :]
    assert np.array_equal(valid, pos < n[..., None]), "-1 fill is not a suffix"
    assert (ids[~valid] == -1).all()
    inc = (ids[..., 1:] > ids[..., :-1]) | ~valid[..., 1:]
    assert inc.all(), "IDs are not strictly ascending"
    assert (np.where(valid, ids, -1).max(-1) <= tg).all(), "an ID lies in the future"
    # the incomplete causal tail is present: the last (tg + 1 - nvis c) valid IDs are nvis c .. tg
    n_tail = tg + 1 - nvis * c
    for k in range(c - 1):  # tail slot k from the end
        has = live & (n_tail > k)
        idx = np.clip(n - 1 - k, 0, W_ - 1)
        got = np.take_along_axis(ids, idx[..., None], -1)[..., 0]
        assert np.array_equal(got[has], tg[has] - k), "causal tail differs"


def _chosen_blocks(row, nvis, c):
    v = row[(row >= 0) & (row < nvis * c)]
    blocks, counts = np.unique(v // c, return_counts=True)
    assert (counts == c).all(), "a chosen block is not whole"
    return blocks


def _assert_valid_topk(ids, ref, tol, lens, budget, c, offset, rows=None):
    """Chosen blocks form a valid top-k of the fp64 scores; returns the number of
    rows whose chosen set differs from the oracle's."""
    B, S_q, _ = ids.shape
    n_best = budget // c
    NB = ref.shape[-1]
    oracle_ids = oracle.select_ids(ref, lens, budget, c, offset)
    differ = 0
    it = rows if rows is not None else [(b, t) for b in range(B) for t in range(S_q)]
    for b, t in it:
        tg = offset + t
        if tg >= lens[b]:
            continue
        nvis = min((tg + 1) // c, NB)
        if nvis <= n_best:
            assert np.array_equal(ids[b, t], oracle_ids[b, t]), (b, t)
            continue
        got = _chosen_blocks(ids[b, t], nvis, c)
        assert got.size == n_best, (b, t, got.size)
        s = ref[b, t, :nvis]
        chosen = np.zeros(nvis, bool)
        chosen[got] = True
        slack = 2 * tol[b, t, :nvis].max()
        assert s[chosen].min() >= s[~chosen].max() - slack, (b, t, s[chosen].min(), s[~chosen].max(), slack)
        if not np.array_equal(ids[b, t], oracle_ids[b, t]):
            differ += 1
    return differ


def _run_fused(case, chunk=None):
    import torch

    import route_sparse_gqa_gb300 as qsa

    w = case.workload
    dev = _dev()
    q = bf16_to_device(case.q, dev)
    k = bf16_to_device(case.k, dev)
    lens = torch.from_numpy(case.lengths).to(dev)
    ids = qsa.select_qsa_token_ids(q, k, lens, w.budget, w.c, query_chunk_size=chunk, query_position_offset=w.offset,
                                   global_sequence_length=w.S_global)
    torch.cuda.synchronize()
    return ids.cpu().numpy()


def _gpu_scores(case):
    import torch

    import route_sparse_gqa_gb300 as qsa

    w = case.workload
    dev = _dev()
    sc = qsa.index_scores(bf16_to_device(case.q, dev), bf16_to_device(case.k, dev),
                          torch.from_numpy(case.lengths).to(dev), w.c, w.offset)
    torch.cuda.synchronize()
    return sc.cpu().numpy().astype(np.float64)


# ------------------------------------------------------------ scores ----

@pytest.mark.parametrize("index", [0, 1])
def test_index_scores_match_oracle(index):
    case = W.make_index_case(index)
    w = case.workload
    qd, kd = f64(case.q), f64(case.k)
    ref = oracle.index_scores(qd, kd, w.c, w.offset)
    got = _gpu_scores(case)
    tol = _score_tol(qd, kd, ref)
    tg = np.arange(w.S_q)[None, :, None] + w.offset
    live = (tg < case.lengths[:, None, None]) & (np.arange(w.n_blocks)[None, None, :] < (tg + 1) // w.c)
    assert np.isfinite(got[live]).all()
    assert np.isnan(got[~live]).all(), "entries outside the visible blocks of live rows were written"
    err = np.abs(got - ref)[live]
    bad = err > tol[live]
    assert not bad.any(), f"{bad.sum()} scores outside tolerance; max err/tol {(err / tol[live]).max():.3g}"


# --------------------------------------------------------- selection ----

def _quantised_scores(rng, B, S_q, NB, step):
    """fp32 scores with many exact ties (values on a grid), some -0.0 and +0.0."""
    x = np.round(rng.standard_normal((B, S_q, NB)).astype(np.float32) / step) * np.float32(step)
    z = x == 0
    x[z] = np.where(rng.random(z.sum()) < 0.5, np.float32(0.0), np.float32(-0.0))
    return x.astype(np.float32)


@pytest.mark.parametrize("B,S_q,c,budget,offset,lens,S_global,step", [
    (2, 777, 4, 64, 0, (777, 500), 777, 0.25),
    (1, 300, 1, 5, 0, (300,), 300, 1.0),
    (2, 200, 7, 20, 100, (300, 250), 300, 0.5),
    (1, 64, 4, 2048, 32704, (32768,), 32768, 1e-3),    # full-size rows: 8176+ visible blocks, 512 chosen
    (1, 64, 4, 2048, 32704, (32768,), 32768, 8.0),     # most scores tie at 0: thousands of keys share one bin
    (1, 32, 4, 2048, 79968, (80000,), 80000, 1e-3),    # 20000 visible blocks: rows walked in chunks
    (1, 32, 4, 16384, 79968, (80000,), 80000, 8.0),    # 4096 chosen, ties, a row too wide to stage
    (1, 50, 4, 3, 0, (50,), 50, 0.5),                  # budget < c: only the causal tails
    (1, 40, 4, 16, 0, (0,), 40, 0.5),                  # every row padding
])
def test_select_from_scores_bit_exact(B, S_q, c, budget, offset, lens, S_global, step):
    import torch

    import route_sparse_gqa_gb300 as qsa

    rng = np.random.default_rng(S_q * 31 + c)
    NB = S_global // c
    sc = _quantised_scores(rng, B, S_q, NB, step)
    want = oracle.select_ids(sc.astype(np.float64), np.asarray(lens), budget, c, offset)
    dev = _dev()
    got = qsa.select_from_scores(torch.from_numpy(sc).to(dev), torch.tensor(lens, dtype=torch.int64, device=dev),
                                 budget, c, offset)
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    assert got.dtype == np.int32
    mism = np.argwhere((got != want).any(-1))
    assert mism.size == 0, f"{len(mism)} rows differ, first {mism[:3].tolist()}"


def test_select_from_scores_all_ties_takes_lowest_blocks():
    import torch

    import route_sparse_gqa_gb300 as qsa

    S, c, budget = 400, 4, 40
    sc = np.zeros((1, S, S // c), np.float32)
    got = qsa.select_from_scores(torch.from_numpy(sc).to(_dev()), torch.tensor([S], device=_dev()), budget, c)
    got = got.cpu().numpy()
    row = got[0, S - 1]
    assert list(row[:budget]) == list(range(budget)) and (row[budget:] == -1).all()


# ----------------------------------------------------------- end to end ----

@pytest.mark.parametrize("index", [0, 1])
def test_select_token_ids_valid_against_oracle(index):
    case = W.make_index_case(index)
    w = case.workload
    ids = _run_fused(case)
    _row_structure(ids, case.lengths, w.budget, w.c, w.offset, w.n_blocks)
    qd, kd = f64(case.q), f64(case.k)
    ref = oracle.index_scores(qd, kd, w.c, w.offset)
    tol = _score_tol(qd, kd, ref)
    differ = _assert_valid_topk(ids, ref, tol, case.lengths, w.budget, w.c, w.offset)
    live = sum(min(w.S_q, max(0, int(L) - w.offset)) for L in case.lengths)
    assert differ <= max(2, live // 100), f"{differ} of {live} rows differ from the oracle's choice"


def test_query_chunks_do_not_change_the_result():
    case = W.make_index_case(1)
    a = _run_fused(case)
    b = _run_fused(case, chunk=1000)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("B,S_q,H,D,c,budget,offset,lens,S_global", [
    (1, 37, 1, 64, 3, 7, 0, (37,), 37),          # H = 1: 256 queries per item, 12 blocks (< one tile)
    (2, 300, 128, 128, 4, 32, 0, (300, 131), 300),  # H = 128: two queries per item
    (1, 513, 16, 64, 2, 100, 0, (513,), 513),     # ragged last item and block tile
    (2, 100, 8, 128, 4, 16, 200, (260, 150), 300),  # CP shard: padding inside, and a whole row of padding
    (1, 3, 8, 64, 4, 16, 0, (3,), 3),             # no complete block anywhere
])
def test_select_token_ids_edge_shapes(B, S_q, H, D, c, budget, offset, lens, S_global):
    import torch

    import route_sparse_gqa_gb300 as qsa

    rng = W.rng_for(0, seed=B * 1000 + S_q + H)
    NB = S_global // c
    qb = W.bf16_normal(rng, (B, S_q, H, D))
    kb = W.bf16_normal(rng, (B, NB, 1, D))
    dev = _dev()
    ids = qsa.select_qsa_token_ids(bf16_to_device(qb, dev), bf16_to_device(kb, dev),
                                   torch.tensor(lens, dtype=torch.int64, device=dev), budget, c,
                                   query_position_offset=offset, global_sequence_length=S_global)
    torch.cuda.synchronize()
    ids = ids.cpu().numpy()
    _row_structure(ids, lens, budget, c, offset, NB)
    qd, kd = f64(qb), f64(kb)
    ref = oracle.index_scores(qd, kd, c, offset)
    _assert_valid_topk(ids, ref, _score_tol(qd, kd, ref), np.asarray(lens), budget, c, offset)


def test_rows_are_already_route_sets():
    """The producer's rows pass through the attention preprocessing unchanged (with the rows-sorted flag the
    preprocessing copies them through)."""
    import torch

    import route_sparse_gqa_gb300 as qsa

    case = W.make_index_case(0)
    w = case.workload
    ids = _run_fused(case)
    dev = _dev()
    routes = torch.from_numpy(ids).to(dev)
    B, S, Hq, Hkv, D = w.B, w.S_q, 8, 1, 256
    q = torch.zeros(B, S, Hq, D, dtype=torch.bfloat16, device=dev)
    kv = torch.zeros(B, S, Hkv, D, dtype=torch.bfloat16, device=dev)
    plan = qsa.preprocess(q, kv, kv, routes, routes_sorted=True)
    sets, counts = plan.route_sets()
    torch.cuda.synchronize()
    assert np.array_equal(sets.cpu().numpy(), ids)
    assert np.array_equal(counts.cpu().numpy(), (ids >= 0).sum(-1))


# ------------------------------------------------------------ full size ----

def _sampled_rows_against_oracle(index, extra):
    case = W.make_index_case(index)
    w = case.workload
    ids = _run_fused(case)
    _row_structure(ids, case.lengths, w.budget, w.c, w.offset, w.n_blocks)
    rng = np.random.default_rng(7)
    sample = sorted(set([t for t in extra if 0 <= t < w.S_q] + [w.S_q - 1] + rng.integers(0, w.S_q, 40).tolist()))
    qd, kd = f64(case.q[:, sample]), f64(case.k)
    for j, t in enumerate(sample):
        ref = oracle.index_scores(qd[:, j:j + 1], kd, w.c, w.offset + t)
        tol = _score_tol(qd[:, j:j + 1], kd, ref)
        _assert_valid_topk(ids[:, t:t + 1], ref, tol, case.lengths, w.budget, w.c, w.offset + t)


def test_full_size_train_step_sampled_rows():
    """B1 S32768 H32 D128 c4 budget2048, launched as the benchmark does: every
    row's structure, and sampled rows against the oracle (scored one row at a
    time through query_position_offset), including the first sparse rows."""
    _sampled_rows_against_oracle(3, [2046, 2047, 2048, 2050, 2051, 2052, 4095])


def test_cp_shard_sampled_rows():
    """Local rows at global offset 24576 against 8192 global blocks."""
    _sampled_rows_against_oracle(2, [0, 1, 8191])


def test_forced_wait_timeout_in_the_score_kernel_is_reported():
    """The score kernel bounds every pipeline wait; the host-side hook
    QSA_DEBUG_WAIT_LIMIT_NS=0 makes them run out at once.  The call must report
    QSA_ERR_TIMEOUT through the workspace status word, and the next normal call
    in the same context must be right."""
    import ctypes
    import os

    import torch

    import route_sparse_gqa_gb300 as qsa
    from route_sparse_gqa_gb300 import _abi

    case = W.make_index_case(0)
    w = case.workload
    dev = _dev()
    q, k = bf16_to_device(case.q, dev), bf16_to_device(case.k, dev)
    lens = torch.from_numpy(case.lengths).to(dev)
    p, qq, kk = qsa.routes._problem(q, k, w.budget, w.c, w.offset, w.S_global)
    lib = _abi.load()
    n = lib.qsa_route_workspace_bytes(ctypes.byref(p))
    ws = torch.full((n,), 0x5A, dtype=torch.uint8, device=dev)  # uninitialised-looking workspace
    ids = torch.empty((w.B, w.S_q, w.budget + w.c - 1), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    os.environ["QSA_DEBUG_WAIT_LIMIT_NS"] = "0"
    try:
        _abi.check(lib.qsa_select_token_ids(ctypes.byref(p), qq.data_ptr(), kk.data_ptr(), lens.data_ptr(),
                                            ws.data_ptr(), n, ids.data_ptr(), stream))
    finally:
        del os.environ["QSA_DEBUG_WAIT_LIMIT_NS"]
    st = lib.qsa_read_device_status(ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(stream))
    assert st == 5, st  # QSA_ERR_TIMEOUT
    assert lib.qsa_read_device_status(ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(stream)) == 0
    # A normal call afterwards, on the same workspace, is right.
    _abi.check(lib.qsa_select_token_ids(ctypes.byref(p), qq.data_ptr(), kk.data_ptr(), lens.data_ptr(),
                                        ws.data_ptr(), n, ids.data_ptr(), stream))
    assert lib.qsa_read_device_status(ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(stream)) == 0
    torch.cuda.synchronize()
    got = ids.cpu().numpy()
    _row_structure(got, case.lengths, w.budget, w.c, w.offset, w.n_blocks)
    qd, kd = f64(case.q), f64(case.k)
    ref = oracle.index_scores(qd, kd, w.c, w.offset)
    _assert_valid_topk(got, ref, _score_tol(qd, kd, ref), case.lengths, w.budget, w.c, w.offset)


def test_strided_index_queries_from_a_fused_projection():
    """The indexer's fused projection yields [B, S, (H + 1) * D]; the queries are a
    strided view of its first H heads.  The producer takes the view as it is and
    returns exactly what it returns for a contiguous copy."""
    import torch

    import route_sparse_gqa_gb300 as qsa

    rng = W.rng_for(0, seed=99)
    B, S, H, D, c, budget = 2, 700, 16, 64, 4, 96
    fused = W.bf16_normal(rng, (B, S, (H + 1) * D))
    kb = W.bf16_normal(rng, (B, S // c, 1, D))
    dev = _dev()
    f = bf16_to_device(fused, dev)
    q_view = f.view(B, S, H + 1, D)[:, :, :H]
    assert not q_view.is_contiguous()
    k = bf16_to_device(kb, dev)
    lens = torch.tensor([S, 555], dtype=torch.int64, device=dev)
    a = qsa.select_qsa_token_ids(q_view, k, lens, budget, c)
    b = qsa.select_qsa_token_ids(q_view.contiguous(), k, lens, budget, c)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    ids = a.cpu().numpy()
    _row_structure(ids, [S, 555], budget, c, 0, S // c)
    qd = f64(np.ascontiguousarray(fused.reshape(B, S, H + 1, D)[:, :, :H]))
    kd = f64(kb)
    ref = oracle.index_scores(qd, kd, c)
    _assert_valid_topk(ids, ref, _score_tol(qd, kd, ref), np.array([S, 555]), budget, c, 0)

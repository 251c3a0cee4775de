"""The seeded workload recipes produce the layouts they claim (CPU only)."""
import numpy as np
import pytest

import oracle
from route_sparse_gqa_gb300 import workloads as W


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-9, -2.5, 3.0e38, 1e-40], np.float32)
    bits = W.bf16_bits_from_f32(x)
    back = W.bf16_bits_to_f32(bits)
    assert back[0] == 1.0
    assert back[1] == 1.0  # exactly halfway, rounds to the even mantissa
    assert back[2] == 1.0 + 2**-7  # 1.5 ulp rounds up
    assert back[3] == -2.5
    assert np.all(np.abs(back - x) <= np.abs(x) * 2**-8 + 1e-38)


def test_generation_is_deterministic():
    a = W.make_case(0)
    b = W.make_case(0)
    for n in ("routes", "q", "k", "v", "do"):
        assert np.array_equal(getattr(a, n), getattr(b, n))


def test_tiny_causal_rows():
    w = W.WORKLOADS[0]
    r = W.make_routes(w, W.rng_for(0))
    assert r.dtype == np.int32 and r.shape == (1, 256, 32)
    ids, counts = oracle.route_sets(r, w.S_kv)
    assert np.all(counts[0, 240:] == 0) and np.all(r[0, 240:] == -1)
    assert np.all(counts[0, :240] > 0)
    assert (r >= w.S_kv).sum() > 0  # out-of-range IDs present
    for i in range(240):  # causal: every valid ID is <= q
        assert ids[0, i, counts[0, i] - 1] <= i
    dup_rows = sum(len(set(x for x in r[0, i] if 0 <= x < 256)) < ((r[0, i] >= 0) & (r[0, i] < 256)).sum()
                   for i in range(240))
    assert dup_rows > 10


def test_right_padded_blocks():
    w = W.WORKLOADS[1]
    r = W.make_routes(w, W.rng_for(1))
    assert r.dtype == np.int32 and r.shape == (2, 4096, 2048)
    assert np.all(r[1, 3000:] == -1)
    ids, counts = oracle.route_sets(r, w.S_kv)
    q = np.arange(4096)
    assert np.all(counts[0] > 0) and np.all(counts[1, :3000] > 0)
    last = np.take_along_axis(ids[0], (counts[0] - 1)[:, None].astype(np.int64), 1)[:, 0]
    assert np.all(last == q)  # the local block always reaches the query itself
    blocks = np.where(ids[0] >= 0, ids[0] // 64, -1)
    nblk = np.array([len(np.unique(b[b >= 0])) for b in blocks[::97]])
    assert np.all(nblk == np.minimum(q[::97] // 64 + 1, 32))


def test_packed_thd_has_pad_segment_and_large_ids():
    w = W.WORKLOADS[2]
    r = W.make_routes(w, W.rng_for(2))
    assert r.dtype == np.int64
    assert (r >= 2**40).sum() > 0.005 * (r >= 0).sum()
    _, counts = oracle.route_sets(r, w.S_kv)
    empty = np.nonzero(counts[0] == 0)[0]
    assert empty.size > 0 and empty[-1] == w.S_q - 1  # the pack tail is a padding segment
    assert np.all(np.diff(empty) == 1)


@pytest.mark.parametrize("index", [3, 4])
def test_long_rows(index):
    w = W.WORKLOADS[index]
    r = W.make_routes(w, W.rng_for(index))
    assert r.shape == (w.B, w.S_q, w.K)
    ids, counts = oracle.route_sets(r, w.S_kv)
    assert np.all(counts > 0) and counts.max() == w.K
    offset = 98304 if index == 3 else 0
    q = np.arange(w.S_q) + offset
    last = np.take_along_axis(ids[0], (counts[0] - 1)[:, None].astype(np.int64), 1)[:, 0]
    assert np.all(last == q)
    if index == 3:
        assert w.B * w.S_q * w.S_kv == 2**32


def test_index_workloads_shapes_and_seeding():
    c0 = W.make_index_case(0)
    c1 = W.make_index_case(0)
    w = c0.workload
    assert c0.q.shape == (w.B, w.S_q, w.H, w.D) and c0.k.shape == (w.B, w.n_blocks, 1, w.D)
    assert np.array_equal(c0.q, c1.q) and np.array_equal(c0.k, c1.k)
    assert list(c0.lengths) == list(w.lengths)
    for iw in W.INDEX_WORKLOADS:  # every local position lies inside the global sequence
        assert iw.offset + iw.S_q <= iw.n_blocks * iw.c + iw.c - 1
        assert max(iw.lengths) <= iw.S_global


def test_bench_route_work_counts_visible_pairs():
    import bench

    w = W.IndexWorkload(9, "t", 2, 37, 60, 20, 4, 64, 3, 6, (50, 30), "t")
    pairs, flop, rows = bench.route_work(w, w.lengths)
    want = 0
    for L in w.lengths:
        for t in range(w.S_q):
            tg = w.offset + t
            if tg < L:
                want += min((tg + 1) // w.c, w.n_blocks)
    assert pairs == want and flop == 2 * w.H * w.D * want
    assert rows == min(w.S_q, 50 - 20) + min(w.S_q, 30 - 20)

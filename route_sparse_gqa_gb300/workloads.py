"""Seeded synthetic workloads for route-set sparse GQA attention.

This module only makes inputs: BF16 tensors drawn from N(0, 1) and int32/int64
route tensors shaped like the layouts the Qwen3.8-Flash-Next pages describe
(right-padded batches, packed THD rows with a padding segment, and
context-parallel local queries against a long gathered K/V).  It holds none of
the attention arithmetic; both the CUDA path and the CPU oracle read exactly the
bytes produced here.

Route recipes (each ID list is built in "generation order": the query's own
64-token block first, then the sampled blocks in the order they were drawn):

* ``tiny-causal-rows`` -- B1 S256 Hq4 Hkv1 D256, int32 K=32.  Query q < 240
  draws min(32, q+1) distinct IDs uniformly from [0, q]; the last 16 queries are
  all -1.  Then each slot of a non-empty row independently becomes, with
  probability 5 %, a copy of one of that row's valid IDs, or with probability
  2 %, an out-of-range ID in [256, 2^31 - 1); finally each row's slots are
  shuffled.
* ``right-padded-blocks`` -- B2 S4096 Hq16 Hkv2, int32 K=2048.  Query q (block
  j = q // 64) takes block j plus min(31, j) distinct blocks drawn uniformly from
  [0, j), expands them to token IDs and keeps IDs <= q.  Sequence 1 has logical
  length 3000: its queries q >= 3000 are all -1.
* ``packed-thd`` -- B1 S16384 Hq16 Hkv2, int64 K=2048.  Document lengths are
  drawn uniformly from [512, 4096] while they still fit; the rest of the row is
  one padding segment with all -1 routes.  Blocks are document-relative and
  causal as above.  Then each slot of a non-empty row becomes, with probability
  10 %, a duplicate of a valid ID of the row, or with probability 1 %, an int64
  value drawn from [2^40, 2^62); rows are shuffled.
* ``cp-long-kv`` -- B1 S_q32768 S_kv131072 Hq16 Hkv2, int64 K=2048.  Local
  query q sits at global position p = 98304 + q; routes are block p // 64 plus 31
  distinct earlier blocks, in global coordinates, keeping IDs <= p.
* ``train-step`` -- B1 S32768 Hq32 Hkv4, int32 K=2048.  Block j plus min(47, j)
  distinct earlier blocks, IDs <= q, truncated to the first 2048 IDs.
* ``right-padded-d128`` (D = 128) and ``right-padded-mha`` (Hq = Hkv = 16):
  variants off the pages' D = 256, G = 8 shapes, with the right-padded-blocks
  route recipe.

Random numbers: ``numpy.random.Generator(PCG64(20261202 + index))``; routes are
drawn first, then Q, K, V and dO, each ``standard_normal(float32)`` rounded to
bfloat16 (round to nearest even).

Route-producer inputs (``INDEX_WORKLOADS``, ``make_index_case``): index queries
``[B,S_q,H,D]`` and compressed keys ``[B,NB,1,D]`` drawn from N(0, 1) and
rounded to bfloat16 (the states the page's indexer feeds the selection are
RMS-normalised and rotated, so unit-variance entries have their scale), plus
right-padded logical lengths.  Generator ``PCG64(20261302 + index)``: queries
first, then keys.
"""
from __future__ import annotations

import dataclasses

import numpy as np

BLOCK = 64
SEED_BASE = 20261202


@dataclasses.dataclass(frozen=True)
class Workload:
    index: int
    name: str
    B: int
    S_q: int
    S_kv: int
    Hq: int
    Hkv: int
    D: int
    K: int
    route_dtype: type
    softmax_scale: float
    summary: str


WORKLOADS = (
    Workload(0, "tiny-causal-rows", 1, 256, 256, 4, 1, 256, 32, np.int32, 1.0 / 16,
             "B1 S256 Hq4 Hkv1 D256, int32 K=32, 5% duplicate / 2% out-of-range slots, 16 empty rows"),
    Workload(1, "right-padded-blocks", 2, 4096, 4096, 16, 2, 256, 2048, np.int32, 1.0 / 16,
             "B2 S4096 Hq16 Hkv2 D256, int32 K=2048, 32 causal 64-token blocks, seq 1 length 3000"),
    Workload(2, "packed-thd", 1, 16384, 16384, 16, 2, 256, 2048, np.int64, 1.0 / 16,
             "B1 S16384 Hq16 Hkv2 D256, int64 K=2048, documents U[512,4096], pad segment, 10% dup / 1% >=2^40"),
    Workload(3, "cp-long-kv", 1, 32768, 131072, 16, 2, 256, 2048, np.int64, 1.0 / 16,
             "B1 S_q32768 S_kv131072 Hq16 Hkv2 D256, int64 K=2048, global offset 98304"),
    Workload(4, "train-step", 1, 32768, 32768, 32, 4, 256, 2048, np.int32, 1.0 / 16,
             "B1 S32768 Hq32 Hkv4 D256, int32 K=2048, 48 causal blocks clipped to 2048 IDs"),
    # Variants beyond the pages' D = 256, G = 8 (D = 128 on the tile kernels, G = 1 on the warp-level
    # kernels); routes as right-padded-blocks.
    Workload(5, "right-padded-d128", 2, 4096, 4096, 16, 2, 128, 2048, np.int32, 1.0 / 128 ** 0.5,
             "B2 S4096 Hq16 Hkv2 D128, routes as right-padded-blocks"),
    Workload(6, "right-padded-mha", 2, 4096, 4096, 16, 16, 256, 2048, np.int32, 1.0 / 16,
             "B2 S4096 Hq16 Hkv16 (G=1) D256, routes as right-padded-blocks"),
    # A quarter-length train-step (same heads and route recipe, inputs still larger than L2): the size the
    # many-pass counter captures run on.
    Workload(7, "train-step-s8192", 1, 8192, 8192, 32, 4, 256, 2048, np.int32, 1.0 / 16,
             "B1 S8192 Hq32 Hkv4 D256, int32 K=2048, 48 causal blocks clipped to 2048 IDs"),
)

_ROWS_PER_PIECE = 2048


@dataclasses.dataclass(frozen=True)
class IndexWorkload:
    index: int
    name: str
    B: int
    S_q: int
    S_global: int
    offset: int  # global position of local query row 0
    H: int
    D: int
    c: int
    budget: int
    lengths: tuple
    summary: str

    @property
    def n_blocks(self) -> int:
        return self.S_global // self.c


INDEX_WORKLOADS = (
    IndexWorkload(0, "index-small", 2, 1000, 1000, 0, 8, 128, 4, 64, (1000, 777),
                  "B2 S1000 H8 D128 c4 budget64, seq 1 length 777"),
    IndexWorkload(1, "index-right-padded", 2, 4096, 4096, 0, 32, 128, 4, 2048, (4096, 3000),
                  "B2 S4096 H32 D128 c4 budget2048, seq 1 length 3000"),
    IndexWorkload(2, "index-cp-shard", 1, 8192, 32768, 24576, 32, 128, 4, 2048, (32768,),
                  "B1 local S_q8192 at global offset 24576 of S32768, H32 D128 c4 budget2048"),
    IndexWorkload(3, "index-train-step", 1, 32768, 32768, 0, 32, 128, 4, 2048, (32768,),
                  "B1 S32768 H32 D128 c4 budget2048 (8192 blocks, 512 chosen per row)"),
)


@dataclasses.dataclass
class IndexCase:
    workload: IndexWorkload
    q: np.ndarray        # uint16 bf16 bits [B, S_q, H, D]
    k: np.ndarray        # uint16 bf16 bits [B, NB, 1, D]
    lengths: np.ndarray  # int64 [B]


def make_index_case(index: int, seed: int | None = None) -> IndexCase:
    w = INDEX_WORKLOADS[index]
    rng = np.random.Generator(np.random.PCG64(SEED_BASE + 100 + index if seed is None else seed))
    q = bf16_normal(rng, (w.B, w.S_q, w.H, w.D))
    k = bf16_normal(rng, (w.B, w.n_blocks, 1, w.D))
    return IndexCase(w, q, k, np.asarray(w.lengths, dtype=np.int64))


def rng_for(index: int, seed: int | None = None) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(SEED_BASE + index if seed is None else seed))


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_normal(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0, 1) float32 draws rounded to bfloat16 bits, drawn in fixed pieces of
    2^24 values so temporaries stay small."""
    out = np.empty(int(np.prod(shape)), np.uint16)
    piece = 1 << 24
    for s in range(0, out.size, piece):
        n = min(piece, out.size - s)
        out[s:s + n] = bf16_bits_from_f32(rng.standard_normal(n, dtype=np.float32))
    return out.reshape(shape)


def _distinct_draws(rng: np.random.Generator, limit: np.ndarray, n_pick: int) -> np.ndarray:
    """Row i: min(n_pick, limit[i]) distinct integers drawn uniformly from [0, limit[i]),
    in draw order, padded with -1.  Shape [len(limit), n_pick]."""
    n = limit.shape[0]
    out = np.full((n, n_pick), -1, np.int64)
    span = int(limit.max()) if n else 0
    if span == 0 or n_pick == 0:
        return out
    keys = rng.random((n, span))
    keys[np.arange(span)[None, :] >= limit[:, None]] = np.inf
    take = min(n_pick, span)
    idx = np.argpartition(keys, take - 1, axis=1)[:, :take] if take < span else np.tile(np.arange(span), (n, 1))
    ksel = np.take_along_axis(keys, idx, 1)
    order = np.argsort(ksel, axis=1, kind="stable")
    idx = np.take_along_axis(idx, order, 1)
    ksel = np.take_along_axis(ksel, order, 1)
    idx[np.isinf(ksel)] = -1
    out[:, :take] = idx
    return out


def _compact(ids: np.ndarray) -> np.ndarray:
    """Move the non-negative entries of each row to the front, keeping their order."""
    order = np.argsort(ids < 0, axis=1, kind="stable")
    return np.take_along_axis(ids, order, 1)


def _block_routes(rng, pos: np.ndarray, base: np.ndarray, n_other: int, K: int) -> np.ndarray:
    """Causal block routes for queries at (document-relative) positions ``pos``:
    the own block pos // 64 plus up to ``n_other`` distinct earlier blocks, each
    expanded to its 64 token IDs (offset by ``base``), keeping IDs whose relative
    position is <= pos, compacted in generation order and cut to K slots."""
    out = np.full((pos.shape[0], K), -1, np.int64)
    for s in range(0, pos.shape[0], _ROWS_PER_PIECE):
        p = pos[s:s + _ROWS_PER_PIECE]
        j = p // BLOCK
        blocks = np.concatenate([j[:, None], _distinct_draws(rng, j, n_other)], axis=1)
        rel = blocks[:, :, None] * BLOCK + np.arange(BLOCK)[None, None, :]
        ok = (blocks[:, :, None] >= 0) & (rel <= p[:, None, None])
        ids = np.where(ok, rel + base[s:s + _ROWS_PER_PIECE, None, None], -1).reshape(p.shape[0], -1)
        ids = _compact(ids)[:, :K]
        out[s:s + _ROWS_PER_PIECE, :ids.shape[1]] = ids
    return out


def _noise(rng, routes: np.ndarray, p_dup: float, p_bad: float, bad_lo: int, bad_hi: int) -> np.ndarray:
    """Per-slot overwrite of non-empty rows (duplicates of the row's own valid IDs,
    or invalid values), then a per-row shuffle of the slots.  Rows are processed
    in pieces to keep temporaries small."""
    n, K = routes.shape
    out = np.empty_like(routes)
    for s in range(0, n, _ROWS_PER_PIECE):
        r = routes[s:s + _ROWS_PER_PIECE]
        m = r.shape[0]
        counts = (r >= 0).sum(1)
        u = rng.random((m, K))
        nonempty = (counts > 0)[:, None]
        dup = nonempty & (u < p_dup)
        bad = nonempty & (u >= p_dup) & (u < p_dup + p_bad)
        pick = (rng.random((m, K)) * np.maximum(counts, 1)[:, None]).astype(np.int64)
        dup_vals = np.take_along_axis(_compact(r), pick, 1)  # valid IDs sit at the front after compaction
        bad_vals = rng.integers(bad_lo, bad_hi, size=(m, K), dtype=np.int64)
        x = np.where(dup, dup_vals, r)
        x = np.where(bad, bad_vals, x)
        perm = np.argsort(rng.random((m, K)), axis=1)
        out[s:s + _ROWS_PER_PIECE] = np.take_along_axis(x, perm, 1)
    return out


def make_routes(w: Workload, rng: np.random.Generator) -> np.ndarray:
    B, S, K = w.B, w.S_q, w.K
    if w.index == 0:
        q = np.arange(S)
        live = q < S - 16
        draws = _distinct_draws(rng, np.where(live, q + 1, 0), K)
        r = _noise(rng, _compact(draws), 0.05, 0.02, w.S_kv, 2**31 - 1)
        return r.reshape(1, S, K).astype(w.route_dtype)
    if w.index in (1, 5, 6):
        out = np.empty((B, S, K), np.int64)
        for b in range(B):
            pos = np.arange(S)
            r = _block_routes(rng, pos, np.zeros(S, np.int64), 31, K)
            if b == 1:
                r[pos >= 3000] = -1
            out[b] = r
        return out.astype(w.route_dtype)
    if w.index == 2:
        starts, lens, t = [], [], 0
        while True:
            L = int(rng.integers(512, 4097))
            if t + L > S:
                break
            starts.append(t)
            lens.append(L)
            t += L
        base = np.full(S, -1, np.int64)
        for s0, L in zip(starts, lens):
            base[s0:s0 + L] = s0
        in_doc = base >= 0
        pos = np.where(in_doc, np.arange(S) - base, 0)
        r = np.full((S, K), -1, np.int64)
        idx = np.nonzero(in_doc)[0]
        r[idx] = _block_routes(rng, pos[idx], base[idx], 31, K)
        r = _noise(rng, r, 0.10, 0.01, 2**40, 2**62)
        return r.reshape(1, S, K).astype(w.route_dtype)
    if w.index == 3:
        pos = 98304 + np.arange(S)
        r = _block_routes(rng, pos, np.zeros(S, np.int64), 31, K)
        return r.reshape(1, S, K).astype(w.route_dtype)
    if w.index in (4, 7):
        pos = np.arange(S)
        r = _block_routes(rng, pos, np.zeros(S, np.int64), 47, K)
        return r.reshape(1, S, K).astype(w.route_dtype)
    raise ValueError(f"no workload {w.index}")


@dataclasses.dataclass
class Case:
    workload: Workload
    routes: np.ndarray  # int32 or int64 [B, S_q, K]
    q: np.ndarray       # uint16 bf16 bits [B, S_q, Hq, D]
    k: np.ndarray       # uint16 bf16 bits [B, S_kv, Hkv, D]
    v: np.ndarray
    do: np.ndarray      # uint16 bf16 bits [B, S_q, Hq, D]


def make_case(index: int, seed: int | None = None) -> Case:
    w = WORKLOADS[index]
    rng = rng_for(index, seed)
    routes = make_routes(w, rng)
    q = bf16_normal(rng, (w.B, w.S_q, w.Hq, w.D))
    k = bf16_normal(rng, (w.B, w.S_kv, w.Hkv, w.D))
    v = bf16_normal(rng, (w.B, w.S_kv, w.Hkv, w.D))
    do = bf16_normal(rng, (w.B, w.S_q, w.Hq, w.D))
    return Case(w, routes, q, k, v, do)

// qsa_fwd_tc.cu -- tile forward of route-set sparse GQA on tcgen05 tensor cores.
//
// Work item = (KV head g, tile of T = 128/G consecutive query rows of one batch
// row).  Its 128 (query, head) rows -- T queries x the G query heads that read
// KV head g -- form the M = 128 rows of every MMA.  The preprocessing pass gave
// the tile the ascending union of its rows' route sets cut into chunks of 64
// keys, with a 64-bit membership mask per (chunk, query).  For every chunk:
//
//   producer warp   loads the chunk's 64 K rows and 64 V rows of head g into
//                   128-byte-swizzled shared memory: four 64-row TMA tile boxes
//                   when the keys form one contiguous run, otherwise TMA
//                   tile::gather4 (four arbitrary rows per instruction); it also
//                   prefetches the next item's Q tile into L2;
//   MMA warp        S = Q K^T (M=128, N=64, K=256) into TMEM with Q as the A
//                   operand in TMEM, and O += P V (M=128, N=256, K=64) into a
//                   TMEM accumulator with P as the A operand in TMEM -- shared
//                   memory only feeds the B operands (K, V);
//   softmax warps   (4 warps, thread i owns TMEM lane / row i) copy each item's
//                   Q rows from global memory into TMEM, read S, apply the
//                   row's membership bits (read from global memory one chunk
//                   ahead), run the online softmax in fp32 (base-2, scale
//                   folded in, lazy rescale of O when the running max grows by
//                   more than 2^8), write P as BF16 into TMEM over the S buffer
//                   it came from, and finally normalise O, store it as BF16 and
//                   write LSE (natural log).
//
// Every K/V row gathered once into shared memory serves all G heads of the
// group and all T queries of the tile that route to it.  Keys a query does not
// route to get P = 0 exactly, so the result is the exact route-set softmax.
//
// TMEM (512 columns): O 0-255 (fp32), Q 256-383 (bf16 pairs), two S/P buffers
// 384-447 and 448-511.  Shared memory: three-stage K and V rings (192 KiB).
//
// Pipelining: every per-chunk barrier is indexed by the chunk's stage (global
// chunk number mod 3).  A K stage is reused once the S MMA that read it has
// completed (the barrier that tells the softmax warps S is ready), a V stage
// once its PV MMA has (the barrier that tells them O is current); the producer
// loads K of chunk c together with V of chunk c-1.  One thread issues every
// MMA, S two chunks ahead of PV (S0 S1 PV0 S2 PV1 S3 ...), and takes the
// waits for each PV(c), S(c+2) pair back to back: a waiting thread stalls
// until the tensor pipe has taken its queued MMAs, so a wait between the two
// groups would leave the pipe idle.  At the end of an item the softmax warps
// load the next item's Q into TMEM (once the last S has read the current one)
// before the epilogue, so the next item's S MMAs overlap it.  A parity wait
// is unambiguous only if the waited phase is the barrier's open one or the one
// just completed; each wait below states why that holds.  Every wait is
// bounded in time; on timeout the kernel records QSA_ERR_TIMEOUT in the
// workspace status word, all roles wind down, in-flight copies and MMAs drain,
// the TMEM is freed and the kernel returns.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>

#include "qsa_tc.cuh"
#include "qsa_tc_ptx.cuh"
#include "qsa_queue.cuh"

namespace qsa {
namespace {

using namespace ptx;

constexpr int kStages = 3;
constexpr int kThreads = 192;  // warps 0-3 softmax, 4 producer, 5 MMA
constexpr int kMaxPairs = kMaxKVPairs;  // (b, g) tensor-map sets per launch
constexpr uint32_t kNumBars = 5 + 5 * kStages + 2 * kQueueRing;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kPanelBytes = kChunkKeys * 128;  // one 64-column (128-byte-wide) panel of a 64-key chunk

// Shared-memory and TMEM layout for head dim D (256, or 128 for the same tiles
// at half the width).  TMEM: O in columns 0..D-1 (fp32), Q in D..D+D/2-1 (bf16
// pairs), then the two S/P buffers of 64 columns.
template <int D>
struct FwdLayout {
    static constexpr int kPanels = D / 64;
    static constexpr uint32_t kKVBytes = kChunkKeys * D * 2;  // per K or V chunk (32 KiB at D = 256)
    static constexpr uint32_t kOffK = 0;
    static constexpr uint32_t kOffV = kOffK + kStages * kKVBytes;
    static constexpr uint32_t kOffBar = kOffV + kStages * kKVBytes;
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
    static constexpr uint32_t kSmemBytes = kOffMisc + 64 + 1024;  // + alignment slack
    static constexpr uint32_t kTmemO = 0, kTmemQ = D, kTmemSP = D + D / 2;  // S/P buffer b at kTmemSP + 64 b
};
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr float kRescaleThreshold = 8.0f;          // log2 units
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct FwdParams {
    CUtensorMap q_map;  // 4-D {D, Hq, S_q, B}, box {64, G, T, 1}: L2 prefetch of Q tiles
    KVMaps kv[kMaxPairs];  // per (b, g): K/V row-gather and 64-row-run maps
    const __nv_bfloat16 *q;
    int64_t qs0, qs1, qs2;
    int64_t B, S_q, Hq, G, T, n_tiles, max_chunks;
    int64_t g0, n_g;     // KV heads handled by this launch
    int32_t head_major;  // work queue order (qsa_queue.cuh)
    int64_t n_items;   // n_g * B * n_tiles
    float sl2;         // softmax_scale * log2(e)
    uint64_t wait_limit_ns;  // bound of every pipeline wait
    const int32_t *tile_nchunks;
    const int32_t *tile_keys;
    const uint64_t *tile_masks;
    const int32_t *order;
    int32_t *sched;  // work queue counters {next, done}
    __nv_bfloat16 *o;
    float *lse;
    const int32_t *choice;  // null, or 1 when the key-major forward runs instead
    DeviceStatus *status;
};

using Item = QueueItem;

// Stage (ring slot, barrier index) and barrier phase parity of global chunk g.  Chunk numbers of one
// CTA stay far below 2^31, so 32-bit arithmetic (a multiply-high for the division) suffices.
__device__ __forceinline__ int stage_of(int64_t g) { return (int)((uint32_t)g % (uint32_t)kStages); }
__device__ __forceinline__ int64_t round_of(int64_t g) { return (int64_t)((uint32_t)g / (uint32_t)kStages); }

// Per-chunk barriers are indexed by the global chunk number c modulo kStages
// (the K/V stage of chunk c); the S/P TMEM buffer of chunk c is c % 2.
struct Bars {
    uint64_t *q_ready, *q_free, *o_free, *drain;
    uint64_t *item_full, *item_empty;  // work queue ring [kQueueRing]
    uint64_t *k_full, *v_full;  // copies of chunk c landed (TMA transaction bytes)
    uint64_t *s_full;           // S(c) complete: softmax may read it, K stage reusable
    uint64_t *p_full;           // P(c) written by the 128 softmax threads
    uint64_t *o_ready;          // PV(c) complete: V stage reusable, O current up to c
};

template <int D>
__device__ __forceinline__ Bars bars_at(uint8_t *smem) {
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + FwdLayout<D>::kOffBar);
    Bars r;
    r.q_ready = b + 0;
    r.q_free = b + 1;
    r.o_free = b + 2;
    r.drain = b + 3;
    r.k_full = b + 5;
    r.v_full = b + 5 + kStages;
    r.s_full = b + 5 + 2 * kStages;
    r.p_full = b + 5 + 3 * kStages;
    r.o_ready = b + 5 + 4 * kStages;
    r.item_full = b + 5 + 5 * kStages;
    r.item_empty = r.item_full + kQueueRing;
    return r;
}

// Loads the 64 K or V rows of one chunk into a stage: one 64-row tile box per
// 64-column panel when the keys form one contiguous run, else 16 lanes x
// tile::gather4 per panel.
template <int D>
__device__ __forceinline__ void load_chunk_rows(uint32_t dst, const CUtensorMap *run_map, const CUtensorMap *rows_map,
                                                uint64_t *bar, bool run, int first, const int4 &kk, int lane) {
    if (run) {
        if (lane == 0)
            for (int kb = 0; kb < FwdLayout<D>::kPanels; ++kb)
                tma_load_2d(dst + kb * kPanelBytes, run_map, bar, kb * 64, first);
    } else if (lane < 16) {
        for (int kb = 0; kb < FwdLayout<D>::kPanels; ++kb)
            tma_gather4(dst + lane * 512 + kb * kPanelBytes, rows_map, bar, kb * 64, kk.x, kk.y, kk.z, kk.w);
    }
}

// Thread r of the softmax warps copies its Q row (D BF16) into TMEM lane r,
// columns kTmemQ..kTmemQ+D/2-1 (column j holds elements 2j and 2j+1).  Rows
// past S_q get zeros.
template <int D>
__device__ __forceinline__ void load_q_row(const FwdParams &p, const Item &it, int qi, int hl, uint32_t trow) {
    const int64_t q = it.t * p.T + qi;
    const bool live = q < p.S_q;
    const uint4 *src = reinterpret_cast<const uint4 *>(p.q + it.b * p.qs0 + q * p.qs1 + (it.g * p.G + hl) * p.qs2);
#pragma unroll 1
    for (int blk = 0; blk < D / 64; ++blk) {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 v = live ? __ldg(src + blk * 8 + i) : make_uint4(0, 0, 0, 0);
            w[4 * i] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
        tmem_st32(trow + FwdLayout<D>::kTmemQ + blk * 32, w);
    }
    tmem_st_wait();
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) tc_fwd_kernel(const __grid_constant__ FwdParams p) {
    if (p.choice && *p.choice == 1) return;  // uniform over the grid
    using L = FwdLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Bars bar = bars_at<D>(smem);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 8);
    volatile int32_t *ring = reinterpret_cast<volatile int32_t *>(smem + L::kOffMisc + 16);  // [kQueueRing]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);

    if (threadIdx.x == 0) {
        mbar_init(bar.q_ready, 128);
        mbar_init(bar.q_free, 1);
        mbar_init(bar.o_free, 128);
        mbar_init(bar.drain, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar.k_full + s, 1);
            mbar_init(bar.v_full + s, 1);
            mbar_init(bar.s_full + s, 1);
            mbar_init(bar.p_full + s, 128);
            mbar_init(bar.o_ready + s, 1);
        }
        for (int s = 0; s < kQueueRing; ++s) {
            mbar_init(bar.item_full + s, 1);
            mbar_init(bar.item_empty + s, 1 + 128);  // the MMA thread and the softmax threads take every item
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) prefetch_tmap(&p.q_map);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int zero = 0;

    auto fail = [&](unsigned where, unsigned info) {
        raise_status(p.status, QSA_ERR_TIMEOUT, where, info, blockIdx.x);
        *abort_flag = 1;
    };
    auto wait = [&](uint64_t *b, int64_t phase) {
        return mbar_wait_warp(b, (uint32_t)(phase & 1), abort_flag, p.wait_limit_ns);
    };

    if (warp == 4) {
        // ---------------- producer ----------------
        int64_t gc = 0;
        int64_t last_k[kStages], last_v[kStages];
        for (int i = 0; i < kStages; ++i) last_k[i] = last_v[i] = -1;
        Item it;
        bool ok = true;
        for (int64_t i = 0; ok; ++i) {
            int32_t idx = -1;
            if (lane == 0) ok = queue_claim(p.sched, p.n_items, ring, bar.item_full, bar.item_empty, i, abort_flag,
                                            p.wait_limit_ns, idx);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            idx = __shfl_sync(0xffffffffu, idx, 0);
            if (!ok || idx < 0) break;
            queue_decode(p, idx, it);
            if (it.nch == 0) continue;
            // Warm L2 with the item's Q tile; the softmax warps copy it into TMEM a little later.
            if (lane == 0)
                for (int kb = 0; kb < L::kPanels; ++kb)
                    tma_prefetch_4d(&p.q_map, kb * 64, (int)(it.g * p.G), (int)(it.t * p.T), (int)it.b);
            const int pair = (int)(it.b * p.n_g + (it.g - p.g0));
            const KVMaps &maps = p.kv[pair];
            const int32_t *keys = p.tile_keys + it.tile * p.max_chunks * kChunkKeys;
            int4 kk_prev = make_int4(0, 0, 0, 0);
            int first_prev = 0;
            bool run_prev = false;
            for (int c = 0; c <= it.nch; ++c) {
                int4 kk = make_int4(0, 0, 0, 0);
                int first = 0;
                bool run = false;
                if (c < it.nch) {
                    const int64_t gk = gc + c;
                    const int sk = stage_of(gk);
                    if (lane < 16) kk = __ldg(reinterpret_cast<const int4 *>(keys + c * kChunkKeys) + lane);
                    first = __shfl_sync(0xffffffffu, kk.x, 0);
                    const int last = __shfl_sync(0xffffffffu, kk.w, 15);
                    run = last - first == kChunkKeys - 1;  // ascending distinct keys: a contiguous run
                    // The stage is free once S of chunk gk - kStages (which read it) has completed.
                    if (gk >= kStages && !wait(bar.s_full + sk, round_of(gk) - 1)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) mbar_arrive_expect_tx(bar.k_full + sk, L::kKVBytes);
                    __syncwarp();
                    load_chunk_rows<D>(sbase + L::kOffK + sk * L::kKVBytes, &maps.k_run, &maps.k_rows, bar.k_full + sk, run,
                                    first, kk, lane);
                    __syncwarp();
                    last_k[sk] = gk;
                }
                if (c > 0) {
                    const int64_t gv = gc + c - 1;
                    const int sv = stage_of(gv);
                    // ... and once PV of chunk gv - kStages has completed.
                    if (gv >= kStages && !wait(bar.o_ready + sv, round_of(gv) - 1)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) mbar_arrive_expect_tx(bar.v_full + sv, L::kKVBytes);
                    __syncwarp();
                    load_chunk_rows<D>(sbase + L::kOffV + sv * L::kKVBytes, &maps.v_run, &maps.v_rows, bar.v_full + sv, run_prev,
                                    first_prev, kk_prev, lane);
                    __syncwarp();
                    last_v[sv] = gv;
                }
                kk_prev = kk;
                first_prev = first;
                run_prev = run;
            }
            gc += it.nch;
        }
        if (!ok && lane == 0) fail(kSiteTileFwdWait, 1);
        if (lane == 0) queue_finish(p.sched);
        // Drain: every issued copy must have landed before the CTA leaves.
        if (lane == 0) {
            bool drained = true;
            for (int i = 0; i < kStages; ++i) {
                if (last_k[i] >= 0)
                    drained &= mbar_wait(bar.k_full + i, (uint32_t)((last_k[i] / kStages) & 1), &zero, kWaitLimitNs);
                if (last_v[i] >= 0)
                    drained &= mbar_wait(bar.v_full + i, (uint32_t)((last_v[i] / kStages) & 1), &zero, kWaitLimitNs);
            }
            if (!drained) fail(kSiteTileFwdWait, 5);
        }
        __syncwarp();
    } else if (warp == 5) {
        // ---------------- MMA issuer (one thread) ----------------
        // Order per item: S(0), S(1), then PV(c), S(c+2) for each c: S runs two chunks ahead so the
        // softmax warps find S ready when they finish a chunk.  The issuing thread executes no
        // warp-collective instruction and takes all waits for a PV(c), S(c+2) pair together: a
        // wait (any shared-memory access) stalls the thread until its queued MMAs have been taken
        // by the tensor pipe, so one wait per pair keeps that pipe fed.
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16(kTileRows, kChunkKeys, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16(kTileRows, D, false, true);
            auto wait1 = [&](uint64_t *b, int64_t phase) {
                return mbar_wait(b, (uint32_t)(phase & 1), abort_flag, p.wait_limit_ns);
            };
            auto issue_s = [&](int64_t g2, bool last_s) {
                const int s = stage_of(g2), sb = (int)(g2 & 1);
                const uint32_t ka = sbase + L::kOffK + s * L::kKVBytes;
                const uint32_t sp = tmem + L::kTmemSP + sb * kChunkKeys;
#pragma unroll
                for (int kb = 0; kb < L::kPanels; ++kb) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t bd = sdesc_sw128(ka + kb * kPanelBytes + k * 32, 16, 1024);
                        mma_bf16_ts(sp, tmem + L::kTmemQ + (kb * 4 + k) * 8, bd, idesc_qk, (kb | k) ? 1u : 0u);
                    }
                }
                mma_commit(bar.s_full + s);
                if (last_s) mma_commit(bar.q_free);  // the item's Q in TMEM is no longer read
            };
            auto issue_pv = [&](int64_t g2, bool first) {
                const int s = stage_of(g2), sb = (int)(g2 & 1);
                const uint32_t va = sbase + L::kOffV + s * L::kKVBytes;
                const uint32_t pa = tmem + L::kTmemSP + sb * kChunkKeys;
#pragma unroll
                for (int k = 0; k < kChunkKeys / 16; ++k) {
                    const uint64_t bd = sdesc_sw128(va + k * 2048, kPanelBytes, 1024);
                    mma_bf16_ts(tmem + L::kTmemO, pa + k * 8, bd, idesc_pv, (first && k == 0) ? 0u : 1u);
                }
                mma_commit(bar.o_ready + s);
            };
            int64_t gc = 0, qc = 0;
            Item it;
            bool ok = true;
            for (int64_t i = 0; ok; ++i) {
                int32_t idx = -1;
                ok = queue_take(ring, bar.item_full, bar.item_empty, i, abort_flag, p.wait_limit_ns, false, idx);
                if (!ok || idx < 0) break;
                queue_decode(p, idx, it);
                if (it.nch == 0) continue;
                const int n = it.nch;
                ok = wait1(bar.q_ready, qc);
                for (int c = 0; ok && c < n && c < 2; ++c) {
                    ok = wait1(bar.k_full + stage_of(gc + c), round_of(gc + c));
                    tc_fence_after();
                    if (ok) issue_s(gc + c, c == n - 1);
                }
                for (int c = 0; ok && c < n; ++c) {
                    const int64_t g2 = gc + c;
                    // One wait per pair: the softmax warps arrive on p_full(c) only after they have also seen
                    // V(c) and, within the item, K(c+2) land, so this barrier covers every operand of PV(c) and
                    // S(c+2).  (Each barrier wait costs this thread a few hundred cycles once it has MMAs queued.)
                    ok = wait1(bar.p_full + stage_of(g2), round_of(g2)) && (c > 0 || qc == 0 || wait1(bar.o_free, qc - 1));
                    tc_fence_after();
                    if (!ok) break;
                    issue_pv(g2, c == 0);
                    if (c + 2 < n) issue_s(g2 + 2, c + 2 == n - 1);
                }
                gc += n;
                ++qc;
            }
            if (!ok) fail(kSiteTileFwdWait, 3);
            // Drain: all issued MMAs complete before the TMEM is released.
            mma_commit(bar.drain);
            if (!mbar_wait(bar.drain, 0, &zero, kWaitLimitNs)) fail(kSiteTileFwdWait, 6);
        }
        __syncwarp();
    } else {
        // ---------------- softmax / Q loader / epilogue (warps 0-3) ----------------
        const int r = threadIdx.x;  // row of the tile = TMEM lane
        const int qi = (int)(r / p.G), hl = (int)(r % p.G);
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        int64_t gc = 0, qc = 0;
        Item it;
        bool ok = true;
        bool have_q = false;  // Q of the current item is already in TMEM
        int64_t pos = 0;      // ring position of the current item
        int32_t idx = -1;
        ok = queue_take(ring, bar.item_full, bar.item_empty, 0, abort_flag, p.wait_limit_ns, true, idx);
        while (ok && idx >= 0) {
            queue_decode(p, idx, it);
            const int64_t q = it.t * p.T + qi;
            const int64_t h = it.g * p.G + hl;
            const bool live = q < p.S_q;
            __nv_bfloat16 *orow = p.o + ((it.b * p.S_q + q) * p.Hq + h) * D;
            if (it.nch == 0) {
                if (live) {
                    const uint4 z = make_uint4(0, 0, 0, 0);
                    for (int i = 0; i < D / 8; ++i) reinterpret_cast<uint4 *>(orow)[i] = z;
                    p.lse[(it.b * p.Hq + h) * p.S_q + q] = -INFINITY;
                }
                ok = queue_take(ring, bar.item_full, bar.item_empty, ++pos, abort_flag, p.wait_limit_ns, true, idx);
                continue;
            }
            if (!have_q) {  // only for the first non-empty item; later ones are loaded ahead
                load_q_row<D>(p, it, qi, hl, trow);
                tc_fence_before();
                mbar_arrive(bar.q_ready);
            }
            const uint64_t *mrow = p.tile_masks + it.tile * p.max_chunks * p.T + qi;
            uint64_t mask_next = __ldg(mrow);
            float m = -INFINITY, l = 0.f;
            for (int c = 0; c < it.nch; ++c, ++gc) {
                const int sb = (int)(gc & 1), st = stage_of(gc);
                const uint32_t sp = trow + L::kTmemSP + sb * kChunkKeys;
                const uint64_t mask = mask_next;
                if (c + 1 < it.nch) mask_next = __ldg(mrow + (c + 1) * p.T);
                // V(c) and, within the item, K(c+2) must have landed before P(c) is released: the MMA thread
                // waits only for P(c) before issuing PV(c) and S(c+2).  V(c) is in shared memory long before
                // S(c) completes (waited here); K(c+2) can only be loaded once S(c-1) has freed its stage, so
                // it is waited for after the softmax math, just before P(c) is released.  Parity safety: the
                // producer reuses a stage only after the S (K) or PV (V) three chunks back completed, and
                // those need P of chunks this thread has not released yet, so neither barrier can be a
                // phase ahead; and the phase before (three chunks back) completed before S(c-1) did.
                if (!wait(bar.v_full + st, round_of(gc))) {
                    ok = false;
                    break;
                }
                if (!wait(bar.s_full + st, round_of(gc))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sr[2][32];
                tmem_ld32(sp, sr[0]);
                tmem_ld32(sp + 32, sr[1]);
                tmem_ld_wait();
                float x[64];
                float mx = -INFINITY;
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    x[j] = ((mask >> j) & 1ull) ? __uint_as_float(sr[j >> 5][j & 31]) * p.sl2 : -INFINITY;
                    mx = fmaxf(mx, x[j]);
                }
                const bool need = (m != -INFINITY) && (mx > m + kRescaleThreshold);
                if (m == -INFINITY) m = mx;  // first keys of this row: nothing accumulated yet
                if (__any_sync(0xffffffffu, need)) {
                    // Rescale O: the previous chunk's PV must have landed in TMEM first.  S(c) is
                    // complete, so every MMA issued before it is too, among them the PV three chunks
                    // back that completed the previous phase of this barrier: the parity wait below
                    // can only mean PV(c-1), and PV(c+2) cannot complete before P(c+2) exists.
                    if (!wait(bar.o_ready + stage_of(gc - 1), round_of(gc - 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const float alpha = need ? ex2(m - mx) : 1.f;
#pragma unroll 1
                    for (int blk = 0; blk < D / 32; ++blk) {
                        uint32_t o[32];
                        tmem_ld32(trow + L::kTmemO + blk * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(trow + L::kTmemO + blk * 32, o);
                    }
                    tmem_st_wait();
                    if (need) {
                        l *= alpha;
                        m = mx;
                    }
                }
                uint32_t pk[32];
                float lsum = 0.f;
#pragma unroll
                for (int j = 0; j < 64; j += 2) {
                    const float p0 = (m == -INFINITY) ? 0.f : ex2(x[j] - m);
                    const float p1 = (m == -INFINITY) ? 0.f : ex2(x[j + 1] - m);
                    lsum += p0 + p1;
                    pk[j >> 1] = pack_bf16(p0, p1);
                }
                l += lsum;
                tmem_st32(sp, pk);  // P over the first half of the S buffer it came from
                tmem_st_wait();
                if (c + 2 < it.nch && !wait(bar.k_full + stage_of(gc + 2), round_of(gc + 2))) {
                    ok = false;
                    break;
                }
                tc_fence_before();
                mbar_arrive(bar.p_full + st);
            }
            if (!ok) break;
            // Take the next item now and, if it has chunks, load its Q once this item's last S has read
            // the current one, so the MMA thread can start it while this epilogue runs.
            int32_t nidx = -1;
            if (!queue_take(ring, bar.item_full, bar.item_empty, pos + 1, abort_flag, p.wait_limit_ns, true, nidx)) {
                ok = false;
                break;
            }
            have_q = false;
            if (nidx >= 0) {
                Item nx;
                queue_decode(p, nidx, nx);
                if (nx.nch > 0) {
                    if (!wait(bar.q_free, qc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    load_q_row<D>(p, nx, qi, hl, trow);
                    tc_fence_before();
                    mbar_arrive(bar.q_ready);
                    have_q = true;
                }
            }
            // Epilogue: O = acc / l (BF16), LSE = ln(sum exp(s)) once the item's last PV has landed.
            if (!wait(bar.o_ready + stage_of(gc - 1), round_of(gc - 1))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int blk = 0; blk < D / 32; ++blk) {
                uint32_t o[32];
                tmem_ld32(trow + L::kTmemO + blk * 32, o);
                tmem_ld_wait();
                if (live) {
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        float f[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(o[i + e]) * inv;
                        reinterpret_cast<uint4 *>(orow + blk * 32 + i)[0] = f32x8_to_bf16(f);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar.o_free);
            if (live) p.lse[(it.b * p.Hq + h) * p.S_q + q] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
            ++qc;
            ++pos;
            idx = nidx;
        }
        if (!ok) fail(kSiteTileFwdWait, 4);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool tc_forward_supported() { return tc_device_ok(); }

bool tc_forward_shape_ok(const AttnArgs &a, const TileArgs &t) {
    return t.T >= 2 && t.T * a.G == kTileRows && a.B <= kMaxPairs && (a.D == 256 || a.D == 128);
}

namespace {
// The dynamic shared-memory limit is a property of the kernel on each device: it is set the
// first time the kernel is launched on a device (devices 0-63 remembered in a bit mask).
template <int D>
cudaError_t set_fwd_smem() {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(tc_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdLayout<D>::kSmemBytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}
}  // namespace

cudaError_t launch_tc_forward(const AttnArgs &a, const TileArgs &t, __nv_bfloat16 *o, float *lse,
                              const int32_t *choice, cudaStream_t s) {
    FwdParams p;
    memset(&p, 0, sizeof(p));
    if (!tc_encode_tile_map(&p.q_map, a.q, a.Hq, a.S_q, a.B, a.qs2, a.qs1, a.qs0, a.G, t.T, a.D))
        return cudaErrorInvalidValue;
    {
        cudaError_t e = a.D == 128 ? set_fwd_smem<128>() : set_fwd_smem<256>();
        if (e != cudaSuccess) return e;
    }
    const int sms = tc_num_sms();
    const int64_t g_per_launch = std::max<int64_t>(1, kMaxPairs / a.B);
    p.q = a.q;
    p.qs0 = a.qs0;
    p.qs1 = a.qs1;
    p.qs2 = a.qs2;
    p.B = a.B;
    p.S_q = a.S_q;
    p.Hq = a.Hq;
    p.G = a.G;
    p.T = t.T;
    p.n_tiles = t.n_tiles;
    p.max_chunks = t.max_chunks;
    p.sl2 = a.scale * kLog2e;
    p.wait_limit_ns = tc_wait_limit_ns(kWaitLimitNs);
    p.tile_nchunks = t.tile_nchunks;
    p.tile_keys = t.tile_keys;
    p.tile_masks = t.tile_masks;
    p.order = t.order;
    p.sched = t.sched;  // forward counters
    p.o = o;
    p.lse = lse;
    p.choice = choice;
    p.status = a.status;
    for (int64_t g0 = 0; g0 < a.Hkv; g0 += g_per_launch) {
        const int64_t n_g = std::min<int64_t>(g_per_launch, a.Hkv - g0);
        p.g0 = g0;
        p.n_g = n_g;
        p.head_major = tc_head_major_order(a, n_g);
        p.n_items = n_g * a.B * t.n_tiles;
        for (int64_t b = 0; b < a.B; ++b)
            for (int64_t gi = 0; gi < n_g; ++gi)
                if (!tc_encode_kv_maps(&p.kv[b * n_g + gi], a, b, g0 + gi)) return cudaErrorInvalidValue;
        const int grid = (int)std::min<int64_t>(p.n_items, sms);
        if (a.D == 128)
            tc_fwd_kernel<128><<<grid, kThreads, FwdLayout<128>::kSmemBytes, s>>>(p);
        else
            tc_fwd_kernel<256><<<grid, kThreads, FwdLayout<256>::kSmemBytes, s>>>(p);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace qsa

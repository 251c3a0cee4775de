// qsa_bwd_tc.cu -- tile backward of route-set sparse GQA on tcgen05 tensor cores.
//
// Same work items as the tile forward: (KV head g, tile of T = 128/G query
// rows); the tile's 128 (query, head) rows are the MMA M.  P is recomputed from
// the forward's LSE (P_j = exp(s_j - LSE)); Delta = <dO, O> per row comes from
// a small kernel beforehand.  Per 64-key chunk of the tile's routed-key union:
//
//   producer warp  gathers V then K rows (TMA tile::gather4) once the previous
//                  chunk's MMAs have released them (single stage each; V is
//                  free early, after the dP MMA);
//   MMA warp       S = Q K^T and dP = dO V^T (M128 N64 K=D) into TMEM;
//                  after the softmax: dQ += dS K (M128 N=D K64, TMEM
//                  accumulator over all chunks of the item), then for each
//                  128-row half of D (one at D = 128): dK^T = Q^T dS and
//                  dV^T = dO^T P (M128 N64 K128,
//                  both operands MN-major straight from the Q/dO tiles and the
//                  P/dS buffers) into TMEM;
//   softmax warps  thread = row: P = mask ? exp2(s*scale*log2e - LSE*log2e) : 0,
//                  dS = scale * P * (dP - Delta), both written as BF16 into
//                  swizzled shared memory; at the end of the item read dQ from
//                  TMEM and store it (BF16);
//   flush warps    thread = one head-dimension index: read a half's dK^T and
//                  dV^T columns (one per chunk key) from TMEM and scatter-add
//                  them into the fp32 dK/dV accumulators -- one coalesced
//                  128-byte reduction per warp, key and matrix.
//
// So each gathered K/V row and each (key, d) accumulator update serves every
// head of the group and every tile query that routes to that key, instead of
// once per (query, head).  Head dim D = 256 or 128.  TMEM (512 columns): dQ
// 0..D-1, S 256-319, dP 320-383, dK^T 384-447, dV^T 448-511.  All waits are bounded (2 s); a
// timeout is recorded in the status word, the roles wind down, in-flight
// copies and MMAs are drained, and the TMEM is freed.
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

constexpr int kThreads = 320;  // warps 0-3 softmax, 4-7 flush, 8 producer, 9 MMA
constexpr int kMaxPairs = kMaxKVPairs;
constexpr uint32_t kPBytes = kTileRows * kChunkKeys * 2;     // 16 KiB
// The Q/dO tiles and the K/V chunks sit in shared memory as 64-column panels
// (128-byte swizzle), so the panel strides do not depend on the head dim.
constexpr uint32_t kTilePanel = kTileRows * 128;  // 16 KiB: 64 columns of a 128-row tile
constexpr uint32_t kKVPanel = kChunkKeys * 128;   // 8 KiB: 64 columns of a 64-key chunk
constexpr uint32_t kBarItemFull = 16;  // work queue ring: full [kQueueRing], then empty [kQueueRing]
constexpr uint32_t kBarItemEmpty = kBarItemFull + kQueueRing;
constexpr uint32_t kNumBars = kBarItemEmpty + kQueueRing;

// Shared-memory layout for head dim D (256, or 128 with the same tiles at half
// the width: 128 KiB instead of 224 KiB).
template <int D>
struct BwdLayout {
    static constexpr int kPanels = D / 64;
    static constexpr int kHalves = D / 128;  // dK^T / dV^T MMAs cover 128 head-dim rows each
    static constexpr uint32_t kTileBytes = kTileRows * D * 2;  // Q or dO tile (64 KiB at D = 256)
    static constexpr uint32_t kKVBytes = kChunkKeys * D * 2;   // K or V chunk (32 KiB at D = 256)
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffDO = kOffQ + kTileBytes;
    static constexpr uint32_t kOffK = kOffDO + kTileBytes;
    static constexpr uint32_t kOffV = kOffK + kKVBytes;
    static constexpr uint32_t kOffP = kOffV + kKVBytes;
    static constexpr uint32_t kOffDS = kOffP + kPBytes;
    static constexpr uint32_t kOffBar = kOffDS + kPBytes;
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
    static constexpr uint32_t kSmemBytes = kOffMisc + 64 + 1024;
};
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemDQ = 0, kTmemS = 256, kTmemDP = 320, kTmemDKT = 384, kTmemDVT = 448;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
    CUtensorMap q_map, do_map;          // 4-D {D, Hq, S_q, B}, box {64, G, T, 1}
    KVMaps kv[kMaxPairs];               // per (b, g): K/V row-gather and 64-row-run maps
    int64_t B, S_q, S_kv, Hq, Hkv, G, T, n_tiles, max_chunks;
    int64_t g0, n_g, n_items;
    int32_t head_major;  // work queue order (qsa_queue.cuh)
    float sl2, scale;
    uint64_t wait_limit_ns;  // bound of every pipeline wait
    const int32_t *tile_nchunks;
    const int32_t *tile_keys;
    const uint64_t *tile_masks;
    const int32_t *order;
    int32_t *sched;  // work queue counters {next, done}
    const float *lse, *delta;
    __nv_bfloat16 *dq;
    float *dk_acc, *dv_acc;
    FxAcc dk_fx, dv_fx;  // deterministic mode: exact accumulators
    const int32_t *gate;  // null, or a device flag: the kernel returns at once when *gate == 1 (key-major runs)
    DeviceStatus *status;
};

using Item = QueueItem;

// kSFull: S of the chunk complete; kSDFull: dP complete too (S is issued first so the softmax can
// start on P while dP runs).
enum BarId {
    kQFull, kQEmpty, kKFull, kKEmpty, kVFull, kVEmpty, kSDFull, kPDSFull, kPDSEmpty, kGradsFull, kFlushDone,
    kDQReady, kDQFree, kDrain, kSFull
};

// D: head dim (128 or 256).  kDet: the flush adds dK/dV into the exact accumulators (FxAcc: bitwise
// reproducible sums).
template <int D, bool kDet>
__global__ void __launch_bounds__(kThreads, 1) tc_bwd_kernel(const __grid_constant__ BwdParams p) {
    if (p.gate && *p.gate == 1) return;  // the key-major backward runs instead (uniform over the grid)
    using L = BwdLayout<D>;
    constexpr uint32_t kOffQ = L::kOffQ, kOffDO = L::kOffDO, kOffK = L::kOffK, kOffV = L::kOffV;
    constexpr uint32_t kOffP = L::kOffP, kOffDS = L::kOffDS, kOffBar = L::kOffBar, kOffMisc = L::kOffMisc;
    constexpr uint32_t kTileBytes = L::kTileBytes, kKVBytes = L::kKVBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 8);
    volatile int32_t *ring = reinterpret_cast<volatile int32_t *>(smem + kOffMisc + 16);  // [kQueueRing]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);

    if (threadIdx.x == 0) {
        const uint32_t counts[kSFull + 1] = {1, 1, 1, 1, 1, 1, 1, 128, 1, 1, 128, 1, 128, 1, 1};
        for (int i = 0; i <= kSFull; ++i) mbar_init(bars + i, counts[i]);
        for (int i = 0; i < kQueueRing; ++i) {
            mbar_init(bars + kBarItemFull + i, 1);
            mbar_init(bars + kBarItemEmpty + i, 32 + 128 + 128);  // MMA warp, softmax and flush threads take every item
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 8 && lane == 0) {
        prefetch_tmap(&p.q_map);
        prefetch_tmap(&p.do_map);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int zero = 0;

    auto fail = [&](unsigned info) {
        raise_status(p.status, QSA_ERR_TIMEOUT, kSiteTileBwdWait, info, blockIdx.x);
        *abort_flag = 1;
    };
    auto wait = [&](int id, int64_t phase) {
        return mbar_wait_warp(bars + id, (uint32_t)(phase & 1), abort_flag, p.wait_limit_ns);
    };

    if (warp == 8) {
        // ---------------- producer ----------------
        int64_t gc = 0, qc = 0, v_issued = 0, k_issued = 0;
        Item it;
        bool ok = true;
        for (int64_t pos = 0; ok; ++pos) {
            int32_t idx = -1;
            if (lane == 0) ok = queue_claim(p.sched, p.n_items, ring, bars + kBarItemFull, bars + kBarItemEmpty, pos,
                                            abort_flag, p.wait_limit_ns, idx);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            idx = __shfl_sync(0xffffffffu, idx, 0);
            if (!ok || idx < 0) break;
            queue_decode(p, idx, it);
            if (it.nch == 0) continue;
            if (qc > 0 && !wait(kQEmpty, qc - 1)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(bars + kQFull, 2 * kTileBytes);
                for (int kb = 0; kb < L::kPanels; ++kb) {
                    tma_load_4d(sbase + kOffQ + kb * kTilePanel, &p.q_map, bars + kQFull, kb * 64,
                                (int)(it.g * p.G), (int)(it.t * p.T), (int)it.b);
                    tma_load_4d(sbase + kOffDO + kb * kTilePanel, &p.do_map, bars + kQFull, kb * 64,
                                (int)(it.g * p.G), (int)(it.t * p.T), (int)it.b);
                }
            }
            ++qc;
            const int pair = (int)(it.b * p.n_g + (it.g - p.g0));
            const KVMaps &maps = p.kv[pair];
            const int32_t *keys = p.tile_keys + it.tile * p.max_chunks * kChunkKeys;
            for (int c = 0; c < it.nch; ++c, ++gc) {
                int4 kk = make_int4(0, 0, 0, 0);
                if (lane < 16) kk = __ldg(reinterpret_cast<const int4 *>(keys + c * kChunkKeys) + lane);
                const int first = __shfl_sync(0xffffffffu, kk.x, 0), last = __shfl_sync(0xffffffffu, kk.w, 15);
                const bool run = last - first == kChunkKeys - 1;  // ascending distinct keys: a contiguous run
                if (gc > 0 && !wait(kVEmpty, gc - 1)) {
                    ok = false;
                    break;
                }
                // One barrier covers the chunk's K and V (the MMA warp waits once): the arrival announces
                // both copies' bytes, V's copy goes out now and K's once its slot is free.
                if (lane == 0) mbar_arrive_expect_tx(bars + kKFull, 2 * kKVBytes);
                __syncwarp();
                if (run) {
                    if (lane == 0)
                        for (int kb = 0; kb < L::kPanels; ++kb)
                            tma_load_2d(sbase + kOffV + kb * kKVPanel, &maps.v_run, bars + kKFull, kb * 64, first);
                } else if (lane < 16) {
                    for (int kb = 0; kb < L::kPanels; ++kb)
                        tma_gather4(sbase + kOffV + lane * 512 + kb * kKVPanel, &maps.v_rows, bars + kKFull,
                                    kb * 64, kk.x, kk.y, kk.z, kk.w);
                }
                __syncwarp();
                ++v_issued;
                if (gc > 0 && !wait(kKEmpty, gc - 1)) {
                    ok = false;
                    break;
                }
                __syncwarp();
                if (run) {
                    if (lane == 0)
                        for (int kb = 0; kb < L::kPanels; ++kb)
                            tma_load_2d(sbase + kOffK + kb * kKVPanel, &maps.k_run, bars + kKFull, kb * 64, first);
                } else if (lane < 16) {
                    for (int kb = 0; kb < L::kPanels; ++kb)
                        tma_gather4(sbase + kOffK + lane * 512 + kb * kKVPanel, &maps.k_rows, bars + kKFull,
                                    kb * 64, kk.x, kk.y, kk.z, kk.w);
                }
                __syncwarp();
                ++k_issued;
            }
        }
        if (!ok && lane == 0) fail(1);
        if (lane == 0) queue_finish(p.sched);
        // Drain every issued copy before the CTA can leave.
        if (lane == 0) {
            bool drained = true;
            // The last chunk's K and V phase; if the producer gave up between the V and the K copy, this
            // wait runs to its bound (the V copy has long landed by then).
            if (v_issued > 0) drained &= mbar_wait(bars + kKFull, (uint32_t)((v_issued - 1) & 1), &zero, kWaitLimitNs);
            (void)k_issued;
            if (qc > 0) drained &= mbar_wait(bars + kQFull, (uint32_t)((qc - 1) & 1), &zero, kWaitLimitNs);
            if (!drained) fail(2);
        }
        __syncwarp();
    } else if (warp == 9) {
        // ---------------- MMA issuer ----------------
        constexpr uint32_t idesc_n64 = idesc_bf16(kTileRows, kChunkKeys, false, false);   // S, dP
        constexpr uint32_t idesc_dq = idesc_bf16(kTileRows, D, false, true);       // dQ += dS K
        constexpr uint32_t idesc_t = idesc_bf16(kTileRows, kChunkKeys, true, true);       // dK^T, dV^T
        int64_t gc = 0, qc = 0, u = 0;
        Item it;
        bool ok = true;
        for (int64_t pos = 0; ok; ++pos) {
            int32_t idx = -1;
            ok = queue_take(ring, bars + kBarItemFull, bars + kBarItemEmpty, pos, abort_flag, p.wait_limit_ns, true, idx);
            if (!ok || idx < 0) break;
            queue_decode(p, idx, it);
            if (it.nch == 0) continue;
            if (!wait(kQFull, qc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int c = 0; c < it.nch; ++c, ++gc) {
                if (!wait(kKFull, gc)) {  // K and V of the chunk
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    // S first (its own completion barrier), then dP.
#pragma unroll
                    for (int kb = 0; kb < L::kPanels; ++kb) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_bf16(tmem + kTmemS, sdesc_sw128(sbase + kOffQ + kb * kTilePanel + k * 32, 16, 1024),
                                     sdesc_sw128(sbase + kOffK + kb * kKVPanel + k * 32, 16, 1024), idesc_n64,
                                     (kb | k) ? 1u : 0u);
                    }
                    mma_commit(bars + kSFull);
#pragma unroll
                    for (int kb = 0; kb < L::kPanels; ++kb) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_bf16(tmem + kTmemDP, sdesc_sw128(sbase + kOffDO + kb * kTilePanel + k * 32, 16, 1024),
                                     sdesc_sw128(sbase + kOffV + kb * kKVPanel + k * 32, 16, 1024), idesc_n64,
                                     (kb | k) ? 1u : 0u);
                    }
                    mma_commit(bars + kSDFull);
                    mma_commit(bars + kVEmpty);
                }
                __syncwarp();
                if (!wait(kPDSFull, gc) || (c == 0 && qc > 0 && !wait(kDQFree, qc - 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
#pragma unroll
                    for (int k = 0; k < kChunkKeys / 16; ++k)
                        mma_bf16(tmem + kTmemDQ, sdesc_sw128(sbase + kOffDS + k * 32, 16, 1024),
                                 sdesc_sw128(sbase + kOffK + k * 2048, kKVPanel, 1024), idesc_dq,
                                 (c == 0 && k == 0) ? 0u : 1u);
                    mma_commit(bars + kKEmpty);
                    if (c == it.nch - 1) mma_commit(bars + kDQReady);
                }
                __syncwarp();
                for (int h = 0; h < L::kHalves; ++h, ++u) {
                    if (u > 0 && !wait(kFlushDone, u - 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
#pragma unroll
                        for (int kk = 0; kk < kTileRows / 16; ++kk) {
                            const uint32_t aoff = (2 * h) * kTilePanel + kk * 2048;
                            mma_bf16(tmem + kTmemDKT, sdesc_sw128(sbase + kOffQ + aoff, kTilePanel, 1024),
                                     sdesc_sw128(sbase + kOffDS + kk * 2048, kPBytes, 1024), idesc_t, kk ? 1u : 0u);
                            mma_bf16(tmem + kTmemDVT, sdesc_sw128(sbase + kOffDO + aoff, kTilePanel, 1024),
                                     sdesc_sw128(sbase + kOffP + kk * 2048, kPBytes, 1024), idesc_t, kk ? 1u : 0u);
                        }
                        mma_commit(bars + kGradsFull);
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (lane == 0) mma_commit(bars + kPDSEmpty);
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) mma_commit(bars + kQEmpty);
            __syncwarp();
            ++qc;
        }
        if (!ok && lane == 0) fail(3);
        if (lane == 0) {
            mma_commit(bars + kDrain);
            if (!mbar_wait(bars + kDrain, 0, &zero, kWaitLimitNs)) fail(4);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ---------------- softmax: P, dS; dQ epilogue ----------------
        const int r = threadIdx.x;
        const int qi = (int)(r / p.G), hl = (int)(r % p.G);
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        int64_t gc = 0, qc = 0;
        Item it;
        bool ok = true;
        for (int64_t pos = 0; ok; ++pos) {
            int32_t idx = -1;
            ok = queue_take(ring, bars + kBarItemFull, bars + kBarItemEmpty, pos, abort_flag, p.wait_limit_ns, true, idx);
            if (!ok || idx < 0) break;
            queue_decode(p, idx, it);
            const int64_t q = it.t * p.T + qi;
            const int64_t h = it.g * p.G + hl;
            const bool live = q < p.S_q;
            __nv_bfloat16 *dqrow = p.dq + ((it.b * p.S_q + q) * p.Hq + h) * D;
            if (it.nch == 0) {
                if (live) {
                    const uint4 z = make_uint4(0, 0, 0, 0);
                    for (int i = 0; i < D / 8; ++i) reinterpret_cast<uint4 *>(dqrow)[i] = z;
                }
                continue;
            }
            const int64_t stat = (it.b * p.Hq + h) * p.S_q + q;
            const float lse2 = live ? p.lse[stat] * kLog2e : 0.f;
            const float delta = live ? p.delta[stat] : 0.f;
            const uint64_t *mrow = p.tile_masks + it.tile * p.max_chunks * p.T + qi;
            uint64_t mask_next = __ldg(mrow);
            for (int c = 0; c < it.nch; ++c, ++gc) {
                const uint64_t mask = mask_next;
                if (c + 1 < it.nch) mask_next = __ldg(mrow + (c + 1) * p.T);
                if (!wait(kSFull, gc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float pf[64];
                {
                    uint32_t sr[2][32];
                    tmem_ld32(trow + kTmemS, sr[0]);
                    tmem_ld32(trow + kTmemS + 32, sr[1]);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 64; ++j)
                        pf[j] = ((mask >> j) & 1ull) ? ex2(__uint_as_float(sr[j >> 5][j & 31]) * p.sl2 - lse2) : 0.f;
                }
                // The previous chunk's gradient MMAs have read the P/dS buffers (long done by now); P goes
                // into shared memory while the dP MMA still runs, so only dS is left once dP lands.
                if (gc > 0 && !wait(kPDSEmpty, gc - 1)) {
                    ok = false;
                    break;
                }
                uint8_t *prow = smem + kOffP + r * 128;
                uint8_t *drow = smem + kOffDS + r * 128;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t w4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) w4[e] = pack_bf16(pf[8 * ch + 2 * e], pf[8 * ch + 2 * e + 1]);
                    *reinterpret_cast<uint4 *>(prow + (ch ^ (r & 7)) * 16) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
                if (!wait(kSDFull, gc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                {
                    uint32_t dr[2][32];
                    tmem_ld32(trow + kTmemDP, dr[0]);
                    tmem_ld32(trow + kTmemDP + 32, dr[1]);
                    tmem_ld_wait();
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        uint32_t w4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 8 * ch + 2 * e;
                            const float d0 = p.scale * pf[j] * (__uint_as_float(dr[j >> 5][j & 31]) - delta);
                            const float d1 = p.scale * pf[j + 1] * (__uint_as_float(dr[(j + 1) >> 5][(j + 1) & 31]) - delta);
                            w4[e] = pack_bf16(d0, d1);
                        }
                        *reinterpret_cast<uint4 *>(drow + (ch ^ (r & 7)) * 16) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bars + kPDSFull);
            }
            if (!ok) break;
            if (!wait(kDQReady, qc)) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int blk = 0; blk < D / 32; ++blk) {
                uint32_t o[32];
                tmem_ld32(trow + kTmemDQ + blk * 32, o);
                tmem_ld_wait();
                if (live) {
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        float f[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(o[i + e]);
                        reinterpret_cast<uint4 *>(dqrow + blk * 32 + i)[0] = f32x8_to_bf16(f);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bars + kDQFree);
            ++qc;
        }
        if (!ok) fail(5);
    } else {
        // ---------------- flush: dK^T / dV^T -> fp32 scatter-add ----------------
        const int quarter = warp & 3;
        const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
        int64_t gc = 0, u = 0;
        Item it;
        bool ok = true;
        for (int64_t pos = 0; ok; ++pos) {
            int32_t idx = -1;
            ok = queue_take(ring, bars + kBarItemFull, bars + kBarItemEmpty, pos, abort_flag, p.wait_limit_ns, true, idx);
            if (!ok || idx < 0) break;
            queue_decode(p, idx, it);
            if (it.nch == 0) continue;
            const int64_t row_stride = p.Hkv * D;
            const int64_t base_off = (it.b * p.S_kv * p.Hkv + it.g) * D + quarter * 32 + lane;
            float *dk_base = kDet ? p.dk_fx.est + base_off : p.dk_acc + base_off;
            float *dv_base = kDet ? p.dv_fx.est + base_off : p.dv_acc + base_off;
            uint32_t *dk_lo = kDet ? p.dk_fx.lo + base_off : nullptr;
            uint32_t *dv_lo = kDet ? p.dv_fx.lo + base_off : nullptr;
            for (int c = 0; c < it.nch; ++c, ++gc) {
                // The chunk's 64 keys, one pair per lane, broadcast below with shuffles.  The loop has no
                // branch: a partial chunk's padding columns have empty membership, so their dK^T/dV^T
                // columns are exact zeros and adding them to the padding key's row changes nothing.
                // Branch-free, the key broadcasts do not wait on one another and the reductions issue
                // back to back.
                const int32_t *keys = p.tile_keys + (it.tile * p.max_chunks + c) * kChunkKeys;
                const int32_t key_lo = __ldg(keys + lane), key_hi = __ldg(keys + 32 + lane);
                for (int h = 0; h < L::kHalves; ++h, ++u) {
                    if (!wait(kGradsFull, u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint32_t a[2][32], v[2][32];
                    tmem_ld32(trow + kTmemDKT, a[0]);
                    tmem_ld32(trow + kTmemDKT + 32, a[1]);
                    tmem_ld32(trow + kTmemDVT, v[0]);
                    tmem_ld32(trow + kTmemDVT + 32, v[1]);
                    tmem_ld_wait();
                    tc_fence_before();
                    mbar_arrive(bars + kFlushDone);
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        const int32_t key = __shfl_sync(0xffffffffu, j < 32 ? key_lo : key_hi, j & 31);
                        const int64_t off = (int64_t)key * row_stride + h * 128;
                        if (kDet) {
                            red_add_fx(dk_base + off, dk_lo + off, __uint_as_float(a[j >> 5][j & 31]));
                            red_add_fx(dv_base + off, dv_lo + off, __uint_as_float(v[j >> 5][j & 31]));
                        } else {
                            red_add_f32(dk_base + off, __uint_as_float(a[j >> 5][j & 31]));
                            red_add_f32(dv_base + off, __uint_as_float(v[j >> 5][j & 31]));
                        }
                    }
                }
                if (!ok) break;
            }
        }
        if (!ok) fail(6);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

namespace {
// The dynamic shared-memory limit is a property of the kernel on each device: it is set the
// first time the kernels are launched on a device (devices 0-63 remembered in a bit mask).
template <int D>
cudaError_t set_bwd_smem() {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(tc_bwd_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             BwdLayout<D>::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tc_bwd_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 BwdLayout<D>::kSmemBytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}
}  // namespace

bool tc_backward_supported() { return tc_device_ok(); }

bool tc_backward_shape_ok(const AttnArgs &a, const TileArgs &t) {
    return t.T >= 2 && t.T * a.G == kTileRows && a.B <= kMaxPairs && (a.D == 256 || a.D == 128);
}

cudaError_t launch_tc_backward(const BwdArgs &bw, const TileArgs &t, const int32_t *gate, cudaStream_t s) {
    const AttnArgs &a = bw.f;
    const int64_t D = a.D;
    BwdParams p;
    memset(&p, 0, sizeof(p));
    if (!tc_encode_tile_map(&p.q_map, a.q, a.Hq, a.S_q, a.B, a.qs2, a.qs1, a.qs0, a.G, t.T, D))
        return cudaErrorInvalidValue;
    if (!tc_encode_tile_map(&p.do_map, bw.dout, a.Hq, a.S_q, a.B, D, a.Hq * D, a.S_q * a.Hq * D, a.G, t.T, D))
        return cudaErrorInvalidValue;
    {
        cudaError_t e = D == 128 ? set_bwd_smem<128>() : set_bwd_smem<256>();
        if (e != cudaSuccess) return e;
    }
    const int sms = tc_num_sms();
    const int64_t g_per_launch = std::max<int64_t>(1, kMaxPairs / a.B);
    p.B = a.B;
    p.S_q = a.S_q;
    p.S_kv = a.S_kv;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.G;
    p.T = t.T;
    p.n_tiles = t.n_tiles;
    p.max_chunks = t.max_chunks;
    p.sl2 = a.scale * kLog2e;
    p.scale = a.scale;
    p.wait_limit_ns = tc_wait_limit_ns(kWaitLimitNs);
    p.tile_nchunks = t.tile_nchunks;
    p.tile_keys = t.tile_keys;
    p.tile_masks = t.tile_masks;
    p.order = t.order;
    p.sched = t.sched + 2;  // backward counters
    p.lse = bw.lse;
    p.delta = bw.delta;
    p.dq = bw.dq;
    p.dk_acc = bw.dk_acc;
    p.dv_acc = bw.dv_acc;
    p.dk_fx = bw.dk_fx;
    p.dv_fx = bw.dv_fx;
    p.gate = gate;
    p.status = a.status;
    for (int64_t g0 = 0; g0 < a.Hkv; g0 += g_per_launch) {
        const int64_t n_g = std::min<int64_t>(g_per_launch, a.Hkv - g0);
        p.g0 = g0;
        p.n_g = n_g;
        p.head_major = tc_head_major_order(bw.f, n_g);
        p.n_items = n_g * a.B * t.n_tiles;
        for (int64_t b = 0; b < a.B; ++b)
            for (int64_t gi = 0; gi < n_g; ++gi)
                if (!tc_encode_kv_maps(&p.kv[b * n_g + gi], a, b, g0 + gi)) return cudaErrorInvalidValue;
        const int grid = (int)std::min<int64_t>(p.n_items, sms);
        const bool det = bw.dk_fx.est != nullptr;
        if (D == 128) {
            if (det)
                tc_bwd_kernel<128, true><<<grid, kThreads, BwdLayout<128>::kSmemBytes, s>>>(p);
            else
                tc_bwd_kernel<128, false><<<grid, kThreads, BwdLayout<128>::kSmemBytes, s>>>(p);
        } else {
            if (det)
                tc_bwd_kernel<256, true><<<grid, kThreads, BwdLayout<256>::kSmemBytes, s>>>(p);
            else
                tc_bwd_kernel<256, false><<<grid, kThreads, BwdLayout<256>::kSmemBytes, s>>>(p);
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace qsa

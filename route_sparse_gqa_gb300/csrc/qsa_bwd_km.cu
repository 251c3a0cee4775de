// qsa_bwd_km.cu -- key-major (reverse-route) backward of route-set sparse GQA on
// tcgen05 tensor cores.
//
// The tile backward walks a query tile's routed keys and scatter-adds dK/dV for
// every (tile, chunk) pair; when a tile's queries share few keys (long prefixes
// with scattered routed blocks) most of each 128-row MMA is masked work and
// most of the scatter traffic carries zeros.  This kernel walks the other way
// (the pages' FA4 preprocessing keeps reverse block lists: fa4_qsa
// _preprocess).  Work item = (KV head g, part of the reverse list of one
// aligned 64-key chunk c of batch row b): up to max_groups groups of T = 128/G
// query rows that route into the chunk, gathered so every MMA row is a routed
// (query, head) pair.  Per item:
//
//   producer warp  loads the chunk's 64 K and V rows once (two 4-D TMA tile
//                  boxes per 64-column panel), then per group the T queries'
//                  Q and dO rows of the G heads of g: one 5-D box per eight
//                  heads of a query covering every panel (4 KiB at D = 256;
//                  small boxes cost the TMA unit about as much per copy as
//                  large ones), empty slots reading zeros past the end of S_q;
//   MMA warp       per group: S = Q K^T and dP = dO V^T (M128 N64 K=D);
//                  after the softmax: dV^T += dO^T P and dK^T += Q^T dS for
//                  every 128-row half of D (M128 N64 K128, accumulated in
//                  TMEM over all groups of the item), then per half
//                  dQ^T = K^T dS^T (M128 N128 K64: D rows, one column per
//                  (query, head) row of the group);
//   softmax warps  thread = row (slot, head): P = mask ? exp2(s*scale*log2e -
//                  LSE*log2e) : 0 and dS = mask ? scale*P*(dP - Delta) : 0,
//                  written as BF16 into swizzled shared memory;
//   flush warps    thread = one head-dimension index of a half: per group and
//                  half, read the group's dQ^T columns from TMEM and add each
//                  row into the fp32 dQ accumulator (one coalesced 128-byte
//                  reduction per warp and row); at the end of the item, add
//                  the chunk's dK^T/dV^T columns into the fp32 dK/dV
//                  accumulators (one reduction per warp, key and matrix).
//
// So dK/dV leave the chip once per (chunk, part) instead of once per (query
// tile, chunk), and every MMA row is a routed pair.  dQ is the scattered side
// now: one fp32 reduction per (routed query, chunk, head, d), exactly the
// useful pairs.  Head dim D = 256 or 128, G a power of two from 8 to 64.  TMEM (512 columns): dK^T per half
// at 0 / 64, dV^T per half after them, dQ^T (128 columns), S (64), dP (64).
// All waits are bounded (2 s); a timeout is recorded in the status word, the
// roles wind down, in-flight copies and MMAs are drained and the TMEM is freed.
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
constexpr uint32_t kPBytes = kTileRows * kChunkKeys * 2;  // 16 KiB: P or dS of one group
// The Q and dO tiles of a group are [8-row block][panel][8 rows][128 B]: an 8-row block is eight heads of
// one query, all D/64 panels (one TMA copy); 8-row blocks follow each other every kBlk8 bytes.
constexpr uint32_t kKVPanel = kChunkKeys * 128;           // 8 KiB: 64 columns of a 64-key chunk
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

// Two tile buffers alternate roles: group gc keeps Q in buffer gc & 1 and dO in the other one, so the buffer
// freed first (dO, after the dV^T MMAs) takes the next group's Q and the Q buffer (after dK^T) its dO.  Each
// buffer is filled and freed once per group.
enum BarId {
    kKVFull, kKVFree, kBufFull0, kBufFull1, kBufFree0, kBufFree1, kSFull, kSDFull, kPFull, kDSFull, kPFree, kDSFree,
    kDQReady, kDQFree, kDKVReady, kDKVFree, kDrain, kNumFixedBars
};
constexpr uint32_t kBarItemFull = kNumFixedBars;  // work queue ring: full [kQueueRing], then empty [kQueueRing]
constexpr uint32_t kBarItemEmpty = kBarItemFull + kQueueRing;
constexpr uint32_t kNumBars = kBarItemEmpty + kQueueRing;

template <int D>
struct KmLayout {
    static constexpr int kPanels = D / 64;
    static constexpr int kHalves = D / 128;
    static constexpr uint32_t kTileBytes = kTileRows * D * 2;  // Q or dO of one group
    static constexpr uint32_t kBlk8 = 8 * D * 2;              // one 8-row block, all panels (4 KiB at D = 256)
    static constexpr uint32_t kKVBytes = kChunkKeys * D * 2;   // K or V of one chunk
    static constexpr uint32_t kOffBuf = 0;  // two tile buffers: Q and dO, alternating (BarId)
    static constexpr uint32_t kOffK = kOffBuf + 2 * kTileBytes;
    static constexpr uint32_t kOffV = kOffK + kKVBytes;
    static constexpr uint32_t kOffP = kOffV + kKVBytes;
    static constexpr uint32_t kOffDS = kOffP + kPBytes;
    static constexpr uint32_t kOffBar = kOffDS + kPBytes;
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
    static constexpr uint32_t kSmemBytes = kOffMisc + 64 + 1024;
    // TMEM columns
    static constexpr uint32_t kTmemDKT = 0;                      // + 64 * half
    static constexpr uint32_t kTmemDVT = 64 * kHalves;           // + 64 * half
    static constexpr uint32_t kTmemDQT = 128 * kHalves;          // 128 columns
    static constexpr uint32_t kTmemS = kTmemDQT + 128;
    static constexpr uint32_t kTmemDP = kTmemS + 64;
};
constexpr uint32_t kTmemCols = 512;

struct KmParams {
    // 5-D {64, Hq, D/64, S_q, B} (64 columns of a panel, head, panel, query, batch), box {64, 8, D/64, 1, 1}:
    // eight heads of one query, every panel, landing as [panel][8 rows][128 B] (one 4 KiB copy).
    CUtensorMap q_map, do_map;
    CUtensorMap k_map, v_map;   // 4-D {D, Hkv, S_kv, B}, box {64, 1, 64, 1}: one chunk of one KV head
    int64_t B, S_q, S_kv, Hq, Hkv, G, T, NC;
    float sl2, scale;
    uint64_t wait_limit_ns;
    const int4 *items;
    const int32_t *queue;
    const int32_t *meta;  // meta[2] = queue length
    const int32_t *e_q;
    const uint64_t *e_mask;
    int32_t *sched;
    const float *lse, *delta;
    float *dq_acc, *dk_acc, *dv_acc;
    FxAcc dq_fx, dk_fx, dv_fx;
    const int32_t *gate;  // null, or a device flag: the kernel returns at once when *gate == 0 (tile runs)
    DeviceStatus *status;
};

struct KmItem {
    int64_t b, g, c;
    int32_t e0, ne, ng;
};

__device__ __forceinline__ void km_decode(const KmParams &p, int32_t idx, KmItem &it) {
    const int32_t v = p.queue[idx];
    const int32_t item = (int32_t)(v / p.Hkv);
    it.g = v % p.Hkv;
    const int4 d = p.items[item];
    it.b = d.x / p.NC;
    it.c = d.x % p.NC;
    it.e0 = d.y;
    it.ne = d.z;
    it.ng = (int32_t)((d.z + p.T - 1) / p.T);
}


template <int D, bool kDet>
__global__ void __launch_bounds__(kThreads, 1) km_bwd_kernel(const __grid_constant__ KmParams p) {
    if (p.gate && *p.gate == 0) return;  // the tile backward runs instead (uniform over the grid)
    using L = KmLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 8);
    volatile int32_t *ring = reinterpret_cast<volatile int32_t *>(smem + L::kOffMisc + 16);  // [kQueueRing]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumFixedBars; ++i) {
            const uint32_t n = (i == kPFull || i == kDSFull || i == kDQFree || i == kDKVFree) ? 128u : 1u;
            mbar_init(bars + i, n);
        }
        for (int i = 0; i < kQueueRing; ++i) {
            mbar_init(bars + kBarItemFull + i, 1);
            mbar_init(bars + kBarItemEmpty + i, 32 + 128 + 128);  // MMA warp, softmax and flush threads
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
        prefetch_tmap(&p.k_map);
        prefetch_tmap(&p.v_map);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int zero = 0;

    auto fail = [&](unsigned info) {
        raise_status(p.status, QSA_ERR_TIMEOUT, kSiteKeyBwdWait, info, blockIdx.x);
        *abort_flag = 1;
    };
    auto wait = [&](int id, int64_t phase) {
        return mbar_wait_warp(bars + id, (uint32_t)(phase & 1), abort_flag, p.wait_limit_ns);
    };

    // Parity of every wait below: each barrier completes once per item (K/V, dK/dV) or per group (the
    // rest) or per (group, half) (dQ^T), and a barrier's next phase needs an action of the waiting role
    // that comes after the wait, so the waited phase is always the open one or the one just completed.
    if (warp == 8) {
        // ---------------- producer ----------------
        const int64_t n_queue = p.meta[2];
        int64_t ic = 0, gc = 0, nfill[2] = {0, 0};
        KmItem it;
        bool ok = true;
        for (int64_t pos = 0; ok; ++pos) {
            int32_t idx = -1;
            if (lane == 0) ok = queue_claim(p.sched, n_queue, ring, bars + kBarItemFull, bars + kBarItemEmpty, pos,
                                            abort_flag, p.wait_limit_ns, idx);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            idx = __shfl_sync(0xffffffffu, idx, 0);
            if (!ok || idx < 0) break;
            km_decode(p, idx, it);
            // The chunk's K and V, once the previous item's last MMA has read the previous chunk.
            if (ic > 0 && !wait(kKVFree, ic - 1)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(bars + kKVFull, 2 * L::kKVBytes);
                for (int kb = 0; kb < L::kPanels; ++kb) {
                    tma_load_4d(sbase + L::kOffK + kb * kKVPanel, &p.k_map, bars + kKVFull, kb * 64, (int)it.g,
                                (int)(it.c * kChunkKeys), (int)it.b);
                    tma_load_4d(sbase + L::kOffV + kb * kKVPanel, &p.v_map, bars + kKVFull, kb * 64, (int)it.g,
                                (int)(it.c * kChunkKeys), (int)it.b);
                }
            }
            __syncwarp();
            ++ic;
            // Lane s: the query of slot s in the next group (loaded one group ahead of its copies).
            auto slot_query = [&](int grp) {
                const int32_t e0 = it.e0 + grp * (int32_t)p.T;
                const int32_t nv = min((int32_t)p.T, it.e0 + it.ne - e0);
                // Slots past the group's queries read rows past the end of S_q: zeros.
                return lane < nv ? __ldg(p.e_q + e0 + lane) : (int)p.S_q;
            };
            int q_next = slot_query(0);
            for (int grp = 0; grp < it.ng; ++grp, ++gc) {
                const int q = q_next;
                if (grp + 1 < it.ng) q_next = slot_query(grp + 1);
                const int qb = (int)(gc & 1);  // Q's buffer; dO goes to the other one
                // 16 8-row blocks per tile (G / 8 per slot): lane i copies block i.
                const int slot = lane / (int)(p.G / 8), h8 = lane % (int)(p.G / 8);
                const int qs = __shfl_sync(0xffffffffu, q, lane < kTileRows / 8 ? slot : 0);
                for (int t = 0; t < 2; ++t) {
                    const int buf = t == 0 ? qb : 1 - qb;
                    // The buffer's previous tile (the other tensor of group gc - 1) is no longer read.
                    if (gc > 0 && !wait(kBufFree0 + buf, gc - 1)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) mbar_arrive_expect_tx(bars + kBufFull0 + buf, L::kTileBytes);
                    ++nfill[buf];
                    __syncwarp();
                    if (lane < kTileRows / 8)
                        tma_load_5d(sbase + buf * L::kTileBytes + (uint32_t)lane * L::kBlk8, t == 0 ? &p.q_map : &p.do_map,
                                    bars + kBufFull0 + buf, 0, (int)(it.g * p.G) + 8 * h8, 0, qs, (int)it.b);
                    __syncwarp();
                }
                if (!ok) break;
            }
        }
        if (!ok && lane == 0) fail(1);
        if (lane == 0) queue_finish(p.sched);
        if (lane == 0) {
            bool drained = true;
            if (ic > 0) drained &= mbar_wait(bars + kKVFull, (uint32_t)((ic - 1) & 1), &zero, kWaitLimitNs);
            // Both buffers' last copies: buffer t's n-th fill completes its phase n - 1.
            for (int t = 0; t < 2; ++t)
                if (nfill[t] > 0)
                    drained &= mbar_wait(bars + kBufFull0 + t, (uint32_t)((nfill[t] - 1) & 1), &zero, kWaitLimitNs);
            if (!drained) fail(2);
        }
        __syncwarp();
    } else if (warp == 9) {
        // ---------------- MMA issuer ----------------
        constexpr uint32_t idesc_n64 = idesc_bf16(kTileRows, kChunkKeys, false, false);  // S, dP
        constexpr uint32_t idesc_t = idesc_bf16(128, kChunkKeys, true, true);           // dK^T, dV^T
        constexpr uint32_t idesc_dqt = idesc_bf16(128, kTileRows, true, false);         // dQ^T
        // The loops over panels and halves stay rolled (only the K steps inside are unrolled): this warp shares
        // a sub-partition's instruction cache with a softmax and a flush warp, and the smaller code measured
        // faster (fewer instruction-fetch stalls) than the fully unrolled sequence.
        int64_t ic = 0, gc = 0, u = 0;
        KmItem it;
        bool ok = true;
        for (int64_t pos = 0; ok; ++pos) {
            int32_t idx = -1;
            ok = queue_take(ring, bars + kBarItemFull, bars + kBarItemEmpty, pos, abort_flag, p.wait_limit_ns, true,
                            idx);
            if (!ok || idx < 0) break;
            km_decode(p, idx, it);
            if (!wait(kKVFull, ic)) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int grp = 0; grp < it.ng; ++grp, ++gc) {
                const uint32_t qa = sbase + (uint32_t)(gc & 1) * L::kTileBytes;        // Q tile
                const uint32_t da = sbase + (uint32_t)((gc + 1) & 1) * L::kTileBytes;  // dO tile
                const int qbar = (int)(gc & 1), dbar = 1 - qbar;
                if (!wait(kBufFull0 + qbar, gc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
#pragma unroll 1
                    for (int kb = 0; kb < L::kPanels; ++kb) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_bf16(tmem + L::kTmemS, sdesc_sw128(qa + kb * 1024 + k * 32, 16, L::kBlk8),
                                     sdesc_sw128(sbase + L::kOffK + kb * kKVPanel + k * 32, 16, 1024), idesc_n64,
                                     (kb | k) ? 1u : 0u);
                    }
                    mma_commit(bars + kSFull);
                }
                __syncwarp();
                if (!wait(kBufFull0 + dbar, gc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
#pragma unroll 1
                    for (int kb = 0; kb < L::kPanels; ++kb) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_bf16(tmem + L::kTmemDP, sdesc_sw128(da + kb * 1024 + k * 32, 16, L::kBlk8),
                                     sdesc_sw128(sbase + L::kOffV + kb * kKVPanel + k * 32, 16, 1024), idesc_n64,
                                     (kb | k) ? 1u : 0u);
                    }
                    mma_commit(bars + kSDFull);
                }
                __syncwarp();
                // dV^T += dO^T P once P is written; on the item's first group the previous item's dK^T/dV^T must
                // have left TMEM.  Then the dO tile's buffer can take the next group's Q.
                if (!wait(kPFull, gc) || (grp == 0 && ic > 0 && !wait(kDKVFree, ic - 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
#pragma unroll 1
                    for (int h = 0; h < L::kHalves; ++h) {
#pragma unroll
                        for (int kk = 0; kk < kTileRows / 16; ++kk) {
                            const uint32_t aoff = (2 * h) * 1024 + kk * 2 * L::kBlk8;  // 16 rows = two 8-row blocks
                            mma_bf16(tmem + L::kTmemDVT + 64 * h, sdesc_sw128(da + aoff, 1024, L::kBlk8),
                                     sdesc_sw128(sbase + L::kOffP + kk * 2048, kPBytes, 1024), idesc_t,
                                     (grp > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    mma_commit(bars + kBufFree0 + dbar);
                    mma_commit(bars + kPFree);
                }
                __syncwarp();
                // dK^T += Q^T dS, then the Q tile's buffer can take the next group's dO.
                if (!wait(kDSFull, gc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
#pragma unroll 1
                    for (int h = 0; h < L::kHalves; ++h) {
#pragma unroll
                        for (int kk = 0; kk < kTileRows / 16; ++kk) {
                            const uint32_t aoff = (2 * h) * 1024 + kk * 2 * L::kBlk8;
                            mma_bf16(tmem + L::kTmemDKT + 64 * h, sdesc_sw128(qa + aoff, 1024, L::kBlk8),
                                     sdesc_sw128(sbase + L::kOffDS + kk * 2048, kPBytes, 1024), idesc_t,
                                     (grp > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    mma_commit(bars + kBufFree0 + qbar);
                }
                __syncwarp();
                for (int h = 0; h < L::kHalves; ++h, ++u) {
                    if (u > 0 && !wait(kDQFree, u - 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
#pragma unroll
                        for (int k = 0; k < kChunkKeys / 16; ++k)
                            mma_bf16(tmem + L::kTmemDQT,
                                     sdesc_sw128(sbase + L::kOffK + (2 * h) * kKVPanel + k * 2048, kKVPanel, 1024),
                                     sdesc_sw128(sbase + L::kOffDS + k * 32, 16, 1024), idesc_dqt, k ? 1u : 0u);
                        mma_commit(bars + kDQReady);
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (lane == 0) {
                    mma_commit(bars + kDSFree);  // the dS buffer is reusable
                    if (grp == it.ng - 1) {
                        mma_commit(bars + kDKVReady);  // the item's dK^T/dV^T are complete
                        mma_commit(bars + kKVFree);    // and its K/V chunk is no longer read
                    }
                }
                __syncwarp();
            }
            if (!ok) break;
            ++ic;
        }
        if (!ok && lane == 0) fail(3);
        if (lane == 0) {
            mma_commit(bars + kDrain);
            if (!mbar_wait(bars + kDrain, 0, &zero, kWaitLimitNs)) fail(4);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ---------------- softmax: P, dS ----------------
        const int r = threadIdx.x;
        const int slot = (int)(r / p.G), hl = (int)(r % p.G);
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        int64_t gc = 0;
        KmItem it;
        bool ok = true;
        for (int64_t pos = 0; ok; ++pos) {
            int32_t idx = -1;
            ok = queue_take(ring, bars + kBarItemFull, bars + kBarItemEmpty, pos, abort_flag, p.wait_limit_ns, true,
                            idx);
            if (!ok || idx < 0) break;
            km_decode(p, idx, it);
            const int64_t h = it.g * p.G + hl;
            for (int grp = 0; grp < it.ng; ++grp, ++gc) {
                const int32_t e = it.e0 + grp * (int32_t)p.T + slot;
                const bool live = e < it.e0 + it.ne;
                const int64_t q = live ? __ldg(p.e_q + e) : 0;
                const uint64_t mask = live ? __ldg(p.e_mask + e) : 0ull;
                const int64_t stat = (it.b * p.Hq + h) * p.S_q + q;
                const float lse2 = live ? __ldg(p.lse + stat) * kLog2e : 0.f;
                const float delta = live ? __ldg(p.delta + stat) : 0.f;
                if (!wait(kSFull, gc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float pf[64];
                {
                    uint32_t sr[2][32];
                    tmem_ld32(trow + L::kTmemS, sr[0]);
                    tmem_ld32(trow + L::kTmemS + 32, sr[1]);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 64; ++j)
                        pf[j] = ((mask >> j) & 1ull) ? ex2(__uint_as_float(sr[j >> 5][j & 31]) * p.sl2 - lse2) : 0.f;
                }
                // P over the previous group's, once its dV^T MMAs have read it; released at once so dV^T
                // runs while dS is computed.
                if (gc > 0 && !wait(kPFree, gc - 1)) {
                    ok = false;
                    break;
                }
                uint8_t *prow = smem + L::kOffP + r * 128;
                uint8_t *drow = smem + L::kOffDS + r * 128;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t w4[4];
#pragma unroll
                    for (int e4 = 0; e4 < 4; ++e4) w4[e4] = pack_bf16(pf[8 * ch + 2 * e4], pf[8 * ch + 2 * e4 + 1]);
                    *reinterpret_cast<uint4 *>(prow + (ch ^ (r & 7)) * 16) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bars + kPFull);
                if (!wait(kSDFull, gc) || (gc > 0 && !wait(kDSFree, gc - 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                {
                    uint32_t dr[2][32];
                    tmem_ld32(trow + L::kTmemDP, dr[0]);
                    tmem_ld32(trow + L::kTmemDP + 32, dr[1]);
                    tmem_ld_wait();
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        uint32_t w4[4];
#pragma unroll
                        for (int e4 = 0; e4 < 4; ++e4) {
                            const int j = 8 * ch + 2 * e4;
                            // A select, not a product with P = 0: rows and keys outside the route set must give
                            // exact zeros whatever dP holds.
                            const float d0 = ((mask >> j) & 1ull)
                                                 ? p.scale * pf[j] * (__uint_as_float(dr[j >> 5][j & 31]) - delta)
                                                 : 0.f;
                            const float d1 = ((mask >> (j + 1)) & 1ull)
                                                 ? p.scale * pf[j + 1] *
                                                       (__uint_as_float(dr[(j + 1) >> 5][(j + 1) & 31]) - delta)
                                                 : 0.f;
                            w4[e4] = pack_bf16(d0, d1);
                        }
                        *reinterpret_cast<uint4 *>(drow + (ch ^ (r & 7)) * 16) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bars + kDSFull);
            }
        }
        if (!ok) fail(5);
    } else {
        // ---------------- flush: dQ^T per group, dK^T / dV^T per item ----------------
        const int quarter = warp & 3;
        const int dl = quarter * 32 + lane;  // head-dimension index within a half = TMEM lane
        const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
        const int gshift = __ffsll(p.G) - 1, gmask = (int)p.G - 1;  // G is a power of two
        int64_t ic = 0, u = 0;
        KmItem it;
        bool ok = true;
        for (int64_t pos = 0; ok; ++pos) {
            int32_t idx = -1;
            ok = queue_take(ring, bars + kBarItemFull, bars + kBarItemEmpty, pos, abort_flag, p.wait_limit_ns, true,
                            idx);
            if (!ok || idx < 0) break;
            km_decode(p, idx, it);
            for (int grp = 0; grp < it.ng; ++grp) {
                const int32_t e0 = it.e0 + grp * (int32_t)p.T;
                const int nv = min((int32_t)p.T, it.e0 + it.ne - e0);
                const int nrows = nv * (int)p.G;
                // Lane s holds slot s's query; row rr of the group is (slot rr / G, head g*G + rr % G).
                const int32_t my_q = lane < nv ? __ldg(p.e_q + e0 + lane) : 0;
                for (int h = 0; h < L::kHalves; ++h, ++u) {
                    if (!wait(kDQReady, u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    float *acc = (kDet ? p.dq_fx.est : p.dq_acc) + h * 128 + dl;
                    // All 128 columns to registers, the TMEM released, then the reductions.  Rows come in blocks
                    // of eight heads of one query (G >= 8): one accumulator row address per block, then eight
                    // reductions at fixed offsets.
                    uint32_t v[4][32];
#pragma unroll
                    for (int b4 = 0; b4 < 4; ++b4) tmem_ld32(trow + L::kTmemDQT + b4 * 32, v[b4]);
                    tmem_ld_wait();
                    tc_fence_before();
                    mbar_arrive(bars + kDQFree);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int r0 = jj * 8;  // first row of the block
                        const int64_t q = __shfl_sync(0xffffffffu, my_q, r0 >> gshift);
                        if (r0 < nrows) {
                            const int64_t off = ((it.b * p.S_q + q) * p.Hq + it.g * p.G + (r0 & gmask)) * D;
#pragma unroll
                            for (int t = 0; t < 8; ++t) {
                                const float x = __uint_as_float(v[jj >> 2][(jj & 3) * 8 + t]);
                                if (kDet) red_add_fx(acc + off + t * D, p.dq_fx.lo + (acc - p.dq_fx.est) + off + t * D, x);
                                else red_add_f32(acc + off + t * D, x);
                            }
                        }
                    }
                }
                if (!ok) break;
            }
            if (!ok) break;
            // The item's dK^T / dV^T: one column per chunk key.
            if (!wait(kDKVReady, ic)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int64_t row_stride = p.Hkv * D;
            const int64_t key0 = it.c * kChunkKeys;
            const int64_t base_off = (it.b * p.S_kv * p.Hkv + it.g) * D + dl;
            const int nkeys = p.S_kv - key0 < kChunkKeys ? (int)(p.S_kv - key0) : kChunkKeys;
            for (int h = 0; h < L::kHalves; ++h) {
                uint32_t a[2][32], w[2][32];
                tmem_ld32(trow + L::kTmemDKT + 64 * h, a[0]);
                tmem_ld32(trow + L::kTmemDKT + 64 * h + 32, a[1]);
                tmem_ld32(trow + L::kTmemDVT + 64 * h, w[0]);
                tmem_ld32(trow + L::kTmemDVT + 64 * h + 32, w[1]);
                tmem_ld_wait();
                if (h == L::kHalves - 1) {
                    tc_fence_before();
                    mbar_arrive(bars + kDKVFree);
                }
                int64_t off = base_off + key0 * row_stride + h * 128;
#pragma unroll
                for (int j = 0; j < kChunkKeys; ++j) {
                    if (j < nkeys) {
                        const float xk = __uint_as_float(a[j >> 5][j & 31]);
                        const float xv = __uint_as_float(w[j >> 5][j & 31]);
                        if (kDet) {
                            red_add_fx(p.dk_fx, off, xk);
                            red_add_fx(p.dv_fx, off, xv);
                        } else {
                            red_add_f32(p.dk_acc + off, xk);
                            red_add_f32(p.dv_acc + off, xv);
                        }
                    }
                    off += row_stride;
                }
            }
            ++ic;
        }
        if (!ok) fail(6);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, kTmemCols);
}

// fp32 dQ accumulator (or the exact pair est/lo) -> BF16 dQ.
template <bool kDet>
__global__ void dq_convert_kernel(const float *acc, FxAcc fx, __nv_bfloat16 *dq, int64_t n8, const int32_t *gate) {
    if (gate && *gate == 0) return;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        float f[8];
        if (kDet) {
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = fx_to_f32(fx.est[8 * i + e], fx.lo[8 * i + e]);
        } else {
            const float4 *a4 = reinterpret_cast<const float4 *>(acc) + 2 * i;
            const float4 x = a4[0], y = a4[1];
            f[0] = x.x, f[1] = x.y, f[2] = x.z, f[3] = x.w, f[4] = y.x, f[5] = y.y, f[6] = y.z, f[7] = y.w;
        }
        reinterpret_cast<uint4 *>(dq)[i] = f32x8_to_bf16(f);
    }
}

template <int D>
cudaError_t set_km_smem() {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(km_bwd_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             KmLayout<D>::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(km_bwd_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 KmLayout<D>::kSmemBytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

}  // namespace

bool km_backward_shape_ok(const AttnArgs &a) {
    const bool pow2 = a.G > 0 && (a.G & (a.G - 1)) == 0;
    return pow2 && a.G >= 8 && a.G <= 64 && (a.D == 256 || a.D == 128);
}

cudaError_t launch_km_backward(const BwdArgs &bw, const KmArgs &k, cudaStream_t s) {
    const AttnArgs &a = bw.f;
    const int64_t D = a.D;
    KmParams p;
    memset(&p, 0, sizeof(p));
    const int64_t T = kTileRows / a.G;
    {
        // Q and dO: eight heads of one query with all D/64 panels in one copy (panel stride 128 bytes).
        const uint32_t box[5] = {64, 8, (uint32_t)(D / 64), 1, 1};
        const int64_t qd[5] = {64, a.Hq, D / 64, a.S_q, a.B};
        const int64_t qst[4] = {a.qs2, 64, a.qs1, a.qs0};
        const int64_t dst[4] = {D, 64, a.Hq * D, a.S_q * a.Hq * D};
        if (!tc_encode_bf16_map(&p.q_map, a.q, 5, qd, qst, box) || !tc_encode_bf16_map(&p.do_map, bw.dout, 5, qd, dst, box))
            return cudaErrorInvalidValue;
    }
    if (!tc_encode_tile_map(&p.k_map, a.k, a.Hkv, a.S_kv, a.B, a.ks2, a.ks1, a.ks0, 1, kChunkKeys, D))
        return cudaErrorInvalidValue;
    if (!tc_encode_tile_map(&p.v_map, a.v, a.Hkv, a.S_kv, a.B, a.vs2, a.vs1, a.vs0, 1, kChunkKeys, D))
        return cudaErrorInvalidValue;
    {
        cudaError_t e = D == 128 ? set_km_smem<128>() : set_km_smem<256>();
        if (e != cudaSuccess) return e;
    }
    p.B = a.B;
    p.S_q = a.S_q;
    p.S_kv = a.S_kv;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.G;
    p.T = T;
    p.NC = k.NC;
    p.sl2 = a.scale * kLog2e;
    p.scale = a.scale;
    p.wait_limit_ns = tc_wait_limit_ns(kWaitLimitNs);
    p.items = k.items;
    p.queue = k.queue;
    p.meta = k.meta;
    p.e_q = k.e_q;
    p.e_mask = k.e_mask;
    p.sched = k.sched;
    p.lse = bw.lse;
    p.delta = bw.delta;
    p.dq_acc = k.dq_acc;
    p.dq_fx = k.dq_fx;
    p.dk_acc = bw.dk_acc;
    p.dv_acc = bw.dv_acc;
    p.dk_fx = bw.dk_fx;
    p.dv_fx = bw.dv_fx;
    p.gate = k.gate;
    p.status = a.status;
    const int grid = tc_num_sms();
    const bool det = bw.dk_fx.est != nullptr;
    if (D == 128) {
        if (det) km_bwd_kernel<128, true><<<grid, kThreads, KmLayout<128>::kSmemBytes, s>>>(p);
        else km_bwd_kernel<128, false><<<grid, kThreads, KmLayout<128>::kSmemBytes, s>>>(p);
    } else {
        if (det) km_bwd_kernel<256, true><<<grid, kThreads, KmLayout<256>::kSmemBytes, s>>>(p);
        else km_bwd_kernel<256, false><<<grid, kThreads, KmLayout<256>::kSmemBytes, s>>>(p);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t n8 = a.B * a.S_q * a.Hq * D / 8;
    const int64_t nb = (n8 + 255) / 256;
    const int blocks = (int)std::min<int64_t>(nb, (int64_t)tc_num_sms() * 16);
    if (det) dq_convert_kernel<true><<<blocks, 256, 0, s>>>(nullptr, k.dq_fx, bw.dq, n8, k.gate);
    else dq_convert_kernel<false><<<blocks, 256, 0, s>>>(k.dq_acc, FxAcc{}, bw.dq, n8, k.gate);
    return cudaGetLastError();
}

}  // namespace qsa

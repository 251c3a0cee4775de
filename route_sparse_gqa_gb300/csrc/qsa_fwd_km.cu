// qsa_fwd_km.cu -- key-major forward of route-set sparse GQA on tcgen05 tensor cores.
//
// The tile forward gives each 128-row MMA the T = 128/G queries of one tile and
// walks the union of their routed keys; when those queries share few keys (long
// prefixes with scattered routed blocks) most (row, key) pairs it computes are
// masked.  This forward walks the reverse lists instead (the same work items as
// the key-major backward: per aligned 64-key chunk, groups of T queries that
// route into it), so every MMA row is a routed (query, head) pair.  A row's
// softmax then spans many work items, so it runs in two passes over the items:
//
//   pass 1 (km_fwd_max_kernel)  S = Q K^T per group; per row the maximum of
//                               scale * s * log2(e) over the chunk's routed
//                               keys, folded into the row's maximum with a
//                               reduction (an order-preserving integer encoding
//                               of the float, so an integer max is the float
//                               max);
//   pass 2 (km_fwd_out_kernel)  S again; P = exp2(s * scale * log2e - max_row),
//                               exact relative to the row's final maximum, so
//                               the partial products of different items add up
//                               directly: O^T += V^T P^T into TMEM, reduced into
//                               an fp32 O accumulator, and sum(P) reduced into
//                               the row's l;
//   finalize                    O = acc / l (BF16), LSE = (max + log2 l) ln 2.
//
// Rows with no valid route keep max = -inf and l = 0: O = 0, LSE = -inf.  Which
// forward runs is decided on the device from the preprocessed routes
// (km_choose_kernel): both are launched, and the one not chosen returns at once.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "qsa_tc.cuh"
#include "qsa_tc_ptx.cuh"
#include "qsa_queue.cuh"

namespace qsa {
namespace {

using namespace ptx;

constexpr uint32_t kKVPanel = kChunkKeys * 128;          // 8 KiB: 64 columns of a 64-key chunk
constexpr uint32_t kPBytes = kTileRows * kChunkKeys * 2;  // 16 KiB: P of one group
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Order-preserving encoding of a float as a signed integer (non-NaN): the
// integer maximum of encodings is the encoding of the float maximum.
__device__ __forceinline__ int32_t enc_max(float f) {
    const int32_t i = __float_as_int(f);
    return i >= 0 ? i : i ^ 0x7FFFFFFF;
}
__device__ __forceinline__ float dec_max(int32_t i) { return __int_as_float(i >= 0 ? i : i ^ 0x7FFFFFFF); }
constexpr int32_t kEncNegInf = (int32_t)(0xFF800000u ^ 0x7FFFFFFFu);  // enc_max(-inf)

__device__ __forceinline__ void red_max_s32(int32_t *addr, int32_t v) {
    asm volatile("red.relaxed.gpu.global.max.s32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

struct KfParams {
    // 5-D {64, Hq, D/64, S_q, B}, box {64, 8, D/64, 1, 1}: eight heads of one query, every panel
    // ([panel][8 rows][128 B], one copy), as in the key-major backward.
    CUtensorMap q_map;
    CUtensorMap k_map, v_map;  // 4-D {D, Hkv, S_kv, B}, box {64, 1, 64, 1}: one chunk of one KV head
    int64_t B, S_q, S_kv, Hq, Hkv, G, T, NC;
    float sl2;  // softmax_scale * log2(e)
    uint64_t wait_limit_ns;
    const int4 *items;
    const int32_t *queue;
    const int32_t *meta;  // meta[2] = queue length
    const int32_t *e_q;
    const uint64_t *e_mask;
    int32_t *sched;   // work queue counters {next, done}
    // Row statistics, [B, S_q, Hq] (a query's heads adjacent, so one warp's reductions share sectors).
    int32_t *mrow;    // encoded row maximum of s * sl2 (row-max pass only)
    float *mref;      // the exponent reference of the bound (used when *need_max == 0)
    // Pairs {sum of P = exp2(s * sl2 - reference), sum of P rounded to BF16}: the first gives the LSE, the
    // second normalises O, whose numerator sums the same rounded P (so a row's weights add up to one and a
    // row with one routed key returns that key's value exactly).
    float *lrow;
    float *o_acc;     // [B, S_q, Hq, D] fp32
    const int32_t *choice;    // 1: this forward runs
    const int32_t *need_max;  // 1: some row's bound is too loose, the row-max pass runs
    DeviceStatus *status;
};

// The exponent reference of row `stat`: the bound, or the exact maximum when the row-max pass ran.
__device__ __forceinline__ float row_reference(const KfParams &p, bool need_max, int64_t stat) {
    return need_max ? dec_max(__ldg(p.mrow + stat)) : __ldg(p.mref + stat);
}

struct KfItem {
    int64_t b, g, c;
    int32_t e0, ne, ng;
};

__device__ __forceinline__ void kf_decode(const KfParams &p, int32_t idx, KfItem &it) {
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

// Ring slot and phase parity of the n-th use of a ring of R slots.
template <int R>
__device__ __forceinline__ int ring_slot(int64_t n) {
    return (int)((uint64_t)n % R);
}
template <int R>
__device__ __forceinline__ uint32_t ring_parity(int64_t n) {
    return (uint32_t)(((uint64_t)n / R) & 1);
}

// Lane i (< 16) issues the copy of 8-row block i of a group's Q tile: eight heads of one query, every
// panel.  Slots past the group's queries read rows past the end of S_q (zeros).
template <int D>
__device__ __forceinline__ void load_q_group(const KfParams &p, const KfItem &it, int grp, uint32_t dst,
                                             uint64_t *bar, int lane) {
    const int32_t e0 = it.e0 + grp * (int32_t)p.T;
    const int32_t nv = min((int32_t)p.T, it.e0 + it.ne - e0);
    const int q = lane < nv ? __ldg(p.e_q + e0 + lane) : (int)p.S_q;
    const int slot = lane / (int)(p.G / 8), h8 = lane % (int)(p.G / 8);
    const int qs = __shfl_sync(0xffffffffu, q, lane < kTileRows / 8 ? slot : 0);
    if (lane < kTileRows / 8)
        tma_load_5d(dst + (uint32_t)lane * (8 * D * 2), &p.q_map, bar, 0, (int)(it.g * p.G) + 8 * h8, 0, qs,
                    (int)it.b);
}

// ---------------------------------------------------------------------------------------------------
// Pass 1: row maxima.  Warps 0-3: thread = row (TMEM lane); warp 4: producer; warp 5: MMA (lane 0).
constexpr int kMaxThreads = 192;
constexpr int kMaxQStages = 3;
constexpr int kMaxSBufs = 4;
enum MaxBar { kMKFull, kMKFree, kMQFull0, kMQFree0 = kMQFull0 + kMaxQStages, kMSFull0 = kMQFree0 + kMaxQStages,
              kMSFree0 = kMSFull0 + kMaxSBufs, kMDrain = kMSFree0 + kMaxSBufs, kMNumFixed };
constexpr uint32_t kMItemFull = kMNumFixed, kMItemEmpty = kMItemFull + kQueueRing, kMNumBars = kMItemEmpty + kQueueRing;

template <int D>
struct MaxLayout {
    static constexpr int kPanels = D / 64;
    static constexpr uint32_t kTileBytes = kTileRows * D * 2;
    static constexpr uint32_t kKBytes = kChunkKeys * D * 2;
    static constexpr uint32_t kOffQ = 0;  // kMaxQStages tiles
    static constexpr uint32_t kOffK = kOffQ + kMaxQStages * kTileBytes;
    static constexpr uint32_t kOffBar = kOffK + kKBytes;
    static constexpr uint32_t kOffMisc = kOffBar + kMNumBars * 8;
    static constexpr uint32_t kSmemBytes = kOffMisc + 64 + 1024;
};

template <int D>
__global__ void __launch_bounds__(kMaxThreads, 1) km_fwd_max_kernel(const __grid_constant__ KfParams p) {
    // The tile forward runs instead, or every row's bound serves as its reference (uniform over the grid).
    if (*p.choice != 1 || *p.need_max == 0) return;
    using L = MaxLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 8);
    volatile int32_t *ring = reinterpret_cast<volatile int32_t *>(smem + L::kOffMisc + 16);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kMNumFixed; ++i) mbar_init(bars + i, (i >= kMSFree0 && i < kMDrain) ? 128u : 1u);
        for (int i = 0; i < kQueueRing; ++i) {
            mbar_init(bars + kMItemFull + i, 1);
            mbar_init(bars + kMItemEmpty + i, 1 + 128);  // the MMA thread and the row threads take every item
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        prefetch_tmap(&p.q_map);
        prefetch_tmap(&p.k_map);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int zero = 0;
    auto fail = [&](unsigned info) {
        raise_status(p.status, QSA_ERR_TIMEOUT, kSiteKeyFwdWait, info, blockIdx.x);
        *abort_flag = 1;
    };
    // Parity: each ring slot completes one phase per use, and a slot's next use needs an action of the
    // waiting role that follows the wait, so the waited phase is the open one or the one just completed.
    if (warp == 4) {
        // ---------------- producer ----------------
        const int64_t n_queue = p.meta[2];
        int64_t ic = 0, gc = 0, last_q[kMaxQStages] = {-1, -1, -1};
        KfItem it;
        bool ok = true;
        for (int64_t pos = 0; ok; ++pos) {
            int32_t idx = -1;
            if (lane == 0) ok = queue_claim(p.sched, n_queue, ring, bars + kMItemFull, bars + kMItemEmpty, pos,
                                            abort_flag, p.wait_limit_ns, idx);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            idx = __shfl_sync(0xffffffffu, idx, 0);
            if (!ok || idx < 0) break;
            kf_decode(p, idx, it);
            if (ic > 0 && !mbar_wait_warp(bars + kMKFree, (uint32_t)((ic - 1) & 1), abort_flag, p.wait_limit_ns)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(bars + kMKFull, L::kKBytes);
                for (int kb = 0; kb < L::kPanels; ++kb)
                    tma_load_4d(sbase + L::kOffK + kb * kKVPanel, &p.k_map, bars + kMKFull, kb * 64, (int)it.g,
                                (int)(it.c * kChunkKeys), (int)it.b);
            }
            __syncwarp();
            ++ic;
            for (int grp = 0; grp < it.ng; ++grp, ++gc) {
                const int st = ring_slot<kMaxQStages>(gc);
                if (gc >= kMaxQStages && !mbar_wait_warp(bars + kMQFree0 + st, ring_parity<kMaxQStages>(gc - kMaxQStages),
                                                         abort_flag, p.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(bars + kMQFull0 + st, L::kTileBytes);
                __syncwarp();
                load_q_group<D>(p, it, grp, sbase + L::kOffQ + st * L::kTileBytes, bars + kMQFull0 + st, lane);
                __syncwarp();
                last_q[st] = gc;
            }
        }
        if (!ok && lane == 0) fail(1);
        if (lane == 0) queue_finish(p.sched);
        if (lane == 0) {
            bool drained = true;
            if (ic > 0) drained &= mbar_wait(bars + kMKFull, (uint32_t)((ic - 1) & 1), &zero, kWaitLimitNs);
            for (int st = 0; st < kMaxQStages; ++st)
                if (last_q[st] >= 0)
                    drained &= mbar_wait(bars + kMQFull0 + st, ring_parity<kMaxQStages>(last_q[st]), &zero, kWaitLimitNs);
            if (!drained) fail(2);
        }
        __syncwarp();
    } else if (warp == 5) {
        // ---------------- MMA issuer (one thread) ----------------
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16(kTileRows, kChunkKeys, false, false);
            constexpr uint32_t kBlk8 = 8 * D * 2;
            auto w1 = [&](int id, uint32_t parity) { return mbar_wait(bars + id, parity, abort_flag, p.wait_limit_ns); };
            int64_t ic = 0, gc = 0;
            KfItem it;
            bool ok = true;
            for (int64_t pos = 0; ok; ++pos) {
                int32_t idx = -1;
                ok = queue_take(ring, bars + kMItemFull, bars + kMItemEmpty, pos, abort_flag, p.wait_limit_ns, false, idx);
                if (!ok || idx < 0) break;
                kf_decode(p, idx, it);
                ok = w1(kMKFull, (uint32_t)(ic & 1));
                for (int grp = 0; ok && grp < it.ng; ++grp, ++gc) {
                    const int st = ring_slot<kMaxQStages>(gc), sb = ring_slot<kMaxSBufs>(gc);
                    ok = w1(kMQFull0 + st, ring_parity<kMaxQStages>(gc)) &&
                         (gc < kMaxSBufs || w1(kMSFree0 + sb, ring_parity<kMaxSBufs>(gc - kMaxSBufs)));
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t qa = sbase + L::kOffQ + st * L::kTileBytes;
#pragma unroll 1
                    for (int kb = 0; kb < L::kPanels; ++kb)
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_bf16(tmem + sb * kChunkKeys, sdesc_sw128(qa + kb * 1024 + k * 32, 16, kBlk8),
                                     sdesc_sw128(sbase + L::kOffK + kb * kKVPanel + k * 32, 16, 1024), idesc_s,
                                     (kb | k) ? 1u : 0u);
                    mma_commit(bars + kMSFull0 + sb);
                    mma_commit(bars + kMQFree0 + st);
                }
                if (!ok) break;
                mma_commit(bars + kMKFree);  // the item's K chunk is no longer read
                ++ic;
            }
            if (!ok) fail(3);
            mma_commit(bars + kMDrain);
            if (!mbar_wait(bars + kMDrain, 0, &zero, kWaitLimitNs)) fail(4);
        }
        __syncwarp();
    } else {
        // ---------------- row maxima (warps 0-3) ----------------
        const int r = threadIdx.x;
        const int slot = (int)(r / p.G), hl = (int)(r % p.G);
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        int64_t gc = 0;
        KfItem it;
        bool ok = true;
        for (int64_t pos = 0; ok; ++pos) {
            int32_t idx = -1;
            ok = queue_take(ring, bars + kMItemFull, bars + kMItemEmpty, pos, abort_flag, p.wait_limit_ns, true, idx);
            if (!ok || idx < 0) break;
            kf_decode(p, idx, it);
            const int64_t h = it.g * p.G + hl;
            for (int grp = 0; grp < it.ng; ++grp, ++gc) {
                const int sb = ring_slot<kMaxSBufs>(gc);
                const int32_t e = it.e0 + grp * (int32_t)p.T + slot;
                const bool live = e < it.e0 + it.ne;
                const uint64_t mask = live ? __ldg(p.e_mask + e) : 0ull;
                const int64_t q = live ? __ldg(p.e_q + e) : 0;
                if (!mbar_wait_warp(bars + kMSFull0 + sb, ring_parity<kMaxSBufs>(gc), abort_flag, p.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sr[2][32];
                tmem_ld32(trow + sb * kChunkKeys, sr[0]);
                tmem_ld32(trow + sb * kChunkKeys + 32, sr[1]);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(bars + kMSFree0 + sb);
                float mx = -INFINITY;
#pragma unroll
                for (int j = 0; j < 64; ++j)
                    if ((mask >> j) & 1ull) mx = fmaxf(mx, __uint_as_float(sr[j >> 5][j & 31]) * p.sl2);
                if (mask) red_max_s32(p.mrow + (it.b * p.S_q + q) * p.Hq + h, enc_max(mx));
            }
        }
        if (!ok) fail(5);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------------------------------
// Pass 2: outputs.  Warps 0-3: P (thread = row); warps 4-7: O flush (thread = head-dimension index of a
// half); warp 8: producer; warp 9: MMA (lane 0).  S is issued two groups ahead of O^T within an item.
constexpr int kOutThreads = 320;
enum OutBar { kOKVFull, kOKVFree, kOQFull0, kOQFree0 = kOQFull0 + 2, kOSFull0 = kOQFree0 + 2, kOSFree0 = kOSFull0 + 2,
              kOPFull0 = kOSFree0 + 2, kOPFree0 = kOPFull0 + 2, kOOReady0 = kOPFree0 + 2, kOOFree0 = kOOReady0 + 3,
              kODrain = kOOFree0 + 3, kONumFixed };
// O^T is produced in units of one 128-row half of D for one group (u = group * D/128 + half), each in one
// of three 128-column TMEM slots (u mod 3), so the MMA can fill the next unit while the flush still reads
// the two before it.
constexpr int kOSlots = 3;
constexpr uint32_t kOItemFull = kONumFixed, kOItemEmpty = kOItemFull + kQueueRing, kONumBars = kOItemEmpty + kQueueRing;

template <int D>
struct OutLayout {
    static constexpr int kPanels = D / 64;
    static constexpr int kHalves = D / 128;
    static constexpr uint32_t kTileBytes = kTileRows * D * 2;
    static constexpr uint32_t kKVBytes = kChunkKeys * D * 2;
    static constexpr uint32_t kOffQ = 0;  // two tiles
    static constexpr uint32_t kOffK = kOffQ + 2 * kTileBytes;
    static constexpr uint32_t kOffV = kOffK + kKVBytes;
    static constexpr uint32_t kOffP = kOffV + kKVBytes;  // two P buffers
    static constexpr uint32_t kOffBar = kOffP + 2 * kPBytes;
    static constexpr uint32_t kOffMisc = kOffBar + kONumBars * 8;
    static constexpr uint32_t kSmemBytes = kOffMisc + 64 + 1024;
    static constexpr uint32_t kTmemO = 0;                // O^T slot s at 128 s
    static constexpr uint32_t kTmemS = 128 * kOSlots;    // two S buffers of 64 columns
};

template <int D>
__global__ void __launch_bounds__(kOutThreads, 1) km_fwd_out_kernel(const __grid_constant__ KfParams p) {
    if (*p.choice != 1) return;
    using L = OutLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 8);
    volatile int32_t *ring = reinterpret_cast<volatile int32_t *>(smem + L::kOffMisc + 16);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kONumFixed; ++i) {
            const bool many = (i >= kOSFree0 && i < kOSFree0 + 2) || (i >= kOPFull0 && i < kOPFull0 + 2) ||
                              (i >= kOOFree0 && i < kOOFree0 + kOSlots);
            mbar_init(bars + i, many ? 128u : 1u);
        }
        for (int i = 0; i < kQueueRing; ++i) {
            mbar_init(bars + kOItemFull + i, 1);
            mbar_init(bars + kOItemEmpty + i, 1 + 128 + 128);  // MMA thread, P threads, flush threads
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp == 8 && lane == 0) {
        prefetch_tmap(&p.q_map);
        prefetch_tmap(&p.k_map);
        prefetch_tmap(&p.v_map);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int zero = 0;
    auto fail = [&](unsigned info) {
        raise_status(p.status, QSA_ERR_TIMEOUT, kSiteKeyFwdWait, 10 + info, blockIdx.x);
        *abort_flag = 1;
    };
    auto waitw = [&](int id, uint32_t parity) { return mbar_wait_warp(bars + id, parity, abort_flag, p.wait_limit_ns); };
    // Parity: as in pass 1, each slot completes one phase per use and its next use needs an action of the
    // waiting role that follows the wait.
    if (warp == 8) {
        // ---------------- producer ----------------
        const int64_t n_queue = p.meta[2];
        int64_t ic = 0, gc = 0, last_q[2] = {-1, -1};
        KfItem it;
        bool ok = true;
        for (int64_t pos = 0; ok; ++pos) {
            int32_t idx = -1;
            if (lane == 0) ok = queue_claim(p.sched, n_queue, ring, bars + kOItemFull, bars + kOItemEmpty, pos,
                                            abort_flag, p.wait_limit_ns, idx);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            idx = __shfl_sync(0xffffffffu, idx, 0);
            if (!ok || idx < 0) break;
            kf_decode(p, idx, it);
            if (ic > 0 && !waitw(kOKVFree, (uint32_t)((ic - 1) & 1))) {
                ok = false;
                break;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(bars + kOKVFull, 2 * L::kKVBytes);
                for (int kb = 0; kb < L::kPanels; ++kb) {
                    tma_load_4d(sbase + L::kOffK + kb * kKVPanel, &p.k_map, bars + kOKVFull, kb * 64, (int)it.g,
                                (int)(it.c * kChunkKeys), (int)it.b);
                    tma_load_4d(sbase + L::kOffV + kb * kKVPanel, &p.v_map, bars + kOKVFull, kb * 64, (int)it.g,
                                (int)(it.c * kChunkKeys), (int)it.b);
                }
            }
            __syncwarp();
            ++ic;
            for (int grp = 0; grp < it.ng; ++grp, ++gc) {
                const int st = ring_slot<2>(gc);
                if (gc >= 2 && !waitw(kOQFree0 + st, ring_parity<2>(gc - 2))) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(bars + kOQFull0 + st, L::kTileBytes);
                __syncwarp();
                load_q_group<D>(p, it, grp, sbase + L::kOffQ + st * L::kTileBytes, bars + kOQFull0 + st, lane);
                __syncwarp();
                last_q[st] = gc;
            }
        }
        if (!ok && lane == 0) fail(1);
        if (lane == 0) queue_finish(p.sched);
        if (lane == 0) {
            bool drained = true;
            if (ic > 0) drained &= mbar_wait(bars + kOKVFull, (uint32_t)((ic - 1) & 1), &zero, kWaitLimitNs);
            for (int st = 0; st < 2; ++st)
                if (last_q[st] >= 0)
                    drained &= mbar_wait(bars + kOQFull0 + st, ring_parity<2>(last_q[st]), &zero, kWaitLimitNs);
            if (!drained) fail(2);
        }
        __syncwarp();
    } else if (warp == 9) {
        // ---------------- MMA issuer (one thread) ----------------
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16(kTileRows, kChunkKeys, false, false);
            constexpr uint32_t idesc_o = idesc_bf16(128, kTileRows, true, false);  // O^T = V^T P^T
            constexpr uint32_t kBlk8 = 8 * D * 2;
            auto w1 = [&](int id, uint32_t parity) { return mbar_wait(bars + id, parity, abort_flag, p.wait_limit_ns); };
            auto issue_s = [&](int64_t g) {
                const int st = ring_slot<2>(g), sb = ring_slot<2>(g);
                if (!w1(kOQFull0 + st, ring_parity<2>(g)) || (g >= 2 && !w1(kOSFree0 + sb, ring_parity<2>(g - 2))))
                    return false;
                tc_fence_after();
                const uint32_t qa = sbase + L::kOffQ + st * L::kTileBytes;
                // Panel loop rolled, K steps unrolled: smaller code for the instruction cache this warp shares.
#pragma unroll 1
                for (int kb = 0; kb < L::kPanels; ++kb)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_bf16(tmem + L::kTmemS + sb * kChunkKeys, sdesc_sw128(qa + kb * 1024 + k * 32, 16, kBlk8),
                                 sdesc_sw128(sbase + L::kOffK + kb * kKVPanel + k * 32, 16, 1024), idesc_s,
                                 (kb | k) ? 1u : 0u);
                mma_commit(bars + kOSFull0 + sb);
                mma_commit(bars + kOQFree0 + st);
                return true;
            };
            int64_t ic = 0, gc = 0, u = 0;
            KfItem it;
            bool ok = true;
            for (int64_t pos = 0; ok; ++pos) {
                int32_t idx = -1;
                ok = queue_take(ring, bars + kOItemFull, bars + kOItemEmpty, pos, abort_flag, p.wait_limit_ns, false, idx);
                if (!ok || idx < 0) break;
                kf_decode(p, idx, it);
                ok = w1(kOKVFull, (uint32_t)(ic & 1));
                tc_fence_after();
                for (int grp = 0; ok && grp < 2 && grp < it.ng; ++grp) ok = issue_s(gc + grp);
                for (int grp = 0; ok && grp < it.ng; ++grp) {
                    const int64_t g = gc + grp;
                    const int pb = ring_slot<2>(g);
                    ok = w1(kOPFull0 + pb, ring_parity<2>(g));
                    for (int h = 0; ok && h < L::kHalves; ++h, ++u) {
                        // The flush has read the slot's previous unit.
                        const int sl = ring_slot<kOSlots>(u);
                        ok = u < kOSlots || w1(kOOFree0 + sl, ring_parity<kOSlots>(u - kOSlots));
                        if (!ok) break;
                        tc_fence_after();
#pragma unroll
                        for (int k = 0; k < kChunkKeys / 16; ++k)
                            mma_bf16(tmem + L::kTmemO + 128 * sl,
                                     sdesc_sw128(sbase + L::kOffV + (2 * h) * kKVPanel + k * 2048, kKVPanel, 1024),
                                     sdesc_sw128(sbase + L::kOffP + pb * kPBytes + k * 32, 16, 1024), idesc_o,
                                     k ? 1u : 0u);
                        mma_commit(bars + kOOReady0 + sl);
                    }
                    if (!ok) break;
                    mma_commit(bars + kOPFree0 + pb);
                    if (grp + 2 < it.ng) ok = issue_s(g + 2);
                }
                if (!ok) break;
                mma_commit(bars + kOKVFree);  // the item's K/V chunk is no longer read
                gc += it.ng;
                ++ic;
            }
            if (!ok) fail(3);
            mma_commit(bars + kODrain);
            if (!mbar_wait(bars + kODrain, 0, &zero, kWaitLimitNs)) fail(4);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ---------------- P = exp2(s - max) (thread = row) ----------------
        const int r = threadIdx.x;
        const int slot = (int)(r / p.G), hl = (int)(r % p.G);
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        const bool need_max = *p.need_max != 0;
        int64_t gc = 0;
        KfItem it;
        bool ok = true;
        for (int64_t pos = 0; ok; ++pos) {
            int32_t idx = -1;
            ok = queue_take(ring, bars + kOItemFull, bars + kOItemEmpty, pos, abort_flag, p.wait_limit_ns, true, idx);
            if (!ok || idx < 0) break;
            kf_decode(p, idx, it);
            const int64_t h = it.g * p.G + hl;
            for (int grp = 0; grp < it.ng; ++grp, ++gc) {
                const int sb = ring_slot<2>(gc);
                const int32_t e = it.e0 + grp * (int32_t)p.T + slot;
                const bool live = e < it.e0 + it.ne;
                const uint64_t mask = live ? __ldg(p.e_mask + e) : 0ull;
                const int64_t q = live ? __ldg(p.e_q + e) : 0;
                const int64_t stat = (it.b * p.S_q + q) * p.Hq + h;
                const float m2 = mask ? row_reference(p, need_max, stat) : 0.f;
                if (!waitw(kOSFull0 + sb, ring_parity<2>(gc))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sr[2][32];
                tmem_ld32(trow + L::kTmemS + sb * kChunkKeys, sr[0]);
                tmem_ld32(trow + L::kTmemS + sb * kChunkKeys + 32, sr[1]);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(bars + kOSFree0 + sb);
                uint32_t pk[32];
                float lsum = 0.f, lsum_b = 0.f;
#pragma unroll
                for (int j = 0; j < 64; j += 2) {
                    const float p0 = ((mask >> j) & 1ull) ? ex2(__uint_as_float(sr[j >> 5][j & 31]) * p.sl2 - m2) : 0.f;
                    const float p1 = ((mask >> (j + 1)) & 1ull)
                                         ? ex2(__uint_as_float(sr[(j + 1) >> 5][(j + 1) & 31]) * p.sl2 - m2)
                                         : 0.f;
                    lsum += p0 + p1;
                    const uint32_t w = pack_bf16(p0, p1);
                    lsum_b += __uint_as_float(w << 16) + __uint_as_float(w & 0xFFFF0000u);
                    pk[j >> 1] = w;
                }
                if (gc >= 2 && !waitw(kOPFree0 + sb, ring_parity<2>(gc - 2))) {
                    ok = false;
                    break;
                }
                uint8_t *prow = smem + L::kOffP + sb * kPBytes + r * 128;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    *reinterpret_cast<uint4 *>(prow + (ch ^ (r & 7)) * 16) =
                        make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bars + kOPFull0 + sb);
                if (mask) red_add_v2_f32(p.lrow + 2 * stat, lsum, lsum_b);
            }
        }
        if (!ok) fail(5);
    } else {
        // ---------------- O^T flush into the fp32 accumulator (thread = head-dimension index) ----------------
        const int quarter = warp & 3;
        const int dl = quarter * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
        const int gshift = __ffsll(p.G) - 1, gmask = (int)p.G - 1;  // G is a power of two, at least 8
        int64_t gc = 0, u = 0;
        KfItem it;
        bool ok = true;
        for (int64_t pos = 0; ok; ++pos) {
            int32_t idx = -1;
            ok = queue_take(ring, bars + kOItemFull, bars + kOItemEmpty, pos, abort_flag, p.wait_limit_ns, true, idx);
            if (!ok || idx < 0) break;
            kf_decode(p, idx, it);
            for (int grp = 0; grp < it.ng; ++grp, ++gc) {
                const int32_t e0 = it.e0 + grp * (int32_t)p.T;
                const int nv = min((int32_t)p.T, it.e0 + it.ne - e0);
                const int nrows = nv * (int)p.G;
                const int32_t my_q = lane < nv ? __ldg(p.e_q + e0 + lane) : 0;  // lane s: slot s's query
                for (int h = 0; h < L::kHalves; ++h, ++u) {
                    const int sl = ring_slot<kOSlots>(u);
                    if (!waitw(kOOReady0 + sl, ring_parity<kOSlots>(u))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // 64 rows at a time (fewer live registers); the TMEM half is released after the second read.
                    float *acc = p.o_acc + h * 128 + dl;
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        uint32_t v[2][32];
                        tmem_ld32(trow + L::kTmemO + 128 * sl + part * 64, v[0]);
                        tmem_ld32(trow + L::kTmemO + 128 * sl + part * 64 + 32, v[1]);
                        tmem_ld_wait();
                        if (part == 1) {
                            tc_fence_before();
                            mbar_arrive(bars + kOOFree0 + sl);
                        }
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) {
                            const int r0 = part * 64 + jj * 8;  // eight heads of one query
                            const int64_t q = __shfl_sync(0xffffffffu, my_q, r0 >> gshift);
                            if (r0 < nrows) {
                                const int64_t off = ((it.b * p.S_q + q) * p.Hq + it.g * p.G + (r0 & gmask)) * D;
#pragma unroll
                                for (int t = 0; t < 8; ++t)
                                    red_add_f32(acc + off + t * D, __uint_as_float(v[jj >> 2][(jj & 3) * 8 + t]));
                            }
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
    if (warp == 9) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------------------------------
// Accumulator set-up and the final division.
// Exponent references without a row-max pass.  By Cauchy-Schwarz every score of row (q, h) satisfies
// s * sl2 <= |sl2| |q_h| max_j |k_j,g| =: m_ref, so P = exp2(s sl2 - m_ref) <= 1 (no overflow, as with
// the exact maximum).  The row's maximum is at least the score s0 of any one routed key (its first one
// here), so m_ref - s0 bounds how far the largest P falls below 1.  While that gap is at most
// kMaxRefGap = 64 for every row, the largest P of a row is >= 2^-64: terms that fall below fp32's normal
// range (2^-126) change l by less than K 2^-62 relative, and products flushed in the tensor core change
// O by less than K 2^-62 absolute, far below the BF16 rounding of the outputs; the results equal those
// with the exact maximum up to rounding.  A row with a wider gap sets *need_max and the row-max pass
// computes exact maxima for all rows.
constexpr float kMaxRefGap = 64.f;

// Largest squared key norm per (batch row, KV head) over all keys (one atomicMax per CTA and head on the
// float bits, which order as unsigned integers for non-negative values).
__global__ void __launch_bounds__(256) km_key_norm_kernel(AttnArgs a, const int32_t *choice, unsigned *kmax2) {
    if (*choice != 1) return;
    __shared__ unsigned smax[64];
    const int lane = threadIdx.x & 31;
    const int64_t Hkv = a.Hkv, nb = a.B * Hkv;
    for (int i = threadIdx.x; i < nb && i < 64; i += blockDim.x) smax[i] = 0u;
    __syncthreads();
    const int64_t n_rows = a.B * a.S_kv * Hkv;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < n_rows; row += warps) {
        const int64_t g = row % Hkv, bj = row / Hkv;
        const int64_t b = bj / a.S_kv, j = bj % a.S_kv;
        float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (lane * 8 < a.D)
            bf16x8_to_f32(*reinterpret_cast<const uint4 *>(a.k + b * a.ks0 + j * a.ks1 + g * a.ks2 + lane * 8), f);
        float n2 = 0.f;
#pragma unroll
        for (int t = 0; t < 8; ++t) n2 = fmaf(f[t], f[t], n2);
        n2 = warp_sum(n2);
        if (lane == 0) {
            const int64_t bg = b * Hkv + g;
            if (nb <= 64) atomicMax(&smax[bg], __float_as_uint(n2));
            else atomicMax(kmax2 + bg, __float_as_uint(n2));
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nb && nb <= 64; i += blockDim.x)
        if (smax[i]) atomicMax(kmax2 + i, smax[i]);
}

// Zeroes the accumulators and the row sums, resets the row maxima, and writes each row's reference: one
// warp per (b, q) and eight heads of one KV head (their Q rows and the key row of the query's first routed
// key are loaded together; lane l holds elements 8l..8l+7).
__global__ void __launch_bounds__(256) km_fwd_init_kernel(KfParams p, AttnArgs a, const int32_t *ids,
                                                          const int32_t *counts, int64_t K,
                                                          const unsigned *kmax2, int force_max,
                                                          int32_t *need_max, int64_t n_o4) {
    if (*p.choice != 1) return;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    float4 *o4 = reinterpret_cast<float4 *>(p.o_acc);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_o4; i += stride)
        o4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (force_max && blockIdx.x == 0 && threadIdx.x == 0) *need_max = 1;
    const int lane = threadIdx.x & 31;
    const int64_t h8n = p.Hq / 8;  // eight-head groups per query (G is a multiple of 8)
    const int64_t n_task = p.B * p.S_q * h8n;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const float asl2 = fabsf(p.sl2);
    const bool on = lane * 8 < a.D;
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < n_task; t += warps) {
        const int64_t bq = t / h8n, h0 = (t % h8n) * 8;
        const int64_t b = bq / p.S_q, q = bq % p.S_q;
        const int64_t g = h0 / p.G;
        const int32_t cnt = __ldg(counts + bq);
        const int32_t j0 = __ldg(ids + bq * K);
        uint4 qv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            qv[j] = on && cnt > 0 ? __ldg(reinterpret_cast<const uint4 *>(a.q + b * a.qs0 + q * a.qs1 + (h0 + j) * a.qs2) + lane)
                                  : make_uint4(0u, 0u, 0u, 0u);
        float kf[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (on && cnt > 0)
            bf16x8_to_f32(__ldg(reinterpret_cast<const uint4 *>(a.k + b * a.ks0 + (int64_t)j0 * a.ks1 + g * a.ks2) + lane), kf);
        float n2[8], dot[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float qf[8];
            bf16x8_to_f32(qv[j], qf);
            n2[j] = 0.f;
            dot[j] = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                n2[j] = fmaf(qf[e], qf[e], n2[j]);
                dot[j] = fmaf(qf[e], kf[e], dot[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            n2[j] = warp_sum(n2[j]);
            dot[j] = warp_sum(dot[j]);
        }
        if (lane < 8) {
            float nj = 0.f, dj = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j == lane) {
                    nj = n2[j];
                    dj = dot[j];
                }
            const int64_t stat = bq * p.Hq + h0 + lane;
            // Rounded up by 2^-10 relative: covers the fp32 rounding of the norms and of the tensor-core dot
            // products (each far below 2^-16 relative of |q| |k|).
            const float mref = asl2 * sqrtf(nj) * sqrtf(__uint_as_float(kmax2[b * p.Hkv + g])) * (1.f + 1.f / 1024.f);
            p.mref[stat] = mref;
            p.mrow[stat] = kEncNegInf;
            reinterpret_cast<float2 *>(p.lrow)[stat] = make_float2(0.f, 0.f);
            if (cnt > 0 && !(mref - dj * p.sl2 <= kMaxRefGap)) *need_max = 1;  // also catches NaN / inf
        }
    }
}

// O = acc / l as BF16 (zero for rows without routes), LSE = (reference + log2 l) ln 2 (natural log, -inf for
// rows without routes).  Each thread converts 16 consecutive elements of a row (four loads in flight).
template <int D>
__global__ void km_fwd_final_kernel(KfParams p, __nv_bfloat16 *o, float *lse) {
    if (*p.choice != 1) return;
    const bool need_max = *p.need_max != 0;
    const int64_t n_rows = p.B * p.S_q * p.Hq;  // (b, q, h) rows of O
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    constexpr int kPer = D / 16;  // threads per row, 16 elements each
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_rows * kPer; i += stride) {
        const int64_t row = i / kPer;  // [B, S_q, Hq]: also the row statistics' index
        const float4 *a4 = reinterpret_cast<const float4 *>(p.o_acc) + 4 * i;
        float4 x[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = a4[j];
        const float2 ls = reinterpret_cast<const float2 *>(p.lrow)[row];
        const float inv = ls.y > 0.f ? 1.f / ls.y : 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float f[8] = {x[2 * j].x * inv, x[2 * j].y * inv, x[2 * j].z * inv, x[2 * j].w * inv,
                                x[2 * j + 1].x * inv, x[2 * j + 1].y * inv, x[2 * j + 1].z * inv, x[2 * j + 1].w * inv};
            reinterpret_cast<uint4 *>(o)[2 * i + j] = f32x8_to_bf16(f);
        }
        if (i % kPer == 0) {
            const int64_t h = row % p.Hq, bq = row / p.Hq;
            const int64_t b = bq / p.S_q, q = bq % p.S_q;
            lse[(b * p.Hq + h) * p.S_q + q] = ls.x > 0.f ? (row_reference(p, need_max, row) + __log2f(ls.x)) * kLn2
                                                         : -INFINITY;
        }
    }
}

template <int D>
cudaError_t set_km_fwd_smem() {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(km_fwd_max_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             MaxLayout<D>::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(km_fwd_out_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 OutLayout<D>::kSmemBytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// One CTA: which forward runs, from the work each path would do.  The tile path computes every (row, key)
// pair of its tiles' chunk unions, one chunk of T queries per unit (a tile's distinct routed keys packed 64
// to a chunk); the key-major path computes only routed
// pairs, one group of T queries per unit, but reduces its outputs through L2, so a group costs about as
// much as kFwdRatio tile chunks.  choice[2], choice[3]: the two unit counts (saturated), for inspection.
constexpr int kFwdRatioNum = 3, kFwdRatioDen = 1;
__global__ void __launch_bounds__(1024) km_choose_kernel(const int32_t *tile_keys, int64_t n_tiles,
                                                         const int32_t *list_start, int64_t n_lists, int64_t slots,
                                                         int force_fwd, int force_bwd, int bwd_num, int bwd_den,
                                                         int32_t *choice) {
    __shared__ unsigned long long tot[2];
    if (threadIdx.x == 0) tot[0] = tot[1] = 0ull;
    __syncthreads();
    unsigned long long a = 0, g = 0;
    for (int64_t i = threadIdx.x; i < n_tiles; i += blockDim.x) a += (unsigned long long)((tile_keys[i] + 63) / 64);
    for (int64_t i = threadIdx.x; i < n_lists; i += blockDim.x)
        g += (unsigned long long)((list_start[i + 1] - list_start[i] + slots - 1) / slots);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        g += __shfl_xor_sync(0xffffffffu, g, o);
    }
    if ((threadIdx.x & 31) == 0) {
        atomicAdd(&tot[0], a);
        atomicAdd(&tot[1], g);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned long long chunks = tot[0], groups = tot[1];
        const int fwd = n_tiles == 0 ? 1 : (groups * kFwdRatioNum < chunks * kFwdRatioDen ? 1 : 0);
        const int bwd = n_tiles == 0 || bwd_den == 0 ? 1 : (groups * bwd_num < chunks * bwd_den ? 1 : 0);
        choice[0] = force_fwd >= 0 ? force_fwd : fwd;
        choice[1] = bwd_den == 0 ? 1 : force_bwd >= 0 ? force_bwd : bwd;
        choice[2] = (int32_t)(chunks < 0x7FFFFFFFull ? chunks : 0x7FFFFFFFull);
        choice[3] = (int32_t)(groups < 0x7FFFFFFFull ? groups : 0x7FFFFFFFull);
    }
}

}  // namespace

// QSA_DEBUG_FORWARD_PATH / QSA_DEBUG_BACKWARD_PATH = "tile" or "keymajor" override the choice (a test hook
// that runs either path on any problem both accept); -1 when unset.
int forced_path(const char *var) {
    const char *env = std::getenv(var);
    if (!env) return -1;
    if (!std::strcmp(env, "tile")) return 0;
    if (!std::strcmp(env, "keymajor")) return 1;
    return -1;
}

bool km_forward_shape_ok(const AttnArgs &a) {
    const bool pow2 = a.G > 0 && (a.G & (a.G - 1)) == 0;
    return pow2 && a.G >= 8 && a.G <= 64 && (a.D == 256 || a.D == 128);
}

cudaError_t launch_km_choose(const int32_t *tile_keys, int64_t n_tiles, const int32_t *list_start,
                             int64_t n_lists, int64_t slots, int64_t D, bool tile_bwd_ok, bool tile_fwd_only,
                             int32_t *choice, cudaStream_t s) {
    // Backward: a key-major group costs about kBwdRatio tile chunks (per unit and KV head: tile 33-34 ns and
    // key-major 35-41 ns at D = 256 on train-step and right-padded; 24 against 32 ns at D = 128).
    const int bwd_num = D == 128 ? 27 : 6, bwd_den = tile_bwd_ok ? (D == 128 ? 20 : 5) : 0;
    km_choose_kernel<<<1, 1024, 0, s>>>(tile_keys, n_tiles, list_start, n_lists, slots,
                                        tile_fwd_only ? 0 : forced_path("QSA_DEBUG_FORWARD_PATH"),
                                        forced_path("QSA_DEBUG_BACKWARD_PATH"),
                                        bwd_num, bwd_den, choice);
    return cudaGetLastError();
}

cudaError_t launch_km_forward(const AttnArgs &a, const KfArgs &k, __nv_bfloat16 *o, float *lse, cudaStream_t s) {
    const int64_t D = a.D;
    KfParams p;
    memset(&p, 0, sizeof(p));
    {
        const uint32_t box[5] = {64, 8, (uint32_t)(D / 64), 1, 1};
        const int64_t qd[5] = {64, a.Hq, D / 64, a.S_q, a.B};
        const int64_t qst[4] = {a.qs2, 64, a.qs1, a.qs0};
        if (!tc_encode_bf16_map(&p.q_map, a.q, 5, qd, qst, box)) return cudaErrorInvalidValue;
    }
    if (!tc_encode_tile_map(&p.k_map, a.k, a.Hkv, a.S_kv, a.B, a.ks2, a.ks1, a.ks0, 1, kChunkKeys, D))
        return cudaErrorInvalidValue;
    if (!tc_encode_tile_map(&p.v_map, a.v, a.Hkv, a.S_kv, a.B, a.vs2, a.vs1, a.vs0, 1, kChunkKeys, D))
        return cudaErrorInvalidValue;
    {
        cudaError_t e = D == 128 ? set_km_fwd_smem<128>() : set_km_fwd_smem<256>();
        if (e != cudaSuccess) return e;
    }
    p.B = a.B;
    p.S_q = a.S_q;
    p.S_kv = a.S_kv;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.G;
    p.T = kTileRows / a.G;
    p.NC = k.NC;
    p.sl2 = a.scale * kLog2e;
    p.wait_limit_ns = tc_wait_limit_ns(kWaitLimitNs);
    p.items = k.items;
    p.queue = k.queue;
    p.meta = k.meta;
    p.e_q = k.e_q;
    p.e_mask = k.e_mask;
    p.mrow = k.mrow;
    p.mref = k.mref;
    p.lrow = k.lrow;
    p.o_acc = k.o_acc;
    p.choice = k.choice;
    p.need_max = k.kbound;
    p.status = a.status;
    const int sms = tc_num_sms();
    const int64_t n_o4 = a.B * a.S_q * a.Hq * D / 4;
    // kbound = {need_max, -, ..., squared key norm maxima from word kKeyNormWord}: cleared, then filled.
    unsigned *kmax2 = reinterpret_cast<unsigned *>(k.kbound + kKeyNormWord);
    cudaError_t e = cudaMemsetAsync(k.kbound, 0, (kKeyNormWord + a.B * a.Hkv) * sizeof(int32_t), s);
    if (e != cudaSuccess) return e;
    km_key_norm_kernel<<<sms * 4, 256, 0, s>>>(a, k.choice, kmax2);
    const char *force = std::getenv("QSA_DEBUG_FORWARD_MAXPASS");
    km_fwd_init_kernel<<<sms * 8, 256, 0, s>>>(p, a, a.ids, a.counts, a.K, kmax2, force && force[0] == '1', k.kbound,
                                                n_o4);
    p.sched = k.sched;
    if (D == 128) km_fwd_max_kernel<128><<<sms, kMaxThreads, MaxLayout<128>::kSmemBytes, s>>>(p);
    else km_fwd_max_kernel<256><<<sms, kMaxThreads, MaxLayout<256>::kSmemBytes, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    p.sched = k.sched + 2;
    if (D == 128) km_fwd_out_kernel<128><<<sms, kOutThreads, OutLayout<128>::kSmemBytes, s>>>(p);
    else km_fwd_out_kernel<256><<<sms, kOutThreads, OutLayout<256>::kSmemBytes, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (D == 128) km_fwd_final_kernel<128><<<sms * 8, 256, 0, s>>>(p, o, lse);
    else km_fwd_final_kernel<256><<<sms * 8, 256, 0, s>>>(p, o, lse);
    return cudaGetLastError();
}

}  // namespace qsa

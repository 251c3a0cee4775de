// qsa_route.cu -- the QSA route producer (select_qsa_token_ids of the
// NeMo-AutoModel Qwen3.8-Flash-Next qsa page): compressed-block index scores
// on tcgen05 tensor cores, then top-k block selection and expansion to
// ascending token IDs.
//
// Scores.  For one batch row the block scores of all query rows are
//   score[t, blk] = sum_h relu(<q[t,h,:], k[blk,:]>) / sqrt(D),
// a dense contraction over D followed by a relu-sum over the H index heads.
// A work item is one batch row's tile of n_q = 256 / H consecutive queries; its
// 256 (query, head) rows form the N = 256 operand of every MMA and stay in
// shared memory for the whole item.  The item walks the visible blocks in
// tiles of 128 (the M = 128 operand): D / 16 MMAs (M=128, N=256, K=16)
// accumulate K_tile * Q_tile^T into TMEM, so TMEM lane i holds block i of the
// tile and the H columns of one query are consecutive.  The relu-sum over heads
// is then a per-thread loop over columns (no cross-lane reduction): each
// epilogue thread turns its block's 128 columns into 128 / H scores.
//
//   warp 0 (producer)  loads the item's Q tile (4-D TMA, box {64, H, n_q, 1})
//                      into one of two Q buffers (the next item's loads while
//                      this one computes) and the K tiles (3-D TMA, box
//                      {64, 128, 1}) into a three-stage ring, all 128-byte
//                      swizzled;
//   warp 1 (MMA)       one thread issues the MMAs into two TMEM accumulators
//                      (256 columns each) alternately;
//   warps 2-9          read an accumulator (warp w: TMEM lanes 32 (w % 4) ..,
//                      column half (w - 2) / 4), release it, and store the
//                      scores (fp32, coalesced along blocks).
//
// Items are claimed from a work queue heaviest first (the last query tiles see
// the most blocks).  Tiles past a row's visible blocks are never computed;
// within the last tile, entries past a query's own visible count are not
// stored.  Every wait is bounded in time: on timeout the kernel records
// QSA_ERR_TIMEOUT in the status word, the roles wind down, the tensor pipe and
// the copies drain, and the TMEM is freed.
//
// Selection.  One CTA per query row.  The row's visible scores are loaded with
// coalesced loads as order-preserving 32-bit keys (raw bits on the product
// path, whose scores are never negative) and transposed through shared memory
// so that each thread holds a contiguous segment of 32 keys in registers (rows
// of up to 8192 visible blocks; longer rows are walked in chunks of 8192,
// re-read from L2 for each pass).  A three-pass radix select with 11-bit
// digits finds the key T of the floor(budget / c)-th best block and how many
// blocks equal to T to keep (lowest indices first): the first pass histograms
// every key, then the keys of its chosen bin are gathered into shared memory
// in index order (when they fit) and the other two passes read only those.
// Blocks in better first-pass bins are all chosen and only the gathered keys
// are compared with T; one block-wide scan of the per-thread counts gives
// every thread the output position of its first chosen block, and a bit mask
// of its chosen keys is walked in index order, so the chosen blocks come out
// ascending.  Each expands to its c token IDs, the incomplete causal tail
// follows, then -1; the row is assembled in shared memory and written with
// coalesced stores.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "../../include/qsa_route.h"
#include "qsa_queue.cuh"
#include "qsa_tc.cuh"
#include "qsa_tc_ptx.cuh"

namespace qsa {
namespace {

using namespace ptx;

// ---------------------------------------------------------------- scores ----
constexpr int kScoreThreads = 320;  // warp 0 producer, 1 MMA, 2-9 epilogue
constexpr int kEpiThreads = 256;
constexpr int kBlkTile = 128;  // blocks per tile (MMA M)
constexpr int kRowsN = 256;    // (query, head) rows per item (MMA N)
constexpr int kScoreStages = 3;  // K tile ring (two Q tiles take the rest of shared memory)
constexpr int kMaxIndexDim = 128;
constexpr uint32_t kTmemCols = 512;  // two accumulators of 256 fp32 columns
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Barrier slots.
enum { kBarQFull, kBarQEmpty = kBarQFull + 2, kBarDrain = kBarQEmpty + 2, kBarKFull, kBarKEmpty = kBarKFull + kScoreStages,
       kBarAccFull = kBarKEmpty + kScoreStages, kBarAccEmpty = kBarAccFull + 2, kBarItemFull = kBarAccEmpty + 2,
       kBarItemEmpty = kBarItemFull + kQueueRing, kNumScoreBars = kBarItemEmpty + kQueueRing };

struct ScoreParams {
    CUtensorMap q_map;  // {D, H, S_q, B}, box {64, H, n_q, 1}
    CUtensorMap k_map;  // {D, NB, B}, box {64, 128, 1}
    int64_t B, S_q, H, D, NB, c, offset;
    int64_t n_q, n_qt, n_items;
    float inv_sqrt_d;
    uint64_t wait_limit_ns;
    const int64_t *seq_len;
    float *scores;  // [B, S_q, NB]
    int32_t *sched;
    DeviceStatus *status;
};

struct ScoreItem {
    int64_t b, t0, t_end;  // live query rows [t0, t_end)
    int n_kt;              // block tiles to compute
};

// Item idx: rank r = idx / B walks query tiles from the last (most visible
// blocks) to the first; b = idx % B.  Dead items (every row padding or no
// visible block) get n_kt = 0.
__device__ __forceinline__ ScoreItem score_item(const ScoreParams &p, int32_t idx) {
    ScoreItem it;
    const int64_t r = idx / p.B;
    it.b = idx % p.B;
    it.t0 = (p.n_qt - 1 - r) * p.n_q;
    const int64_t live_end = min(p.S_q, p.seq_len[it.b] - p.offset);  // rows t with offset + t < len
    it.t_end = min(it.t0 + p.n_q, live_end);
    it.n_kt = 0;
    if (it.t_end > it.t0) {
        const int64_t nvis = min(p.NB, (p.offset + it.t_end) / p.c);  // visible from the last live row
        it.n_kt = (int)((nvis + kBlkTile - 1) / kBlkTile);
    }
    return it;
}

// H (index heads, a power of two up to 128) is a template parameter: each
// epilogue thread then sums fixed runs of H accumulator columns in registers.
template <int H>
__global__ void __launch_bounds__(kScoreThreads, 1) index_score_kernel(const __grid_constant__ ScoreParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t q_panel = kRowsN * 128;    // one 64-column panel of the Q tile
    const uint32_t k_panel = kBlkTile * 128;  // one 64-column panel of a K tile
    const int n_panels = (int)(p.D / 64);
    const uint32_t q_bytes = q_panel * n_panels, k_bytes = k_panel * n_panels;
    const uint32_t off_k = 2 * q_bytes;  // two Q tiles: the next item's loads while this one computes
    const uint32_t off_bar = off_k + kScoreStages * k_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + off_bar);
    uint8_t *misc = smem + off_bar + kNumScoreBars * 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 8);
    volatile int32_t *ring = reinterpret_cast<volatile int32_t *>(misc + 16);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(bars + kBarQFull + b, 1);
            mbar_init(bars + kBarQEmpty + b, 1);
        }
        mbar_init(bars + kBarDrain, 1);
        for (int s = 0; s < kScoreStages; ++s) {
            mbar_init(bars + kBarKFull + s, 1);
            mbar_init(bars + kBarKEmpty + s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bars + kBarAccFull + a, 1);
            mbar_init(bars + kBarAccEmpty + a, kEpiThreads);
        }
        for (int s = 0; s < kQueueRing; ++s) {
            mbar_init(bars + kBarItemFull + s, 1);
            mbar_init(bars + kBarItemEmpty + s, 1 + kEpiThreads);  // the MMA thread and every epilogue thread
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&p.q_map);
        prefetch_tmap(&p.k_map);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int zero = 0;
    auto fail = [&](unsigned info) {
        raise_status(p.status, QSA_ERR_TIMEOUT, kSiteRouteScoreWait, info, blockIdx.x);
        *abort_flag = 1;
    };

    if (warp == 0) {
        // ---------------- producer (lane 0) ----------------
        if (lane == 0) {
            bool ok = true;
            int64_t gk = 0, nq = 0;
            for (int64_t i = 0; ok; ++i) {
                int32_t idx = -1;
                ok = queue_claim(p.sched, p.n_items, ring, bars + kBarItemFull, bars + kBarItemEmpty, i, abort_flag,
                                 p.wait_limit_ns, idx);
                if (!ok || idx < 0) break;
                const ScoreItem it = score_item(p, idx);
                if (it.n_kt == 0) continue;
                // The Q tile is reused once the previous item's last MMAs have completed.
                // Q tiles alternate between two buffers; a buffer is reused once the MMAs of the item two
                // back, its previous user, have completed.
                const int qb = (int)(nq & 1);
                if (nq >= 2 &&
                    !mbar_wait(bars + kBarQEmpty + qb, (uint32_t)((nq / 2 - 1) & 1), abort_flag, p.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(bars + kBarQFull + qb, q_bytes);
                for (int kb = 0; kb < n_panels; ++kb)
                    tma_load_4d(sbase + qb * q_bytes + kb * q_panel, &p.q_map, bars + kBarQFull + qb, kb * 64, 0,
                                (int)it.t0, (int)it.b);
                ++nq;
                for (int kt = 0; kt < it.n_kt; ++kt, ++gk) {
                    const int s = (int)(gk % kScoreStages);
                    if (gk >= kScoreStages &&
                        !mbar_wait(bars + kBarKEmpty + s, (uint32_t)((gk / kScoreStages - 1) & 1), abort_flag,
                                   p.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bars + kBarKFull + s, k_bytes);
                    for (int kb = 0; kb < n_panels; ++kb)
                        tma_load_3d(sbase + off_k + s * k_bytes + kb * k_panel, &p.k_map, bars + kBarKFull + s,
                                    kb * 64, kt * kBlkTile, (int)it.b);
                }
            }
            if (!ok) fail(1);
            queue_finish(p.sched);
            // Drain: every issued copy must have landed before the CTA leaves.
            bool drained = true;
            for (int64_t g = nq > 2 ? nq - 2 : 0; g < nq; ++g)
                drained &= mbar_wait(bars + kBarQFull + (int)(g & 1), (uint32_t)((g / 2) & 1), &zero, kWaitLimitNs);
            for (int64_t g = gk > kScoreStages ? gk - kScoreStages : 0; g < gk; ++g)
                drained &= mbar_wait(bars + kBarKFull + (int)(g % kScoreStages),
                                     (uint32_t)((g / kScoreStages) & 1), &zero, kWaitLimitNs);
            if (!drained) fail(2);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer (lane 0) ----------------
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kBlkTile, kRowsN, false, false);
            bool ok = true, issued = false;
            int64_t gk = 0, ga = 0, nq = 0;
            for (int64_t i = 0; ok; ++i) {
                int32_t idx = -1;
                ok = queue_take(ring, bars + kBarItemFull, bars + kBarItemEmpty, i, abort_flag, p.wait_limit_ns, false,
                                idx);
                if (!ok || idx < 0) break;
                const ScoreItem it = score_item(p, idx);
                if (it.n_kt == 0) continue;
                const int qb = (int)(nq & 1);
                if (!mbar_wait(bars + kBarQFull + qb, (uint32_t)((nq / 2) & 1), abort_flag, p.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kt = 0; kt < it.n_kt; ++kt, ++gk, ++ga) {
                    const int s = (int)(gk % kScoreStages), a = (int)(ga & 1);
                    if (!mbar_wait(bars + kBarKFull + s, (uint32_t)((gk / kScoreStages) & 1), abort_flag,
                                   p.wait_limit_ns) ||
                        (ga >= 2 && !mbar_wait(bars + kBarAccEmpty + a, (uint32_t)((ga / 2 - 1) & 1), abort_flag,
                                               p.wait_limit_ns))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t kt_base = sbase + off_k + s * k_bytes;
                    for (int kb = 0; kb < n_panels; ++kb) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t ad = sdesc_sw128(kt_base + kb * k_panel + k * 32, 16, 1024);
                            const uint64_t bd = sdesc_sw128(sbase + qb * q_bytes + kb * q_panel + k * 32, 16, 1024);
                            mma_bf16(tmem + a * 256, ad, bd, idesc, (kb | k) ? 1u : 0u);
                        }
                    }
                    issued = true;
                    mma_commit(bars + kBarKEmpty + s);
                    mma_commit(bars + kBarAccFull + a);
                }
                if (!ok) break;
                mma_commit(bars + kBarQEmpty + qb);
                ++nq;
            }
            if (!ok) fail(3);
            // Drain the tensor pipe before the TMEM is released.
            if (issued) {
                mma_commit(bars + kBarDrain);
                if (!mbar_wait(bars + kBarDrain, 0, &zero, kWaitLimitNs)) fail(4);
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (warps 2-9) ----------------
        const int quad = warp & 3;          // TMEM lanes 32 quad .. 32 quad + 31
        const int half = (warp - 2) >> 2;   // accumulator columns 128 half .. 128 half + 127
        constexpr int kQPerHalf = 128 / H;  // queries per thread per tile
        bool ok = true;
        int64_t ga = 0;
        for (int64_t i = 0; ok; ++i) {
            int32_t idx = -1;
            ok = queue_take(ring, bars + kBarItemFull, bars + kBarItemEmpty, i, abort_flag, p.wait_limit_ns, true,
                            idx);
            if (!ok || idx < 0) break;
            const ScoreItem it = score_item(p, idx);
            for (int kt = 0; kt < it.n_kt; ++kt, ++ga) {
                const int a = (int)(ga & 1);
                if (!mbar_wait_warp(bars + kBarAccFull + a, (uint32_t)((ga / 2) & 1), abort_flag, p.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t v[4][32];
                const uint32_t taddr = tmem + ((uint32_t)(32 * quad) << 16) + a * 256 + half * 128;
#pragma unroll
                for (int j = 0; j < 4; ++j) tmem_ld32(taddr + j * 32, v[j]);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(bars + kBarAccEmpty + a);
                const int64_t blk = (int64_t)kt * kBlkTile + 32 * quad + lane;
                // blk is visible from t  <=>  blk < floor((offset + t + 1) / c)  <=>  (blk + 1) c <= offset + t + 1.
                const int64_t need = (blk + 1) * p.c - p.offset - 1;  // visible from every t >= need
                const bool blk_ok = blk < p.NB;
#pragma unroll
                for (int qi = 0; qi < kQPerHalf; ++qi) {
                    float acc = 0.f;
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const int j = qi * H + h;
                        acc += fmaxf(__uint_as_float(v[j >> 5][j & 31]), 0.f);
                    }
                    const int64_t t = it.t0 + half * kQPerHalf + qi;
                    if (blk_ok && t < it.t_end && t >= need)
                        p.scores[(it.b * p.S_q + t) * p.NB + blk] = acc * p.inv_sqrt_d;
                }
            }
        }
        if (!ok) fail(5);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------- selection ----
constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kKeysPerThread = 32;                          // a thread's contiguous segment of a chunk
constexpr int64_t kSelChunk = kSelThreads * kKeysPerThread;  // keys held in registers at once
constexpr int kDigitBins = 2048;                            // 11-bit digits: bits 31-21, 20-10, 9-0
constexpr int kStageMax = 12288;                            // output rows up to this width are staged
constexpr int kCandCap = 2048;                              // keys of one first-pass bin kept in shared memory

struct SelParams {
    const float *scores;  // [B, S_q, NB]
    const int64_t *seq_len;
    int32_t *ids;  // [B, S_q, W]
    int64_t S_q;
    // Positions, block counts, token IDs and the row width all fit in 31 bits.
    uint32_t NB, c, offset, n_best, W;
};

// Order-preserving unsigned key of an fp32 score (larger score, larger key).
// Adding +0 first turns -0 into +0, so both zeros get one key.
__device__ __forceinline__ uint32_t score_key(float f) {
    const uint32_t u = __float_as_uint(__fadd_rn(f, 0.0f));
    return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

// Key of a score.  The fused path's scores are relu-sums times a positive
// factor, never negative and never -0, and the bits of a non-negative float
// are already order-preserving.
template <bool kNonNeg>
__device__ __forceinline__ uint32_t key_of(float f) {
    return kNonNeg ? __float_as_uint(f) : score_key(f);
}

// Block-wide exclusive prefix sum of one 32-bit value per thread; `total` gets
// the sum over the block.  Contains two barriers.
__device__ __forceinline__ uint32_t block_scan(uint32_t x, uint32_t *warp_tot, uint32_t &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) {
        const uint32_t t = warp_tot[w];
        before += w < warp ? t : 0u;
        all += t;
    }
    __syncthreads();
    total = all;
    return before + incl - x;
}

// Given a digit histogram, finds the digit d holding the remaining-th largest
// key (counting from the top bin), how many keys of bin d that rank needs, and
// how many keys bin d holds.  In best-first order (position r = bin 2047 - r)
// warp w owns positions 256 w .. 256 w + 255 and lane l eight consecutive ones,
// i.e. the eight bins b0 .. b0 + 7 with b0 = 2040 - 256 w - 8 l, read as two
// 16-byte words; one warp scan of the lanes' sums and the warps' totals give
// every lane the count of better keys.
__device__ __forceinline__ void find_digit(const uint32_t *hist, uint32_t remaining, uint32_t *warp_tot,
                                           uint32_t *s_digit, uint32_t *s_rem, uint32_t *s_cnt) {
    static_assert(kDigitBins == 8 * kSelThreads, "eight bins per thread");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int b0 = kDigitBins - 8 - 256 * warp - 8 * lane;
    const uint4 lo = reinterpret_cast<const uint4 *>(hist + b0)[0];
    const uint4 hi = reinterpret_cast<const uint4 *>(hist + b0)[1];
    const uint32_t cnt[8] = {hi.w, hi.z, hi.y, hi.x, lo.w, lo.z, lo.y, lo.x};  // bins b0 + 7 .. b0
    uint32_t sum = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) sum += cnt[q];
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    uint32_t e = incl - sum;
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) e += w < warp ? warp_tot[w] : 0u;
    if (e < remaining && remaining <= e + sum) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (e + cnt[q] >= remaining) {
                *s_digit = (uint32_t)(b0 + 7 - q);
                *s_rem = remaining - e;
                *s_cnt = cnt[q];
                break;
            }
            e += cnt[q];
        }
    }
    __syncthreads();
}

// A load the compiler may not repeat (the loaded keys are meant to stay in
// registers through every pass, not to be re-read from memory at each use).
__device__ __forceinline__ float load_once(const float *p) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float4 load_once4(const float *p) {
    float4 v;
    asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

// Keys of chunk ch (blocks ch * kSelChunk ..) for this thread's segment;
// returns how many of its kKeysPerThread slots hold visible blocks.  A full
// segment of a 16-byte aligned row is read with 16-byte loads: the 32 lanes of
// a warp read 32 different 128-byte lines per instruction, so wide loads cut
// the L1 transactions fourfold.
template <bool kNonNeg>
__device__ __forceinline__ int load_segment(const float *srow, uint32_t nvis, uint32_t ch,
                                            uint32_t (&k)[kKeysPerThread], bool aligned16) {
    const uint32_t i0 = ch * (uint32_t)kSelChunk + threadIdx.x * kKeysPerThread;
    const int n = i0 >= nvis ? 0 : (int)min(nvis - i0, (uint32_t)kKeysPerThread);
    if (aligned16 && n == kKeysPerThread) {
#pragma unroll
        for (int j = 0; j < kKeysPerThread; j += 4) {
            const float4 v = load_once4(srow + i0 + j);
            k[j] = key_of<kNonNeg>(v.x);
            k[j + 1] = key_of<kNonNeg>(v.y);
            k[j + 2] = key_of<kNonNeg>(v.z);
            k[j + 3] = key_of<kNonNeg>(v.w);
        }
    } else {
#pragma unroll
        for (int j = 0; j < kKeysPerThread; ++j) k[j] = j < n ? key_of<kNonNeg>(load_once(srow + i0 + j)) : 0u;
    }
    return n;
}

// Words of the selection kernel's dynamic shared region.
inline size_t select_smem_words(uint32_t W) {
    const size_t transpose = kSelChunk + kSelChunk / 32;
    const size_t later = 2 * kDigitBins + kCandCap + (W <= (uint32_t)kStageMax ? W : 0);
    return transpose > later ? transpose : later;
}

__device__ __forceinline__ void clear_hist(uint32_t *hist) {
#pragma unroll
    for (int i = threadIdx.x; i < kDigitBins / 4; i += kSelThreads)
        reinterpret_cast<uint4 *>(hist)[i] = make_uint4(0, 0, 0, 0);
}

// Grid (S_q, B): one CTA per query row.
template <bool kNonNeg>
__global__ void __launch_bounds__(kSelThreads, 4) select_kernel(const SelParams p) {
    // One dynamic region, used in turn: a padded transposition buffer for the
    // row's keys while they load; then two digit histograms, the candidate keys
    // and the staged output row (select_smem_words gives its size).
    extern __shared__ __align__(16) uint32_t region[];
    uint32_t(*hist)[kDigitBins] = reinterpret_cast<uint32_t(*)[kDigitBins]>(region);
    uint32_t *cand = region + 2 * kDigitBins;  // keys of the first pass's chosen bin
    int32_t *stage = reinterpret_cast<int32_t *>(region + 2 * kDigitBins + kCandCap);  // the output row
    __shared__ uint32_t warp_tot[kSelWarps];
    __shared__ uint32_t s_digit, s_remaining, s_count;
    const int tid = threadIdx.x;
    const uint32_t t = blockIdx.x, b = blockIdx.y;
    const int64_t row = (int64_t)b * p.S_q + t;
    const uint32_t tg = p.offset + t;
    int32_t *gout = p.ids + row * p.W;
    const bool staged = p.W <= (uint32_t)kStageMax;
    int32_t *out = staged ? stage : gout;
    uint32_t n_out = 0;
    if ((int64_t)tg < p.seq_len[b]) {
        const uint32_t nvis = min(p.NB, (tg + 1) / p.c);
        const uint32_t n_sel = min(nvis, p.n_best);
        n_out = n_sel * p.c + (tg + 1 - nvis * p.c);
        if (nvis <= p.n_best) {
            // Every visible block is chosen: the row is dense causal, 0 .. tg.
            for (uint32_t i = tid; i < n_out; i += kSelThreads) out[i] = (int32_t)i;
        } else {
            const float *srow = p.scores + row * p.NB;
            const uint32_t n_chunks = (nvis + (uint32_t)kSelChunk - 1) / (uint32_t)kSelChunk;
            const bool resident = n_chunks == 1;  // the whole row stays in registers
            uint32_t k[kKeysPerThread];
            const bool a16 = (reinterpret_cast<uintptr_t>(srow) & 15u) == 0;
            int n = 0;
            if (resident) {
                // Coalesced loads (a warp reads 32 consecutive scores), transposed
                // through shared memory into each thread's contiguous segment; one
                // pad word every 32 keys keeps both sides free of bank conflicts.
                const float *src = srow + tid;
                uint32_t *dst = region + tid + (tid >> 5);  // slot of key tid; key tid + 256 j is 264 j further
                if (nvis == (uint32_t)kSelChunk) {
#pragma unroll
                    for (int j = 0; j < kKeysPerThread; ++j) dst[j * 264] = key_of<kNonNeg>(__ldg(src + j * kSelThreads));
                } else {
#pragma unroll
                    for (int j = 0; j < kKeysPerThread; ++j)
                        if ((uint32_t)j * kSelThreads + tid < nvis)
                            dst[j * 264] = key_of<kNonNeg>(__ldg(src + j * kSelThreads));
                }
                __syncthreads();
                const uint32_t i0 = (uint32_t)tid * kKeysPerThread;
                n = i0 >= nvis ? 0 : (int)min(nvis - i0, (uint32_t)kKeysPerThread);
#pragma unroll
                for (int j = 0; j < kKeysPerThread; ++j) k[j] = j < n ? region[i0 + tid + j] : 0u;
                __syncthreads();  // the region becomes the histograms
            }
            // Three radix passes, most significant digit first, find the key T of
            // the n_best-th best block and how many blocks equal to T are kept.
            // The passes alternate between two histograms (the idle one is cleared
            // during the other's pass).  After the first pass, the keys of its chosen
            // bin are gathered into shared memory when they fit, and the other two
            // passes read only those.
            uint32_t prefix = 0, mask = 0, remaining = p.n_best;
            bool use_cand = false;
            uint32_t c_mask = 0, g1_mask = 0, c_cnt = 0, c_at = 0, n_cand = 0;
            clear_hist(hist[0]);
            clear_hist(hist[1]);
            __syncthreads();
#pragma unroll 1
            for (int pass = 0; pass < 3; ++pass) {
                const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
                const uint32_t dmask = pass == 2 ? 0x3FFu : 0x7FFu;
                uint32_t *h = hist[pass & 1];
                if (use_cand) {
                    for (uint32_t i = tid; i < n_cand; i += kSelThreads) {
                        const uint32_t kc = cand[i];
                        if ((kc & mask) == prefix) atomicAdd(&h[(kc >> shift) & dmask], 1u);
                    }
                } else {
                    for (uint32_t ch = 0; ch < n_chunks; ++ch) {
                        if (!resident) n = load_segment<kNonNeg>(srow, nvis, ch, k, a16);
                        if (pass == 0) {
#pragma unroll
                            for (int j = 0; j < kKeysPerThread; ++j)
                                if (j < n) atomicAdd(&h[k[j] >> 21], 1u);
                        } else {
#pragma unroll
                            for (int j = 0; j < kKeysPerThread; ++j)
                                if (j < n && (k[j] & mask) == prefix) atomicAdd(&h[(k[j] >> shift) & dmask], 1u);
                        }
                    }
                }
                __syncthreads();
                find_digit(h, remaining, warp_tot, &s_digit, &s_remaining, &s_count);
                prefix |= s_digit << shift;
                mask |= dmask << shift;
                remaining = s_remaining;
                clear_hist(h);  // read by nobody any more; the pass after next uses it
                if (pass == 0 && resident && s_count <= (uint32_t)kCandCap) {
                    // Gather the chosen bin's keys into shared memory in block order
                    // (thread order = index order) and note, per thread, which keys
                    // went there (c_mask) and which lie in better bins (g1_mask: all
                    // of those are chosen).
#pragma unroll
                    for (int j = 0; j < kKeysPerThread; ++j) {
                        const bool live = j < n;
                        c_mask |= (uint32_t)(live && (k[j] & mask) == prefix) << j;
                        g1_mask |= (uint32_t)(live && (k[j] >> 21) > s_digit) << j;
                    }
                    c_cnt = __popc(c_mask);
                    uint32_t total;
                    c_at = block_scan(c_cnt, warp_tot, total);
                    uint32_t at = c_at;
#pragma unroll
                    for (int j = 0; j < kKeysPerThread; ++j)
                        if ((c_mask >> j) & 1u) cand[at++] = k[j];
                    n_cand = total;
                    use_cand = true;
                    __syncthreads();
                }
            }
            const uint32_t T = prefix, need = remaining;  // keep every key > T and the first `need` keys == T
            // Place the chosen blocks in index order: one block-wide scan of the
            // per-segment counts (key > T, key == T) per chunk gives each thread
            // its first output position and its rank among the ties; a bit mask
            // of the segment's chosen keys is then walked set bit by set bit.
            uint32_t sel_run = 0, eq_run = 0;
            const bool vec4 = staged && p.c == 4;  // whole 16-byte stores into the staged row
            for (uint32_t ch = 0; ch < n_chunks; ++ch) {
                if (!resident) n = load_segment<kNonNeg>(srow, nvis, ch, k, a16);
                uint32_t gt_mask = 0, eq_mask = 0;  // bit j: key j of the segment
                if (use_cand) {
                    // Keys in better bins than the first pass's are all > T; only this
                    // thread's gathered keys (in order, one per set bit of c_mask) need
                    // comparing.
                    gt_mask = g1_mask;
                    uint32_t mm = c_mask;
                    for (uint32_t q = 0; q < c_cnt; ++q) {
                        const uint32_t kc = cand[c_at + q];
                        const uint32_t bit = mm & (0u - mm);
                        mm ^= bit;
                        if (kc > T) gt_mask |= bit;
                        else if (kc == T) eq_mask |= bit;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < kKeysPerThread; ++j) {
                        gt_mask |= (uint32_t)(j < n && k[j] > T) << j;
                        eq_mask |= (uint32_t)(j < n && k[j] == T) << j;
                    }
                }
                const uint32_t eq = __popc(eq_mask);
                uint32_t tot;
                const uint32_t ex = block_scan(__popc(gt_mask) | (eq << 16), warp_tot, tot);
                const uint32_t eq_rank = eq_run + (ex >> 16);  // ties before this segment
                const uint32_t keep = eq_rank >= need ? 0u : min(eq, need - eq_rank);
                while ((uint32_t)__popc(eq_mask) > keep) eq_mask &= ~(1u << (31 - __clz(eq_mask)));
                uint32_t take = gt_mask | eq_mask;
                uint32_t pos = sel_run + (ex & 0xFFFFu) + min(eq_rank, need) - min(eq_run, need);
                const uint32_t i0 = ch * (uint32_t)kSelChunk + tid * kKeysPerThread;
                while (take) {
                    const uint32_t j = (uint32_t)(__ffs(take) - 1);
                    take &= take - 1;
                    if (pos < n_sel) {
                        const int32_t first = (int32_t)((i0 + j) * p.c);
                        if (vec4) {
                            reinterpret_cast<int4 *>(out)[pos] = make_int4(first, first + 1, first + 2, first + 3);
                        } else {
                            int32_t *dst = out + (size_t)pos * p.c;
                            for (uint32_t e = 0; e < p.c; ++e) dst[e] = first + (int32_t)e;
                        }
                    }
                    ++pos;
                }
                const uint32_t eq_tot = tot >> 16;
                sel_run += (tot & 0xFFFFu) + min(eq_run + eq_tot, need) - min(eq_run, need);
                eq_run += eq_tot;
            }
            // Causal tail: the tokens of the incomplete block.
            for (uint32_t i = tid; i < tg + 1 - nvis * p.c; i += kSelThreads)
                out[n_sel * p.c + i] = (int32_t)(nvis * p.c + i);
        }
    }
    if (staged) {
        __syncthreads();
        for (uint32_t i = tid; i < p.W; i += kSelThreads) gout[i] = i < n_out ? stage[i] : -1;
    } else {
        for (uint32_t i = n_out + tid; i < p.W; i += kSelThreads) gout[i] = -1;
    }
}

// --------------------------------------------------------------- host side ----
thread_local char g_msg[384];

qsa_status route_fail(qsa_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return report_error(st, g_msg);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
constexpr size_t kOffStatus = 0, kOffSched = 256, kOffScores = 512;

qsa_status validate_route(const qsa_route_problem *p) {
    if (!p) return route_fail(QSA_ERR_INVALID_ARGUMENT, "problem is null");
    if (p->B <= 0 || p->S_q <= 0 || p->H_index <= 0 || p->D_index <= 0 || p->n_blocks < 0 || p->token_budget < 0 ||
        p->compress_ratio <= 0 || p->query_position_offset < 0)
        return route_fail(QSA_ERR_INVALID_ARGUMENT,
                          "need B, S_q, H_index, D_index, compress_ratio > 0 and n_blocks, token_budget, "
                          "query_position_offset >= 0");
    const int64_t c = p->compress_ratio;
    if (p->query_position_offset + p->S_q > p->n_blocks * c + c - 1)
        return route_fail(QSA_ERR_INVALID_ARGUMENT,
                          "query positions up to %lld lie past the global sequence (%lld blocks of %lld)",
                          (long long)(p->query_position_offset + p->S_q - 1), (long long)p->n_blocks, (long long)c);
    if ((p->H_index & (p->H_index - 1)) != 0 || p->H_index > 128)
        return route_fail(QSA_ERR_UNSUPPORTED, "H_index=%lld: a power of two up to 128 is supported",
                          (long long)p->H_index);
    if (p->D_index != 64 && p->D_index != kMaxIndexDim)
        return route_fail(QSA_ERR_UNSUPPORTED, "D_index=%lld: 64 or 128 is supported", (long long)p->D_index);
    if (p->n_blocks * c + c > 2147483647LL || p->token_budget + c - 1 > 2147483647LL)
        return route_fail(QSA_ERR_UNSUPPORTED, "token IDs or the row width exceed int32");
    if (p->B > 65535 || p->S_q > 2147483647LL)
        return route_fail(QSA_ERR_UNSUPPORTED, "B up to 65535 and S_q up to 2^31 - 1 are supported");
    if (p->q_stride[3] != 1 || p->k_stride[2] != 1)
        return route_fail(QSA_ERR_UNSUPPORTED, "index_queries and compressed_keys need a unit last stride");
    for (int i = 0; i < 3; ++i)
        if (p->q_stride[i] < 0 || p->q_stride[i] % 8 != 0)
            return route_fail(QSA_ERR_UNSUPPORTED, "index_queries stride[%d]=%lld must be a multiple of 8", i,
                              (long long)p->q_stride[i]);
    for (int i = 0; i < 2; ++i)
        if (p->k_stride[i] < 0 || p->k_stride[i] % 8 != 0)
            return route_fail(QSA_ERR_UNSUPPORTED, "compressed_keys stride[%d]=%lld must be a multiple of 8", i,
                              (long long)p->k_stride[i]);
    return QSA_OK;
}

size_t route_ws_bytes(const qsa_route_problem *p) {
    return align256(kOffScores + (size_t)p->B * p->S_q * p->n_blocks * sizeof(float));
}

qsa_status check_route_ws(const qsa_route_problem *p, const void *ws, size_t ws_bytes, size_t need) {
    if (!ws) return route_fail(QSA_ERR_INVALID_ARGUMENT, "workspace is null");
    if (reinterpret_cast<uintptr_t>(ws) % 256 != 0)
        return route_fail(QSA_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
    if (ws_bytes < need)
        return route_fail(QSA_ERR_WORKSPACE_TOO_SMALL, "workspace has %zu bytes, needs %zu", ws_bytes, need);
    return QSA_OK;
}

qsa_status cuda_status(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return QSA_OK;
    return route_fail(QSA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

uint32_t score_smem_bytes(int64_t D) {
    const uint32_t panels = (uint32_t)(D / 64);
    return panels * (2 * kRowsN * 128 + kScoreStages * kBlkTile * 128) + kNumScoreBars * 8 + 64 + 1024;
}

template <int H>
qsa_status launch_score_kernel(const ScoreParams &p, int grid, uint32_t smem, cudaStream_t stream) {
    qsa_status st = cuda_status(
        cudaFuncSetAttribute(index_score_kernel<H>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
        "cudaFuncSetAttribute");
    if (st != QSA_OK) return st;
    index_score_kernel<H><<<grid, kScoreThreads, smem, stream>>>(p);
    return cuda_status(cudaGetLastError(), "index score kernel launch");
}

qsa_status launch_scores(const qsa_route_problem *pr, const void *q, const void *k, const int64_t *seq_len, void *ws,
                         float *scores, cudaStream_t stream) {
    if (!tc_device_ok()) return route_fail(QSA_ERR_UNSUPPORTED, "the score kernel needs an sm_103 GPU");
    ScoreParams p;
    memset(&p, 0, sizeof(p));
    p.B = pr->B;
    p.S_q = pr->S_q;
    p.H = pr->H_index;
    p.D = pr->D_index;
    p.NB = pr->n_blocks;
    p.c = pr->compress_ratio;
    p.offset = pr->query_position_offset;
    p.n_q = kRowsN / p.H;
    p.n_qt = (p.S_q + p.n_q - 1) / p.n_q;
    p.n_items = p.B * p.n_qt;
    p.inv_sqrt_d = (float)(1.0 / std::sqrt((double)p.D));
    p.wait_limit_ns = tc_wait_limit_ns(kWaitLimitNs);
    p.seq_len = seq_len;
    p.scores = scores;
    p.sched = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + kOffSched);
    p.status = reinterpret_cast<DeviceStatus *>(static_cast<char *>(ws) + kOffStatus);
    if (p.n_items > 2147483647LL) return route_fail(QSA_ERR_UNSUPPORTED, "too many query tiles");
    // A fresh status word and work queue for this call (the workspace may be uninitialised memory).
    qsa_status st = cuda_status(cudaMemsetAsync(ws, 0, kOffScores, stream), "cudaMemsetAsync");
    if (st != QSA_OK) return st;
    const int64_t qd[4] = {p.D, p.H, p.S_q, p.B};
    const int64_t qs[3] = {pr->q_stride[2], pr->q_stride[1], pr->q_stride[0]};
    const uint32_t qbox[4] = {64, (uint32_t)p.H, (uint32_t)p.n_q, 1};
    const int64_t kd[3] = {p.D, p.NB, p.B};
    const int64_t ks[2] = {pr->k_stride[1], pr->k_stride[0]};
    const uint32_t kbox[3] = {64, kBlkTile, 1};
    if (p.NB == 0) return QSA_OK;  // no block is ever visible: nothing to score
    if (reinterpret_cast<uintptr_t>(q) % 16 || reinterpret_cast<uintptr_t>(k) % 16)
        return route_fail(QSA_ERR_UNSUPPORTED, "index_queries and compressed_keys need 16-byte aligned bases");
    if (!tc_encode_bf16_map(&p.q_map, q, 4, qd, qs, qbox) || !tc_encode_bf16_map(&p.k_map, k, 3, kd, ks, kbox))
        return route_fail(QSA_ERR_UNSUPPORTED, "tensor map encoding failed for the index operands");
    const uint32_t smem = score_smem_bytes(p.D);
    const int grid = (int)std::min<int64_t>(p.n_items, tc_num_sms());
    switch (p.H) {
        case 1: return launch_score_kernel<1>(p, grid, smem, stream);
        case 2: return launch_score_kernel<2>(p, grid, smem, stream);
        case 4: return launch_score_kernel<4>(p, grid, smem, stream);
        case 8: return launch_score_kernel<8>(p, grid, smem, stream);
        case 16: return launch_score_kernel<16>(p, grid, smem, stream);
        case 32: return launch_score_kernel<32>(p, grid, smem, stream);
        case 64: return launch_score_kernel<64>(p, grid, smem, stream);
        case 128: return launch_score_kernel<128>(p, grid, smem, stream);
        default: return route_fail(QSA_ERR_UNSUPPORTED, "H_index=%lld", (long long)p.H);
    }
}

// nonneg: the scores are known to be >= +0 (they come from the score kernel).
qsa_status launch_select(const qsa_route_problem *pr, const float *scores, const int64_t *seq_len, int32_t *ids,
                         bool nonneg, cudaStream_t stream) {
    SelParams p;
    p.scores = scores;
    p.seq_len = seq_len;
    p.ids = ids;
    p.S_q = pr->S_q;
    p.NB = (uint32_t)pr->n_blocks;
    p.c = (uint32_t)pr->compress_ratio;
    p.offset = (uint32_t)pr->query_position_offset;
    p.n_best = (uint32_t)(pr->token_budget / pr->compress_ratio);
    p.W = (uint32_t)(pr->token_budget + pr->compress_ratio - 1);
    const size_t smem = select_smem_words(p.W) * sizeof(uint32_t);
    if (smem > 48 * 1024) {
        qsa_status st = cuda_status(
            nonneg ? cudaFuncSetAttribute(select_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
                   : cudaFuncSetAttribute(select_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
            "cudaFuncSetAttribute");
        if (st != QSA_OK) return st;
    }
    const dim3 grid((unsigned)pr->S_q, (unsigned)pr->B);
    if (nonneg)
        select_kernel<true><<<grid, kSelThreads, smem, stream>>>(p);
    else
        select_kernel<false><<<grid, kSelThreads, smem, stream>>>(p);
    return cuda_status(cudaGetLastError(), "selection kernel launch");
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

}  // namespace
}  // namespace qsa

using namespace qsa;

extern "C" {

qsa_status qsa_route_check_problem(const qsa_route_problem *problem) { return validate_route(problem); }

int64_t qsa_route_width(const qsa_route_problem *problem) {
    if (validate_route(problem) != QSA_OK) return 0;
    return problem->token_budget + problem->compress_ratio - 1;
}

size_t qsa_route_workspace_bytes(const qsa_route_problem *problem) {
    if (validate_route(problem) != QSA_OK) return 0;
    return route_ws_bytes(problem);
}

qsa_status qsa_index_scores(const qsa_route_problem *p, const void *q, const void *k, const int64_t *seq_len, void *ws,
                            size_t ws_bytes, float *scores, cudaStream_t stream) {
    qsa_status st = validate_route(p);
    if (st != QSA_OK) return st;
    if (!q || (!k && p->n_blocks > 0) || !seq_len || !scores)
        return route_fail(QSA_ERR_INVALID_ARGUMENT, "null tensor pointer");
    st = check_route_ws(p, ws, ws_bytes, kOffScores);
    if (st != QSA_OK) return st;
    return launch_scores(p, q, k, seq_len, ws, scores, stream);
}

qsa_status qsa_select_from_scores(const qsa_route_problem *p, const float *scores, const int64_t *seq_len, void *ws,
                                  size_t ws_bytes, int32_t *ids, cudaStream_t stream) {
    qsa_status st = validate_route(p);
    if (st != QSA_OK) return st;
    if (!scores || !seq_len || !ids) return route_fail(QSA_ERR_INVALID_ARGUMENT, "null tensor pointer");
    st = check_route_ws(p, ws, ws_bytes, kOffScores);
    if (st != QSA_OK) return st;
    return launch_select(p, scores, seq_len, ids, false, stream);
}

qsa_status qsa_select_token_ids(const qsa_route_problem *p, const void *q, const void *k, const int64_t *seq_len,
                                void *ws, size_t ws_bytes, int32_t *ids, cudaStream_t stream) {
    qsa_status st = validate_route(p);
    if (st != QSA_OK) return st;
    if (!q || (!k && p->n_blocks > 0) || !seq_len || !ids)
        return route_fail(QSA_ERR_INVALID_ARGUMENT, "null tensor pointer");
    const size_t need = route_ws_bytes(p);
    st = check_route_ws(p, ws, ws_bytes, need);
    if (st != QSA_OK) return st;
    const size_t id_bytes = (size_t)p->B * p->S_q * (p->token_budget + p->compress_ratio - 1) * sizeof(int32_t);
    if (overlaps(ids, id_bytes, ws, need)) return route_fail(QSA_ERR_INVALID_ARGUMENT, "ids overlap the workspace");
    const size_t q_bytes = 2 * (size_t)((p->B - 1) * p->q_stride[0] + (p->S_q - 1) * p->q_stride[1] +
                                        (p->H_index - 1) * p->q_stride[2] + p->D_index);
    const size_t k_bytes = p->n_blocks > 0 ? 2 * (size_t)((p->B - 1) * p->k_stride[0] +
                                                          (p->n_blocks - 1) * p->k_stride[1] + p->D_index)
                                           : 0;
    if (overlaps(ids, id_bytes, q, q_bytes) || (k && overlaps(ids, id_bytes, k, k_bytes)) ||
        overlaps(ids, id_bytes, seq_len, (size_t)p->B * sizeof(int64_t)))
        return route_fail(QSA_ERR_INVALID_ARGUMENT, "ids overlap an input");
    float *scores = reinterpret_cast<float *>(static_cast<char *>(ws) + kOffScores);
    st = launch_scores(p, q, k, seq_len, ws, scores, stream);
    if (st != QSA_OK) return st;
    return launch_select(p, scores, seq_len, ids, true, stream);
}

}  // extern "C"

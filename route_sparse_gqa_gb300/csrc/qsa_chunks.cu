// qsa_chunks.cu -- key-major (reverse-route) lists for the key-major backward.
//
// The forward and the tile backward walk each query tile's routed keys.  The
// key-major backward walks the other way: per aligned chunk of 64 keys, the
// query rows that route into it (the pages' FA4 preprocessing keeps "forward
// and reverse block lists" for the same reason: fa4_qsa _preprocess).  Built
// from the sorted route sets of route_rows_kernel, with nothing dense in HBM
// beyond one 64-bit word per (block of 64 query rows, chunk):
//
//   chunk_mask_kernel    one CTA per block of 64 query rows: for every chunk,
//                        the bit mask of the block's rows that route into it
//                        (shared-memory table, one atomicOr per (row, chunk));
//   chunk_colscan_kernel one thread per list (b, c): popcounts scanned over the
//                        blocks give each block's offset inside the list, the
//                        list length, and the number of parts (per window);
//   scan_kernel          list starts and part starts (one CTA each);
//   chunk_fill_kernel    one CTA per block again: each (row, chunk) entry goes
//                        to list start + block offset + the number of earlier
//                        rows of the block in the chunk's mask -- so every list
//                        is in ascending query order, whatever the launch order;
//   chunk_items_kernel   one thread per list: parts of at most max_groups
//                        groups of `slots` entries, one window at a time;
//   chunk_queue_kernel   one CTA: parts sorted by window and size (counting
//                        sort, largest first), then the work queue: window by
//                        window, KV head by KV head.
#include <algorithm>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kQueueThreads = 1024;
constexpr int kQueueBins = 8192;
constexpr int kQueueMaxWindows = 1024;  // windows per launch of the queue builder (host guarantees)

__device__ __forceinline__ int block_scan_excl(int x, int *warp_tot, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < nwarps ? warp_tot[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < nwarps) warp_tot[lane] = wi - w;
        if (lane == 31) warp_tot[32] = wi;
    }
    __syncthreads();
    total = warp_tot[32];
    const int r = warp_tot[warp] + incl - x;
    __syncthreads();
    return r;
}

constexpr int kBlockRows = 64;     // query rows per block (one 64-bit row mask)
constexpr int kBlockThreads = 1024;  // 32 warps: two rows of the block each

// Walks the sorted ids of one row and calls emit(c, m) once per chunk c the row
// routes into, with m the mask of the chunk keys it routes to (kMask; 0
// otherwise).  Lane L takes a contiguous range of ceil(n / 32) ids and walks it
// alone, so a run of ids in one chunk costs a compare and an OR per id; runs
// that cross lane boundaries (a chunk's ids split between neighbouring lanes,
// or spanning several lanes of a short row) are joined with one segmented scan
// over the lanes, and emitted by the lane where they end.
// vec4: the row's ids start 16-byte aligned and the row has room up to a multiple of 4 ids past n, so
// lane ranges start at multiples of 4 and are read as int4.
template <bool kMask, typename F>
__device__ __forceinline__ void walk_row_chunks(const int32_t *ids, int n, int lane, bool vec4, F &&emit) {
    if (n <= 0) return;
    const int per = vec4 ? (((n + 31) >> 5) + 3) & ~3 : (n + 31) >> 5;
    const int i0 = min(n, lane * per), i1 = min(n, i0 + per);
    int cf = -1, cl = -1;   // chunks of the lane's first and last runs
    uint64_t mf = 0, ml = 0;  // their key masks
    int nruns = 0;
    constexpr int kBatch = 16;  // ids loaded together (independent loads in flight)
    for (int base = i0; base < i1; base += kBatch) {
        int32_t buf[kBatch];
        if (vec4) {
#pragma unroll
            for (int u = 0; u < kBatch; u += 4) {
                const int4 v = base + u < i1 ? __ldg(reinterpret_cast<const int4 *>(ids + base + u)) : make_int4(0, 0, 0, 0);
                buf[u] = v.x;
                buf[u + 1] = v.y;
                buf[u + 2] = v.z;
                buf[u + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int u = 0; u < kBatch; ++u) buf[u] = base + u < i1 ? __ldg(ids + base + u) : 0;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (base + u >= i1) break;
            const int c = buf[u] >> 6;
            if (c != cl) {
                if (nruns == 1) {
                    cf = cl;
                    mf = ml;
                } else if (nruns > 1) {
                    emit(cl, ml);  // a run that starts and ends inside this lane's range
                }
                cl = c;
                ml = 0;
                ++nruns;
            }
            if (kMask) ml |= 1ull << (buf[u] & 63);
        }
    }
    if (nruns == 1) {
        cf = cl;
        mf = ml;
    }
    const bool single = nruns == 1;
    // Whether the first run continues the previous lane's last run, and whether the next lane's first run
    // continues this lane's last run (empty lanes have cf = cl = -1 and continue nothing).
    const int cl_prev = __shfl_up_sync(0xffffffffu, cl, 1);
    const int cf_next = __shfl_down_sync(0xffffffffu, cf, 1);
    const bool cont_in = nruns > 0 && lane > 0 && cf == cl_prev;
    const bool cont_out = nruns > 0 && lane < 31 && cf_next >= 0 && cf_next == cl;
    uint64_t carry = 0;  // mask of the run this lane's first run continues, over the lanes before it
    if (kMask) {
        // Segmented inclusive OR over the lanes' last runs: a lane whose whole range is one run that continues
        // the previous lane's links to it; any other lane starts a segment.
        uint64_t acc = ml;
        bool head = !(single && cont_in);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t up = __shfl_up_sync(0xffffffffu, acc, o);
            const bool head_up = __shfl_up_sync(0xffffffffu, head, o);
            if (lane >= o && !head) {
                acc |= up;
                head = head_up;
            }
        }
        const uint64_t prev = __shfl_up_sync(0xffffffffu, acc, 1);
        carry = cont_in ? prev : 0ull;
    }
    if (nruns == 0) return;
    if (single) {
        if (!cont_out) emit(cf, mf | carry);
    } else {
        emit(cf, mf | carry);
        if (!cont_out) emit(cl, ml);
    }
}

// One CTA per block of 64 query rows: rmask[block][c] = the block's rows that route into chunk c.
__global__ void __launch_bounds__(kBlockThreads) chunk_mask_kernel(ChunkArgs a) {
    extern __shared__ unsigned long long tbl[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int64_t blk = blockIdx.x;
    const int64_t b = blk / a.n_blk_b, q0 = (blk % a.n_blk_b) * kBlockRows;
    for (int64_t c = threadIdx.x; c < a.NC; c += blockDim.x) tbl[c] = 0ull;
    __syncthreads();
    for (int r = warp; r < kBlockRows && q0 + r < a.S_q; r += nwarps) {
        const int64_t row = b * a.S_q + q0 + r;
        const unsigned long long bit = 1ull << r;
        walk_row_chunks<false>(a.ids + row * a.K, a.counts[row], lane, (a.K & 3) == 0,
                               [&](int c, uint64_t) { atomicOr(&tbl[c], bit); });
    }
    __syncthreads();
    uint64_t *out = a.rmask + blk * a.NC;
    for (int64_t c = threadIdx.x; c < a.NC; c += blockDim.x) out[c] = tbl[c];
}

// One warp per list (b, c): block offsets inside the list (a warp scan over 32
// blocks at a time), the list length (to list_start[l]) and the number of
// parts, window by window (to part_start[l]); both are scanned next.
__global__ void __launch_bounds__(256) chunk_colscan_kernel(ChunkArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t l = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (l >= a.B * a.NC) return;  // whole warps
    const int64_t b = l / a.NC, c = l % a.NC;
    const uint64_t *rm = a.rmask + b * a.n_blk_b * a.NC + c;
    int32_t *ho = a.hoff + b * a.n_blk_b * a.NC + c;
    int32_t run = 0;
    for (int64_t k0 = 0; k0 < a.n_blk_b; k0 += 32) {
        const int64_t k = k0 + lane;
        const int v = k < a.n_blk_b ? __popcll(rm[k * a.NC]) : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (k < a.n_blk_b) ho[k * a.NC] = run + incl - v;
        run += __shfl_sync(0xffffffffu, incl, 31);
    }
    __syncwarp();
    if (lane == 0) {
        const int64_t per = a.max_groups * a.slots;
        int32_t parts = 0;
        for (int64_t w = 0; w < a.n_win_b; ++w) {
            const int64_t k0 = w * a.win_blocks, k1 = k0 + a.win_blocks;
            const int32_t s0 = ho[k0 * a.NC];
            const int32_t s1 = k1 < a.n_blk_b ? ho[k1 * a.NC] : run;
            parts += (int32_t)((s1 - s0 + per - 1) / per);
        }
        a.list_start[l] = run;
        a.part_start[l] = parts;
    }
}

// One CTA per block again: every (row, chunk) entry with its key mask, at the
// list position fixed by the block offset and the row's rank in the block.
__global__ void __launch_bounds__(kBlockThreads) chunk_fill_kernel(ChunkArgs a) {
    extern __shared__ unsigned long long tbl[];
    int32_t *base = reinterpret_cast<int32_t *>(tbl + a.NC);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int64_t blk = blockIdx.x;
    const int64_t b = blk / a.n_blk_b, q0 = (blk % a.n_blk_b) * kBlockRows;
    for (int64_t c = threadIdx.x; c < a.NC; c += blockDim.x) {
        tbl[c] = a.rmask[blk * a.NC + c];
        base[c] = a.list_start[b * a.NC + c] + a.hoff[blk * a.NC + c];
    }
    __syncthreads();
    for (int r = warp; r < kBlockRows && q0 + r < a.S_q; r += nwarps) {
        const int64_t row = b * a.S_q + q0 + r;
        const unsigned long long below = (1ull << r) - 1ull;
        walk_row_chunks<true>(a.ids + row * a.K, a.counts[row], lane, (a.K & 3) == 0, [&](int c, uint64_t m) {
            const int pos = base[c] + __popcll(tbl[c] & below);
            a.e_q[pos] = (int32_t)(q0 + r);
            a.e_mask[pos] = m;
        });
    }
    if (!a.tile_keys) return;
    // The block's query tiles (T = slots rows each): distinct routed keys per tile, the union of its rows'
    // masks summed over the chunks.  The block's entries of chunk c are contiguous in list c and in row
    // order, so each tile's rows form one run there.
    int *tcount = reinterpret_cast<int *>(base + a.NC);
    const int tiles = (kBlockRows + (int)a.slots - 1) / (int)a.slots;
    for (int t = threadIdx.x; t < tiles; t += blockDim.x) tcount[t] = 0;
    __syncthreads();  // also makes the entries written above visible to the whole block
    for (int64_t c = threadIdx.x; c < a.NC; c += blockDim.x) {
        const int n = __popcll(tbl[c]);
        int cur = -1;
        uint64_t u = 0;
        constexpr int kBatch = 4;  // entries loaded together
        for (int i0 = 0; i0 < n; i0 += kBatch) {
            int32_t qv[kBatch];
            uint64_t mv[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                qv[j] = i0 + j < n ? a.e_q[base[c] + i0 + j] : 0;
                mv[j] = i0 + j < n ? a.e_mask[base[c] + i0 + j] : 0ull;
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                if (i0 + j >= n) break;
                const int t = (int)((qv[j] - q0) / a.slots);
                if (t != cur) {
                    if (cur >= 0) atomicAdd(&tcount[cur], __popcll(u));
                    cur = t;
                    u = 0;
                }
                u |= mv[j];
            }
        }
        if (cur >= 0) atomicAdd(&tcount[cur], __popcll(u));
    }
    __syncthreads();
    const int64_t n_tiles_b = (a.S_q + a.slots - 1) / a.slots;
    for (int t = threadIdx.x; t < tiles; t += blockDim.x) {
        const int64_t tg = q0 / a.slots + t;
        if (tg < n_tiles_b) a.tile_keys[b * n_tiles_b + tg] = tcount[t];
    }
}

// One thread per list: its parts, window by window (a window's entries are
// contiguous in the list), each at most max_groups * slots entries.
__global__ void chunk_items_kernel(ChunkArgs a) {
    const int64_t l = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (l >= a.B * a.NC) return;
    const int64_t b = l / a.NC, c = l % a.NC;
    const int32_t per = (int32_t)(a.max_groups * a.slots);
    const int32_t st = a.list_start[l], len = a.list_start[l + 1] - st;
    const int32_t *ho = a.hoff + b * a.n_blk_b * a.NC + c;
    int64_t out = a.part_start[l];
    for (int64_t w = 0; w < a.n_win_b; ++w) {
        const int64_t k0 = w * a.win_blocks, k1 = k0 + a.win_blocks;
        const int32_t s0 = ho[k0 * a.NC];
        const int32_t s1 = k1 < a.n_blk_b ? ho[k1 * a.NC] : len;
        for (int32_t e = s0; e < s1; e += per, ++out) {
            const int32_t n = s1 - e < per ? s1 - e : per;
            if (out < a.cap_items) a.items[out] = make_int4((int32_t)l, st + e, n, (int32_t)(b * a.n_win_b + w));
        }
    }
}

// In-place exclusive scan of x[0..n) by one CTA; x[n] = total, *total_out = total.
__global__ void __launch_bounds__(kScanThreads) scan_kernel(int32_t *x, int64_t n, int32_t *total_out) {
    __shared__ int warp_tot[33];
    constexpr int kPer = 8;
    int carry = 0;
    for (int64_t base = 0; base < n; base += (int64_t)kScanThreads * kPer) {
        int v[kPer];
        int local = 0;
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            const int64_t i = base + (int64_t)threadIdx.x * kPer + e;
            v[e] = i < n ? x[i] : 0;
            local += v[e];
        }
        int total;
        int pos = carry + block_scan_excl(local, warp_tot, total);
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            const int64_t i = base + (int64_t)threadIdx.x * kPer + e;
            if (i < n) x[i] = pos;
            pos += v[e];
        }
        carry += total;
    }
    if (threadIdx.x == 0) {
        x[n] = carry;
        *total_out = carry;
    }
}

// One CTA: items sorted by (window, groups descending) with a counting sort,
// then the queue: for every window, for every KV head, the window's items.
__global__ void __launch_bounds__(kQueueThreads) chunk_queue_kernel(ChunkArgs a) {
    __shared__ int hist[kQueueBins];
    __shared__ int warp_tot[33];
    const int64_t n_items = a.meta[1];
    if (n_items > a.cap_items) {  // cannot happen within the workspace bound; refuse rather than overrun
        if (threadIdx.x == 0) {
            a.meta[2] = 0;
            a.meta[3] = 1;
            raise_status(a.status, QSA_ERR_DEVICE_CHECK, kSiteChunkCapacity, (unsigned)n_items, (unsigned)a.cap_items);
        }
        return;
    }
    const int nbin_w = (int)a.max_groups + 1;
    const int64_t n_win = a.B * a.n_win_b;
    for (int i = threadIdx.x; i < kQueueBins; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    auto bin_of = [&](const int4 &it) {
        const int64_t groups = (it.z + a.slots - 1) / a.slots;
        const int64_t gclamp = groups < a.max_groups ? groups : a.max_groups;
        return (int)(it.w * nbin_w + (a.max_groups - gclamp));
    };
    for (int64_t i = threadIdx.x; i < n_items; i += blockDim.x) atomicAdd(&hist[bin_of(a.items[i])], 1);
    __syncthreads();
    constexpr int kPer = kQueueBins / kQueueThreads;
    int local = 0;
    for (int e = 0; e < kPer; ++e) local += hist[threadIdx.x * kPer + e];
    int total;
    int pos = block_scan_excl(local, warp_tot, total);
    for (int e = 0; e < kPer; ++e) {
        const int h = hist[threadIdx.x * kPer + e];
        hist[threadIdx.x * kPer + e] = pos;
        pos += h;
    }
    __syncthreads();
    // Window starts (item positions) before the scatter moves the bin offsets.
    __shared__ int wstart[kQueueMaxWindows + 1];
    for (int64_t w = threadIdx.x; w <= n_win && w <= kQueueMaxWindows; w += blockDim.x)
        wstart[w] = w < n_win ? hist[w * nbin_w] : (int)n_items;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n_items; i += blockDim.x) {
        const int p = atomicAdd(&hist[bin_of(a.items[i])], 1);
        a.sorted[p] = (int32_t)i;
    }
    __syncthreads();
    const int64_t H = a.Hkv;
    for (int64_t w = 0; w < n_win; ++w) {
        const int64_t ws = wstart[w], we = wstart[w + 1], nw = we - ws;
        for (int64_t j = threadIdx.x; j < nw * H; j += blockDim.x) {
            const int64_t g = j / nw, r = j % nw;
            a.queue[ws * H + j] = (int32_t)(a.sorted[ws + r] * H + g);
        }
    }
    if (threadIdx.x == 0) {
        a.meta[2] = (int32_t)(n_items * H);
        a.meta[3] = 0;
    }
}

}  // namespace

cudaError_t launch_chunk_lists(const ChunkArgs &a, cudaStream_t s) {
    const int64_t n_blk = a.B * a.n_blk_b, n_lists = a.B * a.NC;
    const size_t smem_mask = (size_t)a.NC * sizeof(uint64_t);
    const size_t smem_fill = (size_t)a.NC * (sizeof(uint64_t) + sizeof(int32_t)) + kBlockRows * sizeof(int32_t);
    cudaError_t e = cudaSuccess;
    if (smem_fill > 48 * 1024) {
        e = cudaFuncSetAttribute(chunk_mask_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_mask);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(chunk_fill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_fill);
        if (e != cudaSuccess) return e;
    }
    const unsigned list_blocks = (unsigned)((n_lists + 255) / 256);
    chunk_mask_kernel<<<(unsigned)n_blk, kBlockThreads, smem_mask, s>>>(a);
    chunk_colscan_kernel<<<(unsigned)((n_lists * 32 + 255) / 256), 256, 0, s>>>(a);
    scan_kernel<<<1, kScanThreads, 0, s>>>(a.list_start, n_lists, a.meta + 0);
    scan_kernel<<<1, kScanThreads, 0, s>>>(a.part_start, n_lists, a.meta + 1);
    chunk_fill_kernel<<<(unsigned)n_blk, kBlockThreads, smem_fill, s>>>(a);
    chunk_items_kernel<<<list_blocks, 256, 0, s>>>(a);
    chunk_queue_kernel<<<1, kQueueThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace qsa

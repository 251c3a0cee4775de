// qsa_preprocess.cu -- route preprocessing kernels.
//
// The pages' preprocessing (fa4_qsa _preprocess, _block_kinds, _compact_blocks;
// flex_qsa _routes_to_membership) turns routes into a dense membership table and
// block lists.  Here nothing dense is ever built in HBM:
//
//   route_rows_kernel  one CTA per query row: read the row's K route slots in
//                      their own width (int32 or int64), keep 0 <= id < S_kv
//                      (invalid values, huge int64 included, never reach an
//                      index), mark them in a shared-memory byte map (rows
//                      spread wider: a bitmap) over the row's id range and
//                      read it back in order with coalesced stores (sorted,
//                      repeats gone); a bitonic sort handles rows
//                      whose ids are spread over a very wide range.
//                      Output: ascending unique IDs (int32, -1 tail) + count.
//   route_tiles_kernel one CTA per tile of T consecutive query rows: the union
//                      of the rows' ID sets, ascending, cut into chunks of 64
//                      keys, and for every (chunk, query) a 64-bit mask of the
//                      chunk keys that query routes to.  The union is built a
//                      window of key space at a time in a shared-memory table
//                      of per-key query bitmasks (the membership table, but
//                      only T x W bits of it, never in HBM).
//   route_order_kernel counting sort of tiles by chunk count, heaviest first,
//                      for the attention kernels' static schedule.
#include <algorithm>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kRowThreads = 128;
constexpr int kTileThreads = 512;
constexpr int kTileWindow = 4096;  // keys per window of the shared-memory membership table
constexpr int kTileBatches = 8;   // 32-id batches of one row read per step (independent loads)
constexpr int kRowMapKeys = 16384;       // rows whose ids span at most this many keys: shared-memory byte map
constexpr int kRowWindowBits = 65536;    // wider rows: keys per window of a shared-memory bitmap (8 KiB)
constexpr int kRowMaxWindows = 8;        // still wider rows fall back to the bitonic sort
// Shared memory of the map and bitmap passes: byte map + its bit words + word offsets, or bitmap + offsets.
constexpr size_t kRowSmem = kRowMapKeys + (size_t)kRowMapKeys / 32 * 8 > (size_t)kRowWindowBits / 32 * 8
                                ? kRowMapKeys + (size_t)kRowMapKeys / 32 * 8
                                : (size_t)kRowWindowBits / 32 * 8;
constexpr int kRowCache = 17;          // route slots per thread kept in registers (K <= 17 * kRowThreads)

__device__ __forceinline__ int block_exclusive_scan(int x, int *warp_tot, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nwarps ? warp_tot[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < nwarps) warp_tot[lane] = wi - w;  // exclusive per-warp offsets
        if (lane == 31) warp_tot[32] = wi;
    }
    __syncthreads();
    total = warp_tot[32];
    int r = warp_tot[warp] + incl - x;
    __syncthreads();
    return r;
}

__device__ __forceinline__ int64_t load_route(const RowsArgs &a, int64_t b, int64_t q, int64_t i) {
    const int64_t off = b * a.rs0 + q * a.rs1 + i * a.rs2;
    return a.route_bits == 64 ? static_cast<const int64_t *>(a.routes)[off]
                              : (int64_t) static_cast<const int32_t *>(a.routes)[off];
}

// Bytes b0..b3 of w, each 0 or 1, as the bits 0..3 of a nibble: the product
// puts byte k's value alone at bit 21 + k (the four partial products of each
// byte land on distinct bits, so nothing carries into bits 21..24).
__device__ __forceinline__ uint32_t flag_nibble(uint32_t w) { return ((w * 0x00204081u) >> 21) & 0xFu; }

// Sorting without comparisons.  A row whose valid ids span at most kRowMapKeys
// keys marks them in a shared-memory byte map (plain byte stores: repeated or
// neighbouring ids need no atomics), packed afterwards into 32-key bit words.
// Wider rows set bits of a shared-memory bitmap with atomicOr, a window of
// kRowWindowBits keys at a time.  Either way one block scan of the words'
// popcounts gives every word its output offset, and each warp then writes a
// word's keys as one contiguous run (lane = bit): the ids come out ascending
// with repeats gone, in coalesced stores.  Cost O(K + range/16) for the map,
// O(K + range/32) per bitmap window; rows whose ids span more than
// kRowMaxWindows windows use the bitonic sort instead.
template <bool kTrySorted>
__global__ void __launch_bounds__(kRowThreads, 8) route_rows_kernel(RowsArgs a, int P) {
    extern __shared__ __align__(16) uint32_t rsm[];  // map + words + offsets, bitmap + offsets, or bitonic buffer [P]
    __shared__ int warp_tot[33];
    __shared__ int64_t red_lo[kRowThreads / 32], red_hi[kRowThreads / 32];
    __shared__ int32_t lane0[kRowCache + 1][kRowThreads / 32];  // cached slot j of each warp's lane 0
    __shared__ int n_valid;
    __shared__ bool red_sorted[kRowThreads / 32];
    const int64_t row = blockIdx.x;
    const int64_t b = row / a.S_q, q = row % a.S_q;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    int32_t *out = a.ids + row * a.K;

    // Range of the valid ids (validity tested in the route's own width).  Rows of up to
    // kRowCache * blockDim.x slots are read once and kept in registers for the bitmap pass.
    const bool cached = a.K <= (int64_t)kRowCache * blockDim.x;
    int32_t cache[kRowCache];
    int64_t lo = INT64_MAX, hi = -1;
    if (cached) {
#pragma unroll
        for (int j = 0; j < kRowCache; ++j) {
            const int64_t i = tid + (int64_t)j * blockDim.x;
            const int64_t x = i < a.K ? load_route(a, b, q, i) : -1;
            const bool valid = x >= 0 && x < a.S_kv;
            cache[j] = valid ? (int32_t)x : -1;
            if (valid) {
                lo = min(lo, x);
                hi = max(hi, x);
            }
        }
    } else {
        for (int64_t i = tid; i < a.K; i += blockDim.x) {
            const int64_t x = load_route(a, b, q, i);
            if (x >= 0 && x < a.S_kv) {
                lo = min(lo, x);
                hi = max(hi, x);
            }
        }
    }
    // With QSA_ROUTES_SORTED (kTrySorted), rows that arrive sorted (valid ids strictly ascending, every
    // invalid slot after them, as the route producer writes them) are copied through.  Slot i is checked against slot i + 1: the next lane's slot j
    // (shuffles; the verdict of each warp rides on the range reduction's barrier), or for lane 31 the next
    // warp's lane 0 (slot j + 1 of warp 0 after the last warp), checked only when every warp passed.
    bool warp_sorted = false;
    if (kTrySorted && cached) {
        bool bad = false;
#pragma unroll
        for (int j = 0; j < kRowCache; ++j) {
            const int32_t x = cache[j];
            const int32_t y = __shfl_down_sync(0xffffffffu, x, 1);
            bad |= lane < 31 && ((y >= 0 && x < 0) || (x >= 0 && y >= 0 && y <= x));
            // The thread's own slots, 128 apart, must ascend too: rejects most unsorted rows before any
            // exchange between warps.
            if (j + 1 < kRowCache) bad |= cache[j + 1] >= 0 && (x < 0 || cache[j + 1] <= x);
        }
        warp_sorted = !__any_sync(0xffffffffu, bad);
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < kRowCache; ++j) lane0[j][warp] = cache[j];
        }
        if (tid < nwarps) lane0[kRowCache][tid] = -1;
        if (tid == 0) n_valid = 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
        red_lo[warp] = lo;
        red_hi[warp] = hi;
        if (kTrySorted) red_sorted[warp] = warp_sorted;
    }
    __syncthreads();
    if (kTrySorted && cached) {
        bool all = true;
        for (int w = 0; w < nwarps; ++w) all &= red_sorted[w];
        if (all) {  // uniform over the block
            bool bad = false;
            int nv = 0;
#pragma unroll
            for (int j = 0; j < kRowCache; ++j) {
                const int32_t x = cache[j];
                const int32_t y = warp + 1 < nwarps ? lane0[j][warp + 1] : lane0[j + 1][0];
                bad |= lane == 31 && ((y >= 0 && x < 0) || (x >= 0 && y >= 0 && y <= x));
                nv += x >= 0;
            }
            if (__syncthreads_and(!bad)) {
                atomicAdd(&n_valid, nv);
                __syncthreads();
                const int total = n_valid;
#pragma unroll
                for (int j = 0; j < kRowCache; ++j) {
                    const int64_t i = tid + (int64_t)j * blockDim.x;
                    if (i < a.K) out[i] = cache[j];  // -1 for invalid slots, which all come after the valid ones
                }
                if (tid == 0) a.counts[row] = total;
                return;
            }
        }
    }
    lo = red_lo[0];
    hi = red_hi[0];
    for (int w = 1; w < nwarps; ++w) {
        lo = min(lo, red_lo[w]);
        hi = max(hi, red_hi[w]);
    }
    int total = 0;
    if (hi >= 0 && hi - lo < kRowMapKeys) {
        uint8_t *flags = reinterpret_cast<uint8_t *>(rsm);
        uint32_t *words = rsm + kRowMapKeys / 4;
        int *woff = reinterpret_cast<int *>(words + kRowMapKeys / 32);
        for (int64_t w0 = lo; w0 <= hi; w0 += kRowMapKeys) {  // one pass: the range fits the map
            const int64_t span = (hi - w0 + 1) < kRowMapKeys ? (hi - w0 + 1) : (int64_t)kRowMapKeys;
            const int nwords = (int)((span + 31) / 32);
            for (int i = tid; i < nwords * 2; i += blockDim.x) reinterpret_cast<uint4 *>(flags)[i] = make_uint4(0, 0, 0, 0);
            __syncthreads();
            if (cached) {
#pragma unroll
                for (int j = 0; j < kRowCache; ++j) {
                    const int64_t x = cache[j];
                    if (x >= w0 && x < w0 + span) flags[x - w0] = 1;
                }
            } else {
                for (int64_t i = tid; i < a.K; i += blockDim.x) {
                    const int64_t x = load_route(a, b, q, i);
                    if (x >= w0 && x < w0 + span) flags[x - w0] = 1;
                }
            }
            __syncthreads();
            const int per = (nwords + blockDim.x - 1) / blockDim.x;
            const int s0 = min(nwords, tid * per), s1 = min(nwords, s0 + per);
            int local = 0;
            for (int i = s0; i < s1; ++i) {
                const uint4 *f = reinterpret_cast<const uint4 *>(flags + i * 32);
                const uint4 u = f[0], v = f[1];
                const uint32_t bits = flag_nibble(u.x) | flag_nibble(u.y) << 4 | flag_nibble(u.z) << 8 |
                                      flag_nibble(u.w) << 12 | flag_nibble(v.x) << 16 | flag_nibble(v.y) << 20 |
                                      flag_nibble(v.z) << 24 | flag_nibble(v.w) << 28;
                words[i] = bits;
                local += __popc(bits);
            }
            int win_total;
            int pos = total + block_exclusive_scan(local, warp_tot, win_total);
            for (int i = s0; i < s1; ++i) {
                woff[i] = pos;
                pos += __popc(words[i]);
            }
            __syncthreads();
            for (int g = warp * 32; g < nwords; g += nwarps * 32) {
                const int i = g + lane;
                const uint32_t my_bits = i < nwords ? words[i] : 0u;
                const int my_off = i < nwords ? woff[i] : 0;
                uint32_t nz = __ballot_sync(0xffffffffu, my_bits != 0u);
                while (nz) {
                    const int src = __ffs(nz) - 1;
                    nz &= nz - 1;
                    const uint32_t bits = __shfl_sync(0xffffffffu, my_bits, src);
                    const int off = __shfl_sync(0xffffffffu, my_off, src);
                    if ((bits >> lane) & 1u)
                        out[off + __popc(bits & ((1u << lane) - 1u))] = (int32_t)(w0 + (int64_t)(g + src) * 32 + lane);
                }
            }
            total += win_total;
            __syncthreads();
        }
    } else if (hi >= 0 && (hi - lo) / kRowWindowBits < kRowMaxWindows) {
        uint32_t *words = rsm;
        int *woff = reinterpret_cast<int *>(rsm + kRowWindowBits / 32);
        for (int64_t w0 = lo; w0 <= hi; w0 += kRowWindowBits) {
            const int64_t span = (hi - w0 + 1) < kRowWindowBits ? (hi - w0 + 1) : (int64_t)kRowWindowBits;
            const int nwords = (int)((span + 31) / 32);
            for (int i = tid; i < nwords; i += blockDim.x) words[i] = 0u;
            __syncthreads();
            if (cached) {
#pragma unroll
                for (int j = 0; j < kRowCache; ++j) {
                    const int64_t x = cache[j];
                    if (x >= w0 && x < w0 + span) atomicOr(&words[(x - w0) >> 5], 1u << ((x - w0) & 31));
                }
            } else {
                for (int64_t i = tid; i < a.K; i += blockDim.x) {
                    const int64_t x = load_route(a, b, q, i);
                    if (x >= w0 && x < w0 + span) atomicOr(&words[(x - w0) >> 5], 1u << ((x - w0) & 31));
                }
            }
            __syncthreads();
            const int per = (nwords + blockDim.x - 1) / blockDim.x;
            const int s0 = min(nwords, tid * per), s1 = min(nwords, s0 + per);
            int local = 0;
            for (int i = s0; i < s1; ++i) {
                local += __popc(words[i]);
            }
            int win_total;
            int pos = total + block_exclusive_scan(local, warp_tot, win_total);
            for (int i = s0; i < s1; ++i) {
                woff[i] = pos;
                pos += __popc(words[i]);
            }
            __syncthreads();
            for (int g = warp * 32; g < nwords; g += nwarps * 32) {
                const int i = g + lane;
                const uint32_t my_bits = i < nwords ? words[i] : 0u;
                const int my_off = i < nwords ? woff[i] : 0;
                uint32_t nz = __ballot_sync(0xffffffffu, my_bits != 0u);
                while (nz) {
                    const int src = __ffs(nz) - 1;
                    nz &= nz - 1;
                    const uint32_t bits = __shfl_sync(0xffffffffu, my_bits, src);
                    const int off = __shfl_sync(0xffffffffu, my_off, src);
                    if ((bits >> lane) & 1u)
                        out[off + __popc(bits & ((1u << lane) - 1u))] = (int32_t)(w0 + (int64_t)(g + src) * 32 + lane);
                }
            }
            total += win_total;
            __syncthreads();
        }
    } else if (hi >= 0) {
        int32_t *srt = reinterpret_cast<int32_t *>(rsm);
        for (int i = tid; i < P; i += blockDim.x) {
            int32_t v = INT32_MAX;
            if (i < a.K) {
                const int64_t x = load_route(a, b, q, i);
                if (x >= 0 && x < a.S_kv) v = (int32_t)x;
            }
            srt[i] = v;
        }
        __syncthreads();
        for (int k = 2; k <= P; k <<= 1) {
            for (int j = k >> 1; j > 0; j >>= 1) {
                for (int i = tid; i < P; i += blockDim.x) {
                    const int ixj = i ^ j;
                    if (ixj > i) {
                        const int32_t x = srt[i], y = srt[ixj];
                        if ((x > y) == ((i & k) == 0)) {
                            srt[i] = y;
                            srt[ixj] = x;
                        }
                    }
                }
                __syncthreads();
            }
        }
        const int seg = (P + blockDim.x - 1) / blockDim.x;
        const int s0 = min(P, tid * seg), s1 = min(P, s0 + seg);
        int local = 0;
        for (int i = s0; i < s1; ++i) local += srt[i] != INT32_MAX && (i == 0 || srt[i] != srt[i - 1]);
        int pos = block_exclusive_scan(local, warp_tot, total);
        for (int i = s0; i < s1; ++i)
            if (srt[i] != INT32_MAX && (i == 0 || srt[i] != srt[i - 1])) out[pos++] = srt[i];
    }
    for (int64_t i = total + tid; i < a.K; i += blockDim.x) out[i] = -1;
    if (tid == 0) a.counts[row] = total;
}

// Emit one chunk of 64 union keys: keys, and for each tile query the mask of
// the chunk's keys it routes to.  Executed by one full warp.
__device__ __forceinline__ void emit_chunk(const TilesArgs &a, int64_t tile, int64_t chunk, const uint32_t *cw,
                                           const int32_t *ck) {
    const int lane = threadIdx.x & 31;
    const uint32_t w_lo = cw[lane], w_hi = cw[32 + lane];
    int32_t *keys = a.tile_keys + (tile * a.max_chunks + chunk) * kChunkKeys;
    keys[lane] = ck[lane];
    keys[32 + lane] = ck[32 + lane];
    uint64_t mine = 0;
    for (int qi = 0; qi < a.T; ++qi) {
        const uint32_t lo = __ballot_sync(0xffffffffu, (w_lo >> qi) & 1u);
        const uint32_t hi = __ballot_sync(0xffffffffu, (w_hi >> qi) & 1u);
        if (lane == qi) mine = (uint64_t)lo | ((uint64_t)hi << 32);
    }
    if (lane < a.T) a.tile_masks[(tile * a.max_chunks + chunk) * a.T + lane] = mine;
}

__global__ void __launch_bounds__(kTileThreads) route_tiles_kernel(TilesArgs a) {
    if (a.skip && a.skip[0] == 1 && a.skip[1] == 1) return;
    extern __shared__ uint32_t tsm[];
    uint32_t *mem = tsm;                                              // [W] per-key query bitmask
    uint32_t *cw = mem + kTileWindow;                                 // [W + 64] compacted bitmasks
    int32_t *ck = reinterpret_cast<int32_t *>(cw + kTileWindow + 64);  // [W + 64] compacted keys
    __shared__ int ptr[32], cnt[32], warp_tot[33];
    __shared__ int64_t s_next;
    const int64_t tile = blockIdx.x;
    const int64_t b = tile / a.n_tiles, t = tile % a.n_tiles;
    const int64_t q0 = t * a.T;
    const int nq = (int)(a.T < a.S_q - q0 ? a.T : a.S_q - q0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    if (tid < 32) {
        ptr[tid] = 0;
        cnt[tid] = tid < nq ? a.counts[b * a.S_q + q0 + tid] : 0;
    }
    __syncthreads();
    int carry = 0;
    int64_t nchunks = 0;
    for (;;) {
        if (warp == 0) {
            int64_t nx = INT64_MAX;
            if (lane < nq && ptr[lane] < cnt[lane]) nx = a.ids[(b * a.S_q + q0 + lane) * a.K + ptr[lane]];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) nx = min(nx, __shfl_xor_sync(0xffffffffu, nx, o));
            if (lane == 0) s_next = nx;
        }
        __syncthreads();
        const int64_t w0 = s_next;
        if (w0 == INT64_MAX) break;
        for (int i = tid; i < kTileWindow; i += blockDim.x) mem[i] = 0u;
        __syncthreads();
        for (int qi = warp; qi < nq; qi += nwarps) {
            const int32_t *row = a.ids + (b * a.S_q + q0 + qi) * a.K;
            int p = ptr[qi];
            const int c = cnt[qi];
            // kTileBatches batches of 32 ids per step, loaded independently; ids ascend, so the
            // window ends in the first batch that is not entirely inside it.
            bool more = p < c;
            while (more) {
                int64_t id[kTileBatches];
#pragma unroll
                for (int u = 0; u < kTileBatches; ++u) {
                    const int idx = p + u * 32 + lane;
                    id[u] = idx < c ? (int64_t)row[idx] : INT64_MAX;
                }
                int n_step = 0;
#pragma unroll
                for (int u = 0; u < kTileBatches; ++u) {
                    const bool in = id[u] < w0 + kTileWindow;
                    if (in) atomicOr(&mem[id[u] - w0], 1u << qi);
                    const int n_in = __popc(__ballot_sync(0xffffffffu, in));
                    n_step += n_in;
                    if (n_in < 32) {
                        more = false;
                        break;
                    }
                }
                p += n_step;
                more = more && p < c;
            }
            if (lane == 0) ptr[qi] = p;
        }
        __syncthreads();
        const int per = kTileWindow / kTileThreads;
        const int base = tid * per;
        int local = 0;
        for (int e = 0; e < per; ++e) local += mem[base + e] != 0u;
        int total;
        int pos = carry + block_exclusive_scan(local, warp_tot, total);
        for (int e = 0; e < per; ++e) {
            const uint32_t w = mem[base + e];
            if (w) {
                cw[pos] = w;
                ck[pos] = (int32_t)(w0 + base + e);
                ++pos;
            }
        }
        __syncthreads();
        const int all = carry + total;
        const int full = all / kChunkKeys;
        for (int c = warp; c < full; c += nwarps) {
            if (nchunks + c < a.max_chunks) emit_chunk(a, tile, nchunks + c, cw + c * kChunkKeys, ck + c * kChunkKeys);
        }
        const int rem = all - full * kChunkKeys;
        uint32_t tw = 0;
        int32_t tk = 0;
        if (tid < rem) {
            tw = cw[full * kChunkKeys + tid];
            tk = ck[full * kChunkKeys + tid];
        }
        __syncthreads();
        if (tid < rem) {
            cw[tid] = tw;
            ck[tid] = tk;
        }
        nchunks += full;
        carry = rem;
        __syncthreads();
    }
    if (carry > 0) {
        // Last, partial chunk: pad with the chunk's first key (a valid row to
        // gather) and an empty membership so the padding never contributes.
        if (tid >= carry && tid < kChunkKeys) {
            cw[tid] = 0u;
            ck[tid] = ck[0];
        }
        __syncthreads();
        if (warp == 0 && nchunks < a.max_chunks) emit_chunk(a, tile, nchunks, cw, ck);
        ++nchunks;
    }
    if (tid == 0) a.tile_nchunks[tile] = (int32_t)(nchunks < a.max_chunks ? nchunks : a.max_chunks);
}

constexpr int kOrderThreads = 1024;
constexpr int kOrderBins = 8192;

// Tiles sorted by chunk count, heaviest first (counting sort; ties in any order).
__global__ void __launch_bounds__(kOrderThreads) route_order_kernel(const int32_t *nchunks, int64_t n, int32_t *order,
                                                                    const int32_t *skip) {
    if (skip && skip[0] == 1 && skip[1] == 1) return;
    __shared__ int hist[kOrderBins];
    __shared__ int warp_tot[33];
    for (int i = threadIdx.x; i < kOrderBins; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) atomicAdd(&hist[kOrderBins - 1 - min(nchunks[i], kOrderBins - 1)], 1);
    __syncthreads();
    const int per = kOrderBins / kOrderThreads;
    int local = 0;
    for (int e = 0; e < per; ++e) local += hist[threadIdx.x * per + e];
    int total;
    int pos = block_exclusive_scan(local, warp_tot, total);
    for (int e = 0; e < per; ++e) {
        const int h = hist[threadIdx.x * per + e];
        hist[threadIdx.x * per + e] = pos;
        pos += h;
    }
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
        const int p = atomicAdd(&hist[kOrderBins - 1 - min(nchunks[i], kOrderBins - 1)], 1);
        order[p] = (int32_t)i;
    }
}

}  // namespace

cudaError_t launch_route_rows(const RowsArgs &a, cudaStream_t s) {
    int P = 32;
    while (P < a.K) P <<= 1;
    const size_t smem = std::max<size_t>((size_t)P * sizeof(int32_t), kRowSmem);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(route_rows_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(route_rows_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    if (a.try_sorted) route_rows_kernel<true><<<(unsigned)(a.B * a.S_q), kRowThreads, smem, s>>>(a, P);
    else route_rows_kernel<false><<<(unsigned)(a.B * a.S_q), kRowThreads, smem, s>>>(a, P);
    return cudaGetLastError();
}

cudaError_t launch_route_tiles(const TilesArgs &a, cudaStream_t s) {
    const size_t smem = (size_t)kTileWindow * 4 + 2 * (size_t)(kTileWindow + 64) * 4;
    cudaError_t e = cudaFuncSetAttribute(route_tiles_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t tiles = a.B * a.n_tiles;
    route_tiles_kernel<<<(unsigned)tiles, kTileThreads, smem, s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    route_order_kernel<<<1, kOrderThreads, 0, s>>>(a.tile_nchunks, tiles, a.order, a.skip);
    return cudaGetLastError();
}

}  // namespace qsa

// qsa_api.cu -- host side of the libqsa C ABI (include/qsa.h): validation,
// workspace layout, kernel launches and status reporting.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "qsa_internal.cuh"
#include "qsa_tc.cuh"

namespace qsa {
namespace {

thread_local char g_last_error[512] = "";

qsa_status fail(qsa_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

qsa_status cuda_fail(cudaError_t e, const char *what) {
    return fail(QSA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

qsa_status validate(const qsa_problem *p) {
    if (!p) return fail(QSA_ERR_INVALID_ARGUMENT, "problem is null");
    if (p->B <= 0 || p->S_q <= 0 || p->S_kv <= 0 || p->Hq <= 0 || p->Hkv <= 0 || p->D <= 0 || p->K <= 0)
        return fail(QSA_ERR_INVALID_ARGUMENT, "every dimension must be positive (B=%lld S_q=%lld S_kv=%lld Hq=%lld "
                    "Hkv=%lld D=%lld K=%lld)", (long long)p->B, (long long)p->S_q, (long long)p->S_kv,
                    (long long)p->Hq, (long long)p->Hkv, (long long)p->D, (long long)p->K);
    if (p->Hq % p->Hkv != 0)
        return fail(QSA_ERR_INVALID_ARGUMENT, "Hq=%lld is not a multiple of Hkv=%lld", (long long)p->Hq,
                    (long long)p->Hkv);
    if (!std::isfinite(p->softmax_scale) || !(p->softmax_scale > 0.f))
        return fail(QSA_ERR_INVALID_ARGUMENT, "softmax_scale must be finite and positive (got %g)",
                    (double)p->softmax_scale);
    if (p->route_bits != 32 && p->route_bits != 64)
        return fail(QSA_ERR_INVALID_ARGUMENT, "route_bits must be 32 or 64 (got %d)", p->route_bits);
    if (p->flags & ~(QSA_ROUTES_SORTED | QSA_DETERMINISTIC_FORWARD))
        return fail(QSA_ERR_INVALID_ARGUMENT, "unknown flags 0x%x", p->flags);
    if (p->D != 64 && p->D != 128 && p->D != kHeadDim)
        return fail(QSA_ERR_UNSUPPORTED, "head dim D=%lld: 64, 128 or 256 is supported", (long long)p->D);
    if (p->S_kv > 2147483647LL) return fail(QSA_ERR_UNSUPPORTED, "S_kv=%lld exceeds 2^31-1", (long long)p->S_kv);
    if (p->K > kMaxRouteSlots)
        return fail(QSA_ERR_UNSUPPORTED, "K=%lld route slots exceeds %d", (long long)p->K, kMaxRouteSlots);
    const int64_t *st[3] = {p->q_stride, p->k_stride, p->v_stride};
    const char *nm[3] = {"q", "k", "v"};
    for (int t = 0; t < 3; ++t) {
        if (st[t][3] != 1) return fail(QSA_ERR_UNSUPPORTED, "%s needs a unit last stride (got %lld)", nm[t],
                                       (long long)st[t][3]);
        for (int i = 0; i < 3; ++i)
            if (st[t][i] < 0 || st[t][i] % 8 != 0)
                return fail(QSA_ERR_UNSUPPORTED, "%s stride[%d]=%lld must be a non-negative multiple of 8 elements",
                            nm[t], i, (long long)st[t][i]);
    }
    return QSA_OK;
}

// Key-major backward tuning (qsa_chunks.cu, qsa_bwd_km.cu).
constexpr int64_t kKmMaxGroups = 16;            // groups of 128/G queries per work item at most
constexpr int64_t kKmWindowBytes = 32ll << 20;  // fp32 dQ of one window of queries and one KV head
constexpr int64_t kKmMaskWords = 4ll << 20;     // (64-row block, chunk) mask words at most (32 MiB)
constexpr int64_t kKmMaxChunks = 16384;         // chunks per batch row (S_kv <= 2^20): counters in shared memory
constexpr int64_t kKmMaxWindows = 1024;         // windows per launch of the queue builder
constexpr int64_t kKmQueueBins = 8192;          // its counting-sort bins: windows x (groups + 1)

Layout make_layout(const qsa_problem *p) {
    Layout L{};
    L.G = p->Hq / p->Hkv;
    // The tile path covers power-of-two groups of 4..64 heads (forward: D = 256 or 128; backward:
    // D = 256); the rest runs warp-level.
    L.T = ((p->D == kHeadDim || p->D == 128) && is_pow2(L.G) && L.G >= 4 && L.G <= kTileRows) ? kTileRows / L.G : 0;
    L.n_tiles = L.T ? (p->S_q + L.T - 1) / L.T : 0;
    const int64_t union_cap = L.T ? std::min<int64_t>(L.T * p->K, p->S_kv) : 0;
    L.max_chunks = (union_cap + kChunkKeys - 1) / kChunkKeys;
    const int64_t rows = p->B * p->S_q;
    const int64_t tiles = p->B * L.n_tiles;
    size_t off = 0;
    L.off_status = off;
    off = align256(off + sizeof(DeviceStatus));
    // Work queue counters {next, done}: tile forward, tile backward, key-major backward, key-major forward
    // row-max pass, key-major forward output pass.
    L.off_sched = off;
    off = align256(off + 10 * sizeof(int32_t));
    L.off_counts = off;
    off = align256(off + rows * sizeof(int32_t));
    L.off_ids = off;
    off = align256(off + rows * p->K * sizeof(int32_t));
    L.off_tile_nchunks = off;
    off = align256(off + tiles * sizeof(int32_t));
    L.off_tile_keys = off;
    off = align256(off + tiles * L.max_chunks * kChunkKeys * sizeof(int32_t));
    L.off_tile_masks = off;
    off = align256(off + tiles * L.max_chunks * L.T * sizeof(uint64_t));
    L.off_order = off;
    off = align256(off + tiles * sizeof(int32_t));

    // Key-major backward: reverse lists per aligned 64-key chunk, cut into work items.
    L.NC = (p->S_kv + kChunkKeys - 1) / kChunkKeys;
    if (L.T) {
        const int64_t gd = L.G * p->D;
        const int64_t w_max = std::max<int64_t>(256, kKmWindowBytes / (gd * (int64_t)sizeof(float)));
        L.n_blk_b = (p->S_q + 63) / 64;
        const int64_t wb_max = (w_max + 63) / 64;
        L.n_win_b = (L.n_blk_b + wb_max - 1) / wb_max;
        L.win_blocks = (L.n_blk_b + L.n_win_b - 1) / L.n_win_b;
        L.max_groups = kKmMaxGroups;
        L.cap_entries = rows * std::min<int64_t>(p->K, L.NC);
        L.cap_items = L.cap_entries / (L.max_groups * L.T) + p->B * L.NC * L.n_win_b + 1;
        const int64_t n_win = p->B * L.n_win_b;
        // (The key-major kernels take G = 8..64; with the lists in place the tile lists are built only for the
        // tile forward, so a problem outside that range must not get them.)
        L.km = L.G >= 8 && L.G <= 64 && L.NC <= kKmMaxChunks && p->B * L.n_blk_b * L.NC <= kKmMaskWords && L.cap_entries < INT32_MAX &&
               L.cap_items * p->Hkv < INT32_MAX && n_win <= kKmMaxWindows &&
               n_win * (L.max_groups + 1) <= kKmQueueBins && p->B * L.NC < INT32_MAX && rows * p->Hq < INT32_MAX;
    }
    if (L.km) {
        const int64_t n_lists = p->B * L.NC;
        const size_t words = (size_t)(p->B * L.n_blk_b * L.NC);
        L.off_rmask = off;
        off = align256(off + words * sizeof(uint64_t));
        L.off_hoff = off;
        off = align256(off + words * sizeof(int32_t));
        L.off_list_start = off;
        off = align256(off + (size_t)(n_lists + 1) * sizeof(int32_t));
        L.off_eq = off;
        off = align256(off + (size_t)L.cap_entries * sizeof(int32_t));
        L.off_emask = off;
        off = align256(off + (size_t)L.cap_entries * sizeof(uint64_t));
        L.off_part_start = off;
        off = align256(off + (size_t)(n_lists + 1) * sizeof(int32_t));
        L.off_items = off;
        off = align256(off + (size_t)L.cap_items * 4 * sizeof(int32_t));
        L.off_sorted = off;
        off = align256(off + (size_t)L.cap_items * sizeof(int32_t));
        L.off_queue = off;
        off = align256(off + (size_t)(L.cap_items * p->Hkv) * sizeof(int32_t));
        L.off_kmeta = off;  // {entries, items, queue length, overflow, forward path choice, -, tile chunks, groups}
        off = align256(off + 8 * sizeof(int32_t));
        L.off_tkeys = off;  // distinct routed keys per query tile (the tile forward's cost, for the path choice)
        off = align256(off + (size_t)(p->B * L.n_tiles) * sizeof(int32_t));
        // Key-major forward: row maxima, exponent references and sums, the key norm bound, and the fp32
        // accumulator it shares with the backward's dQ (8 bytes per element for the deterministic
        // backward's exact sums).
        L.off_mrow = off;
        off = align256(off + (size_t)(p->B * p->Hq * p->S_q) * sizeof(int32_t));
        L.off_mref = off;
        off = align256(off + (size_t)(p->B * p->Hq * p->S_q) * sizeof(float));
        L.off_lrow = off;
        off = align256(off + (size_t)(p->B * p->Hq * p->S_q) * 2 * sizeof(float));
        L.off_kbound = off;
        off = align256(off + (size_t)(kKeyNormWord + p->B * p->Hkv) * sizeof(int32_t));
        L.off_dq = off;
        off = align256(off + (size_t)rows * p->Hq * p->D * 8);
    }
    L.fwd_total = off;
    L.off_delta = off;
    off = align256(off + p->B * p->Hq * p->S_q * sizeof(float));
    // dK/dV accumulators: fp32, or (deterministic backward) an fp32 and a 32-bit integer word per element.
    const size_t kv_acc = (size_t)p->B * p->S_kv * p->Hkv * p->D * 8;
    L.off_dk = off;
    off = align256(off + kv_acc);
    L.off_dv = off;
    off = align256(off + kv_acc);
    L.total = off;
    return L;
}

template <typename T>
T *at(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}
template <typename T>
const T *at(const void *ws, size_t off) {
    return reinterpret_cast<const T *>(static_cast<const char *>(ws) + off);
}

// full = true for the backward (every region), false for the preprocessing and the forward (the
// prefix they use).
qsa_status check_ws(const qsa_problem *p, const void *ws, size_t ws_bytes, Layout &L, bool full) {
    qsa_status st = validate(p);
    if (st != QSA_OK) return st;
    if (!ws) return fail(QSA_ERR_INVALID_ARGUMENT, "workspace is null");
    if (reinterpret_cast<uintptr_t>(ws) % 256 != 0)
        return fail(QSA_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
    L = make_layout(p);
    const size_t need = full ? L.total : L.fwd_total;
    if (ws_bytes < need)
        return fail(QSA_ERR_WORKSPACE_TOO_SMALL, "workspace has %zu bytes, %s needs %zu", ws_bytes,
                    full ? "the backward" : "the forward", need);
    return QSA_OK;
}

bool aligned16(const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

// [lo, hi) byte range of a strided [B, S, H, D] bf16 tensor.
void span_of(const void *base, const int64_t *stride, int64_t B, int64_t S, int64_t H, int64_t D, uintptr_t &lo,
             uintptr_t &hi) {
    lo = reinterpret_cast<uintptr_t>(base);
    hi = lo + 2 * (size_t)((B - 1) * stride[0] + (S - 1) * stride[1] + (H - 1) * stride[2] + D);
}

bool overlaps(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

AttnArgs attn_args(const qsa_problem *p, const Layout &L, const void *ws, const void *q, const void *k,
                   const void *v) {
    AttnArgs a{};
    a.B = p->B;
    a.S_q = p->S_q;
    a.S_kv = p->S_kv;
    a.Hq = p->Hq;
    a.Hkv = p->Hkv;
    a.K = p->K;
    a.G = L.G;
    a.D = p->D;
    a.scale = p->softmax_scale;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.k = static_cast<const __nv_bfloat16 *>(k);
    a.v = static_cast<const __nv_bfloat16 *>(v);
    a.qs0 = p->q_stride[0];
    a.qs1 = p->q_stride[1];
    a.qs2 = p->q_stride[2];
    a.ks0 = p->k_stride[0];
    a.ks1 = p->k_stride[1];
    a.ks2 = p->k_stride[2];
    a.vs0 = p->v_stride[0];
    a.vs1 = p->v_stride[1];
    a.vs2 = p->v_stride[2];
    a.ids = at<int32_t>(ws, L.off_ids);
    a.counts = at<int32_t>(ws, L.off_counts);
    a.status = const_cast<DeviceStatus *>(at<DeviceStatus>(ws, L.off_status));
    return a;
}

TileArgs tile_args(const qsa_problem *p, const Layout &L, void *ws) {
    TileArgs t{};
    t.sched = at<int32_t>(ws, L.off_sched);
    t.T = L.T;
    t.n_tiles = L.n_tiles;
    t.max_chunks = L.max_chunks;
    t.tile_nchunks = at<int32_t>(ws, L.off_tile_nchunks);
    t.tile_keys = at<int32_t>(ws, L.off_tile_keys);
    t.tile_masks = at<uint64_t>(ws, L.off_tile_masks);
    t.order = at<int32_t>(ws, L.off_order);
    return t;
}

// The reverse lists' arguments (qsa_chunks.cu) for this problem's workspace.
ChunkArgs chunk_args(const qsa_problem *p, const Layout &L, void *ws) {
    ChunkArgs c{};
    c.B = p->B;
    c.S_q = p->S_q;
    c.S_kv = p->S_kv;
    c.K = p->K;
    c.NC = L.NC;
    c.Hkv = p->Hkv;
    c.n_blk_b = L.n_blk_b;
    c.win_blocks = L.win_blocks;
    c.n_win_b = L.n_win_b;
    c.slots = L.T;
    c.max_groups = L.max_groups;
    c.cap_entries = L.cap_entries;
    c.cap_items = L.cap_items;
    c.ids = at<int32_t>(ws, L.off_ids);
    c.counts = at<int32_t>(ws, L.off_counts);
    c.rmask = at<uint64_t>(ws, L.off_rmask);
    c.hoff = at<int32_t>(ws, L.off_hoff);
    c.list_start = at<int32_t>(ws, L.off_list_start);
    c.e_q = at<int32_t>(ws, L.off_eq);
    c.e_mask = at<uint64_t>(ws, L.off_emask);
    c.part_start = at<int32_t>(ws, L.off_part_start);
    c.items = at<int4>(ws, L.off_items);
    c.sorted = at<int32_t>(ws, L.off_sorted);
    c.queue = at<int32_t>(ws, L.off_queue);
    c.meta = at<int32_t>(ws, L.off_kmeta);
    c.tile_keys = at<int32_t>(ws, L.off_tkeys);
    c.status = at<DeviceStatus>(ws, L.off_status);
    return c;
}

}  // namespace

qsa_status report_error(qsa_status st, const char *msg) { return fail(st, "%s", msg); }

size_t forward_workspace_bytes(const qsa_problem *p) {
    if (validate(p) != QSA_OK) return 0;
    return make_layout(p).fwd_total;
}

}  // namespace qsa

namespace qsa {
namespace {
qsa_status backward_impl(const qsa_problem *p, void *ws, size_t ws_bytes, const void *q, const void *k, const void *v,
                         const void *o, const float *lse, const void *dout, void *dq, void *dk, void *dv,
                         float *dk_f32, float *dv_f32, bool deterministic, cudaStream_t stream) {
    Layout L;
    qsa_status st = check_ws(p, ws, ws_bytes, L, true);
    if (st != QSA_OK) return st;
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv)
        return fail(QSA_ERR_INVALID_ARGUMENT, "null tensor pointer");
    if ((dk_f32 == nullptr) != (dv_f32 == nullptr))
        return fail(QSA_ERR_INVALID_ARGUMENT, "dk_f32 and dv_f32 must both be given or both be null");
    const void *al[] = {q, k, v, o, dout, dq, dk, dv};
    for (const void *x : al)
        if (!aligned16(x)) return fail(QSA_ERR_UNSUPPORTED, "bf16 tensors must be 16-byte aligned");
    if ((dk_f32 && !aligned16(dk_f32)) || (dv_f32 && !aligned16(dv_f32)))
        return fail(QSA_ERR_UNSUPPORTED, "fp32 accumulators must be 16-byte aligned");
    uintptr_t q0, q1, k0, k1, v0, v1;
    span_of(q, p->q_stride, p->B, p->S_q, p->Hq, p->D, q0, q1);
    span_of(k, p->k_stride, p->B, p->S_kv, p->Hkv, p->D, k0, k1);
    span_of(v, p->v_stride, p->B, p->S_kv, p->Hkv, p->D, v0, v1);
    const size_t nq = 2 * (size_t)(p->B * p->S_q * p->Hq * p->D);
    const size_t nkv = 2 * (size_t)(p->B * p->S_kv * p->Hkv * p->D);
    auto u = [](const void *x) { return reinterpret_cast<uintptr_t>(x); };
    const uintptr_t ins[6][2] = {{q0, q1}, {k0, k1}, {v0, v1}, {u(o), u(o) + nq}, {u(dout), u(dout) + nq},
                                 {u(lse), u(lse) + 4 * (size_t)(p->B * p->Hq * p->S_q)}};
    uintptr_t outs[5][2] = {{u(dq), u(dq) + nq}, {u(dk), u(dk) + nkv}, {u(dv), u(dv) + nkv}, {0, 0}, {0, 0}};
    int nout = 3;
    if (dk_f32) {
        outs[3][0] = u(dk_f32);
        outs[3][1] = u(dk_f32) + 2 * nkv;
        outs[4][0] = u(dv_f32);
        outs[4][1] = u(dv_f32) + 2 * nkv;
        nout = 5;
    }
    const uintptr_t w0 = u(ws), w1 = w0 + L.total;
    for (int i = 0; i < nout; ++i) {
        for (auto &r : ins)
            if (overlaps(outs[i][0], outs[i][1], r[0], r[1]))
                return fail(QSA_ERR_INVALID_ARGUMENT, "a gradient output overlaps an input");
        if (overlaps(outs[i][0], outs[i][1], w0, w1))
            return fail(QSA_ERR_INVALID_ARGUMENT, "a gradient output overlaps the workspace");
        for (int j = 0; j < i; ++j)
            if (overlaps(outs[i][0], outs[i][1], outs[j][0], outs[j][1]))
                return fail(QSA_ERR_INVALID_ARGUMENT, "gradient outputs overlap each other");
    }
    BwdArgs b{};
    b.f = attn_args(p, L, ws, q, k, v);
    b.o = static_cast<const __nv_bfloat16 *>(o);
    b.dout = static_cast<const __nv_bfloat16 *>(dout);
    b.lse = lse;
    b.delta = at<float>(ws, L.off_delta);
    b.dq = static_cast<__nv_bfloat16 *>(dq);
    b.dk = static_cast<__nv_bfloat16 *>(dk);
    b.dv = static_cast<__nv_bfloat16 *>(dv);
    const size_t n_kv = (size_t)p->B * p->S_kv * p->Hkv * p->D;
    const size_t n_q = (size_t)p->B * p->S_q * p->Hq * p->D;
    // With reverse lists both backward kernels are launched (when the tile one accepts the problem) and the
    // device-side choice made at preprocessing (choice[1], test hooks included) lets one of them run.
    const bool key_major = L.km && tc_backward_supported() && km_backward_shape_ok(b.f);
    const TileArgs ta = tile_args(p, L, ws);
    const bool tile_ok = L.T && tc_backward_supported() && tc_backward_shape_ok(b.f, ta);
    const int32_t *bwd_choice = at<int32_t>(ws, L.off_kmeta) + 5;
    cudaError_t e;
    if (deterministic) {
        // Fixed-point accumulators in the workspace; the caller's fp32 buffers (if any) receive the sums.
        b.dk_fx.est = at<float>(ws, L.off_dk);
        b.dk_fx.lo = at<uint32_t>(ws, L.off_dk + n_kv * sizeof(float));
        b.dv_fx.est = at<float>(ws, L.off_dv);
        b.dv_fx.lo = at<uint32_t>(ws, L.off_dv + n_kv * sizeof(float));
        b.dk_acc = dk_f32;
        b.dv_acc = dv_f32;
        e = cudaMemsetAsync(at<char>(ws, L.off_dk), 0, n_kv * 8, stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(at<char>(ws, L.off_dv), 0, n_kv * 8, stream);
    } else {
        b.dk_acc = dk_f32 ? dk_f32 : at<float>(ws, L.off_dk);
        b.dv_acc = dv_f32 ? dv_f32 : at<float>(ws, L.off_dv);
        e = cudaMemsetAsync(b.dk_acc, 0, n_kv * sizeof(float), stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(b.dv_acc, 0, n_kv * sizeof(float), stream);
    }
    if (e == cudaSuccess && key_major)
        e = cudaMemsetAsync(at<char>(ws, L.off_dq), 0, n_q * (deterministic ? 8 : 4), stream);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the gradient accumulators");
    e = launch_delta(b, stream);
    if (e != cudaSuccess) return cuda_fail(e, "delta launch");
    if (key_major) {
        const ChunkArgs c = chunk_args(p, L, ws);
        KmArgs k{};
        k.NC = L.NC;
        k.items = c.items;
        k.queue = c.queue;
        k.meta = c.meta;
        k.e_q = c.e_q;
        k.e_mask = c.e_mask;
        k.sched = at<int32_t>(ws, L.off_sched) + 4;
        if (deterministic) {
            k.dq_fx.est = at<float>(ws, L.off_dq);
            k.dq_fx.lo = at<uint32_t>(ws, L.off_dq + n_q * sizeof(float));
        } else {
            k.dq_acc = at<float>(ws, L.off_dq);
        }
        k.gate = tile_ok ? bwd_choice : nullptr;
        if (tile_ok) {
            e = launch_tc_backward(b, ta, bwd_choice, stream);
            if (e != cudaSuccess) return cuda_fail(e, "tile backward launch");
        }
        e = launch_km_backward(b, k, stream);
        if (e != cudaSuccess) return cuda_fail(e, "key-major backward launch");
    } else {
        if (tile_ok) {
            e = launch_tc_backward(b, ta, nullptr, stream);
            if (e != cudaSuccess) return cuda_fail(e, "tile backward launch");
        } else {
            e = launch_rowwise_backward(b, stream);
            if (e != cudaSuccess) return cuda_fail(e, "rowwise backward launch");
        }
    }
    e = launch_convert_dkdv(b, stream);
    if (e != cudaSuccess) return cuda_fail(e, "dK/dV conversion launch");
    return QSA_OK;
}
}  // namespace
}  // namespace qsa

using namespace qsa;

extern "C" {

qsa_status qsa_check_problem(const qsa_problem *problem) { return validate(problem); }

size_t qsa_workspace_bytes(const qsa_problem *problem) {
    if (validate(problem) != QSA_OK) return 0;
    return make_layout(problem).total;
}

qsa_status qsa_preprocess(const qsa_problem *p, const void *routes, void *ws, size_t ws_bytes, cudaStream_t stream) {
    Layout L;
    qsa_status st = check_ws(p, ws, ws_bytes, L, false);
    if (st != QSA_OK) return st;
    if (!routes) return fail(QSA_ERR_INVALID_ARGUMENT, "routes is null");
    if (reinterpret_cast<uintptr_t>(routes) % (p->route_bits / 8) != 0)
        return fail(QSA_ERR_INVALID_ARGUMENT, "routes pointer is not aligned to its element size");
    // Status word and work queue counters (the tile kernels leave the counters reset when they end).
    cudaError_t e = cudaMemsetAsync(at<DeviceStatus>(ws, L.off_status), 0, L.off_counts - L.off_status, stream);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
    RowsArgs r{};
    r.routes = routes;
    r.route_bits = p->route_bits;
    r.B = p->B;
    r.S_q = p->S_q;
    r.S_kv = p->S_kv;
    r.K = p->K;
    r.rs0 = p->r_stride[0];
    r.rs1 = p->r_stride[1];
    r.rs2 = p->r_stride[2];
    r.ids = at<int32_t>(ws, L.off_ids);
    r.counts = at<int32_t>(ws, L.off_counts);
    r.try_sorted = (p->flags & QSA_ROUTES_SORTED) != 0;
    e = launch_route_rows(r, stream);
    if (e != cudaSuccess) return cuda_fail(e, "route_rows launch");
    const int32_t *choice = nullptr;
    if (L.km) {
        // Reverse lists for the key-major kernels, and the forward path choice.
        const ChunkArgs c = chunk_args(p, L, ws);
        e = launch_chunk_lists(c, stream);
        if (e != cudaSuccess) return cuda_fail(e, "reverse route list launch");
        const AttnArgs a = attn_args(p, L, ws, nullptr, nullptr, nullptr);
        const bool tile_bwd_ok = tc_backward_supported() && tc_backward_shape_ok(a, tile_args(p, L, ws));
        e = launch_km_choose(c.tile_keys, p->B * L.n_tiles, c.list_start, p->B * L.NC, L.T, p->D, tile_bwd_ok,
                             (p->flags & QSA_DETERMINISTIC_FORWARD) != 0, c.meta + 4, stream);
        if (e != cudaSuccess) return cuda_fail(e, "path choice launch");
        choice = c.meta + 4;
    }
    if (L.T) {
        TilesArgs t{};
        t.B = p->B;
        t.S_q = p->S_q;
        t.S_kv = p->S_kv;
        t.K = p->K;
        t.T = L.T;
        t.n_tiles = L.n_tiles;
        t.max_chunks = L.max_chunks;
        t.Hkv = p->Hkv;
        t.ids = r.ids;
        t.counts = r.counts;
        t.tile_nchunks = at<int32_t>(ws, L.off_tile_nchunks);
        t.tile_keys = at<int32_t>(ws, L.off_tile_keys);
        t.tile_masks = at<uint64_t>(ws, L.off_tile_masks);
        t.order = at<int32_t>(ws, L.off_order);
        // With reverse lists the tile lists are built only if the device chose a tile kernel in either direction.
        t.skip = choice;
        e = launch_route_tiles(t, stream);
        if (e != cudaSuccess) return cuda_fail(e, "route_tiles launch");
    }
    return QSA_OK;
}

qsa_status qsa_forward(const qsa_problem *p, void *ws, size_t ws_bytes, const void *q, const void *k,
                       const void *v, void *o, float *lse, cudaStream_t stream) {
    Layout L;
    qsa_status st = check_ws(p, ws, ws_bytes, L, false);
    if (st != QSA_OK) return st;
    if (!q || !k || !v || !o || !lse) return fail(QSA_ERR_INVALID_ARGUMENT, "null tensor pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return fail(QSA_ERR_UNSUPPORTED, "q, k, v and o must be 16-byte aligned");
    uintptr_t q0, q1, k0, k1, v0, v1;
    span_of(q, p->q_stride, p->B, p->S_q, p->Hq, p->D, q0, q1);
    span_of(k, p->k_stride, p->B, p->S_kv, p->Hkv, p->D, k0, k1);
    span_of(v, p->v_stride, p->B, p->S_kv, p->Hkv, p->D, v0, v1);
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(o), o1 = o0 + 2 * (size_t)(p->B * p->S_q * p->Hq * p->D);
    const uintptr_t l0 = reinterpret_cast<uintptr_t>(lse), l1 = l0 + 4 * (size_t)(p->B * p->Hq * p->S_q);
    const uintptr_t w0 = reinterpret_cast<uintptr_t>(ws), w1 = w0 + L.fwd_total;
    const uintptr_t in[4][2] = {{q0, q1}, {k0, k1}, {v0, v1}, {w0, w1}};
    for (auto &r : in)
        if (overlaps(o0, o1, r[0], r[1]) || overlaps(l0, l1, r[0], r[1]))
            return fail(QSA_ERR_INVALID_ARGUMENT, "o/lse overlap an input or the workspace");
    if (overlaps(o0, o1, l0, l1)) return fail(QSA_ERR_INVALID_ARGUMENT, "o and lse overlap");
    AttnArgs a = attn_args(p, L, ws, q, k, v);
    cudaError_t e;
    const TileArgs ta = tile_args(p, L, ws);
    if (L.T && tc_forward_supported() && tc_forward_shape_ok(a, ta)) {
        // With reverse lists, the tile and key-major forwards are both launched; the device-side choice
        // made at preprocessing lets one of them run and the other return at once.
        const bool km = L.km && km_forward_shape_ok(a);
        const int32_t *choice = km ? at<int32_t>(ws, L.off_kmeta) + 4 : nullptr;
        e = launch_tc_forward(a, ta, static_cast<__nv_bfloat16 *>(o), lse, choice, stream);
        if (e != cudaSuccess) return cuda_fail(e, "tile forward launch");
        if (km) {
            KfArgs k{};
            k.NC = L.NC;
            k.items = at<int4>(ws, L.off_items);
            k.queue = at<int32_t>(ws, L.off_queue);
            k.meta = at<int32_t>(ws, L.off_kmeta);
            k.e_q = at<int32_t>(ws, L.off_eq);
            k.e_mask = at<uint64_t>(ws, L.off_emask);
            k.sched = at<int32_t>(ws, L.off_sched) + 6;
            k.mrow = at<int32_t>(ws, L.off_mrow);
            k.mref = at<float>(ws, L.off_mref);
            k.lrow = at<float>(ws, L.off_lrow);
            k.kbound = at<int32_t>(ws, L.off_kbound);
            k.o_acc = at<float>(ws, L.off_dq);
            k.choice = choice;
            e = launch_km_forward(a, k, static_cast<__nv_bfloat16 *>(o), lse, stream);
            if (e != cudaSuccess) return cuda_fail(e, "key-major forward launch");
        }
    } else {
        e = launch_rowwise_forward(a, static_cast<__nv_bfloat16 *>(o), lse, stream);
        if (e != cudaSuccess) return cuda_fail(e, "rowwise forward launch");
    }
    return QSA_OK;
}

qsa_status qsa_backward(const qsa_problem *p, void *ws, size_t ws_bytes, const void *q, const void *k, const void *v,
                        const void *o, const float *lse, const void *dout, void *dq, void *dk, void *dv,
                        float *dk_f32, float *dv_f32, cudaStream_t stream) {
    return backward_impl(p, ws, ws_bytes, q, k, v, o, lse, dout, dq, dk, dv, dk_f32, dv_f32, false, stream);
}

qsa_status qsa_backward_deterministic(const qsa_problem *p, void *ws, size_t ws_bytes, const void *q, const void *k,
                                      const void *v, const void *o, const float *lse, const void *dout, void *dq,
                                      void *dk, void *dv, float *dk_f32, float *dv_f32, cudaStream_t stream) {
    return backward_impl(p, ws, ws_bytes, q, k, v, o, lse, dout, dq, dk, dv, dk_f32, dv_f32, true, stream);
}

qsa_status qsa_copy_route_sets(const qsa_problem *p, const void *ws, size_t ws_bytes, int32_t *ids, int32_t *counts,
                               cudaStream_t stream) {
    Layout L;
    qsa_status st = check_ws(p, ws, ws_bytes, L, false);
    if (st != QSA_OK) return st;
    const size_t rows = (size_t)(p->B * p->S_q);
    cudaError_t e = cudaSuccess;
    if (ids)
        e = cudaMemcpyAsync(ids, at<int32_t>(ws, L.off_ids), rows * p->K * sizeof(int32_t), cudaMemcpyDeviceToDevice,
                            stream);
    if (e == cudaSuccess && counts)
        e = cudaMemcpyAsync(counts, at<int32_t>(ws, L.off_counts), rows * sizeof(int32_t), cudaMemcpyDeviceToDevice,
                            stream);
    if (e != cudaSuccess) return cuda_fail(e, "copying route sets");
    return QSA_OK;
}

qsa_status qsa_read_device_status(const void *ws, cudaStream_t stream) {
    if (!ws) return fail(QSA_ERR_INVALID_ARGUMENT, "workspace is null");
    DeviceStatus h{};
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess) e = cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemsetAsync(const_cast<void *>(ws), 0, sizeof(h), stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
    if (h.code == 0) return QSA_OK;
    return fail((qsa_status)h.code, "device reported %s at site %u (info %u, %u)",
                qsa_status_string((qsa_status)h.code), h.where, h.info0, h.info1);
}

const char *qsa_status_string(qsa_status s) {
    switch (s) {
        case QSA_OK: return "QSA_OK";
        case QSA_ERR_INVALID_ARGUMENT: return "QSA_ERR_INVALID_ARGUMENT";
        case QSA_ERR_UNSUPPORTED: return "QSA_ERR_UNSUPPORTED";
        case QSA_ERR_WORKSPACE_TOO_SMALL: return "QSA_ERR_WORKSPACE_TOO_SMALL";
        case QSA_ERR_CUDA: return "QSA_ERR_CUDA";
        case QSA_ERR_TIMEOUT: return "QSA_ERR_TIMEOUT";
        case QSA_ERR_DEVICE_CHECK: return "QSA_ERR_DEVICE_CHECK";
    }
    return "QSA_ERR_UNKNOWN";
}

const char *qsa_last_error(void) { return g_last_error; }

}  // extern "C"

// qsa_rowwise.cu -- warp-level route-set attention: one warp per (query row, head).
//
// This is the general path: any group size G = Hq/Hkv, any route pattern.  A
// CTA owns one (b, q, KV head g); its warps take the group's query heads, so the
// K/V rows they gather for the row's route set are shared through L1.  Each
// lane holds 8 consecutive head dimensions (D = 64, 128 or 256: the first D/8
// lanes hold data, the others zeros, so the warp sums are unchanged).  Scores are warp-reduced dot
// products, the softmax is online in fp32 (base-2 exponent with the scale
// folded in), and LSE is reported in natural-log units.
//
// Backward recomputes P from LSE (P_j = exp(s_j - LSE)), forms dP_j = <dO, V_j>,
// dS_j = P_j (dP_j - Delta) with Delta = <dO, O> per (row, head), writes dQ per
// row and scatter-adds dK/dV in fp32 with vector reductions (red.global.add.v4).
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kUnroll = 4;

__device__ __forceinline__ uint4 ldg16(const __nv_bfloat16 *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }

__device__ __forceinline__ void red_add_v4(float *addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

__global__ void __launch_bounds__(kThreads) rowwise_fwd_kernel(AttnArgs a, __nv_bfloat16 *o, float *lse) {
    const int64_t row = blockIdx.x, g = blockIdx.y;
    const int64_t b = row / a.S_q, qpos = row % a.S_q;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = a.counts[row];
    const int32_t *R = a.ids + row * a.K;
    const float sl2 = a.scale * kLog2e;
    const bool dl = lane * 8 < a.D;  // this lane holds head dimensions
    const __nv_bfloat16 *kbase = a.k + b * a.ks0 + g * a.ks2 + lane * 8;
    const __nv_bfloat16 *vbase = a.v + b * a.vs0 + g * a.vs2 + lane * 8;
    for (int64_t hl = warp; hl < a.G; hl += kWarps) {
        const int64_t h = g * a.G + hl;
        float qf[8], acc[8];
        bf16x8_to_f32(dl ? ldg16(a.q + b * a.qs0 + qpos * a.qs1 + h * a.qs2 + lane * 8) : make_uint4(0, 0, 0, 0), qf);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        float m = -INFINITY, l = 0.f;
        for (int t = 0; t < n; t += kUnroll) {
            int64_t j[kUnroll];
            float s[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                j[u] = t + u < n ? (int64_t)R[t + u] : -1;
                if (t + u < n && (j[u] < 0 || j[u] >= a.S_kv)) {
                    if (lane == 0) raise_status(a.status, QSA_ERR_DEVICE_CHECK, kSiteRowwiseFwdId, (unsigned)row);
                    j[u] = -1;
                }
                float part = 0.f;
                if (j[u] >= 0 && dl) {
                    float kf[8];
                    bf16x8_to_f32(ldg16(kbase + j[u] * a.ks1), kf);
#pragma unroll
                    for (int i = 0; i < 8; ++i) part = fmaf(qf[i], kf[i], part);
                }
                s[u] = part;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) s[u] += __shfl_xor_sync(0xffffffffu, s[u], off);
            }
            float mx = m;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                s[u] = j[u] >= 0 ? s[u] * sl2 : -INFINITY;
                mx = fmaxf(mx, s[u]);
            }
            if (mx == -INFINITY) continue;  // nothing valid in this group of keys yet
            const float alpha = exp2f(m - mx);
            l *= alpha;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] *= alpha;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                if (j[u] < 0) continue;
                const float p = exp2f(s[u] - mx);
                l += p;
                float vf[8];
                bf16x8_to_f32(dl ? ldg16(vbase + j[u] * a.vs1) : make_uint4(0, 0, 0, 0), vf);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmaf(p, vf[i], acc[i]);
            }
            m = mx;
        }
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] *= inv;
        if (dl) *reinterpret_cast<uint4 *>(o + ((row * a.Hq + h) * a.D + lane * 8)) = f32x8_to_bf16(acc);
        if (lane == 0) lse[(b * a.Hq + h) * a.S_q + qpos] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
}

// Delta[b,h,q] = <dO, O> over D, in fp32 from the BF16 forward output.
__global__ void __launch_bounds__(kThreads) delta_kernel(BwdArgs a) {
    const int64_t row = blockIdx.x;
    const int64_t b = row / a.f.S_q, qpos = row % a.f.S_q;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t h = warp; h < a.f.Hq; h += kWarps) {
        float of[8], df[8];
        const bool dl = lane * 8 < a.f.D;
        const int64_t off = (row * a.f.Hq + h) * a.f.D + lane * 8;
        bf16x8_to_f32(dl ? ldg16(a.o + off) : make_uint4(0, 0, 0, 0), of);
        bf16x8_to_f32(dl ? ldg16(a.dout + off) : make_uint4(0, 0, 0, 0), df);
        float part = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) part = fmaf(of[i], df[i], part);
        part = warp_sum(part);
        if (lane == 0) a.delta[(b * a.f.Hq + h) * a.f.S_q + qpos] = part;
    }
}

// kDet: dK/dV contributions go to the exact accumulators (FxAcc: order-independent sums).
template <bool kDet>
__global__ void __launch_bounds__(kThreads) rowwise_bwd_kernel(BwdArgs a) {
    const AttnArgs &f = a.f;
    const int64_t row = blockIdx.x, g = blockIdx.y;
    const int64_t b = row / f.S_q, qpos = row % f.S_q;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = f.counts[row];
    const int32_t *R = f.ids + row * f.K;
    const float sl2 = f.scale * kLog2e;
    const __nv_bfloat16 *kbase = f.k + b * f.ks0 + g * f.ks2 + lane * 8;
    const __nv_bfloat16 *vbase = f.v + b * f.vs0 + g * f.vs2 + lane * 8;
    const bool dl = lane * 8 < f.D;
    float *dkbase = kDet ? nullptr : a.dk_acc + (b * f.S_kv * f.Hkv + g) * f.D + lane * 8;
    float *dvbase = kDet ? nullptr : a.dv_acc + (b * f.S_kv * f.Hkv + g) * f.D + lane * 8;
    for (int64_t hl = warp; hl < f.G; hl += kWarps) {
        const int64_t h = g * f.G + hl;
        float qf[8], df[8], dq[8];
        bf16x8_to_f32(dl ? ldg16(f.q + b * f.qs0 + qpos * f.qs1 + h * f.qs2 + lane * 8) : make_uint4(0, 0, 0, 0), qf);
        bf16x8_to_f32(dl ? ldg16(a.dout + (row * f.Hq + h) * f.D + lane * 8) : make_uint4(0, 0, 0, 0), df);
#pragma unroll
        for (int i = 0; i < 8; ++i) dq[i] = 0.f;
        const float lse2 = n > 0 ? a.lse[(b * f.Hq + h) * f.S_q + qpos] * kLog2e : 0.f;
        const float delta = n > 0 ? a.delta[(b * f.Hq + h) * f.S_q + qpos] : 0.f;
        for (int t = 0; t < n; t += kUnroll) {
            int64_t j[kUnroll];
            float s[kUnroll], dp[kUnroll], kf[kUnroll][8];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                j[u] = t + u < n ? (int64_t)R[t + u] : -1;
                if (t + u < n && (j[u] < 0 || j[u] >= f.S_kv)) {
                    if (lane == 0) raise_status(f.status, QSA_ERR_DEVICE_CHECK, kSiteRowwiseBwdId, (unsigned)row);
                    j[u] = -1;
                }
                float ps = 0.f, pd = 0.f;
                if (j[u] >= 0 && dl) {
                    float vf[8];
                    bf16x8_to_f32(ldg16(kbase + j[u] * f.ks1), kf[u]);
                    bf16x8_to_f32(ldg16(vbase + j[u] * f.vs1), vf);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        ps = fmaf(qf[i], kf[u][i], ps);
                        pd = fmaf(df[i], vf[i], pd);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) kf[u][i] = 0.f;
                }
                s[u] = ps;
                dp[u] = pd;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    s[u] += __shfl_xor_sync(0xffffffffu, s[u], off);
                    dp[u] += __shfl_xor_sync(0xffffffffu, dp[u], off);
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                if (j[u] < 0) continue;
                const float p = exp2f(s[u] * sl2 - lse2);
                const float ds = p * (dp[u] - delta);
#pragma unroll
                for (int i = 0; i < 8; ++i) dq[i] = fmaf(ds, kf[u][i], dq[i]);
                const float c = f.scale * ds;
                if (!dl) continue;
                if (kDet) {
                    const int64_t e0 = ((b * f.S_kv + j[u]) * f.Hkv + g) * f.D + lane * 8;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        red_add_fx(a.dk_fx, e0 + i, c * qf[i]);
                        red_add_fx(a.dv_fx, e0 + i, p * df[i]);
                    }
                } else {
                    float *dkj = dkbase + j[u] * f.Hkv * f.D;
                    float *dvj = dvbase + j[u] * f.Hkv * f.D;
                    red_add_v4(dkj, c * qf[0], c * qf[1], c * qf[2], c * qf[3]);
                    red_add_v4(dkj + 4, c * qf[4], c * qf[5], c * qf[6], c * qf[7]);
                    red_add_v4(dvj, p * df[0], p * df[1], p * df[2], p * df[3]);
                    red_add_v4(dvj + 4, p * df[4], p * df[5], p * df[6], p * df[7]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) dq[i] *= f.scale;
        if (dl) *reinterpret_cast<uint4 *>(a.dq + (row * f.Hq + h) * f.D + lane * 8) = f32x8_to_bf16(dq);
    }
}

__global__ void convert_kernel(const float *dk, const float *dv, __nv_bfloat16 *dkb, __nv_bfloat16 *dvb, int64_t n8) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const float4 *k4 = reinterpret_cast<const float4 *>(dk) + 2 * i;
        const float4 *v4 = reinterpret_cast<const float4 *>(dv) + 2 * i;
        float4 a = k4[0], b = k4[1], c = v4[0], d = v4[1];
        float kf[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        float vf[8] = {c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
        reinterpret_cast<uint4 *>(dkb)[i] = f32x8_to_bf16(kf);
        reinterpret_cast<uint4 *>(dvb)[i] = f32x8_to_bf16(vf);
    }
}

// Exact sums -> bf16 gradients, and fp32 copies when dk32/dv32 are given.
__global__ void convert_fx_kernel(FxAcc dk, FxAcc dv, __nv_bfloat16 *dkb, __nv_bfloat16 *dvb, float *dk32, float *dv32,
                                  int64_t n8) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        float kf[8], vf[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            kf[e] = fx_to_f32(dk.est[8 * i + e], dk.lo[8 * i + e]);
            vf[e] = fx_to_f32(dv.est[8 * i + e], dv.lo[8 * i + e]);
        }
        reinterpret_cast<uint4 *>(dkb)[i] = f32x8_to_bf16(kf);
        reinterpret_cast<uint4 *>(dvb)[i] = f32x8_to_bf16(vf);
        if (dk32) {
            float4 *k4 = reinterpret_cast<float4 *>(dk32) + 2 * i;
            float4 *v4 = reinterpret_cast<float4 *>(dv32) + 2 * i;
            k4[0] = make_float4(kf[0], kf[1], kf[2], kf[3]);
            k4[1] = make_float4(kf[4], kf[5], kf[6], kf[7]);
            v4[0] = make_float4(vf[0], vf[1], vf[2], vf[3]);
            v4[1] = make_float4(vf[4], vf[5], vf[6], vf[7]);
        }
    }
}

}  // namespace

cudaError_t launch_rowwise_forward(const AttnArgs &a, __nv_bfloat16 *o, float *lse, cudaStream_t s) {
    dim3 grid((unsigned)(a.B * a.S_q), (unsigned)a.Hkv);
    rowwise_fwd_kernel<<<grid, kThreads, 0, s>>>(a, o, lse);
    return cudaGetLastError();
}

cudaError_t launch_delta(const BwdArgs &a, cudaStream_t s) {
    delta_kernel<<<(unsigned)(a.f.B * a.f.S_q), kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_rowwise_backward(const BwdArgs &a, cudaStream_t s) {
    dim3 grid((unsigned)(a.f.B * a.f.S_q), (unsigned)a.f.Hkv);
    if (a.dk_fx.est)
        rowwise_bwd_kernel<true><<<grid, kThreads, 0, s>>>(a);
    else
        rowwise_bwd_kernel<false><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_convert_dkdv(const BwdArgs &a, cudaStream_t s) {
    const int64_t n8 = a.f.B * a.f.S_kv * a.f.Hkv * a.f.D / 8;
    int64_t nb = (n8 + 255) / 256;
    int blocks = (int)(nb < 152 * 16 ? nb : 152 * 16);
    if (a.dk_fx.est)
        convert_fx_kernel<<<blocks, 256, 0, s>>>(a.dk_fx, a.dv_fx, a.dk, a.dv, a.dk_acc, a.dv_acc, n8);
    else
        convert_kernel<<<blocks, 256, 0, s>>>(a.dk_acc, a.dv_acc, a.dk, a.dv, n8);
    return cudaGetLastError();
}

}  // namespace qsa

// Attention over a general CSR relation: for every destination row i and head
// h, a softmax over the row's edges e = (j -> i) weighs the source rows v_j.
//
// TIGA-lang attention examples page: the varlen section writes the relation
// as an explicit CSR graph holding exactly the admitted edges, and the GAT
// section's display equation is this operation with a per-edge score
// (out_i = sum_e exp(s_e) / sum_e' exp(s_e') x_j).  The score of an edge is
// either a given field s[e, h] (segment softmax) or the dot-product score
// scale * <q_i, k_j>.  The scan over a row's edges is the online-softmax
// recurrence of the OCANNL "Module Ir.Online_softmax" page (fourth bullet)
// with blocks of 32 edges: per block the new max, the rescale factor, the
// exponentials, the rescaled sum and the value accumulation U += p v.
//
// Gather-bound (each edge reads a row of V, and of K for dot-product scores,
// wherever its source lies), so CUDA cores, not tensor cores.  Two kernels:
//  * row-centric (csr_rows_kernel), for tensors whose rows hold their heads
//    back to back: one warp per destination row gathers whole source rows
//    (all heads, 512 contiguous bytes at H = 4, D = 64 bf16) in 16-byte lane
//    chunks with several edges in flight -- the one the benchmarks run;
// Both take the rows in the caller's row order when one is given (the warps
// in flight at any moment hold consecutive entries of it, so an order that
// keeps rows with shared sources together lets the L2 serve their gathers).
//  * general (csr_fwd_kernel), any strides: one warp per (row, head).  Lane t
//    owns edge t of the current block of 32 (its column index and score) and
//    columns 4 t + 128 c of the D-wide rows (float4 chunks, c < 2, so
//    D <= 256).  Dot-product scores: every lane forms its columns' partial dot
//    with each of the 32 edges' K rows, then a transposing butterfly (31
//    shuffles) leaves lane t with edge t's full dot product.
//
// Malformed relations never cause an out-of-bounds access: a row whose
// offsets decrease or run past the edge count is treated as empty and an edge
// whose source index is out of range is skipped; both set the device status
// word to ATTN_EINVAL.
#include "../../include/attn.h"
#include "common.cuh"

namespace attn {

namespace {

constexpr int kWarps = 8;
constexpr int kChunks = 2;  // float4 column chunks per lane: D <= 256
// Row-centric kernel: edges a warp gathers per step (tunable at compile time).
#ifndef ATTN_CSR_INFLIGHT
#define ATTN_CSR_INFLIGHT 4
#endif

template <typename T>
__device__ __forceinline__ float4 ldg4(const T *p) {
    return load4(p);
}

// The destination row taken in position `r` of the processing order (the
// caller's row_order, else r itself); -1, with the status word set, for an
// entry outside [0, n_dst).  Every lane of a warp asks for the same r.
__device__ __forceinline__ int row_at(const CsrParams &p, int r) {
    if (!p.row_order) return r;
    const int i = __ldg(p.row_order + r);
    if (i < 0 || i >= p.n_dst) {
        if ((threadIdx.x & 31) == 0) report_status(p.status, ATTN_EINVAL);
        return -1;
    }
    return i;
}

template <typename T, typename Tout, bool kDot>
__global__ void __launch_bounds__(32 * kWarps) csr_fwd_kernel(const CsrParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t pairs = (int64_t)p.n_dst * p.H;
    const int64_t stride = (int64_t)gridDim.x * kWarps;
    const T *gv = static_cast<const T *>(p.v);
    const T *gq = static_cast<const T *>(p.q);
    const T *gk = static_cast<const T *>(p.k);
    Tout *go = static_cast<Tout *>(p.o);
    bool live[kChunks];
#pragma unroll
    for (int c = 0; c < kChunks; ++c) live[c] = 4 * (lane + 32 * c) < p.D;

    for (int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); r < pairs; r += stride) {
        const int ri = (int)(r / p.H), h = (int)(r - (int64_t)ri * p.H);
        const int i = row_at(p, ri);
        if (i < 0) continue;  // (warp-uniform) entry outside the rows, reported
        int64_t e0 = __ldg(p.row_ptr + i), e1 = __ldg(p.row_ptr + i + 1);
        if (e0 < 0 || e1 < e0 || e1 > p.n_edges) {
            if (lane == 0) report_status(p.status, ATTN_EINVAL);
            e0 = e1 = 0;  // treated as a row without edges
        }
        float4 qv[kChunks];
        if (kDot) {
#pragma unroll
            for (int c = 0; c < kChunks; ++c)
                qv[c] = live[c] ? ldg4(gq + (int64_t)i * p.q_st + (int64_t)h * p.q_sh + 4 * (lane + 32 * c))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float4 acc[kChunks];
#pragma unroll
        for (int c = 0; c < kChunks; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        float m = -INFINITY, l = 0.f;

        for (int64_t eb = e0; eb < e1; eb += 32) {
            const int cnt = e1 - eb < 32 ? (int)(e1 - eb) : 32;
            const int64_t e = eb + lane;
            int j = -1;
            if (lane < cnt) {
                j = __ldg(p.col + e);
                if (j < 0 || j >= p.n_src) {
                    report_status(p.status, ATTN_EINVAL);
                    j = -1;
                }
            }
            float s;  // this lane's edge score, log2 units (-inf: no edge)
            if (kDot) {
                // partial dots of my columns with the block's K rows, then a
                // transposing butterfly: afterwards d[0] of lane t = edge t's dot
                float d[32];
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const int jt = __shfl_sync(0xffffffffu, j, t);
                    float acc_d = 0.f;
                    if (jt >= 0) {
#pragma unroll
                        for (int c = 0; c < kChunks; ++c) {
                            if (!live[c]) continue;
                            const float4 kv = ldg4(gk + (int64_t)jt * p.k_st + (int64_t)h * p.k_sh + 4 * (lane + 32 * c));
                            acc_d = fmaf(qv[c].x, kv.x, acc_d);
                            acc_d = fmaf(qv[c].y, kv.y, acc_d);
                            acc_d = fmaf(qv[c].z, kv.z, acc_d);
                            acc_d = fmaf(qv[c].w, kv.w, acc_d);
                        }
                    }
                    d[t] = acc_d;
                }
#pragma unroll
                for (int w = 16; w >= 1; w >>= 1) {
                    const bool upper = (lane & w) != 0;
#pragma unroll
                    for (int t = 0; t < w; ++t) {
                        const float send = upper ? d[t] : d[t + w];
                        const float keep = upper ? d[t + w] : d[t];
                        d[t] = keep + __shfl_xor_sync(0xffffffffu, send, w);
                    }
                }
                s = j >= 0 ? d[0] * p.scale_log2 : -INFINITY;
            } else {
                s = j >= 0 ? __ldg(p.scores + e * p.H + h) * kLog2e : -INFINITY;
            }

            // online softmax update over this block of edges
            float bmax = s;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
            const float m_new = fmaxf(m, bmax);
            if (m_new == -INFINITY) continue;  // nothing admitted yet (uniform)
            const float alpha = exp2_approx(m - m_new);
            const float pe = exp2_approx(s - m_new);
            float psum = pe;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
            l = l * alpha + psum;
            m = m_new;
#pragma unroll
            for (int c = 0; c < kChunks; ++c) {
                acc[c].x *= alpha;
                acc[c].y *= alpha;
                acc[c].z *= alpha;
                acc[c].w *= alpha;
            }
            // U += p v over the block's edges, eight row gathers in flight
            for (int t0 = 0; t0 < cnt; t0 += 8) {
                float pt[8];
                int jt[8];
                float4 vv[8][kChunks];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    pt[u] = __shfl_sync(0xffffffffu, pe, (t0 + u) & 31);
                    jt[u] = __shfl_sync(0xffffffffu, j, (t0 + u) & 31);
                    const bool use = t0 + u < cnt && jt[u] >= 0 && pt[u] != 0.f;
#pragma unroll
                    for (int c = 0; c < kChunks; ++c)
                        vv[u][c] = use && live[c]
                                       ? ldg4(gv + (int64_t)jt[u] * p.v_st + (int64_t)h * p.v_sh + 4 * (lane + 32 * c))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
                    if (!use) pt[u] = 0.f;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
#pragma unroll
                    for (int c = 0; c < kChunks; ++c) {
                        acc[c].x = fmaf(pt[u], vv[u][c].x, acc[c].x);
                        acc[c].y = fmaf(pt[u], vv[u][c].y, acc[c].y);
                        acc[c].z = fmaf(pt[u], vv[u][c].z, acc[c].z);
                        acc[c].w = fmaf(pt[u], vv[u][c].w, acc[c].w);
                    }
            }
        }

        const float inv = l > 0.f ? 1.f / l : 0.f;
        Tout *orow = go + (int64_t)i * p.o_st + (int64_t)h * p.o_sh;
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
            if (live[c])
                store4(orow + 4 * (lane + 32 * c),
                       make_float4(acc[c].x * inv, acc[c].y * inv, acc[c].z * inv, acc[c].w * inv));
        if (lane == 0 && p.lse)
            p.lse[(int64_t)h * p.n_dst + i] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
    }
}

// ---- row-centric kernel ------------------------------------------------------
//
// For tensors whose rows hold their H heads back to back (head stride D, token
// stride H * D): one warp per destination row gathers whole source rows, all
// heads at once, in 16-byte chunks (VEC elements; chunk c of a row belongs to
// head c * VEC / D).  LG lanes cover one edge's row (NCL chunks per lane); the
// warp's 32 / LG lane groups ("slots") take different edges, and every slot
// keeps U edges' gathers in flight.  The row's edges are scanned in blocks of
// 32 / LG * U edges with the online-softmax recurrence per head: the block's
// max (over all slots), rescale, exponentials, rescaled sum; each slot keeps
// its own numerator (all slots share one running max, so the numerators add
// up at the end).

template <typename T> struct Vec;
template <> struct Vec<float> {
    static constexpr int N = 4;
    using raw = float4;
    __device__ static void to_f32(const raw &r, float (&f)[4]) { f[0] = r.x; f[1] = r.y; f[2] = r.z; f[3] = r.w; }
};
template <> struct Vec<__half> {
    static constexpr int N = 8;
    using raw = uint4;
    __device__ static void to_f32(const raw &r, float (&f)[8]) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&w[k]));
            f[2 * k] = v.x;
            f[2 * k + 1] = v.y;
        }
    }
};
template <> struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    using raw = uint4;
    __device__ static void to_f32(const raw &r, float (&f)[8]) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[k]));
            f[2 * k] = v.x;
            f[2 * k + 1] = v.y;
        }
    }
};

template <typename T>
__device__ __forceinline__ typename Vec<T>::raw ldg_raw(const T *p) {
    return __ldg(reinterpret_cast<const typename Vec<T>::raw *>(p));
}

template <typename Tout, int N>
__device__ __forceinline__ void store_vec(Tout *dst, const float (&f)[N], float mul) {
#pragma unroll
    for (int k = 0; k < N; k += 4) store4(dst + k, make_float4(f[k] * mul, f[k + 1] * mul, f[k + 2] * mul, f[k + 3] * mul));
}

template <typename T, typename Tout, bool kDot, int LG, int NCL>
__global__ void __launch_bounds__(32 * kWarps) csr_rows_kernel(const CsrParams p) {
    constexpr int VEC = Vec<T>::N;
    constexpr int EP = 32 / LG;      // edge slots per warp
    constexpr int U = ATTN_CSR_INFLIGHT / NCL;  // edges per slot in flight
    constexpr int BLK = EP * U;      // edges per block of the scan
    using raw = typename Vec<T>::raw;
    const int lane = threadIdx.x & 31;
    const int slot = lane / LG, cl = lane % LG;
    const int R = p.H * p.D;         // elements per row (all heads)
    const int NC = R / VEC;          // chunks per row
    const int LPH = p.D / VEC;       // chunks (lanes) per head
    int chunk[NCL], head[NCL];
    bool on[NCL];
#pragma unroll
    for (int k = 0; k < NCL; ++k) {
        chunk[k] = cl + k * LG;
        on[k] = chunk[k] < NC;
        head[k] = on[k] ? chunk[k] * VEC / p.D : 0;
    }
    const T *gv = static_cast<const T *>(p.v);
    const T *gk = static_cast<const T *>(p.k);
    const T *gq = static_cast<const T *>(p.q);
    Tout *go = static_cast<Tout *>(p.o);
    const int64_t stride = (int64_t)gridDim.x * kWarps;

    for (int64_t ri = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); ri < p.n_dst; ri += stride) {
        const int64_t i = row_at(p, (int)ri);
        if (i < 0) continue;  // (warp-uniform) entry outside the rows, reported
        int64_t e0 = __ldg(p.row_ptr + i), e1 = __ldg(p.row_ptr + i + 1);
        if (e0 < 0 || e1 < e0 || e1 > p.n_edges) {
            if (lane == 0) report_status(p.status, ATTN_EINVAL);
            e0 = e1 = 0;  // treated as a row without edges
        }
        float qf[NCL][VEC];
        if (kDot) {
#pragma unroll
            for (int k = 0; k < NCL; ++k) {
                if (on[k]) Vec<T>::to_f32(ldg_raw(gq + i * (int64_t)R + chunk[k] * VEC), qf[k]);
                else
#pragma unroll
                    for (int x = 0; x < VEC; ++x) qf[k][x] = 0.f;
            }
        }
        float acc[NCL][VEC], m[NCL], l[NCL];
#pragma unroll
        for (int k = 0; k < NCL; ++k) {
            m[k] = -INFINITY;
            l[k] = 0.f;
#pragma unroll
            for (int x = 0; x < VEC; ++x) acc[k][x] = 0.f;
        }

        for (int64_t eb = e0; eb < e1; eb += BLK) {
            int j[U];
            raw vr[U][NCL], kr[U][NCL];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t e = eb + u * EP + slot;
                j[u] = -1;
                if (e < e1) {
                    j[u] = __ldg(p.col + e);
                    if (j[u] < 0 || j[u] >= p.n_src) {
                        report_status(p.status, ATTN_EINVAL);
                        j[u] = -1;
                    }
                }
#pragma unroll
                for (int k = 0; k < NCL; ++k) {
                    const bool use = j[u] >= 0 && on[k];
                    vr[u][k] = use ? ldg_raw(gv + (int64_t)j[u] * R + chunk[k] * VEC) : raw{};
                    if (kDot) kr[u][k] = use ? ldg_raw(gk + (int64_t)j[u] * R + chunk[k] * VEC) : raw{};
                }
            }
            // scores (log2 units; -inf where no edge) and the block max per head
            float sc[U][NCL], bmax[NCL];
#pragma unroll
            for (int k = 0; k < NCL; ++k) bmax[k] = -INFINITY;
#pragma unroll
            for (int u = 0; u < U; ++u) {
#pragma unroll
                for (int k = 0; k < NCL; ++k) {
                    float s;
                    if (kDot) {
                        float kf[VEC];
                        Vec<T>::to_f32(kr[u][k], kf);
                        float d = 0.f;
#pragma unroll
                        for (int x = 0; x < VEC; ++x) d = fmaf(qf[k][x], kf[x], d);
                        for (int o = 1; o < LPH; o <<= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
                        s = d * p.scale_log2;
                    } else {
                        const int64_t e = eb + u * EP + slot;
                        s = j[u] >= 0 ? __ldg(p.scores + e * p.H + head[k]) * kLog2e : -INFINITY;
                    }
                    s = j[u] >= 0 ? s : -INFINITY;
                    sc[u][k] = s;
                    bmax[k] = fmaxf(bmax[k], s);
                }
            }
#pragma unroll
            for (int k = 0; k < NCL; ++k)
#pragma unroll
                for (int o = LG; o < 32; o <<= 1) bmax[k] = fmaxf(bmax[k], __shfl_xor_sync(0xffffffffu, bmax[k], o));
#pragma unroll
            for (int k = 0; k < NCL; ++k) {
                // no branch here: the slot sums below shuffle across the whole warp
                const float m_new = fmaxf(m[k], bmax[k]);
                const bool none = m_new == -INFINITY;  // no edge of this head admitted yet
                const float m_ref = none ? 0.f : m_new;
                const float alpha = none ? 1.f : exp2_approx(m[k] - m_new);  // 0 when m = -inf
                float psum = 0.f;
#pragma unroll
                for (int x = 0; x < VEC; ++x) acc[k][x] *= alpha;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const float pe = exp2_approx(sc[u][k] - m_ref);  // 0 for -inf
                    psum += pe;
                    float vf[VEC];
                    Vec<T>::to_f32(vr[u][k], vf);
#pragma unroll
                    for (int x = 0; x < VEC; ++x) acc[k][x] = fmaf(pe, vf[x], acc[k][x]);
                }
#pragma unroll
                for (int o = LG; o < 32; o <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
                l[k] = l[k] * alpha + psum;
                m[k] = m_new;
            }
        }
        // add up the slots' numerators; slot 0 writes the row
#pragma unroll
        for (int k = 0; k < NCL; ++k)
#pragma unroll
            for (int x = 0; x < VEC; ++x)
#pragma unroll
                for (int o = LG; o < 32; o <<= 1) acc[k][x] += __shfl_xor_sync(0xffffffffu, acc[k][x], o);
        if (slot == 0) {
#pragma unroll
            for (int k = 0; k < NCL; ++k) {
                if (!on[k]) continue;
                store_vec<Tout, VEC>(go + i * (int64_t)R + chunk[k] * VEC, acc[k], l[k] > 0.f ? 1.f / l[k] : 0.f);
                if (p.lse && chunk[k] % LPH == 0)
                    p.lse[(int64_t)head[k] * p.n_dst + i] = l[k] > 0.f ? (m[k] + __log2f(l[k])) * kLn2 : -INFINITY;
            }
        }
    }
}

// The row-centric kernel applies when q, k, v, o keep each row's heads back to
// back, D is a multiple of the 16-byte vector and a row has at most 64 chunks
// (and, for dot-product scores, a head's chunks are a power of two).
template <typename T>
int rows_chunks(const CsrParams &p) {
    constexpr int VEC = Vec<T>::N;
    const int64_t R = (int64_t)p.H * p.D;
    auto packed = [&](int64_t st, int64_t sh) { return st == R && sh == p.D; };
    if (p.D % VEC || R / VEC > 64) return 0;
    if (!packed(p.v_st, p.v_sh) || !packed(p.o_st, p.o_sh)) return 0;
    if (!p.scores) {
        const int lph = p.D / VEC;
        if (!packed(p.q_st, p.q_sh) || !packed(p.k_st, p.k_sh) || (lph & (lph - 1))) return 0;
    }
    return (int)(R / VEC);
}

template <typename T, typename Tout, bool kDot>
cudaError_t launch_rows(const CsrParams &p, int nc, cudaStream_t s) {
    const int64_t want = ((int64_t)p.n_dst + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)sm_count() * 8;
    const int grid = (int)(want < cap ? want : cap);
    if (nc <= 8) csr_rows_kernel<T, Tout, kDot, 8, 1><<<grid, 32 * kWarps, 0, s>>>(p);
    else if (nc <= 32) csr_rows_kernel<T, Tout, kDot, 32, 1><<<grid, 32 * kWarps, 0, s>>>(p);
    else csr_rows_kernel<T, Tout, kDot, 32, 2><<<grid, 32 * kWarps, 0, s>>>(p);
    count_launch();
    return cudaGetLastError();
}

template <typename T, typename Tout>
cudaError_t launch_typed(const CsrParams &p, cudaStream_t s) {
    if (const int nc = rows_chunks<T>(p)) {
        if (p.scores) return launch_rows<T, Tout, false>(p, nc, s);
        return launch_rows<T, Tout, true>(p, nc, s);
    }
    const int64_t pairs = (int64_t)p.n_dst * p.H;
    const int64_t want = (pairs + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)sm_count() * 16;
    const int grid = (int)(want < cap ? want : cap);
    if (p.scores) csr_fwd_kernel<T, Tout, false><<<grid, 32 * kWarps, 0, s>>>(p);
    else csr_fwd_kernel<T, Tout, true><<<grid, 32 * kWarps, 0, s>>>(p);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_csr_fwd(const CsrParams &p, cudaStream_t s) {
    if ((int64_t)p.n_dst * p.H == 0) return cudaSuccess;
    if (p.D > 4 * 32 * kChunks) return cudaErrorInvalidValue;
    switch (p.dtype) {
    case ATTN_F16:
        return p.o_dtype == ATTN_F32 ? launch_typed<__half, float>(p, s) : launch_typed<__half, __half>(p, s);
    case ATTN_BF16:
        return p.o_dtype == ATTN_F32 ? launch_typed<__nv_bfloat16, float>(p, s)
                                     : launch_typed<__nv_bfloat16, __nv_bfloat16>(p, s);
    default: return launch_typed<float, float>(p, s);
    }
}

}  // namespace attn

// Merge of partial attention results over disjoint key sets (the split-K
// merge).
//
// Split-K (Vx issue "Chunked-dot Reduce lowering: shorten the reduction
// dependency chain", measurement section: C = 8 key chunks) runs each chunk
// of a query row's keys as its own online-softmax scan.  Chunk c ends with the
// state (m_c, l_c, U_c) of the OCANNL "Module Ir.Online_softmax" page (fourth
// bullet) and stores it normalised, as O_c = U_c / l_c and
// lse_c = m_c + ln l_c.  Softmax over the union of the chunks weighs chunk c
// by exp(lse_c - lse), with lse = ln sum_c exp(lse_c):
//     O = sum_c exp(lse_c - lse) O_c.
// A chunk with lse_c = -inf admits no key and has weight 0 (its O_c is not
// read); a row whose chunks are all -inf gets O = 0, lse = -inf.
//
// HBM-bound: one warp per (query row, head).  Lane c < n_parts reads lse_c;
// the warp reduces max and sum with shuffles; then each lane accumulates
// float4 columns of the weighted partial rows (a 512-byte coalesced read per
// partial at D = 128) and writes the output row once.  Exponentials in base 2
// on the SFU, as in the attention kernels.
#include "../../include/attn.h"
#include "common.cuh"

namespace attn {

namespace {

constexpr int kWarps = 8;
constexpr int kMaxD = 256;

template <typename Tout>
__global__ void __launch_bounds__(32 * kWarps) merge_kernel(const MergeParams p) {
    pdl_trigger();
    pdl_wait();  // the partials come from the kernel before this one
    const int lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)p.n_q * p.H;
    const int64_t stride = (int64_t)gridDim.x * kWarps;
    for (int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); r < rows; r += stride) {
        const int t = (int)(r / p.H), h = (int)(r - (int64_t)t * p.H);
        // lse of the partials, in log2 units; lanes >= n_parts (and the second
        // pass when n_parts > 32) contribute -inf
        float x0 = -INFINITY, x1 = -INFINITY;
        const int64_t lse_off = (int64_t)h * p.n_q + t, lse_st = (int64_t)p.H * p.n_q;
        if (lane < p.n_parts) x0 = __ldg(p.lse_parts + lane * lse_st + lse_off) * kLog2e;
        if (lane + 32 < p.n_parts) x1 = __ldg(p.lse_parts + (lane + 32) * lse_st + lse_off) * kLog2e;
        float mx = fmaxf(x0, x1);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_use = mx == -INFINITY ? 0.f : mx;
        const float w0 = exp2_approx(x0 - m_use), w1 = exp2_approx(x1 - m_use);
        float l = w0 + w1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        const float inv = l > 0.f ? 1.f / l : 0.f;

        Tout *orow = static_cast<Tout *>(p.o) + (int64_t)t * p.o_st + (int64_t)h * p.o_sh;
        const float *prow = p.o_parts + r * p.D;
        // columns 4 lane + 128 i (i < 2 covers D <= 256); every lane takes part
        // in the weight shuffles, columns past D are skipped
        float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
        for (int c = 0; c < p.n_parts; ++c) {
            // weight of partial c, held by lane c % 32
            const float wc = __shfl_sync(0xffffffffu, c < 32 ? w0 : w1, c & 31) * inv;
            if (wc == 0.f) continue;  // uniform across the warp
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int d = 4 * lane + 128 * i;
                if (d >= p.D) break;
                const float4 v = __ldg(reinterpret_cast<const float4 *>(prow + c * p.part_st + d));
                acc[i].x = fmaf(wc, v.x, acc[i].x);
                acc[i].y = fmaf(wc, v.y, acc[i].y);
                acc[i].z = fmaf(wc, v.z, acc[i].z);
                acc[i].w = fmaf(wc, v.w, acc[i].w);
            }
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int d = 4 * lane + 128 * i;
            if (d < p.D) store4(orow + d, acc[i]);
        }
        if (lane == 0 && p.lse) p.lse[lse_off] = mx == -INFINITY ? -INFINITY : (mx + __log2f(l)) * kLn2;
    }
}

}  // namespace

cudaError_t launch_merge(const MergeParams &p, cudaStream_t s) {
    if (p.D > kMaxD || p.n_parts > 64) return cudaErrorInvalidValue;
    const int64_t rows = (int64_t)p.n_q * p.H;
    if (rows == 0) return cudaSuccess;
    const int64_t want = (rows + kWarps - 1) / kWarps;
    const int grid = (int)(want < (int64_t)sm_count() * 16 ? want : (int64_t)sm_count() * 16);
    cudaError_t e;
    switch (p.o_dtype) {
    case ATTN_F16: e = launch_pdl(merge_kernel<__half>, dim3(grid), dim3(32 * kWarps), 0, s, p); break;
    case ATTN_BF16: e = launch_pdl(merge_kernel<__nv_bfloat16>, dim3(grid), dim3(32 * kWarps), 0, s, p); break;
    default: e = launch_pdl(merge_kernel<float>, dim3(grid), dim3(32 * kWarps), 0, s, p); break;
    }
    count_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace attn

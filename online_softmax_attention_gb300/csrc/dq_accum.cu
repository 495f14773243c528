// dQ partial sums of the fused backward (the tensor-core dK/dV kernel also
// accumulates dq with f32 reductions).  The sums live in the workspace laid
// out (H, D/4, n_q, 4) f32: the 4-column group g of query row t of head h is
// the 16 bytes at ((h * D/4 + g) * n_q + t) * 4, so one warp's reduction of a
// group over 32 consecutive query rows covers 512 contiguous bytes.
//
// zero:    the sums are set to 0 before the dK/dV kernel adds to them.
// convert: dq = scale * sums, rounded to grad_dtype, written with dq's
//          strides (a tile of 64 rows x D is transposed through shared memory
//          so that both the reads and the writes are coalesced).
#include "common.cuh"

namespace attn {

namespace {

__global__ void __launch_bounds__(256) dq_zero_kernel(float4 *p, int64_t n4) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride)
        p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

constexpr int kConvRows = 64;

template <typename Tg, int D>
__global__ void __launch_bounds__(256) dq_convert_kernel(const BwdParams p) {
    constexpr int G = D / 4;  // 4-column groups per row
    __shared__ float4 tile[kConvRows][G + 1];
    const int t0 = blockIdx.x * kConvRows, h = blockIdx.y;
    const int rows = min(kConvRows, p.n_q - t0);
    const float4 *src = reinterpret_cast<const float4 *>(p.dq_accum) + (int64_t)h * G * p.n_q + t0;
    for (int i = threadIdx.x; i < kConvRows * G; i += blockDim.x) {
        const int g = i / kConvRows, r = i - g * kConvRows;  // consecutive threads: consecutive rows
        if (r < rows) tile[r][g] = src[(int64_t)g * p.n_q + r];
    }
    __syncthreads();
    Tg *dq = static_cast<Tg *>(p.dq) + (int64_t)h * p.dq_sh;
    for (int i = threadIdx.x; i < kConvRows * G; i += blockDim.x) {
        const int r = i / G, g = i - r * G;  // consecutive threads: consecutive columns of a row
        if (r < rows) {
            const float4 v = tile[r][g];
            store4(dq + (int64_t)(t0 + r) * p.dq_st + 4 * g,
                   make_float4(v.x * p.scale, v.y * p.scale, v.z * p.scale, v.w * p.scale));
        }
    }
}

template <int D>
cudaError_t convert_d(const BwdParams &p, cudaStream_t s) {
    const dim3 grid((p.n_q + kConvRows - 1) / kConvRows, p.H);
    switch (p.grad_dtype) {
    case ATTN_F16: dq_convert_kernel<__half, D><<<grid, 256, 0, s>>>(p); break;
    case ATTN_BF16: dq_convert_kernel<__nv_bfloat16, D><<<grid, 256, 0, s>>>(p); break;
    default: dq_convert_kernel<float, D><<<grid, 256, 0, s>>>(p); break;
    }
    count_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dq_accum_zero(const BwdParams &p, cudaStream_t s) {
    const int64_t n4 = (int64_t)p.n_q * p.H * p.D / 4;
    if (n4 == 0) return cudaSuccess;
    const int64_t want = (n4 + 255) / 256;
    const int blocks = (int)(want < 8LL * sm_count() ? want : 8LL * sm_count());
    dq_zero_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<float4 *>(p.dq_accum), n4);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_dq_accum_convert(const BwdParams &p, cudaStream_t s) {
    if ((int64_t)p.n_q * p.H == 0) return cudaSuccess;
    return p.D == 64 ? convert_d<64>(p, s) : convert_d<128>(p, s);
}

}  // namespace attn

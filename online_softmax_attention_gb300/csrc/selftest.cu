// Self-test hook for the device math helpers the attention kernels use in
// place of SFU instructions, so that tests can compare them with CUDA's own
// functions on the GPU.
#include "../../include/attn.h"
#include "sm100.cuh"

namespace attn {
namespace {

__global__ void exp2_fma2_kernel(const float *__restrict__ x, float *__restrict__ y, int n) {
    const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i + 1 < n) {
        const float2 r = sm100::exp2_fma2(make_float2(x[i], x[i + 1]));
        y[i] = r.x;
        y[i + 1] = r.y;
    } else if (i < n) {
        y[i] = sm100::exp2_fma2(make_float2(x[i], 0.f)).x;
    }
}

}  // namespace
}  // namespace attn

extern "C" int attn_selftest_exp2(const float *x, float *y, int n, void *stream) {
    if (n < 0 || (n > 0 && (!x || !y))) return ATTN_EINVAL;
    if (n == 0) return ATTN_OK;
    const int threads = 256, pairs = (n + 1) / 2;
    attn::exp2_fma2_kernel<<<(pairs + threads - 1) / threads, threads, 0, static_cast<cudaStream_t>(stream)>>>(x, y, n);
    attn::count_launch();
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ECUDA;
}

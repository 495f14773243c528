// Schedule preparation for the persistent attention kernels.
//
// One block validates the cu_seqlens offsets on the device (no host copy of
// them is needed) and writes, for tiles of `block` rows (each counted `splits`
// times under split-K), the prefix of work items per sequence into the workspace; it also resets the dynamic work
// counter.  Inconsistent offsets make the schedule empty and set the device
// status word to ATTN_EINVAL, so the attention kernel that follows does no
// work and reads nothing out of bounds.
#include "../../include/attn.h"
#include "common.cuh"

namespace attn {

namespace {

constexpr int kPrepThreads = 1024;

__global__ void __launch_bounds__(kPrepThreads)
prep_kernel(const int32_t *__restrict__ cu_q, const int32_t *__restrict__ cu_k, int n_seq,
            int n_q, int n_k, int H, int block, int causal, int rows_are_keys, int splits,
            int *hdr, int *prefix, int *status) {
    __shared__ int s_bad;
    __shared__ int s_warp[kPrepThreads / 32];
    __shared__ long long s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_trigger();
    pdl_wait();  // the previous kernel on the stream may still read this schedule block
    if (tid == 0) {
        s_bad = 0;
        s_carry = 0;
    }
    __syncthreads();

    int bad = 0;
    for (int b = tid; b < n_seq; b += kPrepThreads) {
        const int q0 = cu_q ? cu_q[b] : 0, q1 = cu_q ? cu_q[b + 1] : n_q;
        const int k0 = cu_k ? cu_k[b] : 0, k1 = cu_k ? cu_k[b + 1] : n_k;
        if (b == 0 && (q0 != 0 || k0 != 0)) bad = 1;
        if (q1 < q0 || k1 < k0 || q1 > n_q || k1 > n_k) bad = 1;
        if (causal && (q1 - q0) != (k1 - k0)) bad = 1;
    }
    if (bad) atomicOr(&s_bad, 1);
    __syncthreads();
    bad = s_bad;

    for (int base = 0; base < n_seq; base += kPrepThreads) {
        const int b = base + tid;
        int cnt = 0;
        if (b < n_seq && !bad) {
            const int len = rows_are_keys ? ((cu_k ? cu_k[b + 1] - cu_k[b] : n_k))
                                          : ((cu_q ? cu_q[b + 1] - cu_q[b] : n_q));
            cnt = (len + block - 1) / block * H * splits;
        }
        // inclusive scan across the block
        int x = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_warp[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = s_warp[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            s_warp[lane] = w;
        }
        __syncthreads();
        const int incl = x + (warp > 0 ? s_warp[warp - 1] : 0);
        const long long carry = s_carry;
        if (b < n_seq) prefix[b] = (int)(carry + incl - cnt);
        __syncthreads();
        if (tid == kPrepThreads - 1) s_carry = carry + incl;
        __syncthreads();
    }
    if (tid == 0) {
        prefix[n_seq] = (int)s_carry;
        hdr[0] = 0;
        hdr[1] = (int)s_carry;
        if (bad) report_status(status, ATTN_EINVAL);
    }
}

}  // namespace

cudaError_t launch_prep(const int32_t *cu_q, const int32_t *cu_k, int n_seq, int n_q, int n_k,
                        int H, int block, int causal, int rows_are_keys, int splits, Sched sched,
                        int *status, cudaStream_t s) {
    cudaError_t e = launch_pdl(prep_kernel, dim3(1), dim3(kPrepThreads), 0, s, cu_q, cu_k, n_seq, n_q, n_k, H,
                               block, causal, rows_are_keys, splits, sched.hdr,
                               const_cast<int *>(sched.prefix), status);
    count_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace attn

// Device-side helpers shared by the attention kernels: element conversion,
// base-2 exponentials, and the work-item mapping of the persistent scheduler.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/attn.h"
#include "internal.h"

namespace attn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---- programmatic dependent launch ----------------------------------------
// pdl_trigger: the next kernel on the stream (launched with launch_pdl) may
// start once every CTA of this grid has executed it.  pdl_wait: returns once
// the previous grid on the stream has completed and its writes are visible
// (at once when this kernel was launched the ordinary way); a kernel reads no
// global memory before it.

__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- element conversion -------------------------------------------------

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Load 4 consecutive elements (16-byte aligned for f32, 8-byte for 16-bit types).
__device__ __forceinline__ float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 load4(const __half *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ void store4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void store4(__half *p, float4 v) {
    __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&a);
    u.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
}
__device__ __forceinline__ void store4(__nv_bfloat16 *p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&a);
    u.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
}

// 2^x with the SFU (ex2.approx, flush-to-zero).  2^-inf = 0.
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---- persistent scheduler -------------------------------------------------
//
// Work items are (sequence b, head h, tile t, key split c) tuples, numbered
// sequence-major, then head, then tile, then split (c < splits; splits = 1
// without split-K).  prefix[b] = H * splits * (tiles of sequences before b),
// written by the preparation kernel; item w belongs to the last sequence
// whose prefix is <= w.  Tiles of one (b, h) are consecutive so that the CTAs
// running at the same time share K/V in L2; `descending` orders them
// longest-first for the causal relation.

struct WorkItem {
    int b, h, t, ntiles, c;
};

__device__ __forceinline__ WorkItem map_item(int w, const int *prefix, int n_seq, int H,
                                             bool descending, int splits = 1) {
    int lo = 0, hi = n_seq - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(prefix + mid) <= w) lo = mid;
        else hi = mid - 1;
    }
    const int base = __ldg(prefix + lo);
    const int per_head = (__ldg(prefix + lo + 1) - base) / H;  // tiles * splits
    const int r = w - base;
    const int h = r / per_head;
    const int rem = r - h * per_head;
    int t = splits == 1 ? rem : rem / splits;
    const int c = rem - t * splits;
    const int ntiles = per_head / splits;
    if (descending) t = ntiles - 1 - t;
    return {lo, h, t, ntiles, c};
}

// The same mapping for one sequence (no cu_seqlens) of `total` items, which
// needs no prefix from the workspace.
__device__ __forceinline__ WorkItem map_item_single(int w, int total, int H, bool descending,
                                                    int splits = 1) {
    const int per_head = total / H;  // tiles * splits
    const int h = w / per_head;
    const int rem = w - h * per_head;
    int t = splits == 1 ? rem : rem / splits;
    const int c = rem - t * splits;
    const int ntiles = per_head / splits;
    if (descending) t = ntiles - 1 - t;
    return {0, h, t, ntiles, c};
}

// Work-item fetch of the persistent kernels.  Dynamic schedule (static_items
// = 0): items come from the global counter that the preparation kernel reset.
// Static schedule (static_items > 0: one sequence whose items all fit in one
// wave, grid = static_items): CTA i runs item i and nothing else, so neither a
// counter nor a preparation launch is needed.  `k` counts this CTA's fetches.
__device__ __forceinline__ int fetch_item(int *counter, int static_items, int k) {
    if (static_items > 0) return k == 0 ? (int)blockIdx.x : static_items;
    return atomicAdd(counter, 1);
}

// Offsets of sequence b (one sequence when cu is null).
__device__ __forceinline__ void seq_bounds(const int32_t *cu, int total, int b, int &start, int &len) {
    if (cu) {
        start = __ldg(cu + b);
        len = __ldg(cu + b + 1) - start;
    } else {
        start = 0;
        len = total;
    }
}

// Record the first error in the device status word.
__device__ __forceinline__ void report_status(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

}  // namespace attn

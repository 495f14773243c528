// Inline-PTX wrappers for the sm_100-family (sm_103a) features the
// tensor-core attention kernels use: mbarriers, TMA tile loads, and the
// tcgen05 tensor-memory (TMEM) allocator, MMA, commit, loads and stores; and
// the epilogue store of accumulator rows held one row per lane.
//
// Every mbarrier wait is bounded: after `budget` clock cycles it raises the
// CTA's abort flag, records ATTN_ETIMEOUT in the device status word and
// returns false, so a kernel can wind down instead of spinning forever.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include <type_traits>

#include "common.cuh"

namespace attn {
namespace sm100 {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier ---------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One arrival per warp on `bar` (initialised with the number of arriving
// warps) once all 32 lanes have reached this point.  Writes the lanes made
// before -- TMEM stores completed by tcgen05.wait::st and followed by
// tcgen05.fence::before_thread_sync, or shared-memory stores -- are ordered
// before lane 0's release arrive by the warp barrier.  128 or 256 per-thread
// arrivals on one mbarrier serialise; 4 or 8 do not.
__device__ __forceinline__ void mbar_arrive_warp(uint32_t bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-suspending test of the phase (mbarrier.test_wait).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

struct Watchdog {
    long long budget;   // clock cycles per wait
    int *abort_flag;    // shared: set once any wait of the CTA gave up
    int *status;        // global device status word
};

// Budgets below this many cycles (failure-detection tests) are polled with
// test_wait: try_wait may suspend the thread until the phase completes, up to a
// hardware time limit, so a wait that ends within that limit would never see a
// short budget run out.
constexpr long long kPolledBudget = 1ll << 20;

// Wait for the phase of parity `parity` to complete.  Returns false if the
// CTA is aborting (this wait timed out, or another one did).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const Watchdog &wd) {
    if (wd.budget < kPolledBudget) {
        const long long t0 = clock64();
        for (;;) {
            if (mbar_test_wait(bar, parity)) return true;
            if (*reinterpret_cast<volatile int *>(wd.abort_flag)) return false;
            if (clock64() - t0 > wd.budget) {
                *reinterpret_cast<volatile int *>(wd.abort_flag) = 1;
                report_status(wd.status, ATTN_ETIMEOUT);
                return false;
            }
        }
    }
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile int *>(wd.abort_flag)) return false;
        if (clock64() - t0 > wd.budget) {
            *reinterpret_cast<volatile int *>(wd.abort_flag) = 1;
            report_status(wd.status, ATTN_ETIMEOUT);
            return false;
        }
    }
}

// One lane of a converged warp is elected; from_leader() gives its values to
// the other lanes.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n"
        " .reg .pred P;\n"
        " elect.sync _|P, 0xffffffff;\n"
        " selp.u32 %0, 1, 0, P;\n"
        "}\n"
        : "=r"(pred));
    return pred != 0;
}

// The value `v` of the lane for which `lead` is set, for the whole warp.
__device__ __forceinline__ uint32_t from_leader(uint32_t v, bool lead) {
    return __shfl_sync(0xffffffffu, v, __ffs(__ballot_sync(0xffffffffu, lead)) - 1);
}

// An MMA-issuing lane's short, bounded spin (mbarrier.test_wait, which never
// suspends) on a phase that is due within a few hundred cycles; false if it has
// not completed after kIssuerSpin tests, and the warp then waits for it with
// the watchdog.
constexpr int kIssuerSpin = 32;
__device__ __forceinline__ bool mbar_due(uint32_t bar, uint32_t parity) {
    for (int k = 0; k < kIssuerSpin; ++k)
        if (mbar_test_wait(bar, parity)) return true;
    return false;
}

// Position in a ring of N shared-memory slots guarded by full / empty
// mbarriers; `i` counts the uses of the ring.
template <int N>
struct RingPos {
    uint32_t i = 0;
    __device__ __forceinline__ uint32_t slot() const { return i % N; }
    __device__ __forceinline__ uint32_t phase() const { return (i / N) & 1; }
};

__device__ __forceinline__ bool aborting(const Watchdog &wd) {
    return *reinterpret_cast<volatile int *>(wd.abort_flag) != 0;
}

// ---- packed / 3-input FP32 arithmetic (sm_100 family) ------------------------------

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Maximum of n (a multiple of 16) values with eight independent chains.
template <int N>
__device__ __forceinline__ float row_max(const float *v) {
    static_assert(N % 16 == 0, "row_max: N must be a multiple of 16");
    constexpr int L = N / 8;  // values per chain
    float m[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        m[k] = v[k * L];
#pragma unroll
        for (int c = 1; c + 1 < L; c += 2) m[k] = max3f(m[k], v[k * L + c], v[k * L + c + 1]);
        if (L % 2 == 0) m[k] = fmaxf(m[k], v[k * L + L - 1]);
    }
    return max3f(max3f(m[0], m[1], m[2]), max3f(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

// 2^x for a pair, on the FMA and integer pipes instead of the SFU.
// Range reduction (Cody and Waite): n = rint(x) via the 1.5 * 2^23 rounding
// constant, f = x - n in [-1/2, 1/2]; 2^f by a degree-4 polynomial fitted for
// this library (relative minimax on [-1/2, 1/2] with p(0) = 1; max relative
// error 2.9e-6 evaluated in f32); the result's exponent field gets n added.
// x is clamped to [-126, 127], so the result is >= ~2^-126 (never 0): callers
// use it only where no -inf mask applies.  Above 127 it saturates near 2^127
// (finite) instead of carrying the exponent into the sign bit.
__device__ __forceinline__ float2 exp2_fma2(float2 x) {
    constexpr float kRound = 12582912.f;  // 1.5 * 2^23
    x.x = fminf(fmaxf(x.x, -126.f), 127.f);
    x.y = fminf(fmaxf(x.y, -126.f), 127.f);
    const float2 t = __fadd2_rn(x, make_float2(kRound, kRound));
    const float2 n = __fadd2_rn(t, make_float2(-kRound, -kRound));
    const float2 f = __ffma2_rn(n, make_float2(-1.f, -1.f), x);
    float2 p = __ffma2_rn(make_float2(0.00958278402686119f, 0.00958278402686119f), f,
                          make_float2(0.055906277149915695f, 0.055906277149915695f));
    p = __ffma2_rn(p, f, make_float2(0.24024099111557007f, 0.24024099111557007f));
    p = __ffma2_rn(p, f, make_float2(0.6931242346763611f, 0.6931242346763611f));
    p = __ffma2_rn(p, f, make_float2(1.f, 1.f));
    // the low mantissa bits of t hold n; shifting them into the exponent field
    // adds n to it (the rounding constant's own bits shift out entirely)
    return make_float2(__int_as_float(__float_as_int(p.x) + (__float_as_int(t.x) << 23)),
                       __int_as_float(__float_as_int(p.y) + (__float_as_int(t.y) << 23)));
}

// ---- register reallocation between warpgroups ------------------------------------
// All threads of a warpgroup execute the same call.  The counts must add up to
// at most the registers the block was launched with.

template <int N>
__device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

template <int N>
__device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ---- TMA ----------------------------------------------------------------------

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// 3-D tiled load (coordinates innermost first) into shared memory; completes
// `bytes` of transaction count on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *tm, int c0, int c1,
                                            int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// ---- shared / global memory helpers --------------------------------------------

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (tensor-core operand reads, TMA) that a later mbarrier hand-off orders.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// p[0..3] += (a, b, c, d) in global memory, f32, without a return value
// (16-byte aligned p).
__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// ---- tcgen05: TMEM allocation, fences, MMA, commit ------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive once on `bar` when every tcgen05 async operation this thread issued
// before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], 8-bit floating-point operands
// (kind::f8f6f4; the instruction descriptor names the formats)
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand whose
// swizzle atoms (8 rows x 128 bytes) start on 1024-byte boundaries.
//   lbo: byte distance between atoms along the leading (MN for MN-major) axis
//   sbo: byte distance between 8-row groups along the strided axis
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
           (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) |
           (1ull << 46) |   // descriptor version for tcgen05
           (2ull << 61);    // 128-byte swizzle
}

// Advancing a descriptor by `bytes` (a multiple of 16, staying inside the
// 256 KiB shared window) only adds to its start-address field.
__host__ __device__ constexpr uint64_t sdesc_step(uint32_t bytes) { return static_cast<uint64_t>(bytes >> 4); }

// The same advance as a 32-bit add on the descriptor's low word (the
// start-address field cannot carry out of it inside the 256 KiB window).
__device__ __forceinline__ uint64_t sdesc_add(uint64_t d, uint32_t bytes) {
    const uint32_t lo = static_cast<uint32_t>(d) + (bytes >> 4);
    return (d & 0xFFFFFFFF00000000ull) | lo;
}

// Instruction descriptor of tcgen05.mma kind::f16 with an f32 accumulator.
// is_bf16: A and B are bf16 (else f16); b_mn_major: B is N-contiguous.
__host__ __device__ constexpr uint32_t idesc_f16(int is_bf16, int M, int N, int b_mn_major) {
    return (1u << 4) | (static_cast<uint32_t>(is_bf16) << 7) | (static_cast<uint32_t>(is_bf16) << 10) |
           (static_cast<uint32_t>(b_mn_major) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4 with an f32 accumulator
// and A, B both e4m3 (format code 0), K-major.
__host__ __device__ constexpr uint32_t idesc_f8(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ---- tcgen05: TMEM <-> registers (32 lanes x 32 columns of 32 bits per warp) ----

__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}

// Waits for this thread's tcgen05.ld results; the registers pass through the
// asm so that no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]) :: "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// TMEM address of (lane, column) relative to an allocation base.
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
    return base + (lane << 16) + col;
}

// ---- 16-bit packing and row-per-lane stores ---------------------------------------

// Two f32 values rounded to nearest even as one packed 16-bit pair (lo first).
__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
    uint32_t u;
    if (bf16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        u = *reinterpret_cast<uint32_t *>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        u = *reinterpret_cast<uint32_t *>(&v);
    }
    return u;
}

__device__ __forceinline__ void st_piece(float *p, const uint32_t (&w)[8]) {  // 32-byte aligned
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}
template <typename T16>
__device__ __forceinline__ void st_piece(T16 *p, const uint32_t (&w)[4]) {  // 16-byte aligned
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                 "r"(w[3])
                 : "memory");
}

// A warp that read 32 rows of a TMEM accumulator with tcgen05.ld 32x32b holds one
// row per lane, so plain stores would write a few bytes of 32 different rows per
// instruction.  This stores one 32-column chunk of those rows (u: the lane's row
// as f32 bits; each value times `mul`, rounded to T) by cutting it into four
// 8-column pieces that the lanes of each group of four exchange, a 4 x 4
// transpose by xor shuffles: afterwards lane 4g + j holds piece j of rows
// 4g .. 4g + 3, and each store instruction writes eight rows' whole chunks, four
// lanes per row (128 contiguous bytes for f32, 64 for 16-bit types).
//   row0: the warp's first row at the chunk's first column; st: row stride in
//   elements; rows_live: how many of the 32 rows exist (the rest are not
//   written).  All 32 lanes must call it.  f32 pieces are 32-byte stores, so
//   f32 rows that are not 32-byte aligned are written one lane per row instead.
template <typename T>
__device__ __forceinline__ void store_rows_chunk(uint32_t (&u)[32], float mul, T *row0, int64_t st,
                                                 int rows_live, int lane) {
    constexpr int W = sizeof(T) == 4 ? 8 : 4;  // 32-bit words per 8 values
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
#pragma unroll
    for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * mul);
    const bool wide = sizeof(T) < 4 || ((reinterpret_cast<uintptr_t>(row0) & 31) == 0 &&
                                        ((st * (int64_t)sizeof(T)) & 31) == 0);
    if (!wide) {  // the same for every lane of the warp
        if (lane < rows_live) {
            T *dst = row0 + (int64_t)lane * st;
#pragma unroll
            for (int e = 0; e < 32; e += 4)
                store4(dst + e, make_float4(__uint_as_float(u[e]), __uint_as_float(u[e + 1]),
                                            __uint_as_float(u[e + 2]), __uint_as_float(u[e + 3])));
        }
        return;
    }
    uint32_t w[4][W];
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int i = 0; i < W; ++i)
            w[k][i] = W == 8 ? u[8 * k + i]
                             : pack2(__uint_as_float(u[8 * k + 2 * i]), __uint_as_float(u[8 * k + 2 * i + 1]),
                                     kBf16);
    const int gl = lane & 3;
#pragma unroll
    for (int d = 1; d <= 2; d <<= 1) {
        const bool upper = (gl & d) != 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (k & d) continue;
            // the lower lane keeps piece k and sends k | d; the upper keeps k | d and sends k
#pragma unroll
            for (int i = 0; i < W; ++i) {
                const uint32_t send = upper ? w[k][i] : w[k | d][i];
                const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, d);
                if (upper) w[k][i] = recv;
                else w[k | d][i] = recv;
            }
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int r = (lane & ~3) + k;
        if (r < rows_live) st_piece(row0 + (int64_t)r * st + 8 * gl, w[k]);
    }
}

}  // namespace sm100
}  // namespace attn

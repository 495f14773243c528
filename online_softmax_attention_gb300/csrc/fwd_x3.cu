// Forward attention for f32 inputs (D = 64) on the sm_103a tensor cores, with
// f32-level accuracy from bf16 operand splitting.
//
// The recurrence is the one of the OCANNL "Module Ir.Online_softmax" page
// (fourth bullet), scheduled as the 16-bit tensor-core forward: work items of
// 256 query rows in two 128-row tiles that ping-pong between the tensor core
// and their softmax warpgroups, key tiles (here of 64 keys) through TMA rings,
// a persistent grid (or one item per CTA for a short single sequence), bounded
// waits.  What differs is the arithmetic of the two contractions:
//
//  * A prepass kernel splits every f32 input value x into three bf16 parts,
//    x1 = bf16(x), x2 = bf16(x - x1), x3 = bf16(x - x1 - x2) (round to nearest
//    even; each difference is exact in f32), so |x - x1 - x2 - x3| <= 2^-27 |x|.
//  * Each contraction is the sum of the six bf16 products A_a B_b with
//    a + b <= 4 (3-1, 2-2, 1-3, 2-1, 1-2, 1-1: smallest first), accumulated in
//    f32 by the tensor core; every dropped product is below 2^-27 of A B.  For
//    the scores A, B are the parts of Q and K; for the values, the softmax
//    warps split each probability the same way into P1, P2, P3 (bf16, in
//    TMEM) and B is the parts of V.
//  * Each key tile's value contraction starts from zero in TMEM and the
//    softmax warps add that partial to a running U held in registers with f32
//    adds (rounded to nearest), so no rounding of the tensor core's
//    accumulator builds up over the key tiles.
//
// TMEM: query tile t owns [256 t, 256 t + 160): S at [0, 64); after the
// softmax, for key group g of 16 keys (two bf16 per 32-bit column), P1 at
// [16 g, 16 g + 8) and P2 at [16 g + 8, 16 g + 16) (over that group's own S
// columns) and P3 at [64 + 8 g, 64 + 8 g + 8); the key tile's value partial at
// [96, 160).
//
// Shared memory (216 KiB): per query tile Q1, Q2, Q3 (128 x 64 bf16 TMA boxes);
// K ring of 2 stages and V ring of 3 stages, each stage three 64 x 64 parts.
#include <algorithm>
#include <cfloat>

#include "sm100.cuh"
#include "tc.h"

namespace attn {

namespace {

using namespace sm100;

constexpr int D = 64;
constexpr int BM = 128;        // query rows per tile
constexpr int BN = 64;         // keys per key tile
constexpr int NQT = 2;         // query tiles per work item
constexpr int kItemRows = NQT * BM;
constexpr int kThreads = 384;
constexpr int kSchedConsumers = 1 + 8;
constexpr float kRescaleThreshold = 8.f;  // log2 units

constexpr int kParts = 3;                 // bf16 parts of every operand
constexpr int kQPart = BM * D * 2;        // one part of a query tile (16 KiB TMA box)
constexpr int kKVPart = BN * D * 2;       // one part of a key / value tile (8 KiB TMA box)
constexpr int kQBytes = kParts * kQPart;
constexpr int kKBytes = kParts * kKVPart;
constexpr int kVBytes = kParts * kKVPart;
constexpr int kKStages = 2, kVStages = 3;
constexpr int kSmemBytes = NQT * kQBytes + kKStages * kKBytes + kVStages * kVBytes + 1024;
static_assert(kSmemBytes + 1024 <= 232448, "shared memory budget (dynamic + static)");
constexpr int kTmemTile = 256;
constexpr uint32_t kColP3 = 64, kColU = 96;
// the six products A_a B_b with a + b <= 4, smallest first (part indices from 0)
__host__ __device__ constexpr int prod_a(int ch) { return ch == 0 ? 2 : ch == 1 ? 1 : ch == 3 ? 1 : 0; }
__host__ __device__ constexpr int prod_b(int ch) { return ch == 1 ? 1 : ch == 2 ? 2 : ch == 4 ? 1 : 0; }
// registers (from ptxas spill reports): the MMA issuer's six-product chains need
// ~120; the softmax warps keep the running U (64 f32) besides the row state
constexpr int kRegsProducer = 120;
constexpr int kRegsSoftmax = 192;
static_assert(128 * kRegsProducer + 256 * kRegsSoftmax <= kThreads * 168, "register split");

struct X3Args {
    CUtensorMap tq[kParts], tk[kParts], tv[kParts];
    FwdParams p;
};

struct __align__(8) X3Bars {
    uint64_t q_full[NQT], q_empty[NQT];
    uint64_t k_full[kKStages], k_empty[kKStages], v_empty[kVStages];  // k_full: K and V of a key tile
    uint64_t s_full[NQT], p_full[NQT], o_done[NQT], o_free[NQT];
    uint64_t sched_full[2], sched_empty[2];
    uint64_t mma_drain;
};

struct ItemInfo {
    int q_start, Lq, k_start, Lk, h, row0, c, j0;
    int n[NQT];
    int nkv;
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ int total_items(const FwdParams &p) {
    return p.static_items > 0 ? p.static_items : p.sched.hdr[1];
}

__device__ __forceinline__ ItemInfo item_info(const FwdParams &p, int w) {
    const WorkItem it = p.static_items > 0 ? map_item_single(w, p.static_items, p.H, true, p.n_splits)
                                           : map_item(w, p.sched.prefix, p.n_seq, p.H, true, p.n_splits);
    ItemInfo f;
    seq_bounds(p.cu_q, p.n_q, it.b, f.q_start, f.Lq);
    seq_bounds(p.cu_k, p.n_k, it.b, f.k_start, f.Lk);
    f.h = it.h;
    f.c = it.c;
    f.row0 = it.t * kItemRows;
    int full[NQT], most = 0;
#pragma unroll
    for (int t = 0; t < NQT; ++t) {
        const int r0 = f.row0 + BM * t;
        int n = 0;
        if (r0 < f.Lq) n = p.causal ? cdiv(min(f.Lk, r0 + BM), BN) : cdiv(f.Lk, BN);
        full[t] = n;
        most = max(most, n);
    }
    const KeyChunk ch = key_chunk(most, p.n_splits, it.c);
    f.j0 = ch.begin;
    f.nkv = 0;
#pragma unroll
    for (int t = 0; t < NQT; ++t) {
        f.n[t] = max(0, min(full[t], ch.end) - ch.begin);
        f.nkv = max(f.nkv, f.n[t]);
    }
    return f;
}

constexpr long long kDrainCycles = 1ll << 31;
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, long long budget) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > budget) return;
    }
}

// 16 / 8 TMEM columns of 32 bits per lane (32 lanes per warp).
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
}

// Waits for this thread's tcgen05.ld results (the registers pass through the
// asm so that no use of them is scheduled before the wait).
__device__ __forceinline__ void tmem_ld_wait16(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :: "memory");
}

__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

// ---- prepass: f32 -> bf16 parts ----------------------------------------------------

// Splits rows of (tokens, heads, 64) f32 tensors into `parts` contiguous
// (tokens, heads, 64) bf16 arrays each: part 1 = bf16(x), part k+1 = bf16 of
// what parts 1..k leave (round to nearest even; the residuals are exact).
struct SplitJob {
    const float *x;
    int64_t st, sh;
    int tokens, parts;
    __nv_bfloat16 *out;  // parts arrays of tokens * H * 64
};

struct SplitParams {
    SplitJob job[3];
    int H;
};

__global__ void __launch_bounds__(256) split_parts_kernel(const SplitParams sp) {
    pdl_trigger();
    pdl_wait();
    constexpr int C4 = D / 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int j = 0; j < 3; ++j) {
        const SplitJob &jb = sp.job[j];
        const int64_t n4 = (int64_t)jb.tokens * sp.H * C4;
        const int64_t part_elems = (int64_t)jb.tokens * sp.H * D;
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
            const int64_t row = i / C4;
            const int c4 = (int)(i - row * C4);
            const int64_t t = row / sp.H;
            const int h = (int)(row - t * sp.H);
            float4 r = load4(jb.x + t * jb.st + h * jb.sh + 4 * c4);
            __nv_bfloat16 *dst = jb.out + row * D + 4 * c4;
            for (int k = 0; k < jb.parts; ++k) {
                const __nv_bfloat162 a = __floats2bfloat162_rn(r.x, r.y), b = __floats2bfloat162_rn(r.z, r.w);
                uint2 u;
                u.x = *reinterpret_cast<const uint32_t *>(&a);
                u.y = *reinterpret_cast<const uint32_t *>(&b);
                *reinterpret_cast<uint2 *>(dst + k * part_elems) = u;
                const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
                r = make_float4(r.x - fa.x, r.y - fa.y, r.z - fb.x, r.w - fb.y);
            }
        }
    }
}

// ---- warp 0: TMA producer ---------------------------------------------------------

__device__ void producer(const X3Args &a, X3Bars &bars, int *sched_item, uint32_t sQ, uint32_t sK,
                         uint32_t sV, const Watchdog &wd) {
    const FwdParams &p = a.p;
    const int total = total_items(p);
    RingPos<kKStages> kr;
    RingPos<kVStages> vr;
    uint32_t q_uses[NQT] = {0, 0};
    bool q_pending[NQT] = {false, false};
    auto load_kv = [&](int row, int h) -> bool {
        const uint32_t ks = kr.slot(), vs = vr.slot();
        if (!mbar_wait(smem_u32(&bars.k_empty[ks]), kr.phase() ^ 1, wd)) return false;
        if (!mbar_wait(smem_u32(&bars.v_empty[vs]), vr.phase() ^ 1, wd)) return false;
        const uint32_t bar = smem_u32(&bars.k_full[ks]);
        mbar_expect_tx(bar, kKBytes + kVBytes);
#pragma unroll
        for (int g = 0; g < kParts; ++g) tma_load_3d(sK + ks * kKBytes + g * kKVPart, &a.tk[g], 0, row, h, bar);
#pragma unroll
        for (int g = 0; g < kParts; ++g) tma_load_3d(sV + vs * kVBytes + g * kKVPart, &a.tv[g], 0, row, h, bar);
        ++kr.i;
        ++vr.i;
        return true;
    };
    for (int i = 0;; ++i) {
        const int slot = i & 1;
        if (!mbar_wait(smem_u32(&bars.sched_empty[slot]), ((i >> 1) & 1) ^ 1, wd)) break;
        const int w = fetch_item(p.sched.hdr, p.static_items, i);
        sched_item[slot] = w;
        mbar_arrive(smem_u32(&bars.sched_full[slot]));
        if (w >= total) break;
        const ItemInfo f = item_info(p, w);
        bool ok = true;
#pragma unroll
        for (int t = 0; t < NQT; ++t) {
            if (!ok) break;
            if (f.n[t] == 0) continue;
            ok = mbar_wait(smem_u32(&bars.q_empty[t]), (q_uses[t] & 1) ^ 1, wd);
            if (!ok) break;
            const uint32_t bar = smem_u32(&bars.q_full[t]);
            mbar_expect_tx(bar, kQBytes);
#pragma unroll
            for (int g = 0; g < kParts; ++g)
                tma_load_3d(sQ + t * kQBytes + g * kQPart, &a.tq[g], 0, f.q_start + f.row0 + BM * t, f.h, bar);
            ++q_uses[t];
            q_pending[t] = true;
        }
        if (!ok) break;
        for (int j = 0; j < f.nkv && ok; ++j) ok = load_kv(f.k_start + BN * (f.j0 + j), f.h);
        if (!ok) break;
    }
    if (aborting(wd)) {
        const long long budget = kDrainCycles;
        for (uint32_t k = kr.i > (uint32_t)kKStages ? kr.i - kKStages : 0; k < kr.i; ++k)
            drain_wait(smem_u32(&bars.k_full[k % kKStages]), (k / kKStages) & 1, budget);
#pragma unroll
        for (int t = 0; t < NQT; ++t)
            if (q_pending[t]) drain_wait(smem_u32(&bars.q_full[t]), (q_uses[t] - 1) & 1, budget);
    }
}

// ---- warp 1: MMA issuer ------------------------------------------------------------
// Run by all 32 lanes of warp 1 in step (uniform waits; one elected lane issues
// each group of MMAs and the commits), as in the 16-bit forward.

__device__ void mma_issuer(const X3Args &a, X3Bars &bars, const int *sched_item, uint32_t sQ, uint32_t sK,
                           uint32_t sV, uint32_t tmem, const Watchdog &wd) {
    const FwdParams &p = a.p;
    const int total = total_items(p);
    // a negative scale negates Q in the score MMAs (A-negate bit)
    const uint32_t idS = idesc_f16(1, BM, BN, 0) | (p.scale_log2 < 0.f ? (1u << 13) : 0u);
    constexpr uint32_t idO = idesc_f16(1, BM, D, 1);
    uint32_t q_cnt[NQT] = {0, 0}, p_cnt[NQT] = {0, 0}, of_cnt[NQT] = {0, 0};
    RingPos<kKStages> kr;
    RingPos<kVStages> vr;
    const uint64_t q_desc = sdesc_sw128(sQ, 16, 1024);
    const uint64_t k_desc = sdesc_sw128(sK, 16, 1024);
    const uint64_t v_desc = sdesc_sw128(sV, kKVPart, 1024);
    // S_t = sum over the six part products Q_a K_b^T, 4 steps of 16 over D each
    auto issue_s = [&](int t, uint32_t kslot) {
        const uint32_t d = tmem + kTmemTile * t;
        if (elect_one()) {
#pragma unroll
        for (int ch = 0; ch < 6; ++ch) {
            const uint64_t qa = q_desc + sdesc_step(t * kQBytes + prod_a(ch) * kQPart);
            const uint64_t ka = k_desc + sdesc_step(kslot * kKBytes + prod_b(ch) * kKVPart);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t off = sdesc_step(kk * 32);
                mma_ss(d, qa + off, ka + off, idS, ch > 0 || kk > 0);
            }
        }
        tc_commit(smem_u32(&bars.s_full[t]));
        }
        __syncwarp();
    };
    // this key tile's partial U_t = sum over the six part products P_a V_b, from
    // zero; 4 steps of 16 keys (P_a from TMEM, V_b N-major from shared memory)
    auto issue_pv = [&](int t, uint32_t vslot) {
        const uint32_t d = tmem + kTmemTile * t + kColU;
        if (elect_one()) {
#pragma unroll
        for (int ch = 0; ch < 6; ++ch) {
            const uint64_t va = v_desc + sdesc_step(vslot * kVBytes + prod_b(ch) * kKVPart);
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {  // key group kk: 16 keys
                const int a_part = prod_a(ch);
                const uint32_t col = a_part == 0 ? 16 * kk : a_part == 1 ? 16 * kk + 8 : kColP3 + 8 * kk;
                mma_ts(d, tmem + kTmemTile * t + col, va + sdesc_step(kk * 2048), idO, ch > 0 || kk > 0);
            }
        }
        }
        __syncwarp();
    };
    auto wait = [&](uint64_t &bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar), parity, wd));
    };
    // a commit by the lane that issued the MMAs
    auto commit = [&](uint64_t &bar) {
        if (elect_one()) tc_commit(smem_u32(&bar));
        __syncwarp();
    };

    for (int i = 0;; ++i) {
        const int slot = i & 1;
        if (!wait(bars.sched_full[slot], (i >> 1) & 1)) return;
        const int w = sched_item[slot];
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&bars.sched_empty[slot]));
        if (w >= total) return;
        const ItemInfo f = item_info(p, w);
        if (f.nkv == 0) continue;
#pragma unroll
        for (int t = 0; t < NQT; ++t) {
            if (f.n[t] == 0) continue;
            if (!wait(bars.q_full[t], q_cnt[t] & 1)) return;
            ++q_cnt[t];
        }
        const uint32_t ks = kr.slot();
        if (!wait(bars.k_full[ks], kr.phase())) return;
        ++kr.i;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < NQT; ++t) {
            if (f.n[t] == 0) continue;
            issue_s(t, ks);
            if (f.n[t] == 1) commit(bars.q_empty[t]);
        }
        commit(bars.k_empty[ks]);

        for (int j = 0; j < f.nkv; ++j) {
            const uint32_t vs = vr.slot();  // V_j landed with K_j
            ++vr.i;
            bool have_next_k = false;
            uint32_t nks = 0;
#pragma unroll
            for (int t = 0; t < NQT; ++t) {
                if (j >= f.n[t]) continue;
                if (!wait(bars.p_full[t], p_cnt[t] & 1)) return;
                ++p_cnt[t];
                if (j == 0) {
                    // the previous item's epilogue of this tile has read its last partial
                    if (!wait(bars.o_free[t], (of_cnt[t] & 1) ^ 1)) return;
                    ++of_cnt[t];
                }
                tc_fence_after();
                issue_pv(t, vs);
                if (j == f.n[t] - 1) commit(bars.o_done[t]);
                if (j + 1 < f.n[t]) {
                    if (!have_next_k) {
                        nks = kr.slot();
                        if (!wait(bars.k_full[nks], kr.phase())) return;
                        ++kr.i;
                        have_next_k = true;
                        tc_fence_after();
                    }
                    issue_s(t, nks);
                    if (j + 1 == f.n[t] - 1) commit(bars.q_empty[t]);
                }
            }
            commit(bars.v_empty[vs]);
            if (have_next_k) commit(bars.k_empty[nks]);
        }
    }
}

// ---- warps 4-11: softmax and epilogue ------------------------------------------------

// Adds the key tile's value partial (64 f32 TMEM columns of this lane) to U.
__device__ __forceinline__ void add_partial(float (&U)[D], uint32_t u_addr) {
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld_x32(u_addr + 32 * c, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int e = 0; e < 32; ++e) U[32 * c + e] += __uint_as_float(r[e]);
    }
}

__device__ void softmax_wg(const X3Args &a, X3Bars &bars, const int *sched_item, uint32_t tmem, const Watchdog &wd) {
    const FwdParams &p = a.p;
    const int total = total_items(p);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int lrow = 32 * quarter + lane;
    const uint32_t s_addr = tmem_addr(tmem, 32 * quarter, kTmemTile * t);
    const uint32_t u_addr = s_addr + kColU;
    const float sl2 = fmaxf(fabsf(p.scale_log2), FLT_MIN);
    uint32_t s_cnt = 0, o_cnt = 0;
    float *go = static_cast<float *>(p.o);  // f32 inputs store O (and split partials) in f32

    for (int i = 0;; ++i) {
        const int slot = i & 1;
        bool ok = mbar_wait(smem_u32(&bars.sched_full[slot]), (i >> 1) & 1, wd);
        if (!__all_sync(0xffffffffu, ok)) return;
        const int w = sched_item[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars.sched_empty[slot]));
        if (w >= total) return;
        const ItemInfo f = item_info(p, w);
        const int n = t == 0 ? f.n[0] : f.n[1];
        const int r0 = f.row0 + BM * t;
        const int row = r0 + lrow;
        float *orow = go + f.c * p.o_split_st + (int64_t)(f.q_start + row) * p.o_st + (int64_t)f.h * p.o_sh;
        float *lse_at = p.lse ? p.lse + f.c * p.lse_split_st + (int64_t)f.h * p.n_q + f.q_start + row : nullptr;
        if (n == 0) {
            if (r0 < f.Lq && row < f.Lq) {
#pragma unroll 4
                for (int c = 0; c < D; c += 4) store4(orow + c, make_float4(0.f, 0.f, 0.f, 0.f));
                if (lse_at) *lse_at = -INFINITY;
            }
            continue;
        }

        float m = -INFINITY, l = 0.f;
        float U[D];
#pragma unroll
        for (int c = 0; c < D; ++c) U[c] = 0.f;
        for (int j = 0; j < n; ++j) {
            ok = mbar_wait(smem_u32(&bars.s_full[t]), s_cnt & 1, wd);
            ++s_cnt;
            if (!__all_sync(0xffffffffu, ok)) return;
            tc_fence_after();
            // S_j completed after the previous tile's value contraction: add its partial
            if (j > 0) add_partial(U, u_addr);

            const int key0 = BN * (f.j0 + j);
            const bool masked = (p.causal && key0 + BN - 1 > r0) || key0 + BN > f.Lk;
            const int lim = masked ? min(f.Lk - key0, p.causal ? row - key0 + 1 : BN) : BN;  // keys [0, lim)
            // pass 1: the row max over the tile (32 columns at a time)
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_x32(s_addr + 32 * c, r);
                tmem_ld_wait(r);
                float cm = -INFINITY;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float v = __uint_as_float(r[e]);
                    cm = fmaxf(cm, (!masked || 32 * c + e < lim) ? v : -INFINITY);
                }
                mx = fmaxf(mx, cm);
            }
            mx *= sl2;
            const float m_new = fmaxf(m, mx);
            const bool rescale = j > 0 && __any_sync(0xffffffffu, m_new > m + kRescaleThreshold);
            float alpha = 1.f;
            if (j == 0) {
                m = m_new;
            } else if (rescale) {
                alpha = exp2_approx(m - m_new);
                m = m_new;
            }
            const float m_use = m == -INFINITY ? 0.f : m;
            // pass 2: p = 2^(s * scale * log2e - m), split into bf16 parts P1 + P2 + P3,
            // one group of 16 keys at a time; a group's parts overwrite only its own
            // (already read) S columns and the P3 area
            const float2 sc2 = make_float2(sl2, sl2), nm2 = make_float2(-m_use, -m_use);
            const float2 neg1 = make_float2(-1.f, -1.f);
            float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int q16 = 0; q16 < BN / 16; ++q16) {
                uint32_t r[16];
                tmem_ld_x16(s_addr + 16 * q16, r);
                tmem_ld_wait16(r);
                uint32_t p1[8], p2[8], p3[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float2 x = __ffma2_rn(make_float2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1])),
                                                sc2, nm2);
                    float2 pv = make_float2(exp2_approx(x.x), exp2_approx(x.y));
                    if (masked) {
                        if (16 * q16 + 2 * e >= lim) pv.x = 0.f;
                        if (16 * q16 + 2 * e + 1 >= lim) pv.y = 0.f;
                    }
                    acc2 = __fadd2_rn(acc2, pv);
                    const __nv_bfloat162 b1 = __floats2bfloat162_rn(pv.x, pv.y);
                    const float2 r1 = __ffma2_rn(__bfloat1622float2(b1), neg1, pv);
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(r1.x, r1.y);
                    const float2 r2 = __ffma2_rn(__bfloat1622float2(b2), neg1, r1);
                    const __nv_bfloat162 b3 = __floats2bfloat162_rn(r2.x, r2.y);
                    p1[e] = *reinterpret_cast<const uint32_t *>(&b1);
                    p2[e] = *reinterpret_cast<const uint32_t *>(&b2);
                    p3[e] = *reinterpret_cast<const uint32_t *>(&b3);
                }
                tmem_st_x8(s_addr + 16 * q16, p1);
                tmem_st_x8(s_addr + 16 * q16 + 8, p2);
                tmem_st_x8(s_addr + kColP3 + 8 * q16, p3);
            }
            l = l * alpha + (acc2.x + acc2.y);
            if (rescale) {
#pragma unroll
                for (int c = 0; c < D; ++c) U[c] *= alpha;
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive_warp(smem_u32(&bars.p_full[t]));
        }

        // epilogue: the last tile's partial, then O = U / l, lse = (m + log2 l) ln 2
        ok = mbar_wait(smem_u32(&bars.o_done[t]), o_cnt & 1, wd);
        ++o_cnt;
        if (!__all_sync(0xffffffffu, ok)) return;
        tc_fence_after();
        add_partial(U, u_addr);
        tc_fence_before();
        mbar_arrive_warp(smem_u32(&bars.o_free[t]));
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float *wrow0 = go + f.c * p.o_split_st + (int64_t)(f.q_start + r0 + 32 * quarter) * p.o_st +
                      (int64_t)f.h * p.o_sh;
        const int rows_live = min(32, max(0, f.Lq - (r0 + 32 * quarter)));
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t u[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(U[32 * c + e]);
            store_rows_chunk(u, inv, wrow0 + 32 * c, p.o_st, rows_live, lane);
        }
        if (row < f.Lq && lse_at) *lse_at = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
    }
}

__global__ void __launch_bounds__(kThreads, 1) fwd_x3_kernel(const __grid_constant__ X3Args a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ X3Bars bars;
    __shared__ int sched_item[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sQ = (raw + 1023u) & ~1023u;
    const uint32_t sK = sQ + NQT * kQBytes;
    const uint32_t sV = sK + kKStages * kKBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Watchdog wd{a.p.watchdog_cycles, &abort_flag, a.p.status};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int t = 0; t < NQT; ++t) {
            mbar_init(smem_u32(&bars.q_full[t]), 1);
            mbar_init(smem_u32(&bars.q_empty[t]), 1);
            mbar_init(smem_u32(&bars.s_full[t]), 1);
            mbar_init(smem_u32(&bars.p_full[t]), 4);  // one arrival per softmax warp
            mbar_init(smem_u32(&bars.o_done[t]), 1);
            mbar_init(smem_u32(&bars.o_free[t]), 4);
        }
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(smem_u32(&bars.k_full[s]), 1);
            mbar_init(smem_u32(&bars.k_empty[s]), 1);
        }
        for (int s = 0; s < kVStages; ++s) mbar_init(smem_u32(&bars.v_empty[s]), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&bars.sched_full[s]), 1);
            mbar_init(smem_u32(&bars.sched_empty[s]), kSchedConsumers);
        }
        mbar_init(smem_u32(&bars.mma_drain), 1);
        fence_mbar_init();
        for (int g = 0; g < kParts; ++g) {
            prefetch_tmap(&a.tq[g]);
            prefetch_tmap(&a.tk[g]);
            prefetch_tmap(&a.tv[g]);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_base), 512);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    // set-up above overlaps the previous kernel on the stream; inputs are read after this
    pdl_trigger();
    pdl_wait();

    if (warp < 4) {
        regs_dec<kRegsProducer>();
        if (warp == 0) {
            if (lane == 0) producer(a, bars, sched_item, sQ, sK, sV, wd);
        } else if (warp == 1) {
            mma_issuer(a, bars, sched_item, sQ, sK, sV, tmem, wd);  // the whole warp
            if (lane == 0 && aborting(wd)) {  // let issued MMAs finish before TMEM is freed
                tc_commit(smem_u32(&bars.mma_drain));
                drain_wait(smem_u32(&bars.mma_drain), 0, kDrainCycles);
            }
        }
    } else {
        regs_inc<kRegsSoftmax>();
        softmax_wg(a, bars, sched_item, tmem, wd);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

size_t x3_split_bytes(int n_q, int n_k, int H) {
    return (size_t)kParts * ((int64_t)n_q + 2 * (int64_t)n_k) * H * D * 2;
}

bool x3_fwd_supported(const FwdParams &p) {
    return p.dtype == ATTN_F32 && p.D == D && !p.qk_fp8 && !p.prune && p.n_q > 0 && p.n_k > 0 &&
           tc_device_ok();
}

cudaError_t launch_fwd_x3(const FwdParams &p, int num_ctas, cudaStream_t s) {
    if (!p.split_ws) return cudaErrorInvalidValue;
    // the bf16 parts, each a contiguous (tokens, heads, 64) array
    __nv_bfloat16 *base = static_cast<__nv_bfloat16 *>(p.split_ws);
    const int64_t qn = (int64_t)p.n_q * p.H * D, kn = (int64_t)p.n_k * p.H * D;
    __nv_bfloat16 *q_parts = base, *k_parts = q_parts + kParts * qn, *v_parts = k_parts + kParts * kn;
    SplitParams sp;
    sp.H = p.H;
    sp.job[0] = SplitJob{static_cast<const float *>(p.q), p.q_st, p.q_sh, p.n_q, kParts, q_parts};
    sp.job[1] = SplitJob{static_cast<const float *>(p.k), p.k_st, p.k_sh, p.n_k, kParts, k_parts};
    sp.job[2] = SplitJob{static_cast<const float *>(p.v), p.v_st, p.v_sh, p.n_k, kParts, v_parts};
    const int64_t n4 = (qn + kn) / 4;
    const int blocks = (int)std::min<int64_t>((n4 + 255) / 256, (int64_t)sm_count() * 8);
    cudaError_t e = launch_pdl(split_parts_kernel, dim3(blocks), dim3(256), 0, s, sp);
    count_launch();
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    X3Args args;
    args.p = p;
    const int64_t st = (int64_t)p.H * D;
    for (int g = 0; g < kParts; ++g)
        if (!make_tile_map(&args.tq[g], q_parts + g * qn, ATTN_BF16, D, p.n_q, p.H, st, D, BM) ||
            !make_tile_map(&args.tk[g], k_parts + g * kn, ATTN_BF16, D, p.n_k, p.H, st, D, BN) ||
            !make_tile_map(&args.tv[g], v_parts + g * kn, ATTN_BF16, D, p.n_k, p.H, st, D, BN))
            return cudaErrorInvalidValue;
    if (p.o_dtype != ATTN_F32) return cudaErrorInvalidValue;
    auto kern = fwd_x3_kernel;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (num_ctas <= 0) num_ctas = sm_count();
    e = launch_pdl(kern, dim3(num_ctas), dim3(kThreads), kSmemBytes, s, args);
    count_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace attn
